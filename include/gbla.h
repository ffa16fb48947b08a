/*
 * gbla.h — C ABI of the GB300 (sm_103a) Gated Bidirectional Linear Attention
 * (GBLA) layer library, libgbla.so.
 *
 * What the layer computes ("Gated Bidirectional Linear Attention for
 * Generative Retrieval", section "Core method"), per sequence and head h:
 *   Eq. 4  x~ = Conv1d(x);  q = x~ W_Q^h,  k = x~ W_K^h,  v = x~ W_V^h
 *   Eq. 5  g_j = gate(x~_j . w_g^h)  (sigmoid with bias, or softmax over the
 *          sequence, see gbla_gate)
 *   Eq. 6  q~ = phi(q), k~_j = g_j phi(k_j), phi = elu + 1;
 *          S = sum_j k~_j v_j^T (d_h x d_h),  z = sum_j k~_j,
 *          o_i = q~_i^T S / q~_i^T z        (global, non-causal: bidirectional)
 *   Eq. 7  y = RmsNorm(o) (.) gamma (.) SiLU(x~ W_R^h)
 *   "Multi-head" paragraph: each head owns its W_Q^h, W_K^h, W_V^h, w_g^h, W_R^h.
 * The heads' outputs are concatenated: y is [tokens, H*d_h].  No output
 * projection, residual or FFN is part of this library.
 *
 * Conventions shared by every call
 * --------------------------------
 * - Every tensor pointer is a DEVICE pointer owned by the caller.  The library
 *   allocates no device memory: scratch comes from the caller's workspace
 *   `ws` of `ws_bytes` bytes, sized by gbla_workspace_size().  The workspace
 *   need not be zeroed and must be 256-byte aligned.
 * - All calls are asynchronous on the caller's CUDA stream (`stream` is a
 *   cudaStream_t passed as void*; NULL = the legacy default stream).  Calls
 *   that share a workspace must be stream-ordered.  The library keeps no state
 *   between calls; results are deterministic (bitwise reproducible for the same
 *   shape and inputs): no floating-point atomics are used.
 * - Row-major layouts.  Token-major tensors have one row per token: in the
 *   dense and padded forms there are B*L rows (sequence b owns rows b*L ..
 *   b*L+L-1); in the varlen form there are T = L rows and sequence b owns
 *   rows cu_seqlens[b] .. cu_seqlens[b+1]-1.
 * - Weights use the x W convention: W_* is [d, H*d_h] and column block
 *   h*d_h .. h*d_h+d_h-1 belongs to head h; w_g is [d, H].
 * - dtypes: tensors named "(io)" have the shape's io_dtype (fp32 or bf16);
 *   gate values g, logits, den, state and every PARAMETER GRADIENT are fp32.
 *   Accumulation is fp32 everywhere.
 * - Padding and varlen: rows that belong to no sequence (a padded row, i.e.
 *   position >= seq_lens[b]) get zero outputs and zero input gradients.  The
 *   conv window and the state sums never cross a sequence boundary.
 * - Errors: argument errors are detected on the host before anything is
 *   launched and returned as a status.  A launch failure returns
 *   GBLA_ERR_CUDA (gbla_last_error() gives the CUDA text).  Bad sequence data
 *   that only the device can see (cu_seqlens not starting at 0, decreasing,
 *   or not ending at T; seq_lens outside [0, L]) sets an error word in the
 *   workspace, every kernel then skips its work, and gbla_check_device_status()
 *   reports GBLA_ERR_DEVICE_CHECK.  No kernel traps or waits on another CTA.
 *   The tensor-core kernels wait on their own copies and MMAs through
 *   mbarriers; every such wait is bounded, and one that gives up (a device
 *   that stopped making progress) sets a timeout bit in the error word instead
 *   of hanging: gbla_check_device_status() then reports GBLA_ERR_DEVICE_TIMEOUT.
 */
#ifndef GBLA_H
#define GBLA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  GBLA_OK = 0,
  GBLA_ERR_INVALID_ARG = -1,  /* null/misaligned pointer, bad dimension      */
  GBLA_ERR_UNSUPPORTED = -2,  /* a valid shape this build has no kernel for  */
  GBLA_ERR_WORKSPACE = -3,    /* ws NULL, misaligned, or ws_bytes too small  */
  GBLA_ERR_CUDA = -4,         /* a CUDA runtime call or launch failed        */
  GBLA_ERR_DEVICE_CHECK = -5, /* bad sequence data detected on the device   */
  GBLA_ERR_DEVICE_TIMEOUT = -6 /* a kernel's bounded wait gave up            */
} gbla_status;

typedef enum { GBLA_F32 = 0, GBLA_BF16 = 1 } gbla_dtype;

/* Key gate of Eq. 5.  SIGMOID: g = sigmoid(x~ . w_g + b_g) per token and head.
 * SOFTMAX: the pages' g = softmax_j(x~_j . w_g) over the valid tokens of each
 * sequence; its normaliser (and any b_g) cancels between the numerator and
 * denominator of Eq. 5, so the kernels use exp(s_j - m) with a per-sequence
 * running max m and db_g is 0. */
typedef enum { GBLA_GATE_SIGMOID = 0, GBLA_GATE_SOFTMAX = 1 } gbla_gate;

typedef enum {
  GBLA_OP_FORWARD = 0,        /* gbla_forward                                */
  GBLA_OP_BACKWARD = 1,       /* gbla_backward                               */
  GBLA_OP_CORE_FORWARD = 2,   /* bla_core_forward                            */
  GBLA_OP_CORE_BACKWARD = 3,  /* bla_core_backward                           */
  GBLA_OP_DECAY_FORWARD = 4,  /* bla_decay_core_forward                      */
  GBLA_OP_SA_FORWARD = 5      /* sa_core_forward                             */
} gbla_op;

typedef struct {
  int B;       /* batch (dense/padded forms); must be 1 with cu_seqlens       */
  int L;       /* tokens per sequence slot; with cu_seqlens: T, total rows    */
  int d;       /* model width (channels of x)                                 */
  int H;       /* heads                                                       */
  int d_h;     /* head width: bf16 {32, 64, 128}; fp32 1..128                 */
  const int32_t* cu_seqlens; /* device [num_seqs+1] or NULL (varlen form)     */
  int num_seqs;              /* sequences in the varlen form                  */
  const int32_t* seq_lens;   /* device [B] or NULL (padded form: valid rows)  */
  int io_dtype;              /* gbla_dtype                                    */
  int gate;                  /* gbla_gate                                     */
  float rms_eps;             /* RmsNorm epsilon (Eq. 7); e.g. 1e-6            */
} gbla_shape;

/* Bytes of workspace `ws` that call `op` needs for this shape (0 on a shape
 * error; check gbla_validate_shape). */
size_t gbla_workspace_size(const gbla_shape* shape, int op);

/* Bytes of the activation buffer that gbla_forward fills for gbla_backward
 * (x~, the q|k|v|r projections, the gate, the state).  Caller-owned. */
size_t gbla_saved_size(const gbla_shape* shape);

/* Host-side validation of a shape alone; GBLA_OK or the reason. */
gbla_status gbla_validate_shape(const gbla_shape* shape);

/*
 * Layer forward, Eq. 4-7.
 *   x       (io) [rows, d]
 *   conv_w  (io) [d, 4]   depthwise causal taps; tap t multiplies x[l-3+t]
 *   conv_b  (io) [d] or NULL (no bias)
 *   W_q, W_k, W_v, W_r (io) [d, H*d_h]
 *   w_g     (io) [d, H];  b_g (io) [H] or NULL (zero bias)
 *   rms_w   (io) [d_h] or NULL (ones): RmsNorm scale gamma, shared by heads
 *   y       (io) [rows, H*d_h]  output
 *   saved   NULL (inference) or gbla_saved_size() bytes, 256-byte aligned:
 *           filled for gbla_backward
 * bf16 requires every pointer 16-byte aligned and d % 64 == 0.
 */
gbla_status gbla_forward(const gbla_shape* shape, const void* x,
                         const void* conv_w, const void* conv_b,
                         const void* W_q, const void* W_k, const void* W_v,
                         const void* W_r, const void* w_g, const void* b_g,
                         const void* rms_w, void* y, void* saved, void* ws,
                         size_t ws_bytes, void* stream);

/*
 * Layer backward for the scalar <dy, y>: the same inputs as gbla_forward, the
 * `saved` buffer that a training forward of the same inputs filled, and dy
 * (io) [rows, H*d_h].  Outputs (any parameter gradient may be NULL to skip
 * writing it; dx is required):
 *   dx (io) [rows, d];  dconv_w fp32 [d, 4];  dconv_b fp32 [d];
 *   dW_q, dW_k, dW_v, dW_r fp32 [d, H*d_h];  dw_g fp32 [d, H];  db_g fp32 [H];
 *   drms_w fp32 [d_h].
 * Gradients overwrite (they are not accumulated into).
 */
gbla_status gbla_backward(const gbla_shape* shape, const void* x,
                          const void* conv_w, const void* conv_b,
                          const void* W_q, const void* W_k, const void* W_v,
                          const void* W_r, const void* w_g, const void* b_g,
                          const void* rms_w, const void* saved, const void* dy,
                          void* dx, float* dconv_w, float* dconv_b,
                          float* dW_q, float* dW_k, float* dW_v, float* dW_r,
                          float* dw_g, float* db_g, float* drms_w, void* ws,
                          size_t ws_bytes, void* stream);

/*
 * The gated BLA core alone, Eq. 5/6, from raw projections:
 *   q, k, v (io) [rows, H*d_h]  (phi is applied inside)
 *   g       fp32 [rows, H]      gate VALUES g_j >= 0 (not logits)
 *   o       (io) [rows, H*d_h]  o_i = phi(q_i)^T S / phi(q_i)^T z
 *   den     fp32 [rows, H] or NULL: phi(q_i)^T z
 *   state   fp32 [n_seq, H, d_h, d_h+1] or NULL: [S | z] (z = column d_h);
 *           n_seq = B, or num_seqs in the varlen form
 * The shape's d, gate and rms_eps are ignored.
 */
gbla_status bla_core_forward(const gbla_shape* shape, const void* q,
                             const void* k, const void* v, const float* g,
                             void* o, float* den, float* state, void* ws,
                             size_t ws_bytes, void* stream);

/*
 * Backward of bla_core_forward for the scalar <d_o, o>.
 *   d_o (io) [rows, H*d_h];  dq, dk, dv (io) [rows, H*d_h];  dg fp32 [rows, H]
 *   (the gradient with respect to the gate values g).
 * The state is recomputed from q, k, v, g.
 */
gbla_status bla_core_backward(const gbla_shape* shape, const void* q,
                              const void* k, const void* v, const float* g,
                              const void* d_o, void* dq, void* dk, void* dv,
                              float* dg, void* ws, size_t ws_bytes,
                              void* stream);

/*
 * The gated core under LION's decay masks ("Linear Attention for Efficient
 * Bidirectional Sequence Modeling": mask construction and the Lion-d /
 * Lion-s models), with this layer's phi = elu + 1 and key gate (Eq. 5):
 *   M^F_ij = prod_{t=j+1..i} lam_t (j <= i),  M^B_ij = prod_{t=i+1..j} lam_t (j >= i),
 *   M = M^F + M^B - I,
 *   o_i = sum_j M_ij g_j (phi(q_i).phi(k_j)) v_j / sum_j M_ij g_j (phi(q_i).phi(k_j)).
 * Lion-d passes one constant decay for every token (M_ij = lam^|i-j|), Lion-s
 * a decay per token (e.g. sigmoid(W x_t + b)); lam = 1 everywhere is
 * bla_core_forward.  Computed in the bidirectional chunkwise form: 128-row
 * chunks, their local states, a forward and a backward scan over the chunk
 * states, then each chunk's decayed attention plus the two scanned states.
 *   q, k, v (bf16) [rows, H*d_h] (phi is applied inside); g fp32 [rows, H]
 *   gate values >= 0; lam fp32 [rows, H] decays in [0, 1] (lam_t of a
 *   sequence's first token enters no product); o (bf16) [rows, H*d_h];
 *   den fp32 [rows, H] or NULL.
 *   bf16 I/O and d_h = 64 only (GBLA_ERR_UNSUPPORTED otherwise).  Workspace:
 *   gbla_workspace_size(shape, GBLA_OP_DECAY_FORWARD).  The shape's d, gate and
 *   rms_eps are ignored.
 */
gbla_status bla_decay_core_forward(const gbla_shape* shape, const void* q,
                                   const void* k, const void* v, const float* g,
                                   const float* lam, void* o, float* den,
                                   void* ws, size_t ws_bytes, void* stream);

/*
 * The attention of the SA blocks of the hybrid [SA, LA, LA] encoder: the
 * bidirectional softmax attention of Eq. 1 ("Gated Bidirectional Linear
 * Attention for Generative Retrieval", Core method 1; the hybrid encoder
 * interleaves one such block with two GBLA blocks):
 *   o_i = sum_j exp(q_i . k_j / sqrt(d_h)) v_j / sum_j exp(q_i . k_j / sqrt(d_h))
 * over every key j of query i's sequence, per head (no mask: both
 * directions).  Quadratic in the sequence length: the baseline the pages
 * compare GBLA with (Table 5, single-layer latency).
 *   q, k, v, o (bf16) [rows, H*d_h], head h at columns h*d_h .. h*d_h+d_h-1.
 *   Rows of a padded slot past its sequence get o = 0.
 *   bf16 I/O and d_h = 64 only (GBLA_ERR_UNSUPPORTED otherwise).  Workspace:
 *   gbla_workspace_size(shape, GBLA_OP_SA_FORWARD).  The shape's d, gate and
 *   rms_eps are ignored.
 */
gbla_status sa_core_forward(const gbla_shape* shape, const void* q,
                            const void* k, const void* v, void* o, void* ws,
                            size_t ws_bytes, void* stream);

/*
 * bla_core_forward without a caller workspace (the pages have no counterpart:
 * this is a deployment convenience).  Some callers cannot call cudaMalloc or
 * hand the library a scratch buffer: a plugin running inside a host framework
 * that owns all device memory through its own pool and passes only its
 * tensors, or a latency-bound serving loop where an allocation would
 * synchronise the device and stall the other streams.  This entry point
 * allocates nothing: the split-L partial states, combine counters, error word
 * and combined state live in one file-scope device array of 64 MiB
 * (GBLA_NOALLOC_SCRATCH_BYTES) that every GPU which loads the library holds
 * until the process exits.
 *   Arguments, layouts and results are those of bla_core_forward.
 *   GBLA_ERR_WORKSPACE: the shape needs more than 64 MiB of scratch
 *   (gbla_workspace_size(shape, GBLA_OP_CORE_FORWARD) > 64 MiB); nothing runs.
 *   The first call on each device looks up the array's device address
 *   (cudaGetSymbolAddress, with that device current); make that first call
 *   before any stream capture.
 *   Every call on a device shares the one array: calls whose kernels overlap
 *   on the GPU (two streams, or two host threads) race and corrupt each
 *   other's results.  Order them on one stream.  The counters and the error
 *   word are cleared at the start of every call; the error word of the last
 *   call is read by bla_core_noalloc_check_device_status (below).
 */
#define GBLA_NOALLOC_SCRATCH_BYTES ((size_t)64 << 20)
gbla_status bla_core_forward_noalloc(const gbla_shape* shape, const void* q,
                                     const void* k, const void* v,
                                     const float* g, void* o, float* den,
                                     float* state, void* stream);

/* Synchronises `stream` and reads the device error word of the workspace that
 * the last call on it used: GBLA_OK, GBLA_ERR_DEVICE_CHECK (bad cu_seqlens /
 * seq_lens; reported first), GBLA_ERR_DEVICE_TIMEOUT (a bounded wait gave up),
 * or GBLA_ERR_CUDA if the stream itself failed. */
gbla_status gbla_check_device_status(const void* ws, void* stream);

/* gbla_check_device_status for bla_core_forward_noalloc: synchronises
 * `stream` and reads the error word of the library's fixed scratch array on
 * the current device (the last no-allocation call's).  It allocates nothing. */
gbla_status bla_core_noalloc_check_device_status(void* stream);

/* Diagnostic of the timeout path (no counterpart on the pages).  Clears the
 * error word at the start of `ws` (any workspace of at least 16 bytes,
 * 256-byte aligned) and launches one CTA that waits, with the kernels' own
 * bounded mbarrier wait cut to `polls` polls (1 .. 2^20), on a barrier that
 * nothing arrives at.  The wait gives up, sets the timeout bit, and the kernel
 * returns; nothing faults or hangs.  gbla_check_device_status(ws, stream)
 * then reports GBLA_ERR_DEVICE_TIMEOUT.  Asynchronous on `stream`. */
gbla_status gbla_diag_bounded_wait(void* ws, size_t ws_bytes, unsigned polls, void* stream);

/* Static text for a status code. */
const char* gbla_status_string(int status);

/* Text of the last CUDA error seen by this thread (empty if none). */
const char* gbla_last_error(void);

/* Library version, major*10000 + minor*100 + patch. */
int gbla_version(void);

/* Per-launch timing for benchmarks and profiling (no counterpart on the
 * pages).  While enabled, every kernel or memset that a gbla_* / bla_core_*
 * call of the CALLING THREAD launches is bracketed by two CUDA events recorded
 * on that call's stream.  gbla_profiling_read() synchronises on the last
 * event, writes up to `cap` entries (static name strings, milliseconds) and
 * returns the number of launches recorded since the previous read, then
 * clears the record.  Either output array may be NULL.  A name is the step
 * followed by the kernel variant that ran, e.g. "bwd_q[tc]" (5th-generation
 * tensor cores, tcgen05), "bwd_q[mma]" (mma.sync), "bwd_q[f32]" (fp32 I/O),
 * "conv[bulk]" (bulk-copy staged) or "conv[plain]". */
void gbla_profiling_enable(int on);
int gbla_profiling_read(const char** names, float* ms, int cap);

/* Kernel selection of the CALLING THREAD's later calls (no counterpart on the
 * pages).  GBLA_POLICY_AUTO (the default) picks, per step, the kernel that is
 * fastest for the shape: e.g. the state reduction runs on the 5th-generation
 * tensor cores only when every SM gets at least 20 of its 256-row tiles, and
 * on mma.sync otherwise.  GBLA_POLICY_TC takes the tcgen05 kernel wherever it
 * applies (d_h and gate permitting), whatever the size: for tests that check
 * those kernels on small shapes.  GBLA_POLICY_MMA takes the mma.sync kernel
 * of every step that has one beside its tcgen05 kernel: for tests of the
 * mma.sync kernels at the shapes AUTO runs on tcgen05.  Results agree within
 * the tolerances either way.  GBLA_ERR_INVALID_ARG for another value. */
typedef enum { GBLA_POLICY_AUTO = 0, GBLA_POLICY_TC = 1, GBLA_POLICY_MMA = 2 } gbla_policy;
gbla_status gbla_set_kernel_policy(int policy);

#ifdef __cplusplus
}
#endif

#endif /* GBLA_H */
