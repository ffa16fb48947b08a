// Internal interface between the C-ABI host code (api.cu) and the kernels.
// Every launcher returns the cudaError_t of its launch.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"

namespace gbla {

// Row stride (floats) of fp32 state / partial tiles: [S | z | 0 x 7].
__host__ __device__ constexpr int state_ld(int dh) { return dh + 8; }
// Row stride (elements) of the bf16 copy of [S | z | 0 x 15].
__host__ __device__ constexpr int state_bf_ld(int dh) { return dh + 16; }

// Gate input kinds of the state reduction and of the key-side backward.
enum GateKind {
  GATE_VALUES = 0,   // g holds gate values g_j >= 0
  GATE_LOGITS = 1,   // g holds softmax logits s_j; the kernels use exp(s_j - m)
};
// What the key-side backward writes in its gate-gradient slot.
enum GateGrad {
  GG_DG = 0,         // dL/dg (core API), fp32
  GG_SIGMOID = 1,    // dL/ds = dg g (1 - g), io dtype into the dP buffer
  GG_SOFTMAX = 2,    // dL/ds = g' dg with g' = exp(s - m), io dtype into dP
};

// "pre" (the bf16 layer): the projection epilogue has already stored phi(q)
// and phi(k) in place of q and k, so the state kernels skip the feature map;
// the backward uses phi'(x) = min(1, phi(x)) for phi = elu + 1.
struct ReduceArgs {
  int pre;            // k holds phi(k)
  const void* k; const void* v; int64_t ldk, ldv;  // [rows, ld], head h at column h*dh
  const float* g; int64_t ldg; int gate_kind;
  int H, dh;
  SeqDesc seq; Tiling chunks;
  float* partial;     // [chunks*H][dh][state_ld]
  float* partial_m;   // [chunks*H]          (GATE_LOGITS)
  int* counters;      // [n_seq*H], zero on entry
  float* state;       // [n_seq*H][dh][state_ld]
  bf16* state_bf;     // [n_seq*H][dh][state_bf_ld]   (bf16 kernels)
  float* state_m;     // [n_seq*H]           (GATE_LOGITS)
  float* pub_state;   // [n_seq, H, dh, dh+1] or null
  float* center;      // [n_seq*H][dh] or null: centre the state (see combine_state)
  const int* err;
  // tcgen05 kernel: its units are 128-row pieces of `tiles` (n_tiles tiles);
  // one partial slot per (sequence, head) plus one per CTA
  Tiling tiles;
  int partial_slots;
  int* err_out;       // timeout bit of the workspace error word
};

struct ReadoutArgs {
  int pre;                          // q holds phi(q)
  const void* q; int64_t ldq;
  const void* r; int64_t ldr;       // norm only
  const void* rms_w; float eps;     // norm only; rms_w may be null
  const float* state; const bf16* state_bf;
  const float* center;              // [n_seq*H][dh] or null (state is uncentred)
  void* out; int64_t ldo;
  float* den;                       // [rows, H] or null
  float* rsinv;                     // norm, bf16: [rows, H] x {rs, 1/den} (0 on invalid rows) or null
  int H, dh;
  SeqDesc seq; Tiling tiles;
  const int* err;
  int* err_out;                     // tcgen05 kernel: timeout bit of the workspace error word
};

struct BwdQArgs {
  int pre;                          // q holds phi(q)
  const void* q; int64_t ldq;
  const void* r; int64_t ldr;       // norm only
  const void* dy; int64_t lddy;     // norm: dy; core: d_o
  const void* rms_w; float eps;
  const float* state; const bf16* state_bf;
  const float* center;              // [n_seq*H][dh] or null (state is uncentred)
  void* dq; int64_t lddq;
  void* dr; int64_t lddr;           // norm only
  float* gamma_part;                // norm only: [gridDim.x * H][dh] (tcgen05: [gridDim.x][dh])
  float* partial; int* counters;    // dS partials, [n_seq*H] counters
  int partial_slots;                // tcgen05 kernel: slots of `partial` (n_seq H + one per CTA needed)
  float* dstate; bf16* dstate_bf;   // combined [dS | dz]
  int H, dh;
  SeqDesc seq; Tiling chunks;
  Tiling tiles;                     // tcgen05 kernel: its units are 128-row pieces of these tiles
  const float* rsinv;               // tcgen05 kernel: [rows, H] x {rs, 1/den} from the forward
  const int* err;
  int* err_out;                     // tcgen05 kernel: timeout bit of the workspace error word
};

// Bidirectional softmax attention (Eq. 1), the SA blocks of the hybrid encoder.
struct SaArgs {
  const void* q; const void* k; const void* v;  // [T, ld] bf16; head h at columns h*dh
  void* o;                                      // [T, ld] bf16
  int64_t ld;
  int H, dh;
  SeqDesc seq; Tiling tiles;                    // tiles of 256 queries (two MMA tiles)
  const int* err;
  int* err_out;                                 // timeout bit of the workspace error word
};

struct BwdKVArgs {
  int pre;                          // k holds phi(k)
  const void* k; int64_t ldk;
  const void* v; int64_t ldv;
  const float* g; int64_t ldg; int gate_kind;  // GateKind
  const float* state_m;                         // GATE_LOGITS
  const float* dstate; const bf16* dstate_bf;
  const float* center;                         // centre of the forward state, or null
  void* dk; int64_t lddk;
  void* dv; int64_t lddv;
  void* ds; int64_t ldds; int gate_grad;       // GateGrad
  float* bg_part;                              // [gridDim.x * H] (tcgen05: [tiles * tile/128 * H]) or null
  int zero_cols_from, zero_cols_to;            // dP pad columns to clear (head 0 CTAs)
  int H, dh;
  SeqDesc seq; Tiling tiles;
  const int* err;
  int* err_out;                                // tcgen05 kernel: timeout bit of the workspace error word
};

// C[M, N] (+)= sum_k A(m, k) B(n, k).  A is [M][K] (a_kmajor) or [K][M];
// B is [N][K] (b_kmajor) or [K][N].  blockIdx.z splits K into chunks of
// k_split (a multiple of the K tile).
enum GemmEpi {
  EPI_BF16 = 0,       // C bf16
  EPI_F32 = 1,        // C fp32
  EPI_SPLITK = 2,     // fp32 partial C + z * M * ldc
  EPI_PROJ = 3,       // columns < n_main -> bf16 C; the next H columns -> gate (fp32)
  EPI_PROJ_PRE = 4,   // as EPI_PROJ, with phi(q), phi(k) stored in place of q, k
};
struct GemmArgs {
  const void* A; int64_t lda; int a_kmajor;
  const void* B; int64_t ldb; int b_kmajor;
  void* C; int64_t ldc;
  int M, N, K, k_split;
  int epi;
  // EPI_PROJ
  int n_main; const void* bias_g; int gate_mode; float* gate; int64_t ldgate;
  int io_f32;
  int* err;           // workspace error word (bounded device waits that give up set bit 2)
  int hd, dh;         // EPI_PROJ_PRE: H*dh and dh (column -> head)
  int pair;           // tcgen05 GEMM: run CTA pairs (M = 256 MMAs) when there are >= 2 m-tiles
};

struct ConvArgs {
  const void* x; const void* w; const void* b;  // io dtype; b may be null
  void* xt;                                     // io dtype [T, d]
  const void* dxt;                              // backward: io dtype [T, d]
  void* dx;                                     // backward: io dtype [T, d]
  float* part;                                  // backward: [gridDim.x][d][5] (dw 0..3, db)
  int T, d;
  SeqDesc seq;
  const int* err;       // checked on entry (may be null)
  int* err_out;         // workspace error word: a bounded wait that gave up sets kErrTimeout
};

// The core under LION's decay masks (decay.cu): raw q, k, v (bf16, phi
// applied inside), gate values g and decays lam in [0, 1] per row and head.
struct DecayArgs {
  const void* q; const void* k; const void* v; int64_t ld;  // [rows, ld], head h at column h*dh
  const float* g; const float* lam; int64_t ldg;            // [rows, ldg]
  void* o; float* den;                                      // o like q; den [rows, ldg] or null
  bf16* LF; bf16* LB; float* Lam;                           // chunk states [chunks*H][dh][dh+8] bf16, decays [chunks*H]
  bf16* HF; bf16* HB;                                       // scan states [chunks*H][dh][dh+16] bf16
  int H, dh;
  SeqDesc seq; Tiling tiles;                                // tiles: the 128-row chunks
  const int* err;
};

// ---------------------------------------------------------------- launchers
cudaError_t launch_plan(const SeqDesc& s, int ntile, const int* tile_sizes, int32_t* const* prefixes,
                        int* err, cudaStream_t st);

cudaError_t launch_reduce_bf16(const ReduceArgs& a, int grid_x, cudaStream_t st);
// tcgen05 state reduction (reduce_tc.cu): d_h = 64, gate values (sigmoid gate
// or the core API); cudaErrorNotSupported otherwise.
cudaError_t launch_reduce_tc(const ReduceArgs& a, int n_tiles, cudaStream_t st);
cudaError_t launch_readout_bf16(const ReadoutArgs& a, bool norm, int grid_x, cudaStream_t st);
cudaError_t launch_bwd_q_bf16(const BwdQArgs& a, bool norm, int grid_x, cudaStream_t st);
// tcgen05 query-side backward (bwd_q_tc.cu): d_h = 64; the layer's RMSNorm
// epilogue with phi(q) stored (pre), or the core form (q as given: no pre, r,
// rsinv, rms_w, dr or gamma_part); cudaErrorNotSupported otherwise.
// Its CTAs (two per SM) take contiguous ranges of the (128-row tile, head)
// units of a.tiles (n_tiles tiles); *nparts = the dgamma partial rows written.
cudaError_t launch_bwd_q_tc(const BwdQArgs& a, int hd, int n_tiles, int* nparts, cudaStream_t st);
// The same at d_h = 128 (bwd_q_tc128.cu), one CTA per SM.
cudaError_t launch_bwd_q_tc128(const BwdQArgs& a, int hd, int n_tiles, int* nparts, cudaStream_t st);
// tcgen05 readout with the RmsNorm gate (readout_tc.cu): d_h = 64 or 128,
// phi(q) stored (pre), no den output; cudaErrorNotSupported otherwise.
cudaError_t launch_readout_tc(const ReadoutArgs& a, int n_tiles, cudaStream_t st);
// The core form on tcgen05 (q as given, phi applied in shared memory, o and den
// out, no gate); bf16, d_h = 64 or 128.  cudaErrorNotSupported otherwise.
cudaError_t launch_readout_core_tc(const ReadoutArgs& a, int n_tiles, cudaStream_t st);
// tcgen05 key-side backward (bwd_kv_tc.cu): d_h = 64 or 128; phi(k) stored
// with the sigmoid gate (ds = dg g (1 - g)) or softmax logits (ds = dg g,
// g = exp(s - m)) and db_g partials in *nparts rows of bg_part; or the core
// form (k as given, gate values, dg out in fp32, no bg_part).
// cudaErrorNotSupported otherwise.
cudaError_t launch_bwd_kv_tc(const BwdKVArgs& a, int n_tiles, int* nparts, cudaStream_t st);
cudaError_t launch_bwd_kv_bf16(const BwdKVArgs& a, int grid_x, cudaStream_t st);
// tcgen05 softmax attention forward (sa_tc.cu): bf16, d_h = 64, one CTA per
// (256-query block, head), n_blocks blocks (past the last: nothing).
// cudaErrorNotSupported otherwise.
cudaError_t launch_sa_fwd_tc(const SaArgs& a, int n_blocks, cudaStream_t st);

cudaError_t launch_reduce_f32(const ReduceArgs& a, int grid_x, cudaStream_t st);
cudaError_t launch_readout_f32(const ReadoutArgs& a, bool norm, int grid_x, cudaStream_t st);
cudaError_t launch_bwd_q_f32(const BwdQArgs& a, bool norm, int grid_x, cudaStream_t st);
cudaError_t launch_bwd_kv_f32(const BwdKVArgs& a, int grid_x, cudaStream_t st);

cudaError_t launch_gemm_bf16(const GemmArgs& a, cudaStream_t st);
// tcgen05 + TMA GEMM; cudaErrorNotSupported for shapes it does not take.
cudaError_t launch_gemm_tc(const GemmArgs& a, cudaStream_t st);
cudaError_t launch_gemm_f32(const GemmArgs& a, cudaStream_t st);
// Which kernel variant a launcher ran (reported by the per-launch profiler).
enum Variant { VAR_TC = 0, VAR_MMA = 1, VAR_F32 = 2 };
// The GEMM of the layer: tcgen05 where supported, else mma.sync / fp32 SIMT.
inline cudaError_t launch_gemm(const GemmArgs& a, cudaStream_t st, int* variant = nullptr) {
  if (variant) *variant = VAR_TC;
  cudaError_t e = launch_gemm_tc(a, st);
  if (e != cudaErrorNotSupported) return e;
  (void)cudaGetLastError();
  if (variant) *variant = a.io_f32 ? VAR_F32 : VAR_MMA;
  return a.io_f32 ? launch_gemm_f32(a, st) : launch_gemm_bf16(a, st);
}

// *tiled = 1 when the bulk-copy staged bf16 kernel ran, 0 for the plain one.
// The launches of the decay core, in order: the chunks' local states, the
// scans per (sequence, head), the outputs (and, with padding, the zero rows).
// cudaErrorNotSupported unless d_h = 64.
cudaError_t launch_decay_states(const DecayArgs& a, int n_chunks, cudaStream_t st);
cudaError_t launch_decay_scan(const DecayArgs& a, int n_seq, cudaStream_t st);
cudaError_t launch_decay_out(const DecayArgs& a, int n_chunks, cudaStream_t st);
constexpr int kDecayChunk = 128;  // rows per chunk of the decay core

cudaError_t launch_conv_fwd(const ConvArgs& a, bool f32, cudaStream_t st, int* tiled = nullptr);
// Writes the parameter-gradient partials to part[0 .. *nparts)[d][5].
cudaError_t launch_conv_bwd(const ConvArgs& a, bool f32, int* nparts, cudaStream_t st, int* tiled = nullptr);
// Diagnostic: one CTA waits, with the kernels' bounded mbarrier wait limited
// to `polls` polls, on a barrier that nothing arrives at, and sets the
// timeout bit of *err when the wait gives up.
cudaError_t launch_diag_wait(int* err, unsigned polls, cudaStream_t st);
// Rows of the part buffer the backward may use, at most.
int conv_bwd_parts_max(int T);
// bf16 kernels staged through shared memory by bulk copies (conv.cu); usable
// when conv_tile_ok (16-byte aligned rows).
bool conv_tile_ok(const ConvArgs& a, bool bwd);
int conv_tile_parts(int T, int d);
int conv_tile_parts_max(int T);
cudaError_t launch_conv_fwd_tile(const ConvArgs& a, cudaStream_t st);
cudaError_t launch_conv_bwd_tile(const ConvArgs& a, int nparts, cudaStream_t st);
int sm_count();  // of the current device, cached

// Packs W_q | W_k | W_v | W_r | w_g into Wp [d][np] (row-major, zero-padded
// past 4*H*dh + H columns); also clears zero_bytes (a multiple of 4) at zero
// when zero is not null.
cudaError_t launch_pack_weights(const void* const* W, const void* w_g, int d, int H, int dh,
                                bool f32, void* Wp, int np, void* zero, size_t zero_bytes, cudaStream_t st);

// Fixed-order column sums of partial arrays, up to three in one launch: job
// j adds rows k = 0 .. S-1 of part[k * stride + i] for i < n; mode 0 writes
// out[i]; mode 1 (conv parameters, i = 5 c + t) writes t < 4 to out[4 c + t]
// and t = 4 to out2[c] (either may be null).
struct ColsumJob {
  const float* part; int S; int64_t stride, n;
  float* out; float* out2; int mode;
};
// The split-K sum of the weight gradient: part [S][d][np] fp32 -> dW_q, dW_k,
// dW_v, dW_r [d][H*dh] and dw_g [d][H] (out[m] may be null); fixed order.
struct ScatterJob {
  const float* part; int S, d, np, H, dh;
  float* out[5];
  int blocks;  // set by launch_colsums
};
struct ColsumJobs {
  ColsumJob j[3];
  int n;
  ScatterJob sc;  // part == null: none
};
// The scatter job (if any) and the column sums in one launch.
cudaError_t launch_colsums(ColsumJobs js, cudaStream_t st);

}  // namespace gbla
