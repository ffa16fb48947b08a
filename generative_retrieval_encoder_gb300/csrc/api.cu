// C ABI of the GBLA library (include/gbla.h): argument validation, workspace
// layout, tiling choices and the launch sequence of every entry point.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdio>
#include <cstring>
#include <string>
#include <vector>

#include "../../include/gbla.h"
#include "kernels.h"
#include "mbarrier.cuh"

using namespace gbla;

namespace {

thread_local std::string g_last_error;
thread_local int g_policy = GBLA_POLICY_AUTO;  // gbla_set_kernel_policy

constexpr size_t kAlign = 256;

size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }
int cdiv(int a, int b) { return (a + b - 1) / b; }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

// Per-launch profiler names of the GEMMs, by Variant: the projection, dx~ and dW GEMMs.
const char* const kGemmNames[3][3] = {
    {"projection gemm[tc]", "projection gemm[mma]", "projection gemm[f32]"},
    {"dx~ gemm[tc]", "dx~ gemm[mma]", "dx~ gemm[f32]"},
    {"dW gemm[tc]", "dW gemm[mma]", "dW gemm[f32]"},
};

// Everything derived from a shape: sequence form, tilings, buffer sizes.
struct Plan {
  bool f32;
  int B, L, d, H, dh, T, n_seq, mode;
  int HD, N1, NP;        // H*dh, 4*H*dh + H, N1 padded to 64
  int chunk, chunk_per_seq, n_chunks;  // state-reduction chunks (grid.x)
  int tile, tile_per_seq, n_tiles;     // readout / key-side tiles (grid.x)
  int wsplit, n_wsplit;                // dW split over rows
  int conv_blocks;
  int sms;               // SMs of the current device
  int max_grid;          // CTAs of a range-split kernel the workspace provides for (>= 2 x SMs)
  size_t io;             // bytes per io element
};

gbla_status make_plan(const gbla_shape* s, Plan& p) {
  if (!s) return GBLA_ERR_INVALID_ARG;
  if (s->io_dtype != GBLA_F32 && s->io_dtype != GBLA_BF16) return GBLA_ERR_INVALID_ARG;
  if (s->gate != GBLA_GATE_SIGMOID && s->gate != GBLA_GATE_SOFTMAX) return GBLA_ERR_INVALID_ARG;
  if (s->B < 1 || s->L < 1 || s->d < 1 || s->H < 1 || s->d_h < 1) return GBLA_ERR_INVALID_ARG;
  if (!(s->rms_eps >= 0.f)) return GBLA_ERR_INVALID_ARG;
  if (s->cu_seqlens && s->seq_lens) return GBLA_ERR_INVALID_ARG;
  if (s->cu_seqlens && (s->B != 1 || s->num_seqs < 1)) return GBLA_ERR_INVALID_ARG;
  p.f32 = s->io_dtype == GBLA_F32;
  p.io = p.f32 ? 4 : 2;
  p.B = s->B; p.L = s->L; p.d = s->d; p.H = s->H; p.dh = s->d_h;
  p.sms = sm_count();
  p.max_grid = std::max(512, 2 * p.sms);
  const int kSMs = p.sms;
  if (p.f32) {
    if (p.dh % 4 != 0 || p.dh > 128) return GBLA_ERR_UNSUPPORTED;
  } else {
    if (p.dh != 32 && p.dh != 64 && p.dh != 128) return GBLA_ERR_UNSUPPORTED;
  }
  const long long T = s->cu_seqlens ? (long long)s->L : (long long)s->B * s->L;
  if (T > (8LL << 20)) return GBLA_ERR_UNSUPPORTED;  // grid rows of the GEMMs
  if ((long long)s->H * s->d_h > 65536) return GBLA_ERR_UNSUPPORTED;
  p.T = (int)T;
  p.mode = s->cu_seqlens ? SEQ_VARLEN : (s->seq_lens ? SEQ_PADDED : SEQ_DENSE);
  p.n_seq = s->cu_seqlens ? s->num_seqs : s->B;
  p.HD = p.H * p.dh;
  p.N1 = 4 * p.HD + p.H;
  p.NP = (p.N1 + 63) / 64 * 64;
  const int pairs = p.n_seq * p.H;
  const int cg = p.f32 ? 64 : 128;  // chunk granule: the row tile of the query-side backward
  if (p.mode == SEQ_VARLEN) {
    const long long want = ((long long)p.T * p.H + kSMs - 1) / kSMs;
    p.chunk = (int)std::min<long long>(2048, std::max<long long>(256, (want + cg - 1) / cg * cg));
    p.chunk_per_seq = 0;
    p.n_chunks = cdiv(p.T, p.chunk) + p.n_seq;
  } else {
    // Chunks per sequence: one CTA per (chunk, head) of the state reduction
    // and the query-side backward, two resident per SM.  Take the split with
    // the least work on the busiest SM: its CTAs x (tiles per CTA + one tile
    // for start-up and the combine), at 3.7 time units a tile when two CTAs
    // share the SM and 4.5 when one runs alone (measured per-tile times of the
    // query-side backward).
    const int tiles = cdiv(p.L, cg);
    long long best_cost = -1;
    int best_tpc = tiles;
    for (int per = 1; per <= std::min(tiles, 64); ++per) {
      const int tpc = cdiv(tiles, per);
      const long long ctas = (long long)pairs * cdiv(tiles, tpc);
      const long long per_sm = (ctas + kSMs - 1) / kSMs;
      const long long cost = per_sm >= 2 ? per_sm * (tpc + 1) * 37 : (long long)(tpc + 1) * 45;
      if (best_cost < 0 || cost < best_cost) {
        best_cost = cost;
        best_tpc = tpc;
      }
    }
    p.chunk = best_tpc * cg;
    p.chunk_per_seq = cdiv(p.L, p.chunk);
    p.n_chunks = p.chunk_per_seq * p.n_seq;
  }
  p.tile = p.f32 ? 64 : (p.dh == 128 ? 128 : 256);
  if (p.mode == SEQ_VARLEN) {
    p.tile_per_seq = 0;
    p.n_tiles = cdiv(p.T, p.tile) + p.n_seq;
  } else {
    p.tile_per_seq = cdiv(p.L, p.tile);
    p.n_tiles = p.tile_per_seq * p.n_seq;
  }
  // dW = x~^T dP: split the T rows so that output tiles x splits fill whole
  // waves of the GPU (tiles of the bf16 tensor-core GEMM: 128 x 256; of the
  // fp32 GEMM: 64 x 64), each split at least 1024 rows.
  const int tiles = p.f32 ? cdiv(p.d, 64) * cdiv(p.NP, 64) : cdiv(p.d, 128) * cdiv(p.NP, 256);
  const int max_split = std::max(1, std::min(16, p.T / 1024));
  int want_split = 1;
  double best = -1.0;
  for (int sp = 1; sp <= max_split; ++sp) {
    const int units = tiles * sp;
    const double eff = (double)units / ((double)cdiv(units, kSMs) * kSMs);
    if (eff > best + 0.02) { best = eff; want_split = sp; }  // the smallest split within 2% of the best
  }
  p.wsplit = cdiv(cdiv(p.T, want_split), 64) * 64;
  p.n_wsplit = cdiv(p.T, p.wsplit);
  p.conv_blocks = conv_bwd_parts_max(p.T);
  return GBLA_OK;
}

gbla_status check_layer_shape(const Plan& p) {
  if (p.d % (p.f32 ? 4 : 64) != 0) return GBLA_ERR_UNSUPPORTED;
  return GBLA_OK;
}

// Byte layout of a workspace (or of the saved buffer), in order.
struct Layout {
  size_t err, cnt_f, cnt_b, pre_c, pre_t;
  size_t partial, partial_m, state, state_bf, state_m, center;
  size_t xt, P, gate, Wt;
  size_t Wp, dP, dxt, dW, dstate, dstate_bf, gamma_part, bg_part, conv_part;
  size_t pre_d, LF, LB, lamc, HF, HB;  // the decay core: its chunks' prefix, chunk and scan states
  size_t total;
};

// 256-query blocks (per sequence) of the softmax attention.
constexpr int kSaBlock = 256;
int sa_blocks(const Plan& p) {
  return p.mode == SEQ_VARLEN ? cdiv(p.T, kSaBlock) + p.n_seq : cdiv(p.L, kSaBlock) * p.n_seq;
}

// Chunks (128 rows, per sequence) of the decay core.
int decay_chunks(const Plan& p) {
  return p.mode == SEQ_VARLEN ? cdiv(p.T, kDecayChunk) + p.n_seq : cdiv(p.L, kDecayChunk) * p.n_seq;
}

struct Cursor {
  size_t off = 0;
  size_t take(size_t bytes) { const size_t o = off; off = align_up(off + bytes); return o; }
};


size_t state_bytes(const Plan& p) { return (size_t)p.n_seq * p.H * p.dh * state_ld(p.dh) * 4; }
size_t state_bf_bytes(const Plan& p) { return (size_t)p.n_seq * p.H * p.dh * state_bf_ld(p.dh) * 2; }

// Saved activations of a training forward: x~, P = [q|k|v|r], gate, state.
struct SavedLayout { size_t xt, P, gate, state, state_bf, state_m, center, rsinv, total; };
size_t center_bytes(const Plan& p) { return (size_t)p.n_seq * p.H * p.dh * 4; }
SavedLayout saved_layout(const Plan& p) {
  Cursor c;
  SavedLayout s;
  s.xt = c.take((size_t)p.T * p.d * p.io);
  s.P = c.take((size_t)p.T * 4 * p.HD * p.io);
  s.gate = c.take((size_t)p.T * p.H * 4);
  s.state = c.take(state_bytes(p));
  s.state_bf = c.take(state_bf_bytes(p));
  s.state_m = c.take((size_t)p.n_seq * p.H * 4);
  s.center = c.take(center_bytes(p));
  s.rsinv = c.take((size_t)p.T * p.H * 8);  // per row and head: RMSNorm rs and 1/den of the readout
  s.total = c.off;
  return s;
}

// Partial-state slots: one per (chunk, head) for the split-L kernels; the
// tcgen05 query-side backward takes one per (sequence, head) plus one per CTA
// (a CTA boundary inside a (sequence, head)).
int partial_slots(const Plan& p) { return std::max(p.n_chunks * p.H, p.n_seq * p.H + p.max_grid); }

Layout ws_layout(const Plan& p, int op) {
  Cursor c;
  Layout l;
  std::memset(&l, 0xff, sizeof(l));
  const size_t cnt = (size_t)p.n_seq * p.H * 4;
  l.err = c.take(16 + 2 * cnt);  // err word, then forward and backward counters
  l.cnt_f = l.err + 16;
  l.cnt_b = l.cnt_f + cnt;
  if (p.mode == SEQ_VARLEN) {
    l.pre_c = c.take((size_t)(p.n_seq + 1) * 4);
    l.pre_t = c.take((size_t)(p.n_seq + 1) * 4);
  }
  if (op != GBLA_OP_SA_FORWARD) {  // split-L partial states (every kernel but the softmax attention)
    l.partial = c.take((size_t)partial_slots(p) * p.dh * state_ld(p.dh) * 4);
    l.partial_m = c.take((size_t)p.n_chunks * p.H * 4);
  }
  if (op == GBLA_OP_FORWARD) {  // inference forward keeps its activations here
    l.state = c.take(state_bytes(p));
    l.state_bf = c.take(state_bf_bytes(p));
    l.state_m = c.take((size_t)p.n_seq * p.H * 4);
    l.center = c.take(center_bytes(p));
    l.xt = c.take((size_t)p.T * p.d * p.io);
    l.P = c.take((size_t)p.T * 4 * p.HD * p.io);
    l.gate = c.take((size_t)p.T * p.H * 4);
    l.Wt = c.take((size_t)p.d * p.NP * p.io);  // packed W_all [d][NP]
  } else if (op == GBLA_OP_BACKWARD) {
    l.Wp = c.take((size_t)p.d * p.NP * p.io);
    l.dP = c.take((size_t)p.T * p.NP * p.io);
    l.dxt = c.take((size_t)p.T * p.d * p.io);
    l.dW = c.take((size_t)p.n_wsplit * p.d * p.NP * 4);
    l.dstate = c.take(state_bytes(p));
    l.dstate_bf = c.take(state_bf_bytes(p));
    l.gamma_part = c.take((size_t)std::max(p.n_chunks * p.H, p.max_grid) * p.dh * 4);
    // db_g partial rows: two per tile (tcgen05 kernel) or one per chunk
    l.bg_part = c.take((size_t)std::max(2 * p.n_tiles, p.n_chunks) * p.H * 4);
    l.conv_part = c.take((size_t)p.conv_blocks * p.d * 5 * 4);
  } else if (op == GBLA_OP_SA_FORWARD) {
    if (p.mode == SEQ_VARLEN) l.pre_d = c.take((size_t)(p.n_seq + 1) * 4);
  } else if (op == GBLA_OP_DECAY_FORWARD) {
    const size_t ch = (size_t)decay_chunks(p) * p.H;
    if (p.mode == SEQ_VARLEN) l.pre_d = c.take((size_t)(p.n_seq + 1) * 4);
    l.LF = c.take(ch * p.dh * state_ld(p.dh) * 2);
    l.LB = c.take(ch * p.dh * state_ld(p.dh) * 2);
    l.lamc = c.take(ch * 4);
    l.HF = c.take(ch * p.dh * state_bf_ld(p.dh) * 2);
    l.HB = c.take(ch * p.dh * state_bf_ld(p.dh) * 2);
  } else {  // core forward / backward
    l.state = c.take(state_bytes(p));
    l.state_bf = c.take(state_bf_bytes(p));
    l.state_m = c.take((size_t)p.n_seq * p.H * 4);
    l.center = c.take(center_bytes(p));
    if (op == GBLA_OP_CORE_BACKWARD) {
      l.dstate = c.take(state_bytes(p));
      l.dstate_bf = c.take(state_bf_bytes(p));
    }
  }
  l.total = c.off;
  return l;
}

template <typename T>
T* at(void* base, size_t off) {
  return reinterpret_cast<T*>(static_cast<char*>(base) + off);
}

gbla_status cuda_fail(cudaError_t e, const char* what) {
  g_last_error = std::string(what) + ": " + cudaGetErrorString(e);
  return GBLA_ERR_CUDA;
}

// Per-launch timing (gbla_profiling_*): when on, every launch of this thread
// is bracketed by two CUDA events recorded on the call's stream.
struct ProfRecord { const char* name; cudaEvent_t t0, t1; };
struct Profiler {
  bool on = false;
  std::vector<ProfRecord> rec;
  std::vector<cudaEvent_t> pool;
  cudaEvent_t event() {
    if (!pool.empty()) { cudaEvent_t e = pool.back(); pool.pop_back(); return e; }
    cudaEvent_t e = nullptr;
    cudaEventCreate(&e);
    return e;
  }
};
thread_local Profiler g_prof;

#define GBLA_CHECK(call, what)                                         \
  do {                                                                 \
    cudaEvent_t t0_ = nullptr;                                         \
    if (g_prof.on) { t0_ = g_prof.event(); cudaEventRecord(t0_, c.st); } \
    cudaError_t e_ = (call);                                           \
    if (g_prof.on) {                                                   \
      cudaEvent_t t1_ = g_prof.event();                                \
      cudaEventRecord(t1_, c.st);                                      \
      g_prof.rec.push_back({what, t0_, t1_});                          \
    }                                                                  \
    if (e_ != cudaSuccess) return cuda_fail(e_, what);                 \
  } while (0)

struct Ctx {
  Plan p;
  Layout l;
  SeqDesc seq;
  Tiling chunks, tiles;
  int* err;          // workspace error word (always valid)
  const int* kerr;   // what the state / conv kernels read: err, or null in the dense form
  cudaStream_t st;
  int pre = 0;       // P holds [phi(q) | phi(k) | v | r] (the bf16 layer)
  // The error word and counters to clear, when the call's first kernel (the
  // weight pack) clears them instead of a memset; null once cleared.
  void* zero = nullptr;
  size_t zero_bytes = 0;
};

// The bf16 layer applies the feature map phi = elu + 1 to q and k in the
// projection epilogue, so the state kernels read phi(q) and phi(k) directly.
bool layer_pre(const Plan& p, const gbla_shape*) { return !p.f32; }

// zero_in_pack: the caller's first kernel is the weight pack, which then
// clears the error word and counters (dense batches: no sequence-data check
// runs before it).
gbla_status begin(const gbla_shape* s, int op, void* ws, size_t ws_bytes, void* stream, Ctx& c,
                  bool zero_in_pack = false) {
  gbla_status r = make_plan(s, c.p);
  if (r != GBLA_OK) return r;
  c.l = ws_layout(c.p, op);
  if (!ws || (reinterpret_cast<uintptr_t>(ws) % kAlign) != 0 || ws_bytes < c.l.total) return GBLA_ERR_WORKSPACE;
  c.st = static_cast<cudaStream_t>(stream);
  const Plan& p = c.p;
  c.seq.mode = p.mode;
  c.seq.n_seq = p.n_seq;
  c.seq.L = p.mode == SEQ_VARLEN ? p.T : p.L;
  c.seq.T = p.T;
  c.seq.lens = s->seq_lens;
  c.seq.cu = s->cu_seqlens;
  c.chunks.tile = p.chunk;
  c.chunks.per_seq = p.chunk_per_seq;
  c.chunks.prefix = p.mode == SEQ_VARLEN ? at<int32_t>(ws, c.l.pre_c) : nullptr;
  c.tiles.tile = p.tile;
  c.tiles.per_seq = p.tile_per_seq;
  c.tiles.prefix = p.mode == SEQ_VARLEN ? at<int32_t>(ws, c.l.pre_t) : nullptr;
  c.err = at<int>(ws, c.l.err);
  // Only the varlen and padded forms have sequence data to check on the
  // device; in the dense form the kernels skip the error-word read.
  c.kerr = p.mode == SEQ_DENSE ? nullptr : c.err;
  const size_t zero_bytes = c.l.cnt_b + (size_t)p.n_seq * p.H * 4 - c.l.err;
  if (zero_in_pack && p.mode == SEQ_DENSE) {
    c.zero = at<char>(ws, c.l.err);
    c.zero_bytes = zero_bytes;
  } else {
    GBLA_CHECK(cudaMemsetAsync(at<char>(ws, c.l.err), 0, zero_bytes, c.st), "memset");
  }
  if (p.mode != SEQ_DENSE) {
    const int ts[2] = {p.chunk, p.tile};
    int32_t* pre[2] = {const_cast<int32_t*>(c.chunks.prefix), const_cast<int32_t*>(c.tiles.prefix)};
    GBLA_CHECK(launch_plan(c.seq, p.mode == SEQ_VARLEN ? 2 : 0, ts, pre, c.err, c.st), "plan");
  }
  return GBLA_OK;
}

// State reduction + combine.  The bf16 path centres the state on the
// k~-weighted mean of v (center); the fp32 path keeps it uncentred.
// The layer's bf16 readout: the tcgen05 kernel where it applies.
// The mma.sync readout loads a (sequence, head) state per CTA: it takes a
// chunk of rows (up to 2048) per CTA, not a tile, so that the load is spread
// over more rows.  Every row is written by its own index, whatever the tiling.
cudaError_t launch_readout_chunks_bf16(const ReadoutArgs& ra, bool norm, const Tiling& chunks, int n_chunks,
                                       cudaStream_t st) {
  ReadoutArgs rc = ra;
  rc.tiles = chunks;
  return launch_readout_bf16(rc, norm, n_chunks, st);
}

// The core readout: tcgen05 where it applies (unless the policy asks for
// mma.sync), else the mma.sync kernel over the chunks.
cudaError_t launch_readout_core_bf16(const ReadoutArgs& ra, int n_tiles, const Tiling& chunks, int n_chunks,
                                     cudaStream_t st, const char** name) {
  if (g_policy != GBLA_POLICY_MMA) {
    const cudaError_t e = launch_readout_core_tc(ra, n_tiles, st);
    if (e != cudaErrorNotSupported) {
      *name = "readout[tc]";
      return e;
    }
    (void)cudaGetLastError();
  }
  *name = "readout[mma]";
  return launch_readout_chunks_bf16(ra, false, chunks, n_chunks, st);
}

cudaError_t launch_readout_layer_bf16(const ReadoutArgs& ra, int n_tiles, const Tiling& chunks, int n_chunks,
                                      cudaStream_t st, const char** nm) {
  if (g_policy != GBLA_POLICY_MMA) {
    *nm = "readout[tc]";
    const cudaError_t e = launch_readout_tc(ra, n_tiles, st);
    if (e != cudaErrorNotSupported) return e;
    (void)cudaGetLastError();
  }
  *nm = "readout[mma]";
  return launch_readout_chunks_bf16(ra, true, chunks, n_chunks, st);
}

// The layer's bf16 key-side backward: the tcgen05 kernel where it applies;
// *bg_rows = the rows of db_g partials written.
// The mma.sync key-side backward, like the readout, takes a chunk of rows per
// CTA (one load of [dS | dz] for up to 2048 rows).  Its db_g partials are one
// row per CTA: n_chunks <= 2 n_tiles rows, which the partial buffer holds.
cudaError_t launch_bwd_kv_chunks_bf16(const BwdKVArgs& kv, const Tiling& chunks, int n_chunks, cudaStream_t st) {
  BwdKVArgs kc = kv;
  kc.tiles = chunks;
  return launch_bwd_kv_bf16(kc, n_chunks, st);
}

// The core's query-side backward: tcgen05 where it applies (d_h = 64; unless
// the policy asks for mma.sync), else the mma.sync kernel.
cudaError_t launch_bwd_q_core_bf16(const BwdQArgs& q, int hd, int n_tiles, const Ctx& c, const char** nm) {
  if (g_policy != GBLA_POLICY_MMA) {
    int parts = 0;
    const cudaError_t e = launch_bwd_q_tc(q, hd, n_tiles, &parts, c.st);
    if (e != cudaErrorNotSupported) {
      *nm = "bwd_q[tc]";
      return e;
    }
    (void)cudaGetLastError();
  }
  *nm = "bwd_q[mma]";
  return launch_bwd_q_bf16(q, false, c.p.n_chunks, c.st);
}

// The core's key-side backward: tcgen05 where it applies (unless the policy
// asks for mma.sync), else the mma.sync kernel over the chunks.
cudaError_t launch_bwd_kv_core_bf16(const BwdKVArgs& kv, int n_tiles, const Ctx& c, const char** nm) {
  if (g_policy != GBLA_POLICY_MMA) {
    int parts = 0;
    const cudaError_t e = launch_bwd_kv_tc(kv, n_tiles, &parts, c.st);
    if (e != cudaErrorNotSupported) {
      *nm = "bwd_kv[tc]";
      return e;
    }
    (void)cudaGetLastError();
  }
  *nm = "bwd_kv[mma]";
  return launch_bwd_kv_chunks_bf16(kv, c.chunks, c.p.n_chunks, c.st);
}

cudaError_t launch_bwd_kv_layer_bf16(const BwdKVArgs& kv, int n_tiles, const Tiling& chunks, int n_chunks,
                                     int* bg_rows, cudaStream_t st, const char** nm) {
  if (g_policy != GBLA_POLICY_MMA) {
    *nm = "bwd_kv[tc]";
    const cudaError_t e = launch_bwd_kv_tc(kv, n_tiles, bg_rows, st);
    if (e != cudaErrorNotSupported) return e;
    (void)cudaGetLastError();
  }
  *nm = "bwd_kv[mma]";
  *bg_rows = n_chunks;
  return launch_bwd_kv_chunks_bf16(kv, chunks, n_chunks, st);
}

// The layer's bf16 query-side backward: the tcgen05 kernel where it applies.
// *gamma_rows = the rows of dgamma partials written.
cudaError_t launch_bwd_q_layer_bf16(const BwdQArgs& q, int hd, int n_chunks, int n_tiles, int* gamma_rows,
                                    cudaStream_t st, const char** nm) {
  if (g_policy != GBLA_POLICY_MMA) {
    *nm = "bwd_q[tc]";
    cudaError_t e = launch_bwd_q_tc(q, hd, n_tiles, gamma_rows, st);
    if (e != cudaErrorNotSupported) return e;
    (void)cudaGetLastError();
    e = launch_bwd_q_tc128(q, hd, n_tiles, gamma_rows, st);
    if (e != cudaErrorNotSupported) return e;
    (void)cudaGetLastError();
  }
  *nm = "bwd_q[mma]";
  *gamma_rows = n_chunks * q.H;
  return launch_bwd_q_bf16(q, true, n_chunks, st);
}

// The bf16 state reduction: the tcgen05 kernel where it applies (gate values,
// d_h = 64) and either each SM streams at least 20 of its 256-row tiles or
// phi(k) is not stored (the core entry points: the mma.sync kernel then
// applies phi in registers, 65 against 61 us at 13 tiles an SM), else the
// mma.sync kernel (softmax logits, other d_h; and shorter batches of the
// layer, where the tcgen05 kernel's fixed start and final drain outweigh its
// faster stream: measured 51 against 47 us at 13 tiles an SM, 80 against 81
// at 27, 129 against 132 at 54).
cudaError_t launch_reduce_layer_bf16(const ReduceArgs& a, int n_chunks, int n_tiles, int sms, cudaStream_t st,
                                     const char** nm) {
  const long long units = (long long)a.seq.T * a.H / 256;
  if (((units >= 20LL * sms || !a.pre) && g_policy != GBLA_POLICY_MMA) || g_policy == GBLA_POLICY_TC) {
    *nm = "reduce[tc]";
    const cudaError_t e = launch_reduce_tc(a, n_tiles, st);
    if (e != cudaErrorNotSupported) return e;
    (void)cudaGetLastError();
  }
  *nm = "reduce[mma]";
  return launch_reduce_bf16(a, n_chunks, st);
}

gbla_status run_reduce(Ctx& c, const void* k, const void* v, int64_t ld, const float* g, int gate_kind, float* state,
                       bf16* state_bf, float* state_m, float* pub_state, float* center, void* ws) {
  const Plan& p = c.p;
  ReduceArgs a{};
  a.k = k; a.v = v; a.ldk = ld; a.ldv = ld;
  a.g = g; a.ldg = p.H; a.gate_kind = gate_kind;
  a.H = p.H; a.dh = p.dh;
  a.seq = c.seq; a.chunks = c.chunks;
  a.partial = at<float>(ws, c.l.partial);
  a.partial_m = at<float>(ws, c.l.partial_m);
  a.counters = at<int>(ws, c.l.cnt_f);
  a.state = state; a.state_bf = state_bf; a.state_m = state_m; a.pub_state = pub_state;
  a.pre = c.pre;
  a.center = p.f32 ? nullptr : center;
  a.err = c.kerr;
  a.tiles = c.tiles;
  a.partial_slots = partial_slots(p);
  a.err_out = c.err;
  const char* nm = "reduce[f32]";
  GBLA_CHECK(p.f32 ? launch_reduce_f32(a, p.n_chunks, c.st) : launch_reduce_layer_bf16(a, p.n_chunks, p.n_tiles, p.sms, c.st, &nm),
             nm);
  return GBLA_OK;
}

}  // namespace

extern "C" {

gbla_status gbla_validate_shape(const gbla_shape* shape) {
  Plan p;
  return make_plan(shape, p);
}

size_t gbla_workspace_size(const gbla_shape* shape, int op) {
  Plan p;
  if (make_plan(shape, p) != GBLA_OK) return 0;
  if (op < GBLA_OP_FORWARD || op > GBLA_OP_SA_FORWARD) return 0;
  return ws_layout(p, op).total;
}

size_t gbla_saved_size(const gbla_shape* shape) {
  Plan p;
  if (make_plan(shape, p) != GBLA_OK) return 0;
  return saved_layout(p).total;
}

gbla_status gbla_forward(const gbla_shape* shape, const void* x, const void* conv_w, const void* conv_b,
                         const void* W_q, const void* W_k, const void* W_v, const void* W_r, const void* w_g,
                         const void* b_g, const void* rms_w, void* y, void* saved, void* ws, size_t ws_bytes,
                         void* stream) {
  Plan p0;
  gbla_status r = make_plan(shape, p0);
  if (r != GBLA_OK) return r;
  if ((r = check_layer_shape(p0)) != GBLA_OK) return r;
  const void* req[] = {x, conv_w, W_q, W_k, W_v, W_r, w_g, y};
  for (const void* q : req)
    if (!q || !aligned16(q)) return GBLA_ERR_INVALID_ARG;
  for (const void* q : {conv_b, b_g, rms_w})
    if (q && !aligned16(q)) return GBLA_ERR_INVALID_ARG;
  if (saved && (reinterpret_cast<uintptr_t>(saved) % kAlign) != 0) return GBLA_ERR_INVALID_ARG;
  Ctx c;
  if ((r = begin(shape, GBLA_OP_FORWARD, ws, ws_bytes, stream, c, true)) != GBLA_OK) return r;
  const Plan& p = c.p;
  const Layout& l = c.l;
  void *xt, *P;
  float *gate, *state, *state_m, *center;
  bf16* state_bf;
  if (saved) {
    const SavedLayout s = saved_layout(p);
    xt = at<char>(saved, s.xt); P = at<char>(saved, s.P); gate = at<float>(saved, s.gate);
    state = at<float>(saved, s.state); state_bf = at<bf16>(saved, s.state_bf); state_m = at<float>(saved, s.state_m);
    center = at<float>(saved, s.center);
  } else {
    xt = at<char>(ws, l.xt); P = at<char>(ws, l.P); gate = at<float>(ws, l.gate);
    state = at<float>(ws, l.state); state_bf = at<bf16>(ws, l.state_bf); state_m = at<float>(ws, l.state_m);
    center = at<float>(ws, l.center);
  }
  if (p.f32) center = nullptr;
  // packed weights first: the pack also clears the error word and counters (dense batches)
  const void* W[4] = {W_q, W_k, W_v, W_r};
  void* Wt = at<char>(ws, l.Wt);
  GBLA_CHECK(launch_pack_weights(W, w_g, p.d, p.H, p.dh, p.f32, Wt, p.NP, c.zero, c.zero_bytes, c.st), "pack");
  // Eq. 4: conv
  ConvArgs ca{};
  ca.x = x; ca.w = conv_w; ca.b = conv_b; ca.xt = xt; ca.T = p.T; ca.d = p.d; ca.seq = c.seq; ca.err = c.kerr; ca.err_out = c.err;
  int tiled = 0;
  GBLA_CHECK(launch_conv_fwd(ca, p.f32, c.st, &tiled), tiled ? "conv[bulk]" : "conv[plain]");
  c.pre = layer_pre(p, shape) ? 1 : 0;
  // Eq. 4, 5, 7: projections and gate
  GemmArgs ga{};
  ga.A = xt; ga.lda = p.d; ga.a_kmajor = 1;
  ga.B = Wt; ga.ldb = p.NP; ga.b_kmajor = 0;  // B(n, k) = W_all[k][n]: N-major
  ga.C = P; ga.ldc = 4 * p.HD;
  ga.M = p.T; ga.N = p.N1; ga.K = p.d; ga.k_split = (p.d + 31) / 32 * 32;
  ga.epi = c.pre ? EPI_PROJ_PRE : EPI_PROJ; ga.n_main = 4 * p.HD; ga.hd = p.HD; ga.dh = p.dh;
  ga.bias_g = shape->gate == GBLA_GATE_SIGMOID ? b_g : nullptr;
  ga.gate_mode = shape->gate == GBLA_GATE_SIGMOID ? 0 : 1; ga.gate = gate; ga.ldgate = p.H; ga.io_f32 = p.f32;
  ga.err = c.err;
  ga.pair = 1;  // CTA pairs: each CTA loads half of B, a third less operand traffic per SM
  int var = VAR_TC;
  GBLA_CHECK(launch_gemm(ga, c.st, &var), kGemmNames[0][var]);
  // Eq. 5/6: state
  const size_t es = p.io;
  const char* Pc = static_cast<const char*>(P);
  r = run_reduce(c, Pc + p.HD * es, Pc + 2 * p.HD * es, 4 * p.HD, gate,
                 shape->gate == GBLA_GATE_SIGMOID ? GATE_VALUES : GATE_LOGITS, state, state_bf, state_m, nullptr,
                 center, ws);
  if (r != GBLA_OK) return r;
  // Eq. 5/6 readout fused with Eq. 7
  ReadoutArgs ra{};
  ra.q = P; ra.ldq = 4 * p.HD;
  ra.r = Pc + 3 * p.HD * es; ra.ldr = 4 * p.HD;
  ra.rms_w = rms_w; ra.eps = shape->rms_eps;
  ra.state = state; ra.state_bf = state_bf; ra.center = center; ra.pre = c.pre;
  ra.out = y; ra.ldo = p.HD; ra.den = nullptr;
  ra.rsinv = (saved && !p.f32) ? at<float>(saved, saved_layout(p).rsinv) : nullptr;
  ra.H = p.H; ra.dh = p.dh; ra.seq = c.seq; ra.tiles = c.tiles; ra.err = c.kerr; ra.err_out = c.err;
  const char* nm = "readout[f32]";
  GBLA_CHECK(p.f32 ? launch_readout_f32(ra, true, p.n_tiles, c.st)
                   : launch_readout_layer_bf16(ra, p.n_tiles, c.chunks, p.n_chunks, c.st, &nm),
             nm);
  return GBLA_OK;
}

gbla_status gbla_backward(const gbla_shape* shape, const void* x, const void* conv_w, const void* conv_b,
                          const void* W_q, const void* W_k, const void* W_v, const void* W_r, const void* w_g,
                          const void* b_g, const void* rms_w, const void* saved, const void* dy, void* dx,
                          float* dconv_w, float* dconv_b, float* dW_q, float* dW_k, float* dW_v, float* dW_r,
                          float* dw_g, float* db_g, float* drms_w, void* ws, size_t ws_bytes, void* stream) {
  (void)conv_b; (void)b_g;
  Plan p0;
  gbla_status r = make_plan(shape, p0);
  if (r != GBLA_OK) return r;
  if ((r = check_layer_shape(p0)) != GBLA_OK) return r;
  const void* req[] = {x, conv_w, W_q, W_k, W_v, W_r, w_g, saved, dy, dx};
  for (const void* q : req)
    if (!q || !aligned16(q)) return GBLA_ERR_INVALID_ARG;
  if (rms_w && !aligned16(rms_w)) return GBLA_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(saved) % kAlign) != 0) return GBLA_ERR_INVALID_ARG;
  Ctx c;
  if ((r = begin(shape, GBLA_OP_BACKWARD, ws, ws_bytes, stream, c, true)) != GBLA_OK) return r;
  const Plan& p = c.p;
  const Layout& l = c.l;
  const SavedLayout s = saved_layout(p);
  const size_t es = p.io;
  const char* P = at<const char>(const_cast<void*>(saved), s.P);
  const void* xt = at<const char>(const_cast<void*>(saved), s.xt);
  const float* gate = at<const float>(const_cast<void*>(saved), s.gate);
  char* dP = at<char>(ws, l.dP);
  const bool sig = shape->gate == GBLA_GATE_SIGMOID;
  const int pre = layer_pre(p, shape) ? 1 : 0;
  // gamma_part and bg_part: every CTA of bwd_q / bwd_kv writes its row (zeros when it has no rows)
  const void* W[4] = {W_q, W_k, W_v, W_r};
  GBLA_CHECK(launch_pack_weights(W, w_g, p.d, p.H, p.dh, p.f32, at<char>(ws, l.Wp), p.NP, c.zero, c.zero_bytes, c.st),
             "pack");
  // Eq. 7 + Eq. 5/6 query side: dr, dq, [dS | dz]
  BwdQArgs q{};
  q.q = P; q.ldq = 4 * p.HD;
  q.r = P + 3 * p.HD * es; q.ldr = 4 * p.HD;
  q.dy = dy; q.lddy = p.HD;
  q.rms_w = rms_w; q.eps = shape->rms_eps;
  q.state = at<const float>(const_cast<void*>(saved), s.state);
  q.state_bf = at<const bf16>(const_cast<void*>(saved), s.state_bf);
  const float* center = p.f32 ? nullptr : at<const float>(const_cast<void*>(saved), s.center);
  q.center = center;
  q.pre = pre;
  q.dq = dP; q.lddq = p.NP;
  q.dr = dP + 3 * p.HD * es; q.lddr = p.NP;
  q.gamma_part = at<float>(ws, l.gamma_part);
  q.partial = at<float>(ws, l.partial); q.counters = at<int>(ws, l.cnt_b);
  q.dstate = at<float>(ws, l.dstate); q.dstate_bf = at<bf16>(ws, l.dstate_bf);
  q.rsinv = at<const float>(const_cast<void*>(saved), s.rsinv);
  q.H = p.H; q.dh = p.dh; q.seq = c.seq; q.chunks = c.chunks; q.tiles = c.tiles; q.err = c.kerr; q.err_out = c.err;
  q.partial_slots = partial_slots(p);
  int gamma_rows = p.n_chunks * p.H;
  const char* nm = "bwd_q[f32]";
  GBLA_CHECK(p.f32 ? launch_bwd_q_f32(q, true, p.n_chunks, c.st)
                   : launch_bwd_q_layer_bf16(q, p.HD, p.n_chunks, p.n_tiles, &gamma_rows, c.st, &nm),
             nm);
  // key side: dk, dv, ds
  BwdKVArgs kv{};
  kv.k = P + p.HD * es; kv.ldk = 4 * p.HD;
  kv.v = P + 2 * p.HD * es; kv.ldv = 4 * p.HD;
  kv.g = gate; kv.ldg = p.H; kv.gate_kind = sig ? GATE_VALUES : GATE_LOGITS;
  kv.state_m = at<const float>(const_cast<void*>(saved), s.state_m);
  kv.dstate = at<float>(ws, l.dstate); kv.dstate_bf = at<bf16>(ws, l.dstate_bf);
  kv.center = center;
  kv.pre = pre;
  kv.dk = dP + p.HD * es; kv.lddk = p.NP;
  kv.dv = dP + 2 * p.HD * es; kv.lddv = p.NP;
  kv.ds = dP; kv.ldds = p.NP; kv.gate_grad = sig ? GG_SIGMOID : GG_SOFTMAX;
  // ds of head h lands in column 4*H*dh + h: offset the pointer, keep the stride
  kv.ds = dP + (size_t)4 * p.HD * es;
  kv.zero_cols_from = kv.zero_cols_to = 0;  // the pad columns of dP are never read
  kv.bg_part = at<float>(ws, l.bg_part);
  kv.H = p.H; kv.dh = p.dh; kv.seq = c.seq; kv.tiles = c.tiles; kv.err = c.kerr; kv.err_out = c.err;
  int bg_rows = p.n_tiles;
  nm = "bwd_kv[f32]";
  GBLA_CHECK(p.f32 ? launch_bwd_kv_f32(kv, p.n_tiles, c.st)
                   : launch_bwd_kv_layer_bf16(kv, p.n_tiles, c.chunks, p.n_chunks, &bg_rows, c.st, &nm),
             nm);
  // Eq. 4 projections backward: dx~ = dP W_all^T, dW_all = x~^T dP
  GemmArgs g1{};
  g1.A = dP; g1.lda = p.NP; g1.a_kmajor = 1;
  g1.B = at<char>(ws, l.Wp); g1.ldb = p.NP; g1.b_kmajor = 1;
  g1.C = at<char>(ws, l.dxt); g1.ldc = p.d;  // dx~ in the io dtype
  // K = N1, not the padded NP: the pad columns of dP and W_all are never read (the
  // tensor-core GEMM's loads zero-fill past N1), so nothing needs to clear them
  g1.M = p.T; g1.N = p.d; g1.K = p.N1; g1.k_split = p.N1; g1.epi = p.f32 ? EPI_F32 : EPI_BF16; g1.io_f32 = p.f32;
  g1.err = c.err;
  g1.pair = 1;  // long K: the operand feed limits, CTA pairs halve it per SM
  int var = VAR_TC;
  GBLA_CHECK(launch_gemm(g1, c.st, &var), kGemmNames[1][var]);
  GemmArgs g2{};
  g2.A = xt; g2.lda = p.d; g2.a_kmajor = 0;
  g2.B = dP; g2.ldb = p.NP; g2.b_kmajor = 0;
  g2.C = at<float>(ws, l.dW); g2.ldc = p.NP;
  g2.M = p.d; g2.N = p.N1; g2.K = p.T; g2.k_split = p.wsplit; g2.epi = EPI_SPLITK; g2.io_f32 = p.f32; g2.err = c.err;
  g2.pair = 1;  // long K: the operand feed limits, CTA pairs halve it per SM
  GBLA_CHECK(launch_gemm(g2, c.st, &var), kGemmNames[2][var]);

  // Eq. 4 conv backward
  ConvArgs ca{};
  ca.x = x; ca.w = conv_w; ca.dxt = at<char>(ws, l.dxt); ca.dx = dx; ca.part = at<float>(ws, l.conv_part);
  ca.T = p.T; ca.d = p.d; ca.seq = c.seq; ca.err = c.kerr; ca.err_out = c.err;
  int nparts = 0, tiled = 0;
  GBLA_CHECK(launch_conv_bwd(ca, p.f32, &nparts, c.st, &tiled), tiled ? "conv bwd[bulk]" : "conv bwd[plain]");
  // the parameter gradients from their partials, one launch: W_all, conv taps and bias, gamma, b_g
  ColsumJobs js{};
  js.sc.part = at<float>(ws, l.dW);  // and the split-K sum of the weight gradient
  js.sc.S = p.n_wsplit; js.sc.d = p.d; js.sc.np = p.NP; js.sc.H = p.H; js.sc.dh = p.dh;
  js.sc.out[0] = dW_q; js.sc.out[1] = dW_k; js.sc.out[2] = dW_v; js.sc.out[3] = dW_r; js.sc.out[4] = dw_g;
  if (dconv_w || dconv_b)
    js.j[js.n++] = ColsumJob{ca.part, nparts, (int64_t)p.d * 5, (int64_t)p.d * 5, (float*)dconv_w, (float*)dconv_b, 1};
  if (drms_w) js.j[js.n++] = ColsumJob{q.gamma_part, gamma_rows, p.dh, p.dh, (float*)drms_w, nullptr, 0};
  if (db_g) js.j[js.n++] = ColsumJob{kv.bg_part, bg_rows, p.H, p.H, (float*)db_g, nullptr, 0};
  GBLA_CHECK(launch_colsums(js, c.st), "param grads");
  return GBLA_OK;
}

gbla_status bla_core_forward(const gbla_shape* shape, const void* q, const void* k, const void* v, const float* g,
                             void* o, float* den, float* state, void* ws, size_t ws_bytes, void* stream) {
  for (const void* ptr : {q, k, v, (const void*)g, (const void*)o})
    if (!ptr || !aligned16(ptr)) return GBLA_ERR_INVALID_ARG;
  for (const void* ptr : {(const void*)den, (const void*)state})
    if (ptr && !aligned16(ptr)) return GBLA_ERR_INVALID_ARG;
  Ctx c;
  gbla_status r = begin(shape, GBLA_OP_CORE_FORWARD, ws, ws_bytes, stream, c);
  if (r != GBLA_OK) return r;
  const Plan& p = c.p;
  float* st = at<float>(ws, c.l.state);
  bf16* sbf = at<bf16>(ws, c.l.state_bf);
  float* center = p.f32 ? nullptr : at<float>(ws, c.l.center);
  r = run_reduce(c, k, v, p.HD, g, GATE_VALUES, st, sbf, at<float>(ws, c.l.state_m), state, center, ws);
  if (r != GBLA_OK) return r;
  ReadoutArgs ra{};
  ra.q = q; ra.ldq = p.HD;
  ra.state = st; ra.state_bf = sbf; ra.center = center;
  ra.out = o; ra.ldo = p.HD; ra.den = den;
  ra.H = p.H; ra.dh = p.dh; ra.seq = c.seq; ra.tiles = c.tiles; ra.err = c.kerr;
  const char* nm = "readout[f32]";
  GBLA_CHECK(p.f32 ? launch_readout_f32(ra, false, p.n_tiles, c.st)
                   : launch_readout_core_bf16(ra, p.n_tiles, c.chunks, p.n_chunks, c.st, &nm),
             nm);
  return GBLA_OK;
}

gbla_status bla_core_backward(const gbla_shape* shape, const void* q, const void* k, const void* v, const float* g,
                              const void* d_o, void* dq, void* dk, void* dv, float* dg, void* ws, size_t ws_bytes,
                              void* stream) {
  for (const void* ptr : {q, k, v, (const void*)g, d_o, (const void*)dq, (const void*)dk, (const void*)dv, (const void*)dg})
    if (!ptr || !aligned16(ptr)) return GBLA_ERR_INVALID_ARG;
  Ctx c;
  gbla_status r = begin(shape, GBLA_OP_CORE_BACKWARD, ws, ws_bytes, stream, c);
  if (r != GBLA_OK) return r;
  const Plan& p = c.p;
  float* st = at<float>(ws, c.l.state);
  bf16* sbf = at<bf16>(ws, c.l.state_bf);
  float* center = p.f32 ? nullptr : at<float>(ws, c.l.center);
  r = run_reduce(c, k, v, p.HD, g, GATE_VALUES, st, sbf, at<float>(ws, c.l.state_m), nullptr, center, ws);
  if (r != GBLA_OK) return r;
  BwdQArgs a{};
  a.q = q; a.ldq = p.HD; a.dy = d_o; a.lddy = p.HD;
  a.state = st; a.state_bf = sbf; a.center = center;
  a.dq = dq; a.lddq = p.HD;
  a.partial = at<float>(ws, c.l.partial); a.counters = at<int>(ws, c.l.cnt_b);
  a.dstate = at<float>(ws, c.l.dstate); a.dstate_bf = at<bf16>(ws, c.l.dstate_bf);
  a.H = p.H; a.dh = p.dh; a.seq = c.seq; a.chunks = c.chunks; a.tiles = c.tiles; a.err = c.kerr; a.err_out = c.err;
  a.partial_slots = partial_slots(p);
  const char* nmq = "bwd_q[f32]";
  GBLA_CHECK(p.f32 ? launch_bwd_q_f32(a, false, p.n_chunks, c.st) : launch_bwd_q_core_bf16(a, p.HD, p.n_tiles, c, &nmq),
             nmq);
  BwdKVArgs kv{};
  kv.k = k; kv.ldk = p.HD; kv.v = v; kv.ldv = p.HD;
  kv.g = g; kv.ldg = p.H; kv.gate_kind = GATE_VALUES;
  kv.dstate = a.dstate; kv.dstate_bf = a.dstate_bf; kv.center = center;
  kv.dk = dk; kv.lddk = p.HD; kv.dv = dv; kv.lddv = p.HD;
  kv.ds = dg; kv.ldds = p.H; kv.gate_grad = GG_DG;
  kv.H = p.H; kv.dh = p.dh; kv.seq = c.seq; kv.tiles = c.tiles; kv.err = c.kerr;
  const char* nm = "bwd_kv[f32]";
  GBLA_CHECK(p.f32 ? launch_bwd_kv_f32(kv, p.n_tiles, c.st) : launch_bwd_kv_core_bf16(kv, p.n_tiles, c, &nm), nm);
  return GBLA_OK;
}

gbla_status bla_decay_core_forward(const gbla_shape* shape, const void* q, const void* k, const void* v,
                                   const float* g, const float* lam, void* o, float* den, void* ws, size_t ws_bytes,
                                   void* stream) {
  for (const void* ptr : {q, k, v, (const void*)g, (const void*)lam, (const void*)o})
    if (!ptr || !aligned16(ptr)) return GBLA_ERR_INVALID_ARG;
  if (den && !aligned16(den)) return GBLA_ERR_INVALID_ARG;
  Plan p0;
  gbla_status r = make_plan(shape, p0);
  if (r != GBLA_OK) return r;
  if (p0.f32 || p0.dh != 64) return GBLA_ERR_UNSUPPORTED;
  Ctx c;
  if ((r = begin(shape, GBLA_OP_DECAY_FORWARD, ws, ws_bytes, stream, c)) != GBLA_OK) return r;
  const Plan& p = c.p;
  DecayArgs a{};
  a.q = q; a.k = k; a.v = v; a.ld = p.HD;
  a.g = g; a.lam = lam; a.ldg = p.H;
  a.o = o; a.den = den;
  a.LF = at<bf16>(ws, c.l.LF); a.LB = at<bf16>(ws, c.l.LB); a.Lam = at<float>(ws, c.l.lamc);
  a.HF = at<bf16>(ws, c.l.HF); a.HB = at<bf16>(ws, c.l.HB);
  a.H = p.H; a.dh = p.dh; a.seq = c.seq; a.err = c.kerr;
  a.tiles.tile = kDecayChunk;
  a.tiles.per_seq = p.mode == SEQ_VARLEN ? 0 : cdiv(p.L, kDecayChunk);
  a.tiles.prefix = p.mode == SEQ_VARLEN ? at<int32_t>(ws, c.l.pre_d) : nullptr;
  if (p.mode == SEQ_VARLEN) {
    const int ts[1] = {kDecayChunk};
    int32_t* pre[1] = {at<int32_t>(ws, c.l.pre_d)};
    GBLA_CHECK(launch_plan(c.seq, 1, ts, pre, c.err, c.st), "plan");
  }
  GBLA_CHECK(launch_decay_states(a, decay_chunks(p), c.st), "decay states[mma]");
  GBLA_CHECK(launch_decay_scan(a, p.n_seq, c.st), "decay scan");
  GBLA_CHECK(launch_decay_out(a, decay_chunks(p), c.st), "decay out[mma]");
  return GBLA_OK;
}

gbla_status sa_core_forward(const gbla_shape* shape, const void* q, const void* k, const void* v, void* o, void* ws,
                            size_t ws_bytes, void* stream) {
  for (const void* ptr : {q, k, v, (const void*)o})
    if (!ptr || !aligned16(ptr)) return GBLA_ERR_INVALID_ARG;
  Plan p0;
  gbla_status r = make_plan(shape, p0);
  if (r != GBLA_OK) return r;
  if (p0.f32 || p0.dh != 64) return GBLA_ERR_UNSUPPORTED;
  Ctx c;
  if ((r = begin(shape, GBLA_OP_SA_FORWARD, ws, ws_bytes, stream, c)) != GBLA_OK) return r;
  const Plan& p = c.p;
  SaArgs a{};
  a.q = q; a.k = k; a.v = v; a.o = o; a.ld = p.HD;
  a.H = p.H; a.dh = p.dh; a.seq = c.seq; a.err = c.kerr; a.err_out = c.err;
  a.tiles.tile = kSaBlock;
  a.tiles.per_seq = p.mode == SEQ_VARLEN ? 0 : cdiv(p.L, kSaBlock);
  a.tiles.prefix = p.mode == SEQ_VARLEN ? at<int32_t>(ws, c.l.pre_d) : nullptr;
  if (p.mode == SEQ_VARLEN) {
    const int ts[1] = {kSaBlock};
    int32_t* pre[1] = {at<int32_t>(ws, c.l.pre_d)};
    GBLA_CHECK(launch_plan(c.seq, 1, ts, pre, c.err, c.st), "plan");
  }
  GBLA_CHECK(launch_sa_fwd_tc(a, sa_blocks(p), c.st), "sa[tc]");
  return GBLA_OK;
}

gbla_status gbla_check_device_status(const void* ws, void* stream) {
  if (!ws) return GBLA_ERR_WORKSPACE;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int err = 0;
  cudaError_t e = cudaMemcpyAsync(&err, ws, sizeof(int), cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return cuda_fail(e, "check_device_status");
  if (err & 1) return GBLA_ERR_DEVICE_CHECK;
  if (err & kErrTimeout) return GBLA_ERR_DEVICE_TIMEOUT;
  return err ? GBLA_ERR_DEVICE_CHECK : GBLA_OK;
}

gbla_status gbla_diag_bounded_wait(void* ws, size_t ws_bytes, unsigned polls, void* stream) {
  if (!ws || (reinterpret_cast<uintptr_t>(ws) % kAlign) != 0 || ws_bytes < 16) return GBLA_ERR_WORKSPACE;
  if (polls < 1 || polls > (1u << 20)) return GBLA_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemsetAsync(ws, 0, sizeof(int), st);
  if (e == cudaSuccess) e = launch_diag_wait(static_cast<int*>(ws), polls, st);
  if (e != cudaSuccess) return cuda_fail(e, "diag_bounded_wait");
  return GBLA_OK;
}

const char* gbla_status_string(int status) {
  switch (status) {
    case GBLA_OK: return "GBLA_OK";
    case GBLA_ERR_INVALID_ARG: return "GBLA_ERR_INVALID_ARG: null or misaligned pointer, or bad dimension";
    case GBLA_ERR_UNSUPPORTED: return "GBLA_ERR_UNSUPPORTED: no kernel for this shape (d_h, d alignment or size)";
    case GBLA_ERR_WORKSPACE: return "GBLA_ERR_WORKSPACE: workspace NULL, not 256-byte aligned, or too small";
    case GBLA_ERR_CUDA: return "GBLA_ERR_CUDA: a CUDA call failed (see gbla_last_error)";
    case GBLA_ERR_DEVICE_CHECK: return "GBLA_ERR_DEVICE_CHECK: bad cu_seqlens / seq_lens detected on the device";
    case GBLA_ERR_DEVICE_TIMEOUT:
      return "GBLA_ERR_DEVICE_TIMEOUT: a kernel's bounded wait for its copies or MMAs gave up; results are invalid";
    default: return "unknown gbla_status";
  }
}

const char* gbla_last_error(void) { return g_last_error.c_str(); }

void gbla_profiling_enable(int on) { g_prof.on = on != 0; }

gbla_status gbla_set_kernel_policy(int policy) {
  if (policy != GBLA_POLICY_AUTO && policy != GBLA_POLICY_TC && policy != GBLA_POLICY_MMA) return GBLA_ERR_INVALID_ARG;
  g_policy = policy;
  return GBLA_OK;
}

int gbla_profiling_read(const char** names, float* ms, int cap) {
  const int n = (int)g_prof.rec.size();
  if (n > 0) cudaEventSynchronize(g_prof.rec.back().t1);
  for (int i = 0; i < n; ++i) {
    ProfRecord& r = g_prof.rec[i];
    if (i < cap) {
      float t = -1.f;
      if (cudaEventElapsedTime(&t, r.t0, r.t1) != cudaSuccess) t = -1.f;
      if (names) names[i] = r.name;
      if (ms) ms[i] = t;
    }
    g_prof.pool.push_back(r.t0);
    g_prof.pool.push_back(r.t1);
  }
  g_prof.rec.clear();
  return n;
}

int gbla_version(void) { return 100; }

}  // extern "C"
