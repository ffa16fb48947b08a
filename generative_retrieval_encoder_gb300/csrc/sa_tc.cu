// Bidirectional softmax attention, the SA blocks of the hybrid [SA, LA, LA]
// encoder ("Gated Bidirectional Linear Attention for Generative Retrieval",
// Core method 1, Eq. 1, and the hybrid-encoder paragraph), on the
// 5th-generation tensor cores, bf16 I/O, d_h = 64:
//   o_i = sum_j exp(q_i . k_j / sqrt(d_h)) v_j / sum_j exp(q_i . k_j / sqrt(d_h))
// over every key j of query i's sequence (no mask: both directions).
//
// One CTA per (256-query block of a sequence, head): two 128-query tiles a
// and b that share every key and value tile of the sequence.  Per key tile
// j (128 keys):
//   S_t = Q_t K_j^T                  tcgen05 -> TMEM (128 columns per tile t)
//   softmax (one thread per query row, a reference m of the exponentials and
//   the sum l in the log2 domain): P_t = 2^(S_t log2(e)/sqrt(d_h) - m) in bf16
//   into shared memory; m moves (and the accumulator is rescaled by
//   2^(m_old - m_new)) only when the row's maximum passes m by more than 8
//   [O_t | l_t] += P_t [V_j | 1]     tcgen05 -> TMEM (80 columns per tile t)
// and o = O / l at the end: the sum l accumulates on the tensor cores from
// the same bf16 weights as the numerator (a constant block with a column of
// ones is B's second atom).  Roles: a producer warp (TMA: the two Q tiles,
// then K_j and V_j through a 3-stage ring), an S warp (S_a(j+1), S_b(j+1) as
// soon as the softmax holds S(j) in registers: the tensor cores compute the
// next scores while the softmax of the current ones runs), a PV warp (PV_a(j),
// PV_b(j) once P is written; two issuing threads issue the short MMAs twice
// as fast as one), and two groups of four softmax warps (tile a, tile b).
// Keys past the end of the sequence are
// masked; queries past it are computed but not stored, and rows of a padded
// slot past the sequence receive zeros.
//
// Every mbarrier wait is bounded; after one gives up, the kernel finishes its
// loops without waiting, sets the timeout bit of the error word, waits
// (bounded) for its copies and MMAs, frees its TMEM and returns.
#include "pdl.cuh"
#include "kernels.h"
#include "tcgen05.cuh"

namespace gbla {
namespace {

constexpr int D = 64;                 // d_h
constexpr int BQ = 128;               // queries per tile (MMA M); two tiles a CTA
constexpr int BK = 128;               // keys per tile (MMA N of S, K of PV)
constexpr int TILE = 128 * 128;       // [128 rows][64 bf16], one 128-byte swizzle block, 16 KB
constexpr int KST = 3;                // K / V ring stages
constexpr int O_Q = 0;                          // Q_a | Q_b
constexpr int O_KV = O_Q + 2 * TILE;            // KST x (K | V)
constexpr int O_P = O_KV + KST * 2 * TILE;      // P_a | P_b, each two 64-key atoms
constexpr int O_ONE = O_P + 2 * 2 * TILE;      // [128 key rows][64]: 1 in column 0, the sum column of PV
constexpr int O_BAR = O_ONE + TILE;
// qfull, kvfull[KST], kvempty[KST], sfull[2], sfree[2], pfull[2], oready[2]
constexpr int NBAR = 1 + 2 * KST + 8;
constexpr int O_SLOT = O_BAR + 8 * NBAR;
constexpr int O_FAIL = O_SLOT + 4;
constexpr int SMEM = O_FAIL + 4 + 1024;         // + alignment slack
constexpr int ON = D + 16;                      // PV's N: the 64 value columns and the sum column (+ pad)
constexpr int TMEM_COLS = 512;                  // S_a | S_b | O_a | O_b (128 + 128 + 80 + 80)
constexpr int NSW = 8;                          // softmax warps (4 a tile)
constexpr int NTH = (NSW + 3) * 32;             // + producer, S issuer, PV issuer
static_assert(SMEM <= 227 * 1024, "shared memory");

__device__ __forceinline__ uint32_t swz_off(int row, int chunk) {
  return (uint32_t)(row * 128 + ((chunk ^ (row & 7)) << 4));
}
// max(a, b, c): the three-input form of max.f32
__device__ __forceinline__ float max3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// The unit of a CTA: 256 queries of sequence b, head blockIdx.y.
struct SaUnit {
  int b, len, rows;   // sequence, its valid rows, rows of its slot
  int q0;             // first query of the block inside the sequence
  size_t base;        // first row of the sequence
};

__global__ void __launch_bounds__(NTH, 1)
    k_sa_fwd_tc(const SaArgs a, const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                const __grid_constant__ CUtensorMap tmV) {
  if (threadIdx.x == 0) {  // the descriptors load while the previous kernel finishes
    tma_prefetch_map(&tmQ);
    tma_prefetch_map(&tmK);
    tma_prefetch_map(&tmV);
  }
  pdl_enter();
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_align1024(smem_raw);
  const uint32_t sbase = smem_u32(smem);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (a.err && *a.err) return;
  const int h = blockIdx.y;
  SaUnit u;
  {
    int row0, nvalid, tin;
    if (!map_tile(a.seq, a.tiles, blockIdx.x, u.b, row0, nvalid, tin)) return;
    u.len = nvalid;
    u.rows = slot_rows(a.seq, nvalid);
    u.q0 = tin * 2 * BQ;
    u.base = (size_t)row0;
  }
  bf16* out = (bf16*)a.o;
  if (u.q0 >= u.len) {  // slot rows past the sequence only: zeros
    const int nr = min(2 * BQ, u.rows - u.q0);
    for (int idx = tid; idx < nr * (D / 8); idx += NTH) {
      const int r = idx / (D / 8), c = idx % (D / 8);
      *reinterpret_cast<uint4*>(out + (u.base + u.q0 + r) * a.ld + (size_t)h * D + 8 * c) = make_uint4(0u, 0u, 0u, 0u);
    }
    return;
  }
  const int nk = (u.len + BK - 1) / BK;  // key tiles of the sequence

  const uint32_t bar0 = sbase + O_BAR;
  const uint32_t QFULL = bar0;
  auto KVFULL = [&](int s) { return bar0 + 8 * (1 + s); };
  auto KVEMPTY = [&](int s) { return bar0 + 8 * (1 + KST + s); };
  auto SFULL = [&](int t) { return bar0 + 8 * (1 + 2 * KST + t); };
  auto SFREE = [&](int t) { return bar0 + 8 * (3 + 2 * KST + t); };
  auto PFULL = [&](int t) { return bar0 + 8 * (5 + 2 * KST + t); };
  auto OREADY = [&](int t) { return bar0 + 8 * (7 + 2 * KST + t); };
  uint32_t* slot = reinterpret_cast<uint32_t*>(smem + O_SLOT);
  volatile int* fail = reinterpret_cast<volatile int*>(smem + O_FAIL);
  if (tid == 0) {
    mbar_init(QFULL, 1);
    for (int s = 0; s < KST; ++s) {
      mbar_init(KVFULL(s), 1);
      mbar_init(KVEMPTY(s), 2);  // the commits after the stage's last S and last PV
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(SFULL(t), 1);
      mbar_init(SFREE(t), 4);    // the tile's four softmax warps
      mbar_init(PFULL(t), 4);
      mbar_init(OREADY(t), 1);
    }
    mbar_init_fence();
    *fail = 0;
  }
  if (warp == NSW + 1) tmem_alloc(smem_u32(slot), TMEM_COLS);
  // the ones block: bf16 1.0 in column 0 of each row (its swizzled chunk), 0 elsewhere
  for (int idx = tid; idx < 128 * 8; idx += NTH) {
    const int r = idx >> 3, c = idx & 7;
    *reinterpret_cast<uint4*>(smem + O_ONE + r * 128 + c * 16) =
        make_uint4(c == (r & 7) ? 0x3F80u : 0u, 0u, 0u, 0u);
  }
  fence_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *slot;
  auto tS = [&](int t) { return tmem + 128 * t; };
  auto tO = [&](int t) { return tmem + 256 + ON * t; };
  auto sQ = [&](int t) { return sbase + O_Q + t * TILE; };
  auto sK = [&](int s) { return sbase + O_KV + s * 2 * TILE; };
  auto sV = [&](int s) { return sbase + O_KV + s * 2 * TILE + TILE; };
  auto sP = [&](int t) { return sbase + O_P + t * 2 * TILE; };

  if (warp == NSW) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      mbar_expect_tx(QFULL, 2 * TILE);
      tma_load_2d(sQ(0), &tmQ, QFULL, h * D, (int)(u.base + u.q0));
      tma_load_2d(sQ(1), &tmQ, QFULL, h * D, (int)(u.base + u.q0 + BQ));
      int last[KST] = {0, 0, 0};
      for (int j = 0; j < nk; ++j) {
        const int s = j % KST;
        if (j >= KST && !mbar_wait(KVEMPTY(s), ((j / KST) - 1) & 1, fail)) break;
        mbar_expect_tx(KVFULL(s), 2 * TILE);
        tma_load_2d(sK(s), &tmK, KVFULL(s), h * D, (int)(u.base + (size_t)j * BK));
        tma_load_2d(sV(s), &tmV, KVFULL(s), h * D, (int)(u.base + (size_t)j * BK));
        last[s] = j + 1;
      }
      if (*fail) {  // let the copies still in flight land
        for (uint32_t it = 0; it < kPollLimit && !mbar_try_wait(QFULL, 0); ++it) {
        }
        for (int s = 0; s < KST; ++s)
          if (last[s] > 0)
            for (uint32_t it = 0; it < kPollLimit && !mbar_try_wait(KVFULL(s), (uint32_t)((last[s] - 1) / KST) & 1);
                 ++it) {
            }
      }
    }
  } else if (warp == NSW + 1) {
    // ------------------------------------------------------------ S issuer
    // S and PV have one issuing warp each: a thread issues an MMA about every
    // 50 cycles, so that one thread alone cannot keep up with MMAs this short
    // (64 and 52 cycles of tensor-core work).  The whole warp runs each loop,
    // so that its waits and descriptor arithmetic stay warp-uniform; one lane
    // issues the MMAs and commits.
    const uint32_t id_s = idesc_bf16(BQ, BK, false, false);
    // S_t = Q_t K_j^T: K = d_h.  A = Q_t K-major (+32 B per 16 features); B = K_j K-major (rows = keys).
    auto issue_s = [&](int t, int j) {
      const uint64_t da = sdesc(sQ(t), 16, 1024), db = sdesc(sK(j % KST), 16, 1024);
      if (lane == 0) {
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) tc_mma(tS(t), da + 2 * kk, db + 2 * kk, id_s, kk > 0);
        tc_commit(SFULL(t));
      }
      __syncwarp();
    };
    bool ok = mbar_wait(QFULL, 0, fail) && mbar_wait(KVFULL(0), 0, fail);
    for (int j = 0; j < nk && ok; ++j) {
      // S_t(j) once the softmax holds S_t(j - 1) in registers
      if (j > 0) ok = mbar_wait(KVFULL(j % KST), (j / KST) & 1, fail);
      for (int t = 0; t < 2 && ok; ++t) {
        if (j > 0) ok = mbar_wait(SFREE(t), (j - 1) & 1, fail);
        if (!ok) break;
        tc_fence_after();
        issue_s(t, j);
      }
      if (ok && lane == 0) tc_commit(KVEMPTY(j % KST));  // K_j read by both tiles' S
      __syncwarp();
    }
  } else if (warp == NSW + 2) {
    // ----------------------------------------------------------- PV issuer
    const uint32_t id_o = idesc_bf16(BQ, ON, false, true);
    // [O_t | l_t] += P_t [V_j | 1]: K = keys.  A = P_t K-major (two 64-key atoms); B N-major
    // (16 key rows = 2048 B), its second 64-column atom the ones block (LBO apart).
    auto issue_pv = [&](int t, int j) {
      const int s = j % KST;
      const uint64_t da = sdesc(sP(t), 16, 1024), db = sdesc(sV(s), sbase + O_ONE - sV(s), 1024);
      const uint32_t acc0 = j > 0 ? 1u : 0u;
      if (lane == 0) {
#pragma unroll
        for (int kk = 0; kk < BK / 16; ++kk)
          tc_mma(tO(t), da + (kk >> 2) * (TILE >> 4) + 2 * (kk & 3), db + 128 * kk, id_o, kk > 0 ? 1u : acc0);
        tc_commit(OREADY(t));
      }
      __syncwarp();
    };
    bool ok = true;
    for (int j = 0; j < nk && ok; ++j) {
      ok = mbar_wait(KVFULL(j % KST), (j / KST) & 1, fail);  // V_j in shared memory
      for (int t = 0; t < 2 && ok; ++t) {
        ok = mbar_wait(PFULL(t), j & 1, fail);
        if (!ok) break;
        tc_fence_after();
        issue_pv(t, j);
      }
      if (ok && lane == 0) tc_commit(KVEMPTY(j % KST));  // V_j read by both tiles' PV
      __syncwarp();
    }
    // every MMA this warp issued has finished once the last OREADY completes
    for (int t = 0; t < 2; ++t)
      for (uint32_t it = 0; it < kPollLimit && !mbar_try_wait(OREADY(t), (uint32_t)(nk - 1) & 1) && !*fail; ++it) {
      }
  } else {
    // --------------------------------------------------------- softmax
    const int t = warp >> 2, wq = warp & 3;  // query tile, TMEM lane quarter
    const int i = wq * 32 + lane;            // row of the tile = TMEM lane
    const uint32_t lrow = (uint32_t)(wq * 32) << 16;
    const float sl2 = 1.4426950408889634f / 8.f;  // log2(e) / sqrt(d_h)
    // m: the reference of the exponentials (log2 domain), moved only when the
    // row's maximum exceeds it by more than 8, so that most key tiles need no
    // rescale of O; the weights then stay below 2^8, well inside bf16 and fp32.
    float m = -INFINITY;
    uint8_t* pt = smem + O_P + t * 2 * TILE;
    for (int j = 0; j < nk; ++j) {
      const int kv = u.len - j * BK;  // valid keys of this tile (>= 1; >= BK but for the last)
      const bool full = kv >= BK;
      mbar_wait(SFULL(t), j & 1, fail);
      tc_fence_after();
      // the row's 128 scores into registers, one wait; S_t is then free for the next tile
      uint32_t sv[BK / 32][32];
#pragma unroll
      for (int c4 = 0; c4 < BK / 32; ++c4) tmem_ld32_async(tS(t) + lrow + 32 * c4, sv[c4]);
      asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
      for (int c4 = 0; c4 < BK / 32; ++c4) tmem_tie32(sv[c4]);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(SFREE(t));
      // the row's maximum over the valid keys
      float mx = -INFINITY;
#pragma unroll
      for (int c4 = 0; c4 < BK / 32; ++c4) {
        if (full) {
#pragma unroll
          for (int c = 0; c < 32; c += 2) mx = max3(mx, __uint_as_float(sv[c4][c]), __uint_as_float(sv[c4][c + 1]));
        } else {
#pragma unroll
          for (int c = 0; c < 32; ++c)
            if (32 * c4 + c < kv) mx = fmaxf(mx, __uint_as_float(sv[c4][c]));
        }
      }
      const float mt = mx * sl2;
      const bool move = mt > m + 8.f;  // always on the first tile (m = -inf)
      const float mnew = move ? mt : m;
      const float alpha = ex2(m - mnew);  // 0 on the first tile, 1 when m stays
      m = mnew;
      // P = 2^(s log2(e)/sqrt(d_h) - m) in bf16, into registers before the wait below
      uint32_t pw[BK / 2];
#pragma unroll
      for (int c4 = 0; c4 < BK / 32; ++c4) {
#pragma unroll
        for (int c = 0; c < 32; c += 2) {
          const int key = 32 * c4 + c;
          const float2 xa = __ffma2_rn(make_float2(__uint_as_float(sv[c4][c]), __uint_as_float(sv[c4][c + 1])),
                                       make_float2(sl2, sl2), make_float2(-m, -m));
          float p0 = ex2(xa.x);
          float p1 = ex2(xa.y);
          if (!full) {
            p0 = key < kv ? p0 : 0.f;
            p1 = key + 1 < kv ? p1 : 0.f;
          }
          pw[key / 2] = pack_bf16(p0, p1);
        }
      }
      // the accumulator and P_t are free once PV_t of the previous tile is done
      if (j > 0) {
        mbar_wait(OREADY(t), (j - 1) & 1, fail);
        tc_fence_after();
        if (__any_sync(0xffffffffu, move)) {  // rescale [O_t | l_t] by 2^(m_old - m_new)
#pragma unroll
          for (int c2 = 0; c2 < D / 32; ++c2) {
            uint32_t ov[32];
            tmem_ld32(tO(t) + lrow + 32 * c2, ov);
#pragma unroll
            for (int c = 0; c < 32; ++c) ov[c] = __float_as_uint(__uint_as_float(ov[c]) * alpha);
            tmem_st32(tO(t) + lrow + 32 * c2, ov);
          }
          uint32_t lv[8];
          tmem_ld8(tO(t) + lrow + D, lv);
          lv[0] = __float_as_uint(__uint_as_float(lv[0]) * alpha);
          tmem_st8(tO(t) + lrow + D, lv);
          tmem_st_wait();
        }
      }
#pragma unroll
      for (int chunk = 0; chunk < BK / 8; ++chunk)
        *reinterpret_cast<uint4*>(pt + (chunk >> 3) * TILE + swz_off(i, chunk & 7)) =
            make_uint4(pw[4 * chunk], pw[4 * chunk + 1], pw[4 * chunk + 2], pw[4 * chunk + 3]);
      fence_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(PFULL(t));
    }
    // o = O / l, staged over the tile's Q rows (every S_t has been computed), stored as whole lines
    mbar_wait(OREADY(t), (nk - 1) & 1, fail);
    tc_fence_after();
    uint32_t lv[8];
    tmem_ld8(tO(t) + lrow + D, lv);
    const float inv = 1.f / __uint_as_float(lv[0]);
    uint8_t* qt = smem + O_Q + t * TILE;
#pragma unroll
    for (int c2 = 0; c2 < D / 32; ++c2) {
      uint32_t ov[32];
      tmem_ld32(tO(t) + lrow + 32 * c2, ov);
#pragma unroll
      for (int c8 = 0; c8 < 4; ++c8) {
        const int c = 8 * c8;
        *reinterpret_cast<uint4*>(qt + swz_off(i, 4 * c2 + c8)) =
            make_uint4(pack_bf16(__uint_as_float(ov[c]) * inv, __uint_as_float(ov[c + 1]) * inv),
                       pack_bf16(__uint_as_float(ov[c + 2]) * inv, __uint_as_float(ov[c + 3]) * inv),
                       pack_bf16(__uint_as_float(ov[c + 4]) * inv, __uint_as_float(ov[c + 5]) * inv),
                       pack_bf16(__uint_as_float(ov[c + 6]) * inv, __uint_as_float(ov[c + 7]) * inv));
      }
    }
    __syncwarp();
    {
      const int ch = lane & 7;
#pragma unroll
      for (int it = 0; it < 8; ++it) {
        const int rr = wq * 32 + 4 * it + (lane >> 3);  // row of the tile
        const int q = u.q0 + t * BQ + rr;              // query inside the sequence
        if (q < u.rows) {
          const uint4 v = q < u.len ? *reinterpret_cast<const uint4*>(qt + swz_off(rr, ch)) : make_uint4(0u, 0u, 0u, 0u);
          *reinterpret_cast<uint4*>(out + (u.base + q) * a.ld + (size_t)h * D + 8 * ch) = v;
        }
      }
    }
  }
  __syncwarp();  // single-lane roles rejoin their warps: the CTA barrier below is warp-aligned
  __syncthreads();
  const bool bad = *fail != 0;
  tc_fence_before();
  __syncthreads();
  if (warp == NSW + 1) tmem_dealloc(tmem, TMEM_COLS);
  if (bad && tid == 0 && a.err_out) atomicOr(a.err_out, kErrTimeout);
}

}  // namespace

cudaError_t launch_sa_fwd_tc(const SaArgs& a, int n_blocks, cudaStream_t st) {
  auto al16 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; };
  if (a.dh != D || !al16(a.q) || !al16(a.k) || !al16(a.v) || !al16(a.o) || a.ld % 8 || a.seq.T <= 0 ||
      n_blocks <= 0 || a.tiles.tile != 2 * BQ)
    return cudaErrorNotSupported;
  CUtensorMap tmQ, tmK, tmV;
  const uint64_t cols = (uint64_t)a.H * D;
  if (!make_map(&tmQ, a.q, cols, (uint64_t)a.seq.T, (uint64_t)a.ld, 64, BQ, false) ||
      !make_map(&tmK, a.k, cols, (uint64_t)a.seq.T, (uint64_t)a.ld, 64, BK, false) ||
      !make_map(&tmV, a.v, cols, (uint64_t)a.seq.T, (uint64_t)a.ld, 64, BK, false))
    return cudaErrorNotSupported;
  cudaError_t e = cudaFuncSetAttribute(k_sa_fwd_tc, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM);
  if (e != cudaSuccess) return e;
  return launch_pdl(k_sa_fwd_tc, dim3(n_blocks, a.H), dim3(NTH), SMEM, st, a, tmQ, tmK, tmV);
}

}  // namespace gbla
