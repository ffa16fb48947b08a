// Blackwell tensor-core GEMM for the projection GEMMs of the GBLA layer:
//   C[M, N] = sum_k A(m, k) B(n, k), bf16 operands, fp32 accumulation in TMEM.
//
// Persistent and warp-specialised: one CTA per SM walks a static list of
// 128 x 256 output tiles (x K splits).
//   warp 0 (one lane)  TMA producer: cp.async.bulk.tensor loads (128-byte
//                      swizzle) into a shared-memory ring (full/empty
//                      mbarriers) of 4 stages, or 6 on a CTA pair, whose CTAs
//                      each hold half of B;
//   warp 1 (one lane)  MMA issuer: tcgen05.mma M = 128 (one CTA) or 256 (a
//                      CTA pair, cta_group::2), N <= 256, K = 16, into one of
//                      two TMEM accumulators (2 x 256 columns),
//                      tcgen05.commit frees ring stages and hands a finished
//                      accumulator to the epilogue;
//   warps 2-9          epilogue: tcgen05.ld of their 32-lane quarter and
//                      column half, release the accumulator, convert and
//                      store (bf16 / fp32 / split partial / projection + gate).
//                      bf16 columns go 64 at a time through a per-warp staging
//                      block, so that each warp store writes four whole
//                      128-byte row segments instead of 32 scattered 16-byte
//                      pieces.
// So the epilogue of tile i overlaps the MMAs of tile i + 1.  Operands may be
// K-major ([rows][K]) or M/N-major ([K][rows], the weight-gradient GEMM
// x~^T dP and the forward GEMM's packed weights).  With two or more m-tiles
// the CTAs run as pairs (clusters of two).
//
// Every mbarrier wait gives up after a bounded number of polls; the kernel then
// sets bit 2 of the workspace error word, waits (bounded) for the copies and
// MMAs it issued, frees its TMEM and returns.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <atomic>

#include "pdl.cuh"
#include "kernels.h"
#include "mbarrier.cuh"
#include "tcgen05.cuh"

namespace gbla {
namespace {

constexpr int PBM = 128, PBN = 256, PBK = 64;
constexpr int A_TILE = PBM * PBK * 2;  // 16 KB
constexpr int B_TILE = PBN * PBK * 2;  // 32 KB
constexpr int EPW = 8;                    // epilogue warps: two per TMEM lane quarter, one column half each
constexpr int STG = 4096;                 // per epilogue warp: [32 rows][64 bf16], 16-byte chunks XOR-swizzled
constexpr int STG_ALL = EPW * STG;
constexpr int SMEM_P = 4 * (A_TILE + B_TILE) + STG_ALL + 1024 + 256;
constexpr int NTHREADS = 64 + 32 * EPW;
// Work units: (k split z, m-tile group, n-tile), a group being `cl` adjacent
// m-tiles that the CTAs of one cluster take (rank r the m-tile cl g + r).
struct TileSched {
  int tiles_m, tiles_n, splits, cl, groups_m, total;  // total = units
  __device__ void decode(int t, int rank, int& z, int& mt, int& nt) const {
    z = t / (groups_m * tiles_n);
    const int r = t - z * groups_m * tiles_n;
    const int g = r / tiles_n;
    nt = r - g * tiles_n;
    mt = g * cl + rank;
  }
};

// phi(x) = elu(x) + 1 = max(x, 0) + exp(min(x, 0)), the exponential as
// 2^(x log2 e) on the hardware ex2 approximation (relative error ~2^-22,
// far below the bf16 rounding of the stored value).
__device__ __forceinline__ float phi_elu1(float x) {
  float e;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(e) : "f"(fminf(x, 0.f) * 1.4426950408889634f));
  return fmaxf(x, 0.f) + e;
}

// One 32-column chunk of a finished accumulator row to global memory.
__device__ __forceinline__ void store_chunk(const GemmArgs& a, int m, int n, int z, const uint32_t (&r)[32]) {
  const int Hg = a.N - a.n_main;
  if (a.epi == EPI_PROJ_PRE && n < a.n_main) {
    // [q | k | v | r] column blocks of width H*dh, H*dh a multiple of 32: a
    // 32-column chunk lies in one block.  q, k -> phi(.), v and r unchanged.
    const int blk = n / a.hd;  // the same for every lane of the warp
    bf16* C = (bf16*)a.C + (size_t)m * a.ldc + n;
    if (blk < 2) {  // phi = elu + 1
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        float f[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          f[j] = phi_elu1(__uint_as_float(r[8 * q + j]));
        }
        uint4 u;
        u.x = pack_bf16(f[0], f[1]); u.y = pack_bf16(f[2], f[3]);
        u.z = pack_bf16(f[4], f[5]); u.w = pack_bf16(f[6], f[7]);
        reinterpret_cast<uint4*>(C)[q] = u;
      }
    } else {
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        uint4 u;
        u.x = pack_bf16(__uint_as_float(r[8 * q + 0]), __uint_as_float(r[8 * q + 1]));
        u.y = pack_bf16(__uint_as_float(r[8 * q + 2]), __uint_as_float(r[8 * q + 3]));
        u.z = pack_bf16(__uint_as_float(r[8 * q + 4]), __uint_as_float(r[8 * q + 5]));
        u.w = pack_bf16(__uint_as_float(r[8 * q + 6]), __uint_as_float(r[8 * q + 7]));
        reinterpret_cast<uint4*>(C)[q] = u;
      }
    }
    return;
  }
  if (a.epi == EPI_BF16 || (a.epi == EPI_PROJ && n < a.n_main)) {
    bf16* C = (bf16*)a.C + (size_t)m * a.ldc + n;
    const int lim = a.epi == EPI_PROJ ? a.n_main : a.N;
    if (n + 32 <= lim) {
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        uint4 u;
        u.x = pack_bf16(__uint_as_float(r[8 * q + 0]), __uint_as_float(r[8 * q + 1]));
        u.y = pack_bf16(__uint_as_float(r[8 * q + 2]), __uint_as_float(r[8 * q + 3]));
        u.z = pack_bf16(__uint_as_float(r[8 * q + 4]), __uint_as_float(r[8 * q + 5]));
        u.w = pack_bf16(__uint_as_float(r[8 * q + 6]), __uint_as_float(r[8 * q + 7]));
        reinterpret_cast<uint4*>(C)[q] = u;
      }
    } else {
#pragma unroll
      for (int j = 0; j < 32; ++j)
        if (n + j < lim) C[j] = __float2bfloat16_rn(__uint_as_float(r[j]));
    }
  } else if (a.epi == EPI_PROJ || a.epi == EPI_PROJ_PRE) {  // the gate columns
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      const int hh = n + j - a.n_main;
      if (hh >= 0 && hh < Hg) {
        float s = __uint_as_float(r[j]);
        if (a.bias_g) s += __bfloat162float(((const bf16*)a.bias_g)[hh]);
        a.gate[(size_t)m * a.ldgate + hh] = a.gate_mode == 0 ? 1.f / (1.f + __expf(-s)) : s;
      }
    }
  } else {
    float* C = (float*)a.C + (a.epi == EPI_SPLITK ? (size_t)z * a.M * a.ldc : 0) + (size_t)m * a.ldc + n;
    if (n + 32 <= a.N) {
#pragma unroll
      for (int q = 0; q < 8; ++q)
        reinterpret_cast<float4*>(C)[q] = make_float4(__uint_as_float(r[4 * q]), __uint_as_float(r[4 * q + 1]),
                                                      __uint_as_float(r[4 * q + 2]), __uint_as_float(r[4 * q + 3]));
    } else {
#pragma unroll
      for (int j = 0; j < 32; ++j)
        if (n + j < a.N) C[j] = __uint_as_float(r[j]);
    }
  }
}

// Ring geometry per variant.  CL = 1: one CTA, 4 stages of A (16 KB) + B
// (32 KB).  CL = 2: a CTA pair runs M = 256 MMAs (cta_group::2); each CTA
// holds its 128 rows of A and half of B's columns, so a stage is 32 KB and 6
// of them fit.
template <int CL>
struct Ring {
  static constexpr int ST = CL == 2 ? 6 : 4;
  static constexpr int B_ST = CL == 2 ? B_TILE / 2 : B_TILE;  // B bytes per stage and CTA
  static constexpr int BYTES = ST * (A_TILE + B_ST);
};
static_assert(Ring<1>::BYTES == Ring<2>::BYTES, "one shared-memory layout for both variants");

// CL = 2: the even CTA of each pair (rank 0) issues the MMAs; both CTAs' copies
// complete on its full barriers (expect-tx armed by its producer for the
// pair's bytes); its commits arrive, multicast, on both CTAs' empty and
// accumulator-full barriers; both CTAs' epilogue warps release an accumulator
// by remote arrivals on its accumulator-empty barrier.
template <bool AMN, bool BMN, int CL>
__global__ void __launch_bounds__(NTHREADS, 1)
    k_gemm_tc(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
              const GemmArgs a, const TileSched ts, int wide_ok) {
  if (threadIdx.x == 0) {  // the descriptors load while the previous kernel finishes
    tma_prefetch_map(&tmA);
    tma_prefetch_map(&tmB);
  }
  pdl_enter();  // the previous kernel's outputs are visible from here on
  using RG = Ring<CL>;
  constexpr int ST = RG::ST;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_align1024(smem_raw);
  const uint32_t sA = smem_u32(smem), sB = sA + ST * A_TILE;
  const uint32_t stg = sA + RG::BYTES;  // epilogue staging of bf16 output boxes
  const uint32_t bars = stg + STG_ALL;
  const uint32_t full = bars, empty = bars + 8 * ST, accf = bars + 16 * ST, acce = accf + 16, drain = acce + 16;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + RG::BYTES + STG_ALL + 16 * ST + 40);
  __shared__ int s_fail;
  __shared__ int s_issued[ST];  // last ring use issued per stage (+1), for the drain

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int rank = CL == 2 ? (int)cluster_ctarank() : 0;
  const bool leader = rank == 0;  // issues the MMAs
  const int cid = blockIdx.x / CL, ncl = gridDim.x / CL;
  constexpr uint16_t kPair = 3;
  if (threadIdx.x == 0) {
    for (int s = 0; s < ST; ++s) {
      mbar_init(full + 8 * s, 1);
      mbar_init(empty + 8 * s, 1);
      s_issued[s] = 0;
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(accf + 8 * b, 1);
      mbar_init(acce + 8 * b, EPW * CL);  // one arrival per epilogue warp of the pair
    }
    mbar_init(drain, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    s_fail = 0;
  }
  if (warp == 1) {  // CL = 2: one warp of each CTA of the pair allocates, collectively
    if (CL == 2) {
      asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                   "r"(2 * PBN));
      asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;");
    } else {
      asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                   "r"(2 * PBN));
      asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
  }
  tc_fence_before();
  if (CL == 2) cluster_sync();  // the pair's barriers and TMEM exist before either CTA uses them
  else __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  volatile int* fail = &s_fail;
  // The barriers this CTA's copies complete on, and its accumulator releases go to.
  const uint32_t full_dst = CL == 2 ? mapa_shared(full, 0) : full;
  const uint32_t acce_dst = CL == 2 ? mapa_shared(acce, 0) : acce;

  if (warp == 0) {
    if (lane == 0) {  // ---------------------------------------------- producer
      uint32_t kt = 0;
      for (int t = cid; t < ts.total && !*fail; t += ncl) {
        int z, mt, nt;
        ts.decode(t, rank, z, mt, nt);
        const int m0 = mt * PBM, n0 = nt * PBN;
        const int ncols = min(PBN, a.N - n0);
        const int mma_n = (ncols + 15) / 16 * 16;
        // CL = 2: this CTA holds columns [n0 + rank nh, + nh) of the MMA's N
        const int nh = mma_n / CL, nb0 = n0 + rank * nh;
        const int nbox = BMN ? (CL == 2 ? (nh + 63) / 64 : PBN / 64) : 1;
        const uint32_t bbytes = BMN ? (uint32_t)nbox * (B_TILE / 4) : (uint32_t)RG::B_ST;
        const int kbeg = z * a.k_split, kend = min(a.K, kbeg + a.k_split);
        for (int k0 = kbeg; k0 < kend; k0 += PBK, ++kt) {
          const int s = kt % ST;
          const uint32_t use = kt / ST;
          if (use > 0 && !mbar_wait(empty + 8 * s, (use - 1) & 1, fail)) break;
          if (leader) mbar_expect_tx(full + 8 * s, (uint32_t)CL * (A_TILE + bbytes));
          s_issued[s] = (int)use + 1;
          const uint32_t da = sA + s * A_TILE, db = sB + s * RG::B_ST, fb = full_dst + 8 * s;
          if (CL == 2) {
            if (AMN) {
              tma_load_2d_pair(da, &tmA, fb, m0, k0);
              tma_load_2d_pair(da + A_TILE / 2, &tmA, fb, m0 + 64, k0);
            } else {
              tma_load_2d_pair(da, &tmA, fb, k0, m0);
            }
            if (BMN) {
              for (int j = 0; j < nbox; ++j) tma_load_2d_pair(db + j * (B_TILE / 4), &tmB, fb, nb0 + 64 * j, k0);
            } else {
              tma_load_2d_pair(db, &tmB, fb, k0, nb0);
            }
          } else {
            if (AMN) {
              tma_load_2d(da, &tmA, fb, m0, k0);
              tma_load_2d(da + A_TILE / 2, &tmA, fb, m0 + 64, k0);
            } else {
              tma_load_2d(da, &tmA, fb, k0, m0);
            }
            if (BMN) {
#pragma unroll
              for (int j = 0; j < PBN / 64; ++j) tma_load_2d(db + j * (B_TILE / 4), &tmB, fb, n0 + 64 * j, k0);
            } else {
              tma_load_2d(db, &tmB, fb, k0, n0);
            }
          }
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && leader) {  // ------------------------------------ MMA issuer
      uint32_t kt = 0;
      int i = 0;
      for (int t = cid; t < ts.total && !*fail; t += ncl, ++i) {
        int z, mt, nt;
        ts.decode(t, rank, z, mt, nt);
        const int n0 = nt * PBN;
        const int ncols = min(PBN, a.N - n0);
        const int mma_n = (ncols + 15) / 16 * 16;
        const uint32_t idesc = idesc_bf16(PBM * CL, mma_n, AMN, BMN);
        const int kbeg = z * a.k_split, kend = min(a.K, kbeg + a.k_split);
        const int b = i & 1;
        const uint32_t u = (uint32_t)i >> 1;
        if (u > 0 && !mbar_wait(acce + 8 * b, (u - 1) & 1, fail)) break;
        tc_fence_after();
        const uint32_t d = tmem + b * PBN;
        bool first = true;
        bool ok = true;
        for (int k0 = kbeg; k0 < kend; k0 += PBK, ++kt) {
          const int s = kt % ST;
          if (!mbar_wait(full + 8 * s, (kt / ST) & 1, fail)) { ok = false; break; }
          tc_fence_after();
          const uint32_t ta = sA + s * A_TILE, tb = sB + s * RG::B_ST;
#pragma unroll
          for (int kk = 0; kk < PBK / 16; ++kk) {
            // K-major: advance 32 B inside the 128-byte swizzled row.  M/N-major:
            // advance 16 k-rows (2 x 1024-byte swizzle atoms); 64-wide M/N
            // chunks of the tile are LBO = 8 KB apart.
            const uint64_t da = AMN ? sdesc(ta + kk * 2048, 8192, 1024) : sdesc(ta + kk * 32, 16, 1024);
            const uint64_t db = BMN ? sdesc(tb + kk * 2048, 8192, 1024) : sdesc(tb + kk * 32, 16, 1024);
            if (CL == 2) tc_mma_pair(d, da, db, idesc, first ? 0u : 1u);
            else tc_mma(d, da, db, idesc, first ? 0u : 1u);
            first = false;
          }
          if (CL == 2) tc_commit_pair_mc(empty + 8 * s, kPair);
          else tc_commit(empty + 8 * s);
        }
        if (!ok) break;
        if (CL == 2) tc_commit_pair_mc(accf + 8 * b, kPair);
        else tc_commit(accf + 8 * b);
      }
      if (CL == 2) tc_commit_pair(drain);  // completes once every MMA issued above has finished
      else tc_commit(drain);
      for (uint32_t k = 0; k < kPollLimit && !mbar_try_wait(drain, 0); ++k) {
      }
    }
  } else {  // ------------------------------------------------------- epilogue
    const int q = warp & 3;  // TMEM lane quarter this warp may access
    const int row = q * 32 + lane;
    const int ew = warp - 2, c_lo = (ew >> 2) * (PBN / 2), c_hi = c_lo + PBN / 2;  // this warp's columns
    int i = 0;
    auto release = [&](int b) {  // hand accumulator b back to the MMA issuer
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if (CL == 2) mbar_arrive_cluster(acce_dst + 8 * b);
        else mbar_arrive(acce + 8 * b);
      }
    };
    for (int t = cid; t < ts.total && !*fail; t += ncl, ++i) {
      int z, mt, nt;
      ts.decode(t, rank, z, mt, nt);
      const int m0 = mt * PBM, n0 = nt * PBN;
      const int ncols = min(PBN, a.N - n0);
      const int kbeg = z * a.k_split, kend = min(a.K, kbeg + a.k_split);
      const int b = i & 1;
      if (!mbar_wait(accf + 8 * b, ((uint32_t)i >> 1) & 1, fail)) break;
      tc_fence_after();
      const int m = m0 + row;
      if (kend > kbeg) {
        const uint32_t taddr = tmem + ((uint32_t)(q * 32) << 16) + b * PBN;
        const int cend = min(ncols, c_hi);
        if (c_lo >= cend) release(b);  // nothing in this warp's half
        for (int c = c_lo; c < cend;) {
          const int n = n0 + c;
          // 64 bf16 columns at once through the staging rows, unless they reach
          // past the bf16 columns (uniform per warp)
          const bool wide = wide_ok && c + 64 <= cend && ((a.epi == EPI_BF16 && n + 64 <= a.N) ||
                                               ((a.epi == EPI_PROJ || a.epi == EPI_PROJ_PRE) && n + 64 <= a.n_main));
          if (!wide) {
            uint32_t r[32];
            tmem_ld32(taddr + c, r);       // warp-collective: every lane runs it
            if (c + 32 >= cend) release(b);  // last chunk read
            if (m < a.M) store_chunk(a, m, n, z, r);
            c += 32;
            continue;
          }
          // phi on the q and k blocks: n is a multiple of 64 and so is 2 hd
          // (hd a multiple of 32), so the 64 columns lie on one side
          const bool phi = a.epi == EPI_PROJ_PRE && n < 2 * a.hd;
          uint32_t w[32];
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            uint32_t r[32];
            tmem_ld32(taddr + c + 32 * h, r);
            if (phi) {
#pragma unroll
              for (int j = 0; j < 16; ++j)
                w[16 * h + j] = pack_bf16(phi_elu1(__uint_as_float(r[2 * j])), phi_elu1(__uint_as_float(r[2 * j + 1])));
            } else {
#pragma unroll
              for (int j = 0; j < 16; ++j) w[16 * h + j] = pack_bf16(__uint_as_float(r[2 * j]), __uint_as_float(r[2 * j + 1]));
            }
          }
          if (c + 64 >= cend) release(b);
          // this lane's row into the staging rows (chunk j of row r at chunk j ^ (r & 7))
          const uint32_t sw = stg + (uint32_t)(ew * STG);
#pragma unroll
          for (int j = 0; j < 8; ++j)
            asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(sw + lane * 128 + ((j ^ (lane & 7)) << 4)),
                         "r"(w[4 * j]), "r"(w[4 * j + 1]), "r"(w[4 * j + 2]), "r"(w[4 * j + 3])
                         : "memory");
          __syncwarp();
          // eight lanes per row: each warp store writes four whole 128-byte row segments
          bf16* Cb = (bf16*)a.C;
          const int ch = lane & 7;
#pragma unroll
          for (int it = 0; it < 8; ++it) {
            const int rr = 4 * it + (lane >> 3), gm = m0 + 32 * q + rr;
            uint4 v;
            asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                         : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                         : "r"(sw + rr * 128 + ((ch ^ (rr & 7)) << 4)));
            if (gm < a.M) *reinterpret_cast<uint4*>(Cb + (size_t)gm * a.ldc + n + 8 * ch) = v;
          }
          __syncwarp();
          c += 64;
        }
      } else {
        release(b);
        if (m < a.M && a.epi == EPI_SPLITK)
          for (int j = c_lo; j < min(ncols, c_hi); ++j)
            ((float*)a.C)[(size_t)z * a.M * a.ldc + (size_t)m * a.ldc + n0 + j] = 0.f;
      }
    }
  }

  __syncwarp();  // single-lane roles rejoin their warps: the CTA barrier below is warp-aligned
  __syncthreads();
  if (*fail) {
    if (threadIdx.x == 0) {
      if (a.err) atomicOr(a.err, kErrTimeout);
      // wait (bounded) for the last copy issued into each ring stage (all of
      // the pair's copies complete on the leader's barriers)
      if (leader)
        for (int s = 0; s < ST; ++s) {
          const int u = s_issued[s];
          if (u > 0)
            for (uint32_t k = 0; k < kPollLimit && !mbar_try_wait(full + 8 * s, (uint32_t)(u - 1) & 1); ++k) {
            }
        }
    }
    __syncwarp();
    __syncthreads();
  }
  tc_fence_before();
  if (CL == 2) cluster_sync();  // no copy, MMA or arrival of the pair still targets this CTA
  else __syncthreads();
  if (warp == 1) {
    if (CL == 2) asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(2 * PBN));
    else asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(2 * PBN));
  }
}

}  // namespace

PFN_cuTensorMapEncodeTiled_v12000 encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

// 2-D bf16 tensor map over a row-major [outer][inner] array (row pitch ld
// elements), box {box_inner, box_outer}, 128-byte swizzle, zero fill out of bounds.
bool make_map(CUtensorMap* m, const void* ptr, uint64_t inner, uint64_t outer, uint64_t ld, uint32_t box_inner,
              uint32_t box_outer, bool wide_promotion) {
  auto enc = encoder();
  if (!enc) return false;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {ld * 2};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t es[2] = {1, 1};
  const CUtensorMapL2promotion promo =
      wide_promotion ? CU_TENSOR_MAP_L2_PROMOTION_L2_256B : CU_TENSOR_MAP_L2_PROMOTION_L2_128B;
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, promo, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
         CUDA_SUCCESS;
}

int sm_count() {
  // Per device, looked up once.  Without a usable device (a host that only
  // sizes workspaces) the GB300's 152 SMs stand in, so that the sizes a
  // host computes agree with those of the GPU it targets.
  constexpr int kMaxDev = 256;
  static std::atomic<int> n[kMaxDev] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) {
    (void)cudaGetLastError();
    return 152;
  }
  int v = n[dev].load(std::memory_order_relaxed);
  if (v <= 0) {
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0) {
      (void)cudaGetLastError();
      v = 152;
    }
    n[dev].store(v, std::memory_order_relaxed);
  }
  return v;
}

// cudaErrorNotSupported when the shape is outside what this kernel handles
// (the caller then uses the mma.sync GEMM).
cudaError_t launch_gemm_tc(const GemmArgs& a, cudaStream_t st) {
  if (a.io_f32 || a.M <= 0 || a.N <= 0 || a.K <= 0) return cudaErrorNotSupported;
  if (a.k_split % PBK != 0 && a.k_split < a.K) return cudaErrorNotSupported;
  const bool amn = !a.a_kmajor, bmn = !a.b_kmajor;
  if ((reinterpret_cast<uintptr_t>(a.A) | reinterpret_cast<uintptr_t>(a.B)) & 15) return cudaErrorNotSupported;
  if ((a.lda % 8) || (a.ldb % 8)) return cudaErrorNotSupported;
  if (a.epi == EPI_PROJ && a.n_main % 32) return cudaErrorNotSupported;
  if (a.epi == EPI_PROJ_PRE && (a.n_main != 4 * a.hd || a.hd % 32)) return cudaErrorNotSupported;
  TileSched ts;
  ts.tiles_m = (a.M + PBM - 1) / PBM;
  ts.tiles_n = (a.N + PBN - 1) / PBN;
  ts.splits = (a.K + a.k_split - 1) / a.k_split;
  ts.cl = a.pair && ts.tiles_m >= 2 ? 2 : 1;  // CTA pairs on adjacent m-tiles
  ts.groups_m = (ts.tiles_m + ts.cl - 1) / ts.cl;
  ts.total = ts.groups_m * ts.tiles_n * ts.splits;
  CUtensorMap ta, tb;
  // B boxes: N-major 64 x 64 (four per tile); K-major 64 x 256, or 64 x 128 (one half) in pairs
  const bool okA = amn ? make_map(&ta, a.A, (uint64_t)a.M, (uint64_t)a.K, (uint64_t)a.lda, 64, PBK)
                       : make_map(&ta, a.A, (uint64_t)a.K, (uint64_t)a.M, (uint64_t)a.lda, PBK, PBM);
  const bool okB = bmn ? make_map(&tb, a.B, (uint64_t)a.N, (uint64_t)a.K, (uint64_t)a.ldb, 64, PBK)
                       : make_map(&tb, a.B, (uint64_t)a.K, (uint64_t)a.N, (uint64_t)a.ldb, PBK, PBN / ts.cl);
  if (!okA || !okB) return cudaErrorNotSupported;
  // 16-byte row stores of the staged bf16 output (see the epilogue)
  const int wide_ok = (reinterpret_cast<uintptr_t>(a.C) & 15) == 0 && a.ldc % 8 == 0 ? 1 : 0;
  const int slots = sm_count() / ts.cl;  // clusters resident at once (one CTA per SM)
  const int grid = ts.cl * (ts.total < slots ? ts.total : slots);
  cudaError_t e;
#define GBLA_CASE(AMN, BMN)                                                                                  \
  if (amn == AMN && bmn == BMN) {                                                                            \
    if (ts.cl == 1) {                                                                                        \
      if ((e = cudaFuncSetAttribute(k_gemm_tc<AMN, BMN, 1>, cudaFuncAttributeMaxDynamicSharedMemorySize,     \
                                    SMEM_P)) != cudaSuccess)                                                 \
        return e;                                                                                            \
      return launch_pdl(k_gemm_tc<AMN, BMN, 1>, dim3(grid), dim3(NTHREADS), SMEM_P, st, ta, tb, a, ts, wide_ok); \
    }                                                                                                        \
    if ((e = cudaFuncSetAttribute(k_gemm_tc<AMN, BMN, 2>, cudaFuncAttributeMaxDynamicSharedMemorySize,       \
                                  SMEM_P)) != cudaSuccess)                                                   \
      return e;                                                                                              \
    cudaLaunchConfig_t cfg = {};                                                                             \
    cfg.gridDim = dim3(grid);                                                                                \
    cfg.blockDim = dim3(NTHREADS);                                                                           \
    cfg.dynamicSmemBytes = SMEM_P;                                                                           \
    cfg.stream = st;                                                                                         \
    cudaLaunchAttribute attr[2];                                                                             \
    attr[0].id = cudaLaunchAttributeClusterDimension;                                                        \
    attr[0].val.clusterDim.x = 2;                                                                            \
    attr[0].val.clusterDim.y = 1;                                                                            \
    attr[0].val.clusterDim.z = 1;                                                                            \
    attr[1] = pdl_attribute();                                                                               \
    cfg.attrs = attr;                                                                                        \
    cfg.numAttrs = 2;                                                                                        \
    return cudaLaunchKernelEx(&cfg, k_gemm_tc<AMN, BMN, 2>, ta, tb, a, ts, wide_ok);                        \
  }
  GBLA_CASE(false, false) GBLA_CASE(true, true) GBLA_CASE(false, true) GBLA_CASE(true, false)
#undef GBLA_CASE
  return cudaErrorNotSupported;
}

}  // namespace gbla
