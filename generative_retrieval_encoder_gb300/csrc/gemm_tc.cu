// Blackwell tensor-core GEMM for the projection GEMMs of the GBLA layer:
//   C[M, N] = sum_k A(m, k) B(n, k), bf16 operands, fp32 accumulation in TMEM.
// tcgen05.mma (cta_group::1, M = 128, N <= 128, K = 16) issued by one thread,
// operands staged by TMA (cp.async.bulk.tensor, 128-byte swizzle) through a
// 3-stage mbarrier pipeline, accumulator read back with tcgen05.ld for the
// epilogue (the same epilogue kinds as the mma.sync GEMM: bf16 / fp32 / split
// over K / projection + gate).  Operands may be K-major ([rows][K]) or
// M/N-major ([K][rows]); the latter is the weight-gradient GEMM x~^T dP.
//
// Every wait on an mbarrier gives up after a bounded number of polls; the
// kernel then sets bit 2 of the workspace error word, drains the copies it
// issued (again bounded), frees its TMEM and returns without storing.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "kernels.h"

namespace gbla {
namespace {

constexpr int TBM = 128, TBN = 128, TBK = 64, TSTAGES = 3;
constexpr int OP_BYTES = TBM * TBK * 2;  // one operand tile: 16 KB
constexpr int SMEM_TC = TSTAGES * 2 * OP_BYTES + 1024 + 256;
constexpr uint32_t kPollLimit = 1u << 24;
constexpr int kErrTimeout = 2;

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count));
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
// Bounded wait: false if the phase did not complete within kPollLimit polls.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity) {
  for (uint32_t i = 0; i < kPollLimit; ++i)
    if (mbar_try_wait(bar, parity)) return true;
  return false;
}
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, uint32_t bar, int x, int y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4}], [%2];"
      ::"r"(dst), "l"(map), "r"(bar), "r"(x), "r"(y)
      : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Shared-memory matrix descriptor: 128-byte swizzle, descriptor version 1.
__device__ __forceinline__ uint64_t sdesc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFF) >> 4);
  d |= (uint64_t)((lbo >> 4) & 0x3FFF) << 16;
  d |= (uint64_t)((sbo >> 4) & 0x3FFF) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)2 << 61;  // SWIZZLE_128B
  return d;
}
// Instruction descriptor, kind::f16: D fp32, A and B bf16, M x N tile.
__device__ __forceinline__ uint32_t idesc_bf16(int M, int N, bool a_mn, bool b_mn) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((a_mn ? 1u : 0u) << 15) | ((b_mn ? 1u : 0u) << 16) |
         ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}
__device__ __forceinline__ void tc_mma(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n"
      ::"r"(d_tmem), "l"(a), "l"(b), "r"(idesc), "r"(acc));
}
__device__ __forceinline__ void tc_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// A (AMN = false): tiles [TBM rows][TBK] loaded as one TMA box {TBK, TBM}.
// A (AMN = true) : tiles [TBK rows (k)][TBM] loaded as two boxes {64, TBK}
//                  (64 M-elements x 64 k-rows each, 8 KB apart).
// Same for B with TBN.
template <bool AMN, bool BMN>
__global__ void __launch_bounds__(128, 2)
    k_gemm_tc(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB, const GemmArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sA = smem_u32(smem), sB = sA + TSTAGES * OP_BYTES;
  const uint32_t bar0 = sB + TSTAGES * OP_BYTES;  // full[s] at bar0 + 8 s, empty[s] at +8 (TSTAGES + s), done after
  const uint32_t full = bar0, empty = bar0 + 8 * TSTAGES, done = bar0 + 16 * TSTAGES;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + 2 * TSTAGES * OP_BYTES + 16 * TSTAGES + 8);
  __shared__ int s_fail;
  __shared__ int s_issued;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n0 = blockIdx.x * TBN, m0 = blockIdx.y * TBM;
  const int kbeg = blockIdx.z * a.k_split;
  const int kend = min(a.K, kbeg + a.k_split);
  const int nk = (kend - kbeg + TBK - 1) / TBK;
  const int ncols = min(TBN, a.N - n0);
  const int mma_n = (ncols + 15) / 16 * 16;

  if (threadIdx.x == 0) {
    for (int s = 0; s < TSTAGES; ++s) {
      mbar_init(full + 8 * s, 1);
      mbar_init(empty + 8 * s, 1);
    }
    mbar_init(done, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    s_fail = 0;
    s_issued = 0;
  }
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                 "r"(TBN));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (threadIdx.x == 0) {  // TMA producer
    int kt = 0;
    for (; kt < nk; ++kt) {
      const int s = kt % TSTAGES;
      if (kt >= TSTAGES && !mbar_wait(empty + 8 * s, ((kt / TSTAGES) & 1) ^ 1)) {
        s_fail = 1;
        break;
      }
      const int k0 = kbeg + kt * TBK;
      mbar_expect_tx(full + 8 * s, 2 * OP_BYTES);
      const uint32_t da = sA + s * OP_BYTES, db = sB + s * OP_BYTES;
      if (AMN) {
        tma_load_2d(da, &tmA, full + 8 * s, m0, k0);
        tma_load_2d(da + OP_BYTES / 2, &tmA, full + 8 * s, m0 + 64, k0);
      } else {
        tma_load_2d(da, &tmA, full + 8 * s, k0, m0);
      }
      if (BMN) {
        tma_load_2d(db, &tmB, full + 8 * s, n0, k0);
        tma_load_2d(db + OP_BYTES / 2, &tmB, full + 8 * s, n0 + 64, k0);
      } else {
        tma_load_2d(db, &tmB, full + 8 * s, k0, n0);
      }
    }
    s_issued = kt;
  } else if (threadIdx.x == 32) {  // MMA issuer
    const uint32_t idesc = idesc_bf16(TBM, mma_n, AMN, BMN);
    for (int kt = 0; kt < nk; ++kt) {
      const int s = kt % TSTAGES;
      if (!mbar_wait(full + 8 * s, (kt / TSTAGES) & 1)) {
        s_fail = 1;
        break;
      }
      tc_fence_after();
      const uint32_t ta = sA + s * OP_BYTES, tb = sB + s * OP_BYTES;
#pragma unroll
      for (int kk = 0; kk < TBK / 16; ++kk) {
        // K-major: advance 32 B inside the 128-byte swizzled row.  M/N-major:
        // advance 16 k-rows (2 x 1024-byte swizzle atoms); the two 64-wide
        // halves of the tile are LBO = 8 KB apart.
        const uint64_t da = AMN ? sdesc(ta + kk * 2048, OP_BYTES / 2, 1024) : sdesc(ta + kk * 32, 16, 1024);
        const uint64_t db = BMN ? sdesc(tb + kk * 2048, OP_BYTES / 2, 1024) : sdesc(tb + kk * 32, 16, 1024);
        tc_mma(tmem, da, db, idesc, (kt | kk) != 0 ? 1u : 0u);
      }
      tc_commit(empty + 8 * s);  // the stage is free once these MMAs have read it
    }
    tc_commit(done);  // arrives when every MMA issued above has completed
  }
  __syncwarp();
  if (!mbar_wait(done, 0)) s_fail = 1;
  tc_fence_after();
  __syncthreads();
  if (s_fail) {  // uniform across the CTA
    if (threadIdx.x == 0) {
      if (a.err) atomicOr(a.err, kErrTimeout);
      // drain the copies this CTA issued so that none lands after it exits
      const int issued = s_issued;
      for (int kt = max(0, issued - TSTAGES); kt < issued; ++kt)
        mbar_wait(full + 8 * (kt % TSTAGES), (kt / TSTAGES) & 1);
    }
  } else if (nk > 0) {
    const int m = m0 + warp * 32 + lane;
    const uint32_t trow = tmem + ((uint32_t)(warp * 32) << 16);
    const int Hg = a.N - a.n_main;
    for (int c = 0; c < ncols; c += 16) {
      uint32_t r[16];
      tmem_ld16(trow + c, r);  // warp-collective: every lane runs it, rows past M included
      const int n = n0 + c;
      if (m < a.M) {
      if (a.epi == EPI_BF16 || (a.epi == EPI_PROJ && n < a.n_main)) {
        bf16* C = (bf16*)a.C + (size_t)m * a.ldc + n;
        const int lim = a.epi == EPI_PROJ ? a.n_main : a.N;
        if (n + 16 <= lim) {
          uint4 u0, u1;
          u0.x = pack_bf16(__uint_as_float(r[0]), __uint_as_float(r[1]));
          u0.y = pack_bf16(__uint_as_float(r[2]), __uint_as_float(r[3]));
          u0.z = pack_bf16(__uint_as_float(r[4]), __uint_as_float(r[5]));
          u0.w = pack_bf16(__uint_as_float(r[6]), __uint_as_float(r[7]));
          u1.x = pack_bf16(__uint_as_float(r[8]), __uint_as_float(r[9]));
          u1.y = pack_bf16(__uint_as_float(r[10]), __uint_as_float(r[11]));
          u1.z = pack_bf16(__uint_as_float(r[12]), __uint_as_float(r[13]));
          u1.w = pack_bf16(__uint_as_float(r[14]), __uint_as_float(r[15]));
          reinterpret_cast<uint4*>(C)[0] = u0;
          reinterpret_cast<uint4*>(C)[1] = u1;
        } else {
          for (int j = 0; j < 16 && n + j < lim; ++j) C[j] = __float2bfloat16_rn(__uint_as_float(r[j]));
        }
      } else if (a.epi == EPI_PROJ) {
        for (int j = 0; j < 16; ++j) {
          const int hh = n + j - a.n_main;
          if (hh < 0 || hh >= Hg) continue;
          float s = __uint_as_float(r[j]);
          if (a.bias_g) s += __bfloat162float(((const bf16*)a.bias_g)[hh]);
          a.gate[(size_t)m * a.ldgate + hh] = a.gate_mode == 0 ? 1.f / (1.f + __expf(-s)) : s;
        }
      } else {
        float* C = (float*)a.C + (a.epi == EPI_SPLITK ? (size_t)blockIdx.z * a.M * a.ldc : 0) + (size_t)m * a.ldc + n;
        if (n + 16 <= a.N) {
#pragma unroll
          for (int j = 0; j < 4; ++j)
            reinterpret_cast<float4*>(C)[j] = make_float4(__uint_as_float(r[4 * j]), __uint_as_float(r[4 * j + 1]),
                                                          __uint_as_float(r[4 * j + 2]), __uint_as_float(r[4 * j + 3]));
        } else {
          for (int j = 0; j < 16 && n + j < a.N; ++j) C[j] = __uint_as_float(r[j]);
        }
      }
      }  // m < M
    }
  } else {
    // empty K range (split past K): this split's partial is zero
    const int m = m0 + warp * 32 + lane;
    if (a.epi == EPI_SPLITK && m < a.M)
      for (int j = 0; j < ncols; ++j) ((float*)a.C)[(size_t)blockIdx.z * a.M * a.ldc + (size_t)m * a.ldc + n0 + j] = 0.f;
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(TBN));
}

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
              uint32_t box_outer) {
  auto enc = encoder();
  if (!enc) return false;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {ld * 2};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t es[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

// cudaErrorNotSupported when the shape is outside what this kernel handles
// (the caller then uses the mma.sync GEMM).
cudaError_t launch_gemm_tc(const GemmArgs& a, cudaStream_t st) {
  if (a.io_f32 || a.M <= 0 || a.N <= 0 || a.K <= 0) return cudaErrorNotSupported;
  if (a.k_split % TBK != 0 && a.k_split < a.K) return cudaErrorNotSupported;
  const bool amn = !a.a_kmajor, bmn = !a.b_kmajor;
  if ((reinterpret_cast<uintptr_t>(a.A) | reinterpret_cast<uintptr_t>(a.B)) & 15) return cudaErrorNotSupported;
  if ((a.lda % 8) || (a.ldb % 8)) return cudaErrorNotSupported;
  CUtensorMap ta, tb;
  const bool okA = amn ? make_map(&ta, a.A, (uint64_t)a.M, (uint64_t)a.K, (uint64_t)a.lda, 64, TBK)
                       : make_map(&ta, a.A, (uint64_t)a.K, (uint64_t)a.M, (uint64_t)a.lda, TBK, TBM);
  const bool okB = bmn ? make_map(&tb, a.B, (uint64_t)a.N, (uint64_t)a.K, (uint64_t)a.ldb, 64, TBK)
                       : make_map(&tb, a.B, (uint64_t)a.K, (uint64_t)a.N, (uint64_t)a.ldb, TBK, TBN);
  if (!okA || !okB) return cudaErrorNotSupported;
  const int splits = (a.K + a.k_split - 1) / a.k_split;
  const dim3 grid((a.N + TBN - 1) / TBN, (a.M + TBM - 1) / TBM, splits);
  cudaError_t e;
#define GBLA_CASE(AMN, BMN)                                                                                   \
  if (amn == AMN && bmn == BMN) {                                                                             \
    if ((e = cudaFuncSetAttribute(k_gemm_tc<AMN, BMN>, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_TC)) != \
        cudaSuccess)                                                                                          \
      return e;                                                                                               \
    k_gemm_tc<AMN, BMN><<<grid, 128, SMEM_TC, st>>>(ta, tb, a);                                               \
    return cudaGetLastError();                                                                                \
  }
  GBLA_CASE(false, false) GBLA_CASE(true, true) GBLA_CASE(false, true) GBLA_CASE(true, false)
#undef GBLA_CASE
  return cudaErrorNotSupported;
}

}  // namespace gbla
