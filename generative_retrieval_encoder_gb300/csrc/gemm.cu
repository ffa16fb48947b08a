// Projection GEMMs of the GBLA layer, C[M, N] = sum_k A(m, k) B(n, k):
//   forward   [Q | K | V | R | s] = x~ [W_Q W_K W_V W_R w_g]          (Eq. 4, 5, 7)
//             epilogue: bf16 projections, gate g = sigmoid(s + b_g) or logit s
//   backward  dx~ = dP W_all^T                                         (fp32 out)
//             dW_all = x~^T dP   (split over rows, fixed-order sum after)
// bf16: mma.sync m16n8k16 tensor-core tiles 128 x 128 x 32, 8 warps, 4-stage
// cp.async pipeline, swizzled smem, ldmatrix (.trans for M/N-major operands).
// fp32: a plain SIMT tile GEMM with the same argument contract.
#include "kernels.h"

namespace gbla {
namespace {

constexpr int BM = 128, BN = 128, BK = 32, STAGES = 4;
constexpr int TILE_B = BM * BK * 2;  // bytes of one operand tile
constexpr int SMEM = STAGES * 2 * TILE_B;

template <bool AK, bool BKM>
__global__ void __launch_bounds__(256) k_gemm_bf16(const GemmArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int wm = warp & 1, wn = warp >> 1;  // 2 x 4 warps, warp tile 64 x 32
  const int n0 = blockIdx.x * BN, m0 = blockIdx.y * BM;
  const int kbeg = blockIdx.z * a.k_split;
  const int kend = min(a.K, kbeg + a.k_split);
  const int nk = (kend - kbeg + BK - 1) / BK;
  const bf16* A = (const bf16*)a.A;
  const bf16* B = (const bf16*)a.B;

  auto load = [&](int stage, int kt) {
    const int k0 = kbeg + kt * BK;
    const uint32_t ab = smem_u32(smem + stage * 2 * TILE_B), bb = ab + TILE_B;
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const int i = tid + u * 256;
      if (AK) {  // [BM rows m][BK]
        const int r = i >> 2, c = i & 3;
        const bool ok = (m0 + r < a.M) && (k0 + c * 8 < kend);
        cp_async16(ab + swz<4>(r, c), ok ? A + (size_t)(m0 + r) * a.lda + k0 + c * 8 : A, ok ? 16 : 0);
      } else {   // [BK rows k][BM]
        const int r = i >> 4, c = i & 15;
        const bool ok = (k0 + r < kend) && (m0 + c * 8 < a.M);
        cp_async16(ab + swz<16>(r, c), ok ? A + (size_t)(k0 + r) * a.lda + m0 + c * 8 : A, ok ? 16 : 0);
      }
      if (BKM) {
        const int r = i >> 2, c = i & 3;
        const bool ok = (n0 + r < a.N) && (k0 + c * 8 < kend);
        cp_async16(bb + swz<4>(r, c), ok ? B + (size_t)(n0 + r) * a.ldb + k0 + c * 8 : B, ok ? 16 : 0);
      } else {
        const int r = i >> 4, c = i & 15;
        const bool ok = (k0 + r < kend) && (n0 + c * 8 < a.N);
        cp_async16(bb + swz<16>(r, c), ok ? B + (size_t)(k0 + r) * a.ldb + n0 + c * 8 : B, ok ? 16 : 0);
      }
    }
  };

  float acc[4][4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j][0] = acc[i][j][1] = acc[i][j][2] = acc[i][j][3] = 0.f;

#pragma unroll
  for (int s = 0; s < STAGES - 1; ++s) {
    if (s < nk) load(s, s);
    cp_async_commit();
  }
  const int mi = lane >> 3, rr = lane & 7;
  for (int kt = 0; kt < nk; ++kt) {
    cp_async_wait<STAGES - 2>();
    __syncthreads();
    {
      const int kn = kt + STAGES - 1;
      if (kn < nk) load(kn % STAGES, kn);
      cp_async_commit();
    }
    const int st = kt % STAGES;
    const uint32_t ab = smem_u32(smem + st * 2 * TILE_B), bb = ab + TILE_B;
#pragma unroll
    for (int kk = 0; kk < BK / 16; ++kk) {
      uint32_t af[4][4], bfr[4][2];
#pragma unroll
      for (int mt = 0; mt < 4; ++mt) {
        const int mb = wm * 64 + mt * 16;
        if (AK)
          ldsm_x4(ab + swz<4>(mb + ((mi & 1) << 3) + rr, 2 * kk + (mi >> 1)), af[mt][0], af[mt][1], af[mt][2], af[mt][3]);
        else
          ldsm_x4_t(ab + swz<16>(kk * 16 + ((mi >> 1) << 3) + rr, mb / 8 + (mi & 1)), af[mt][0], af[mt][1], af[mt][2],
                    af[mt][3]);
      }
#pragma unroll
      for (int np = 0; np < 2; ++np) {
        const int nb = wn * 32 + np * 16;
        if (BKM)
          ldsm_x4(bb + swz<4>(nb + ((mi >> 1) << 3) + rr, 2 * kk + (mi & 1)), bfr[2 * np][0], bfr[2 * np][1],
                  bfr[2 * np + 1][0], bfr[2 * np + 1][1]);
        else
          ldsm_x4_t(bb + swz<16>(kk * 16 + ((mi & 1) << 3) + rr, nb / 8 + (mi >> 1)), bfr[2 * np][0], bfr[2 * np][1],
                    bfr[2 * np + 1][0], bfr[2 * np + 1][1]);
      }
#pragma unroll
      for (int mt = 0; mt < 4; ++mt)
#pragma unroll
        for (int nt = 0; nt < 4; ++nt)
          mma_bf16(acc[mt][nt], af[mt][0], af[mt][1], af[mt][2], af[mt][3], bfr[nt][0], bfr[nt][1]);
    }
  }
  cp_async_wait<0>();

  const int g = lane >> 2, t4 = lane & 3;
  const int Hg = a.N - a.n_main;
#pragma unroll
  for (int mt = 0; mt < 4; ++mt)
#pragma unroll
    for (int hr = 0; hr < 2; ++hr) {
      const int m = m0 + wm * 64 + mt * 16 + g + hr * 8;
      if (m >= a.M) continue;
#pragma unroll
      for (int nt = 0; nt < 4; ++nt) {
        const int n = n0 + wn * 32 + nt * 8 + 2 * t4;
        const float v0 = acc[mt][nt][2 * hr], v1 = acc[mt][nt][2 * hr + 1];
        if (a.epi == EPI_PROJ_PRE && n < a.n_main) {  // [phi(q) | phi(k) | v | r]; a pair lies in one block
          const bool ph = n < 2 * a.hd;
          const float w0 = ph ? phi_f(v0) : v0, w1 = ph ? phi_f(v1) : v1;
          *reinterpret_cast<uint32_t*>((bf16*)a.C + (size_t)m * a.ldc + n) = pack_bf16(w0, w1);
          continue;
        }
        // n is even and n_main a multiple of 8: a pair never straddles n_main
        if (a.epi == EPI_BF16 || (a.epi == EPI_PROJ && n < a.n_main)) {
          bf16* C = (bf16*)a.C + (size_t)m * a.ldc + n;
          const int nlim = a.epi == EPI_PROJ ? a.n_main : a.N;
          if (n + 1 < nlim) *reinterpret_cast<uint32_t*>(C) = pack_bf16(v0, v1);
          else if (n < nlim) C[0] = __float2bfloat16_rn(v0);
        } else if (a.epi == EPI_PROJ || a.epi == EPI_PROJ_PRE) {
#pragma unroll
          for (int q = 0; q < 2; ++q) {
            const int hh = n + q - a.n_main;
            if (hh < 0 || hh >= Hg) continue;
            float s = q ? v1 : v0;
            if (a.bias_g) s += __bfloat162float(((const bf16*)a.bias_g)[hh]);
            a.gate[(size_t)m * a.ldgate + hh] = a.gate_mode == 0 ? 1.f / (1.f + __expf(-s)) : s;
          }
        } else {
          float* C = (float*)a.C + (a.epi == EPI_SPLITK ? (size_t)blockIdx.z * a.M * a.ldc : 0) +
                     (size_t)m * a.ldc + n;
          if (n + 1 < a.N) *reinterpret_cast<float2*>(C) = make_float2(v0, v1);
          else if (n < a.N) C[0] = v0;
        }
      }
    }
}

// ------------------------------------------------------------------ fp32
constexpr int FB = 64, FK = 16;

__global__ void __launch_bounds__(256) k_gemm_f32(const GemmArgs a) {
  __shared__ float As[FK][FB + 1], Bs[FK][FB + 1];
  const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
  const int n0 = blockIdx.x * FB, m0 = blockIdx.y * FB;
  const int kbeg = blockIdx.z * a.k_split;
  const int kend = min(a.K, kbeg + a.k_split);
  const float* A = (const float*)a.A;
  const float* B = (const float*)a.B;
  float acc[4][4] = {};
  for (int k0 = kbeg; k0 < kend; k0 += FK) {
    for (int i = tid; i < FK * FB; i += 256) {
      const int kk = a.a_kmajor ? i % FK : i / FB, mm = a.a_kmajor ? i / FK : i % FB;
      const int m = m0 + mm, k = k0 + kk;
      As[kk][mm] = (m < a.M && k < kend) ? (a.a_kmajor ? A[(size_t)m * a.lda + k] : A[(size_t)k * a.lda + m]) : 0.f;
      const int kb = a.b_kmajor ? i % FK : i / FB, nn = a.b_kmajor ? i / FK : i % FB;
      const int n = n0 + nn, k2 = k0 + kb;
      Bs[kb][nn] = (n < a.N && k2 < kend) ? (a.b_kmajor ? B[(size_t)n * a.ldb + k2] : B[(size_t)k2 * a.ldb + n]) : 0.f;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < FK; ++kk) {
      float av[4], bv[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) { av[i] = As[kk][ty * 4 + i]; bv[i] = Bs[kk][tx * 4 + i]; }
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] += av[i] * bv[j];
    }
    __syncthreads();
  }
  const int Hg = a.N - a.n_main;
  for (int i = 0; i < 4; ++i) {
    const int m = m0 + ty * 4 + i;
    if (m >= a.M) continue;
    for (int j = 0; j < 4; ++j) {
      const int n = n0 + tx * 4 + j;
      if (n >= a.N) continue;
      float v = acc[i][j];
      if (a.epi == EPI_PROJ) {
        if (n < a.n_main) {
          ((float*)a.C)[(size_t)m * a.ldc + n] = v;
        } else if (n - a.n_main < Hg) {
          if (a.bias_g) v += ((const float*)a.bias_g)[n - a.n_main];
          a.gate[(size_t)m * a.ldgate + n - a.n_main] = a.gate_mode == 0 ? 1.f / (1.f + expf(-v)) : v;
        }
      } else {
        ((float*)a.C)[(a.epi == EPI_SPLITK ? (size_t)blockIdx.z * a.M * a.ldc : 0) + (size_t)m * a.ldc + n] = v;
      }
    }
  }
}

}  // namespace

cudaError_t launch_gemm_bf16(const GemmArgs& a, cudaStream_t st) {
  const int splits = (a.K + a.k_split - 1) / a.k_split;
  const dim3 grid((a.N + BN - 1) / BN, (a.M + BM - 1) / BM, splits);
  cudaError_t e;
#define GBLA_CASE(AK, BKM)                                                                           \
  if (a.a_kmajor == AK && a.b_kmajor == BKM) {                                                       \
    if ((e = cudaFuncSetAttribute(k_gemm_bf16<AK, BKM>, cudaFuncAttributeMaxDynamicSharedMemorySize, \
                                  SMEM)) != cudaSuccess)                                             \
      return e;                                                                                      \
    k_gemm_bf16<AK, BKM><<<grid, 256, SMEM, st>>>(a);                                                \
    return cudaGetLastError();                                                                       \
  }
  GBLA_CASE(1, 1) GBLA_CASE(0, 0) GBLA_CASE(1, 0) GBLA_CASE(0, 1)
#undef GBLA_CASE
  return cudaErrorInvalidValue;
}

cudaError_t launch_gemm_f32(const GemmArgs& a, cudaStream_t st) {
  const int splits = (a.K + a.k_split - 1) / a.k_split;
  const dim3 grid((a.N + FB - 1) / FB, (a.M + FB - 1) / FB, splits);
  k_gemm_f32<<<grid, 256, 0, st>>>(a);
  return cudaGetLastError();
}

}  // namespace gbla
