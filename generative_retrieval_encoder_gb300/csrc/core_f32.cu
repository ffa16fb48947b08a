// fp32 GBLA state kernels: the same four steps as the bf16 kernels (reduce +
// deterministic combine, readout with optional fused RmsNorm gate, bwd_q with
// the [dS | dz] reduction, bwd_kv), in plain fp32 FMA arithmetic for fp32 I/O.
// Any d_h that is a multiple of 4 up to 128.
//
// "Gated Bidirectional Linear Attention for Generative Retrieval", section
// "Core method", Eq. 5-7 (see core_bf16.cu for the step-by-step formulas).
#include "core_common.cuh"

namespace gbla {
namespace {

constexpr unsigned FULL = 0xffffffffu;
constexpr int FT = 32;      // rows per smem tile
constexpr int NI = 65;      // ceil(128 * 129 / 256): state entries per thread

__device__ __forceinline__ float phi_x(float x) { return x > 0.f ? x + 1.f : expf(x); }
__device__ __forceinline__ float dphi_x(float x) { return x > 0.f ? 1.f : expf(x); }
__device__ __forceinline__ float sig_x(float x) { return 1.f / (1.f + expf(-x)); }

__device__ __forceinline__ float warp_sum(float v) {
  for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(FULL, v, o);
  return v;
}

// Writes this CTA's [dh][dh+1] accumulator (entry idx = tid + 256 i) as a
// partial with row stride state_ld(dh) and zero padding columns.
__device__ void write_partial(float* P, const float (&acc)[NI], int dh) {
  const int LD = state_ld(dh), W = dh + 1;
#pragma unroll
  for (int i = 0; i < NI; ++i) {
    const int idx = threadIdx.x + 256 * i;
    if (idx < dh * W) P[(idx / W) * LD + idx % W] = acc[i];
  }
  for (int idx = threadIdx.x; idx < dh * (LD - W); idx += 256)
    P[(idx / (LD - W)) * LD + W + idx % (LD - W)] = 0.f;
}

// acc[i] += sum_{r < rows} A[r][e_i] * B[r][f_i],  A [rows][dh], B [rows][dh+1].
__device__ __forceinline__ void accum_outer(float (&acc)[NI], const float* A, const float* B, int dh,
                                            int rows) {
  const int W = dh + 1;
#pragma unroll
  for (int i = 0; i < NI; ++i) {
    const int idx = threadIdx.x + 256 * i;
    if (idx < dh * W) {
      const int e = idx / W, f = idx % W;
      float s = acc[i];
      for (int r = 0; r < rows; ++r) s += A[r * dh + e] * B[r * W + f];
      acc[i] = s;
    }
  }
}

__global__ void __launch_bounds__(256) k_reduce_f32(const ReduceArgs a) {
  extern __shared__ float sm[];
  __shared__ float red8[8];
  const int dh = a.dh, W = dh + 1;
  float* kt = sm;            // [FT][dh]  g phi(k)
  float* vt = sm + FT * dh;  // [FT][dh+1]  [v | 1]
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (a.err && *a.err) return;
  int b, row0, nvalid, cin;
  if (!map_tile(a.seq, a.chunks, blockIdx.x, b, row0, nvalid, cin)) return;
  const int h = blockIdx.y, H = a.H;
  const int c0 = cin * a.chunks.tile;
  const int n_in = max(0, min(a.chunks.tile, nvalid - c0));
  const bool logits = a.gate_kind == GATE_LOGITS;
  const size_t rb = (size_t)row0 + c0;
  const float* kp = (const float*)a.k + rb * a.ldk + (size_t)h * dh;
  const float* vp = (const float*)a.v + rb * a.ldv + (size_t)h * dh;
  const float* gp = a.g + rb * a.ldg + h;
  float mch = 0.f;
  if (logits) {
    float m = -INFINITY;
    for (int i = tid; i < n_in; i += 256) m = fmaxf(m, gp[(size_t)i * a.ldg]);
    for (int o = 16; o; o >>= 1) m = fmaxf(m, __shfl_xor_sync(FULL, m, o));
    if (lane == 0) red8[warp] = m;
    __syncthreads();
    m = red8[0];
    for (int w = 1; w < 8; ++w) m = fmaxf(m, red8[w]);
    mch = m;
  }
  float acc[NI];
#pragma unroll
  for (int i = 0; i < NI; ++i) acc[i] = 0.f;
  for (int t0 = 0; t0 < n_in; t0 += FT) {
    const int rows = min(FT, n_in - t0);
    for (int i = tid; i < rows * dh; i += 256) {
      const int r = i / dh, e = i % dh;
      const float gv = gp[(size_t)(t0 + r) * a.ldg];
      kt[i] = (logits ? expf(gv - mch) : gv) * phi_x(kp[(size_t)(t0 + r) * a.ldk + e]);
    }
    for (int i = tid; i < rows * W; i += 256) {
      const int r = i / W, f = i % W;
      vt[i] = f < dh ? vp[(size_t)(t0 + r) * a.ldv + f] : 1.f;
    }
    __syncthreads();
    accum_outer(acc, kt, vt, dh, rows);
    __syncthreads();
  }
  write_partial(a.partial + ((size_t)blockIdx.x * H + h) * dh * state_ld(dh), acc, dh);
  if (logits && tid == 0) a.partial_m[(size_t)blockIdx.x * H + h] = n_in > 0 ? mch : -INFINITY;
  int first, count;
  seq_tiles(a.seq, a.chunks, b, first, count);
  if (!arrive_last(a.counters + (size_t)b * H + h, count)) return;
  combine_state(a.partial, a.partial_m, first, count, H, h, dh, b * H + h, logits, a.state, nullptr,
                a.state_m, a.pub_state);
}

// Loads [S | z] (rows e, dh+1 columns) of one (sequence, head) into smem.
__device__ __forceinline__ void load_state(float* S, const float* src, int dh) {
  const int W = dh + 1, LD = state_ld(dh);
  for (int i = threadIdx.x; i < dh * W; i += blockDim.x) S[i] = src[(i / W) * LD + i % W];
}

template <bool NORM>
__global__ void __launch_bounds__(256) k_readout_f32(const ReadoutArgs a) {
  extern __shared__ float sm[];
  const int dh = a.dh, W = dh + 1;
  float* S = sm;             // [dh][dh+1]
  float* qs = sm + dh * W;   // [8][dh]
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (a.err && *a.err) return;
  int b, row0, nvalid, tin;
  if (!map_tile(a.seq, a.tiles, blockIdx.x, b, row0, nvalid, tin)) return;
  const int h = blockIdx.y, H = a.H;
  const int R0 = tin * a.tiles.tile;
  const int nrows = min(a.tiles.tile, slot_rows(a.seq, nvalid) - R0);
  if (nrows <= 0) return;
  const int nval = max(0, min(nrows, nvalid - R0));
  load_state(S, a.state + (size_t)(b * H + h) * dh * state_ld(dh), dh);
  __syncthreads();
  float* q = qs + warp * dh;
  for (int r = warp; r < nrows; r += 8) {
    const size_t row = (size_t)row0 + R0 + r;
    const bool valid = r < nval;
    float* outp = (float*)a.out + row * a.ldo + (size_t)h * dh;
    if (!valid) {
      for (int f = lane; f < dh; f += 32) outp[f] = 0.f;
      if (a.den && lane == 0) a.den[row * H + h] = 0.f;
      continue;
    }
    for (int e = lane; e < dh; e += 32) q[e] = phi_x(((const float*)a.q)[row * a.ldq + (size_t)h * dh + e]);
    __syncwarp();
    float dpart = 0.f;
    for (int e = lane; e < dh; e += 32) dpart += q[e] * S[e * W + dh];
    const float den = warp_sum(dpart);
    float o[4];
    float ss = 0.f;
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int f = lane + 32 * u;
      o[u] = 0.f;
      if (f < dh) {
        float n = 0.f;
        for (int e = 0; e < dh; ++e) n += q[e] * S[e * W + f];
        o[u] = n / den;
        ss += o[u] * o[u];
      }
    }
    if (NORM) {
      const float rs = rsqrtf(warp_sum(ss) / dh + a.eps);
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int f = lane + 32 * u;
        if (f < dh) {
          const float rv = ((const float*)a.r)[row * a.ldr + (size_t)h * dh + f];
          const float gm = a.rms_w ? ((const float*)a.rms_w)[f] : 1.f;
          o[u] = o[u] * rs * gm * rv * sig_x(rv);
        }
      }
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int f = lane + 32 * u;
      if (f < dh) outp[f] = o[u];
    }
    if (a.den && lane == 0) a.den[row * H + h] = den;
    __syncwarp();
  }
}

template <bool NORM>
__global__ void __launch_bounds__(256) k_bwd_q_f32(const BwdQArgs a) {
  extern __shared__ float sm[];
  __shared__ float gred[8][128];
  const int dh = a.dh, W = dh + 1;
  float* S = sm;                // [dh][dh+1]
  float* qt = S + dh * W;       // [FT][dh]    phi(q)
  float* dnt = qt + FT * dh;    // [FT][dh+1]  [dn | dden]
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (a.err && *a.err) return;
  int b, row0, nvalid, cin;
  if (!map_tile(a.seq, a.chunks, blockIdx.x, b, row0, nvalid, cin)) {  // no chunk: a zero dgamma partial
    if (a.gamma_part)
      for (int f = tid; f < dh; f += blockDim.x) a.gamma_part[((size_t)blockIdx.x * a.H + blockIdx.y) * dh + f] = 0.f;
    return;
  }
  const int h = blockIdx.y, H = a.H;
  const int c0 = cin * a.chunks.tile;
  const int nrows = max(0, min(a.chunks.tile, slot_rows(a.seq, nvalid) - c0));
  const int nval = max(0, min(nrows, nvalid - c0));
  load_state(S, a.state + (size_t)(b * H + h) * dh * state_ld(dh), dh);
  float gacc[4] = {0.f, 0.f, 0.f, 0.f};
  float acc[NI];
#pragma unroll
  for (int i = 0; i < NI; ++i) acc[i] = 0.f;
  __syncthreads();
  for (int t0 = 0; t0 < nrows; t0 += FT) {
    const int rows = min(FT, nrows - t0);
    for (int r = warp; r < rows; r += 8) {
      const int rel = t0 + r;
      const size_t row = (size_t)row0 + c0 + rel;
      const bool valid = rel < nval;
      float* qr = qt + r * dh;
      float* dr_ = dnt + r * W;
      float* dqp = (float*)a.dq + row * a.lddq + (size_t)h * dh;
      float* drp = NORM ? (float*)a.dr + row * a.lddr + (size_t)h * dh : nullptr;
      const float* qin = (const float*)a.q + row * a.ldq + (size_t)h * dh;
      if (!valid) {
        for (int e = lane; e < dh; e += 32) { qr[e] = 0.f; dqp[e] = 0.f; if (NORM) drp[e] = 0.f; }
        for (int f = lane; f < W; f += 32) dr_[f] = 0.f;
        continue;
      }
      for (int e = lane; e < dh; e += 32) qr[e] = phi_x(qin[e]);
      __syncwarp();
      float dpart = 0.f;
      for (int e = lane; e < dh; e += 32) dpart += qr[e] * S[e * W + dh];
      const float den = warp_sum(dpart);
      float o[4], dO[4];
      float ss = 0.f;
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int f = lane + 32 * u;
        o[u] = 0.f;
        if (f < dh) {
          float n = 0.f;
          for (int e = 0; e < dh; ++e) n += qr[e] * S[e * W + f];
          o[u] = n / den;
          ss += o[u] * o[u];
        }
      }
      const float* yin = (const float*)a.dy + row * a.lddy + (size_t)h * dh;
      if (NORM) {
        const float rs = rsqrtf(warp_sum(ss) / dh + a.eps);
        const float* rin = (const float*)a.r + row * a.ldr + (size_t)h * dh;
        float uu[4], m = 0.f;
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int f = lane + 32 * u;
          uu[u] = 0.f; dO[u] = 0.f;
          if (f < dh) {
            const float rv = rin[f], yv = yin[f];
            const float gm = a.rms_w ? ((const float*)a.rms_w)[f] : 1.f;
            const float sg = sig_x(rv), av = rv * sg;
            uu[u] = o[u] * rs;
            gacc[u] += yv * uu[u] * av;
            drp[f] = yv * uu[u] * gm * sg * (1.f + rv * (1.f - sg));
            dO[u] = yv * gm * av;
            m += dO[u] * uu[u];
          }
        }
        m = warp_sum(m) / dh;
#pragma unroll
        for (int u = 0; u < 4; ++u) dO[u] = rs * (dO[u] - uu[u] * m);
      } else {
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int f = lane + 32 * u;
          dO[u] = f < dh ? yin[f] : 0.f;
        }
      }
      float dot = 0.f;
#pragma unroll
      for (int u = 0; u < 4; ++u) dot += dO[u] * o[u];
      const float dden = -warp_sum(dot) / den;
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int f = lane + 32 * u;
        if (f < dh) dr_[f] = dO[u] / den;
      }
      if (lane == 0) dr_[dh] = dden;
      __syncwarp();
      for (int e = lane; e < dh; e += 32) {
        float s = S[e * W + dh] * dden;
        for (int f = 0; f < dh; ++f) s += S[e * W + f] * dr_[f];
        dqp[e] = s * dphi_x(qin[e]);
      }
      __syncwarp();
    }
    __syncthreads();
    accum_outer(acc, qt, dnt, dh, rows);
    __syncthreads();
  }
  if (NORM) {
    for (int u = 0; u < 4; ++u)
      if (lane + 32 * u < dh) gred[warp][lane + 32 * u] = gacc[u];
    __syncthreads();
    for (int f = tid; f < dh; f += 256) {
      float v = 0.f;
      for (int w = 0; w < 8; ++w) v += gred[w][f];
      a.gamma_part[((size_t)blockIdx.x * H + h) * dh + f] = v;
    }
  }
  write_partial(a.partial + ((size_t)blockIdx.x * H + h) * dh * state_ld(dh), acc, dh);
  int first, count;
  seq_tiles(a.seq, a.chunks, b, first, count);
  if (!arrive_last(a.counters + (size_t)b * H + h, count)) return;
  combine_state(a.partial, nullptr, first, count, H, h, dh, b * H + h, false, a.dstate, nullptr, nullptr,
                nullptr);
}

__global__ void __launch_bounds__(256) k_bwd_kv_f32(const BwdKVArgs a) {
  extern __shared__ float sm[];
  __shared__ float bred[8];
  const int dh = a.dh, W = dh + 1;
  float* S = sm;                 // [dh][dh+1]  [dS | dz]
  float* ks = S + dh * W;        // [8][dh] g phi(k)
  float* vs = ks + 8 * dh;       // [8][dh] v
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (a.err && *a.err) return;
  int b, row0, nvalid, tin;
  if (!map_tile(a.seq, a.tiles, blockIdx.x, b, row0, nvalid, tin)) {  // no tile: a zero db_g partial
    if (a.bg_part && tid == 0) a.bg_part[(size_t)blockIdx.x * a.H + blockIdx.y] = 0.f;
    return;
  }
  const int h = blockIdx.y, H = a.H;
  const int R0 = tin * a.tiles.tile;
  const int nrows = min(a.tiles.tile, slot_rows(a.seq, nvalid) - R0);
  if (nrows <= 0) {
    if (a.bg_part && tid == 0) a.bg_part[(size_t)blockIdx.x * H + h] = 0.f;
    return;
  }
  const int nval = max(0, min(nrows, nvalid - R0));
  const bool logits = a.gate_kind == GATE_LOGITS;
  const float mseq = logits ? a.state_m[b * H + h] : 0.f;
  load_state(S, a.dstate + (size_t)(b * H + h) * dh * state_ld(dh), dh);
  __syncthreads();
  float bsum = 0.f;
  float* kr = ks + warp * dh;
  float* vr = vs + warp * dh;
  for (int r = warp; r < nrows; r += 8) {
    const size_t row = (size_t)row0 + R0 + r;
    const bool valid = r < nval;
    float* dkp = (float*)a.dk + row * a.lddk + (size_t)h * dh;
    float* dvp = (float*)a.dv + row * a.lddv + (size_t)h * dh;
    float* dsp = (float*)a.ds + row * a.ldds + h;
    if (h == 0 && a.zero_cols_to > a.zero_cols_from)
      for (int c = a.zero_cols_from + lane; c < a.zero_cols_to; c += 32)
        ((float*)a.ds)[row * a.ldds + c] = 0.f;
    if (!valid) {
      for (int e = lane; e < dh; e += 32) { dkp[e] = 0.f; dvp[e] = 0.f; }
      if (lane == 0) *dsp = 0.f;
      continue;
    }
    float gv = a.g[row * a.ldg + h];
    if (logits) gv = expf(gv - mseq);
    const float* kin = (const float*)a.k + row * a.ldk + (size_t)h * dh;
    const float* vin = (const float*)a.v + row * a.ldv + (size_t)h * dh;
    for (int e = lane; e < dh; e += 32) { kr[e] = gv * phi_x(kin[e]); vr[e] = vin[e]; }
    __syncwarp();
    float dgp = 0.f;
    for (int e = lane; e < dh; e += 32) {
      float s = S[e * W + dh];
      for (int f = 0; f < dh; ++f) s += S[e * W + f] * vr[f];
      dgp += phi_x(kin[e]) * s;
      dkp[e] = gv * s * dphi_x(kin[e]);
    }
    for (int f = lane; f < dh; f += 32) {
      float s = 0.f;
      for (int e = 0; e < dh; ++e) s += S[e * W + f] * kr[e];
      dvp[f] = s;
    }
    const float dg = warp_sum(dgp);
    float o = dg;
    if (a.gate_grad == GG_SIGMOID) o = dg * gv * (1.f - gv);
    else if (a.gate_grad == GG_SOFTMAX) o = gv * dg;
    if (lane == 0) *dsp = o;
    bsum += o;
    __syncwarp();
  }
  if (a.bg_part) {
    if (lane == 0) bred[warp] = bsum;
    __syncthreads();
    if (tid == 0) {
      float s = 0.f;
      for (int w = 0; w < 8; ++w) s += bred[w];
      a.bg_part[(size_t)blockIdx.x * H + h] = s;
    }
  }
}

template <typename K>
cudaError_t prep(K kernel, int smem) {
  return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
}

}  // namespace

cudaError_t launch_reduce_f32(const ReduceArgs& a, int grid_x, cudaStream_t st) {
  const int smem = (FT * a.dh + FT * (a.dh + 1)) * 4;
  cudaError_t e = prep(k_reduce_f32, smem);
  if (e != cudaSuccess) return e;
  k_reduce_f32<<<dim3(grid_x, a.H), 256, smem, st>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_readout_f32(const ReadoutArgs& a, bool norm, int grid_x, cudaStream_t st) {
  const int smem = (a.dh * (a.dh + 1) + 8 * a.dh) * 4;
  cudaError_t e = norm ? prep(k_readout_f32<true>, smem) : prep(k_readout_f32<false>, smem);
  if (e != cudaSuccess) return e;
  if (norm) k_readout_f32<true><<<dim3(grid_x, a.H), 256, smem, st>>>(a);
  else k_readout_f32<false><<<dim3(grid_x, a.H), 256, smem, st>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_bwd_q_f32(const BwdQArgs& a, bool norm, int grid_x, cudaStream_t st) {
  const int smem = (a.dh * (a.dh + 1) + FT * a.dh + FT * (a.dh + 1)) * 4;
  cudaError_t e = norm ? prep(k_bwd_q_f32<true>, smem) : prep(k_bwd_q_f32<false>, smem);
  if (e != cudaSuccess) return e;
  if (norm) k_bwd_q_f32<true><<<dim3(grid_x, a.H), 256, smem, st>>>(a);
  else k_bwd_q_f32<false><<<dim3(grid_x, a.H), 256, smem, st>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_bwd_kv_f32(const BwdKVArgs& a, int grid_x, cudaStream_t st) {
  const int smem = (a.dh * (a.dh + 1) + 16 * a.dh) * 4;
  cudaError_t e = prep(k_bwd_kv_f32, smem);
  if (e != cudaSuccess) return e;
  k_bwd_kv_f32<<<dim3(grid_x, a.H), 256, smem, st>>>(a);
  return cudaGetLastError();
}

}  // namespace gbla
