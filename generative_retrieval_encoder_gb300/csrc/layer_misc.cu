// Layer kernels around the state contractions: the sequence plan (varlen
// tile prefix sums + validation), the depthwise causal Conv1d of Eq. 4 and its
// backward, weight packing, and fixed-order reductions of per-block partial
// gradients.
#include "kernels.h"

namespace gbla {
namespace {

// ------------------------------------------------------------------ plan
// One CTA of 1024 threads.  Varlen: checks cu[0] == 0, cu[n] == T and
// cu[b+1] >= cu[b]; writes prefix_i[b+1] = sum_{b' <= b} max(1, ceil(len_b' /
// tile_i)).  Padded: checks 0 <= lens[b] <= L.  Violations set *err = 1.
__global__ void __launch_bounds__(1024) k_plan(SeqDesc s, int ntile, int t0, int t1, int t2,
                                               int32_t* p0, int32_t* p1, int32_t* p2, int* err) {
  __shared__ int wsum[32];
  __shared__ int carry[3];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int n = s.n_seq;
  if (s.mode == SEQ_PADDED) {
    for (int b = tid; b < n; b += 1024)
      if (s.lens[b] < 0 || s.lens[b] > s.L) atomicOr(err, 1);
    return;
  }
  if (s.mode != SEQ_VARLEN) return;
  if (tid == 0) {
    if (s.cu[0] != 0 || s.cu[n] != s.T) atomicOr(err, 1);
    carry[0] = carry[1] = carry[2] = 0;
  }
  const int ts[3] = {t0, t1, t2};
  int32_t* ps[3] = {p0, p1, p2};
  if (tid < ntile) ps[tid][0] = 0;
  __syncthreads();
  for (int base = 0; base < n; base += 1024) {
    const int b = base + tid;
    int len = 0;
    if (b < n) {
      len = s.cu[b + 1] - s.cu[b];
      if (len < 0) { atomicOr(err, 1); len = 0; }
    }
    for (int i = 0; i < ntile; ++i) {
      int v = b < n ? max(1, (len + ts[i] - 1) / ts[i]) : 0;
      for (int o = 1; o < 32; o <<= 1) {  // inclusive warp scan
        const int y = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += y;
      }
      if (lane == 31) wsum[warp] = v;
      __syncthreads();
      if (warp == 0) {
        int w = wsum[lane];
        for (int o = 1; o < 32; o <<= 1) {
          const int y = __shfl_up_sync(0xffffffffu, w, o);
          if (lane >= o) w += y;
        }
        wsum[lane] = w;
      }
      __syncthreads();
      const int incl = v + (warp > 0 ? wsum[warp - 1] : 0) + carry[i];
      if (b < n) ps[i][b + 1] = incl;
      __syncthreads();
      if (tid == 1023) carry[i] = incl;
      __syncthreads();
    }
  }
}

// Walks the rows of the sequences: for row l gives the first row s0 of its
// sequence, the end of its valid rows vend and the end of its slot send.
struct SeqCursor {
  const SeqDesc& s;
  int b, s0, vend, send;
  __device__ explicit SeqCursor(const SeqDesc& sd) : s(sd), b(0), s0(0), vend(0), send(0) {}
  __device__ void seek(int l) {
    if (s.mode != SEQ_VARLEN) {
      b = l / s.L;
      s0 = b * s.L;
      send = s0 + s.L;
      vend = s0 + (s.mode == SEQ_PADDED ? s.lens[b] : s.L);
    } else {
      int lo = 0, hi = s.n_seq - 1;  // last b with cu[b] <= l
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (s.cu[mid] <= l) lo = mid; else hi = mid - 1;
      }
      b = lo;
      while (b + 1 < s.n_seq && s.cu[b + 1] <= l) ++b;  // skip empty sequences
      s0 = s.cu[b];
      vend = send = s.cu[b + 1];
    }
  }
};

template <typename T> struct Vec;
template <> struct Vec<bf16> { static constexpr int N = 8; typedef uint4 U; };
template <> struct Vec<float> { static constexpr int N = 4; typedef float4 U; };

template <typename T>
__device__ __forceinline__ void vload(const T* p, float* out) {
  typedef typename Vec<T>::U U;
  const U u = *reinterpret_cast<const U*>(p);
  const T* e = reinterpret_cast<const T*>(&u);
#pragma unroll
  for (int i = 0; i < Vec<T>::N; ++i) out[i] = to_f<T>(e[i]);
}
template <typename T>
__device__ __forceinline__ void vstore(T* p, const float* in) {
  typedef typename Vec<T>::U U;
  U u;
  T* e = reinterpret_cast<T*>(&u);
#pragma unroll
  for (int i = 0; i < Vec<T>::N; ++i) e[i] = from_f<T>(in[i]);
  *reinterpret_cast<U*>(p) = u;
}

constexpr int RUN = 16;   // rows per thread, forward conv
constexpr int RUNB = 64;  // rows per block, backward conv

// Eq. 4 Conv1d (depthwise, causal, kernel 4):
//   x~[l, c] = b[c] + sum_t w[c, t] x[l - 3 + t, c]   (rows before the sequence start read 0)
// Each thread owns VEC channels and RUN consecutive rows (sliding window).
template <typename T>
__global__ void __launch_bounds__(128) k_conv_fwd(const ConvArgs a) {
  constexpr int V = Vec<T>::N;
  if (*a.err) return;
  const int c0 = (blockIdx.y * 128 + threadIdx.x) * V;
  if (c0 >= a.d) return;
  const int r0 = blockIdx.x * RUN, r1 = min(a.T, r0 + RUN);
  if (r0 >= r1) return;
  const T* x = (const T*)a.x;
  T* xt = (T*)a.xt;
  float w[V][4], bias[V];
#pragma unroll
  for (int i = 0; i < V; ++i) {
#pragma unroll
    for (int t = 0; t < 4; ++t) w[i][t] = to_f<T>(((const T*)a.w)[(size_t)(c0 + i) * 4 + t]);
    bias[i] = a.b ? to_f<T>(((const T*)a.b)[c0 + i]) : 0.f;
  }
  SeqCursor cur(a.seq);
  cur.seek(r0);
  float p3[V], p2[V], p1[V], xc[V];
#pragma unroll
  for (int i = 0; i < V; ++i) p3[i] = p2[i] = p1[i] = 0.f;
  if (r0 - 3 >= cur.s0) vload<T>(x + (size_t)(r0 - 3) * a.d + c0, p3);
  if (r0 - 2 >= cur.s0) vload<T>(x + (size_t)(r0 - 2) * a.d + c0, p2);
  if (r0 - 1 >= cur.s0) vload<T>(x + (size_t)(r0 - 1) * a.d + c0, p1);
  for (int l = r0; l < r1; ++l) {
    if (l >= cur.send) {
      cur.seek(l);
#pragma unroll
      for (int i = 0; i < V; ++i) p3[i] = p2[i] = p1[i] = 0.f;
    }
    float o[V];
    if (l < cur.vend) {
      vload<T>(x + (size_t)l * a.d + c0, xc);
#pragma unroll
      for (int i = 0; i < V; ++i) o[i] = bias[i] + w[i][0] * p3[i] + w[i][1] * p2[i] + w[i][2] * p1[i] + w[i][3] * xc[i];
    } else {
#pragma unroll
      for (int i = 0; i < V; ++i) { xc[i] = 0.f; o[i] = 0.f; }
    }
    vstore<T>(xt + (size_t)l * a.d + c0, o);
#pragma unroll
    for (int i = 0; i < V; ++i) { p3[i] = p2[i]; p2[i] = p1[i]; p1[i] = xc[i]; }
  }
}

// Backward of Eq. 4 Conv1d.  For rows l of a sequence (valid rows [s0, vend)):
//   dx[l]   = sum_t w[t] dx~[l + 3 - t]   (terms with l + 3 - t < vend)
//   dw[t]  += x[l - 3 + t] dx~[l];   db += dx~[l]
// Block bx owns rows [bx RUNB, bx RUNB + RUNB); each thread VEC channels.
// Per-block parameter partials go to part[bx][c][0..4].
template <typename T>
__global__ void __launch_bounds__(128) k_conv_bwd(const ConvArgs a) {
  constexpr int V = Vec<T>::N;
  if (*a.err) return;
  const int c0 = (blockIdx.y * 128 + threadIdx.x) * V;
  if (c0 >= a.d) return;
  const int r0 = blockIdx.x * RUNB, r1 = min(a.T, r0 + RUNB);
  const T* x = (const T*)a.x;
  float w[V][4];
#pragma unroll
  for (int i = 0; i < V; ++i)
#pragma unroll
    for (int t = 0; t < 4; ++t) w[i][t] = to_f<T>(((const T*)a.w)[(size_t)(c0 + i) * 4 + t]);
  float dw[V][4], db[V];
#pragma unroll
  for (int i = 0; i < V; ++i) { db[i] = 0.f; dw[i][0] = dw[i][1] = dw[i][2] = dw[i][3] = 0.f; }
  auto ldg = [&](int row, float* out) {  // dx~ row (fp32)
    const float4* p = reinterpret_cast<const float4*>(a.dxt + (size_t)row * a.d + c0);
#pragma unroll
    for (int i = 0; i < V / 4; ++i) {
      const float4 u = p[i];
      out[4 * i] = u.x; out[4 * i + 1] = u.y; out[4 * i + 2] = u.z; out[4 * i + 3] = u.w;
    }
  };
  if (r0 < r1) {
    SeqCursor cur(a.seq);
    cur.seek(r0);
    float p3[V], p2[V], p1[V], xc[V];  // x[l-3], x[l-2], x[l-1], x[l]
    float g0[V], g1[V], g2[V], g3[V];  // dx~[l .. l+3]
    auto reset = [&](int l) {
#pragma unroll
      for (int i = 0; i < V; ++i) p3[i] = p2[i] = p1[i] = g0[i] = g1[i] = g2[i] = 0.f;
      if (l - 3 >= cur.s0 && l - 3 < cur.vend) vload<T>(x + (size_t)(l - 3) * a.d + c0, p3);
      if (l - 2 >= cur.s0 && l - 2 < cur.vend) vload<T>(x + (size_t)(l - 2) * a.d + c0, p2);
      if (l - 1 >= cur.s0 && l - 1 < cur.vend) vload<T>(x + (size_t)(l - 1) * a.d + c0, p1);
      if (l < cur.vend) ldg(l, g0);
      if (l + 1 < cur.vend) ldg(l + 1, g1);
      if (l + 2 < cur.vend) ldg(l + 2, g2);
    };
    reset(r0);
    for (int l = r0; l < r1; ++l) {
      if (l >= cur.send) {
        cur.seek(l);
        reset(l);
      }
      float o[V];
      if (l < cur.vend) {
        vload<T>(x + (size_t)l * a.d + c0, xc);
#pragma unroll
        for (int i = 0; i < V; ++i) g3[i] = 0.f;
        if (l + 3 < cur.vend) ldg(l + 3, g3);
#pragma unroll
        for (int i = 0; i < V; ++i) {
          o[i] = w[i][3] * g0[i] + w[i][2] * g1[i] + w[i][1] * g2[i] + w[i][0] * g3[i];
          dw[i][0] += p3[i] * g0[i];
          dw[i][1] += p2[i] * g0[i];
          dw[i][2] += p1[i] * g0[i];
          dw[i][3] += xc[i] * g0[i];
          db[i] += g0[i];
        }
      } else {
#pragma unroll
        for (int i = 0; i < V; ++i) { o[i] = 0.f; xc[i] = 0.f; g3[i] = 0.f; }
      }
      vstore<T>((T*)a.dx + (size_t)l * a.d + c0, o);
#pragma unroll
      for (int i = 0; i < V; ++i) {
        p3[i] = p2[i]; p2[i] = p1[i]; p1[i] = xc[i];
        g0[i] = g1[i]; g1[i] = g2[i]; g2[i] = g3[i];
      }
    }
  }
  float* P = a.part + (size_t)blockIdx.x * a.d * 5;
#pragma unroll
  for (int i = 0; i < V; ++i) {
#pragma unroll
    for (int t = 0; t < 4; ++t) P[(size_t)(c0 + i) * 5 + t] = dw[i][t];
    P[(size_t)(c0 + i) * 5 + 4] = db[i];
  }
}

// Wt[n][c] (n < 4*H*dh + H) and/or Wp[c][n] (n < np, zero past 4*H*dh + H).
template <typename T>
__global__ void k_pack(const T* Wq, const T* Wk, const T* Wv, const T* Wr, const T* wg, int d, int H,
                       int dh, T* Wt, T* Wp, int np) {
  const int HD = H * dh, N1 = 4 * HD + H;
  const size_t total = (size_t)d * np;
  const T* Ws[4] = {Wq, Wk, Wv, Wr};
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < total; i += (size_t)gridDim.x * blockDim.x) {
    const int c = (int)(i / np), n = (int)(i % np);
    T v = from_f<T>(0.f);
    if (n < 4 * HD) v = Ws[n / HD][(size_t)c * HD + n % HD];
    else if (n < N1) v = wg[(size_t)c * H + n - 4 * HD];
    if (Wp) Wp[i] = v;
    if (Wt && n < N1) Wt[(size_t)n * d + c] = v;
  }
}

// Column sums of a [S][stride] partial array in a fixed order: block b owns
// columns 32 b .. 32 b + 31; warp w adds rows w, w + 32, w + 64, ... (lanes
// read 32 consecutive floats); then warp 0 adds the 32 warp sums in order.
// mode 0: out[i];  mode 1 (conv parameters, i = 5 c + t): t < 4 -> out[4 c + t], else out2[c].
__global__ void __launch_bounds__(1024) k_colsum(const float* part, int S, int64_t stride, int64_t n, float* out,
                                                 float* out2, int mode) {
  __shared__ float red[32][33];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t i = (int64_t)blockIdx.x * 32 + lane;
  float s = 0.f;
  if (i < n)
    for (int k = warp; k < S; k += 32) s += part[(int64_t)k * stride + i];
  red[warp][lane] = s;
  __syncthreads();
  if (warp == 0 && i < n) {
    float t = 0.f;
    for (int w = 0; w < 32; ++w) t += red[w][lane];
    if (mode == 0) {
      out[i] = t;
    } else {
      const int64_t c = i / 5, q = i % 5;
      if (q < 4) { if (out) out[c * 4 + q] = t; }
      else if (out2) out2[c] = t;
    }
  }
}

__global__ void k_scatter_dw(const float* part, int S, int d, int np, int H, int dh, float* o0, float* o1,
                             float* o2, float* o3, float* o4) {
  const int HD = H * dh;
  float* outs[4] = {o0, o1, o2, o3};
  const size_t total = (size_t)d * np;
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < total; i += (size_t)gridDim.x * blockDim.x) {
    const int c = (int)(i / np), n = (int)(i % np);
    if (n >= 4 * HD + H) continue;
    float s = 0.f;
    for (int k = 0; k < S; ++k) s += part[(size_t)k * total + i];
    if (n < 4 * HD) {
      if (outs[n / HD]) outs[n / HD][(size_t)c * HD + n % HD] = s;
    } else if (o4) {
      o4[(size_t)c * H + n - 4 * HD] = s;
    }
  }
}

int grid_for(size_t n) { const size_t g = (n + 255) / 256; return (int)(g < 2432 ? (g > 0 ? g : 1) : 2432); }

}  // namespace

cudaError_t launch_plan(const SeqDesc& s, int ntile, const int* tile_sizes, int32_t* const* prefixes,
                        int* err, cudaStream_t st) {
  k_plan<<<1, 1024, 0, st>>>(s, ntile, tile_sizes[0], ntile > 1 ? tile_sizes[1] : 1,
                             ntile > 2 ? tile_sizes[2] : 1, prefixes[0], ntile > 1 ? prefixes[1] : nullptr,
                             ntile > 2 ? prefixes[2] : nullptr, err);
  return cudaGetLastError();
}

cudaError_t launch_conv_fwd(const ConvArgs& a, bool f32, cudaStream_t st) {
  const int V = f32 ? 4 : 8;
  const dim3 grid((a.T + RUN - 1) / RUN, (a.d / V + 127) / 128);
  if (f32) k_conv_fwd<float><<<grid, 128, 0, st>>>(a);
  else k_conv_fwd<bf16><<<grid, 128, 0, st>>>(a);
  return cudaGetLastError();
}

int conv_bwd_blocks(int T) { return (T + RUNB - 1) / RUNB; }

cudaError_t launch_conv_bwd(const ConvArgs& a, bool f32, int nblk, cudaStream_t st) {
  const int V = f32 ? 4 : 8;
  const dim3 grid(nblk, (a.d / V + 127) / 128);
  if (f32) k_conv_bwd<float><<<grid, 128, 0, st>>>(a);
  else k_conv_bwd<bf16><<<grid, 128, 0, st>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_pack_weights(const void* const* W, const void* w_g, int d, int H, int dh, bool f32,
                                void* Wt, void* Wp, int np, cudaStream_t st) {
  const int grid = grid_for((size_t)d * np);
  if (f32)
    k_pack<float><<<grid, 256, 0, st>>>((const float*)W[0], (const float*)W[1], (const float*)W[2],
                                        (const float*)W[3], (const float*)w_g, d, H, dh, (float*)Wt,
                                        (float*)Wp, np);
  else
    k_pack<bf16><<<grid, 256, 0, st>>>((const bf16*)W[0], (const bf16*)W[1], (const bf16*)W[2],
                                       (const bf16*)W[3], (const bf16*)w_g, d, H, dh, (bf16*)Wt, (bf16*)Wp, np);
  return cudaGetLastError();
}

cudaError_t launch_sum_parts(const float* part, int S, int64_t stride, int64_t n, float* out, cudaStream_t st) {
  k_colsum<<<(unsigned)((n + 31) / 32), 1024, 0, st>>>(part, S, stride, n, out, nullptr, 0);
  return cudaGetLastError();
}

cudaError_t launch_scatter_dw(const float* part, int S, int d, int np, int H, int dh, float* const* outs,
                              cudaStream_t st) {
  k_scatter_dw<<<grid_for((size_t)d * np), 256, 0, st>>>(part, S, d, np, H, dh, outs[0], outs[1], outs[2],
                                                         outs[3], outs[4]);
  return cudaGetLastError();
}

cudaError_t launch_conv_param_grads(const float* part, int S, int d, float* dw, float* db, cudaStream_t st) {
  k_colsum<<<(unsigned)((d * 5 + 31) / 32), 1024, 0, st>>>(part, S, (int64_t)d * 5, (int64_t)d * 5, dw, db, 1);
  return cudaGetLastError();
}

}  // namespace gbla
