// Layer kernels around the state contractions: the sequence plan (varlen
// tile prefix sums + validation), the depthwise causal Conv1d of Eq. 4 and its
// backward, weight packing, and fixed-order reductions of per-block partial
// gradients.
#include <algorithm>

#include "kernels.h"
#include "pdl.cuh"
#include "tcgen05.cuh"

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

constexpr int RUN = 16;    // rows per thread, forward conv
constexpr int RUNB = 4;    // rows per inner run, backward conv
constexpr int BW_ROWGROUPS = 4;  // backward: row groups per block (block = 64 channel vectors x 4)

template <typename T>
__device__ __forceinline__ typename Vec<T>::U vraw(const T* p) {
  return *reinterpret_cast<const typename Vec<T>::U*>(p);
}
template <typename T>
__device__ __forceinline__ void vcvt(const typename Vec<T>::U& u, float* out) {
  const T* e = reinterpret_cast<const T*>(&u);
#pragma unroll
  for (int i = 0; i < Vec<T>::N; ++i) out[i] = to_f<T>(e[i]);
}

// The 4 taps of channels c0 .. c0 + V - 1 (w is [d][4], contiguous: 4 vector
// loads) and their biases (b may be null).
template <typename T>
__device__ __forceinline__ void load_taps(const T* w, const T* b, int c0, float (&wt)[Vec<T>::N][4],
                                          float (&bias)[Vec<T>::N]) {
  constexpr int V = Vec<T>::N;
  typedef typename Vec<T>::U U;
  const U* wp = reinterpret_cast<const U*>(w + (size_t)c0 * 4);
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    float f[V];
    vcvt<T>(wp[j], f);
#pragma unroll
    for (int i = 0; i < V; ++i) wt[(j * V + i) / 4][(j * V + i) % 4] = f[i];
  }
  if (b) {
    vcvt<T>(*reinterpret_cast<const U*>(b + c0), bias);
  } else {
#pragma unroll
    for (int i = 0; i < V; ++i) bias[i] = 0.f;
  }
}

// Eq. 4 Conv1d (depthwise, causal, kernel 4):
//   x~[l, c] = b[c] + sum_t w[c, t] x[l - 3 + t, c]   (rows before the sequence start read 0)
// Work item = (channel vector, run of RUN rows); consecutive threads take
// consecutive channel vectors (coalesced).  The RUN + 3 input rows of a run
// are loaded up front so that all of them are in flight together.
template <typename T>
__global__ void __launch_bounds__(256) k_conv_fwd(const ConvArgs a) {
  constexpr int V = Vec<T>::N;
  typedef typename Vec<T>::U U;
  if (a.err && *a.err) return;
  const int CV = a.d / V;
  const long long item = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  const int cv = (int)(item % CV);
  const int r0 = (int)(item / CV) * RUN;
  if (r0 >= a.T) return;
  const int c0 = cv * V;
  const T* x = (const T*)a.x;
  T* xt = (T*)a.xt;
  U raw[RUN + 3];
#pragma unroll
  for (int j = 0; j < RUN + 3; ++j) {
    const int l = r0 - 3 + j;
    if (l >= 0 && l < a.T) raw[j] = vraw<T>(x + (size_t)l * a.d + c0);
    else raw[j] = U{};
  }
  float w[V][4], bias[V];
  load_taps<T>((const T*)a.w, (const T*)a.b, c0, w, bias);
  SeqCursor cur(a.seq);
  cur.seek(r0);
#pragma unroll
  for (int i = 0; i < RUN; ++i) {
    const int l = r0 + i;
    if (l < a.T) {
      if (l >= cur.send) cur.seek(l);
      float o[V];
#pragma unroll
      for (int c = 0; c < V; ++c) o[c] = 0.f;
      if (l < cur.vend) {
#pragma unroll
        for (int c = 0; c < V; ++c) o[c] = bias[c];
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          if (l - 3 + t >= cur.s0) {
            float xv[V];
            vcvt<T>(raw[i + t], xv);
#pragma unroll
            for (int c = 0; c < V; ++c) o[c] += w[c][t] * xv[c];
          }
        }
      }
      vstore<T>(xt + (size_t)l * a.d + c0, o);
    }
  }
}

// Backward of Eq. 4 Conv1d.  For rows l of a sequence (valid rows [s0, vend)):
//   dx[l]   = sum_t w[t] dx~[l + 3 - t]   (terms with l + 3 - t < vend)
//   dw[t]  += x[l - 3 + t] dx~[l];   db += dx~[l]
// Block (bx, by): 64 channel vectors x 4 row groups over rows
// [by rows_per_block, ...); a row group takes runs of RUNB rows, loading the
// run's x and dx~ rows up front.  The 4 row groups' parameter partials are
// added in a fixed order into part[by][c][0..4].
template <typename T>
__global__ void __launch_bounds__(256) k_conv_bwd(const ConvArgs a, int rows_per_block) {
  constexpr int V = Vec<T>::N;
  typedef typename Vec<T>::U U;
  __shared__ float red[BW_ROWGROUPS - 1][64][5 * V];
  if (a.err && *a.err) return;
  const int CV = a.d / V;
  const int tx = threadIdx.x & 63, rg = threadIdx.x >> 6;
  const int cv = blockIdx.x * 64 + tx;
  const bool active = cv < CV;
  const int c0 = cv * V;
  const int rb0 = blockIdx.y * rows_per_block, rb1 = min(a.T, rb0 + rows_per_block);
  const T* x = (const T*)a.x;
  const T* gx = (const T*)a.dxt;
  float dw[V][4], db[V];
#pragma unroll
  for (int i = 0; i < V; ++i) { db[i] = 0.f; dw[i][0] = dw[i][1] = dw[i][2] = dw[i][3] = 0.f; }
  if (active) {
    float w[V][4], nobias[V];
    load_taps<T>((const T*)a.w, nullptr, c0, w, nobias);
    SeqCursor cur(a.seq);
    for (int r0 = rb0 + rg * RUNB; r0 < rb1; r0 += BW_ROWGROUPS * RUNB) {
      U xr[RUNB + 3], gr[RUNB + 3];  // x[r0-3 .. r0+RUNB-1], dx~[r0 .. r0+RUNB+2]
#pragma unroll
      for (int j = 0; j < RUNB + 3; ++j) {
        const int lx = r0 - 3 + j, lg = r0 + j;
        xr[j] = (lx >= 0 && lx < a.T) ? vraw<T>(x + (size_t)lx * a.d + c0) : U{};
        gr[j] = (lg < a.T) ? vraw<T>(gx + (size_t)lg * a.d + c0) : U{};
      }
      cur.seek(r0);
#pragma unroll
      for (int i = 0; i < RUNB; ++i) {
        const int l = r0 + i;
        if (l < rb1) {
          if (l >= cur.send) cur.seek(l);
          float o[V];
#pragma unroll
          for (int c = 0; c < V; ++c) o[c] = 0.f;
          if (l < cur.vend) {
            float g0[V];
            vcvt<T>(gr[i], g0);
#pragma unroll
            for (int k = 1; k < 4; ++k) {  // dx~[l + k] feeds tap 3 - k
              if (l + k < cur.vend) {
                float gk[V];
                vcvt<T>(gr[i + k], gk);
#pragma unroll
                for (int c = 0; c < V; ++c) o[c] += w[c][3 - k] * gk[c];
              }
            }
#pragma unroll
            for (int c = 0; c < V; ++c) {
              o[c] += w[c][3] * g0[c];
              db[c] += g0[c];
            }
#pragma unroll
            for (int t = 0; t < 4; ++t) {
              if (l - 3 + t >= cur.s0) {
                float xv[V];
                vcvt<T>(xr[i + t], xv);
#pragma unroll
                for (int c = 0; c < V; ++c) dw[c][t] += xv[c] * g0[c];
              }
            }
          }
          vstore<T>((T*)a.dx + (size_t)l * a.d + c0, o);
        }
      }
    }
  }
  if (rg > 0 && active) {
#pragma unroll
    for (int c = 0; c < V; ++c) {
#pragma unroll
      for (int t = 0; t < 4; ++t) red[rg - 1][tx][5 * c + t] = dw[c][t];
      red[rg - 1][tx][5 * c + 4] = db[c];
    }
  }
  __syncthreads();
  if (rg == 0 && active) {
    float* P = a.part + (size_t)blockIdx.y * a.d * 5;
#pragma unroll
    for (int c = 0; c < V; ++c) {
#pragma unroll
      for (int t = 0; t < 5; ++t) {
        float s = t < 4 ? dw[c][t] : db[c];
        for (int g = 0; g < BW_ROWGROUPS - 1; ++g) s += red[g][tx][5 * c + t];
        P[(size_t)(c0 + c) * 5 + t] = s;
      }
    }
  }
}

// Wp[c][n] = [W_q | W_k | W_v | W_r | w_g | 0][c][n] for n < np, 16 bytes
// per thread: row c = blockIdx.y, vectors blockIdx.x * 256 + threadIdx.x of it
// (no 64-bit index division).  np and H*dh are multiples of the vector width,
// so a vector lies in one block; `vec`: the W_* rows are 16-byte aligned.
template <typename T>
__global__ void __launch_bounds__(256) k_pack(const T* Wq, const T* Wk, const T* Wv, const T* Wr, const T* wg,
                                              int d, int H, int dh, T* Wp, int np, int vec, uint32_t* zero,
                                              int zero_words) {
  pdl_enter();  // the previous kernel's outputs are visible from here on
  constexpr int V = 16 / sizeof(T);
  typedef uint4 U;
  if (zero && blockIdx.x == 0 && blockIdx.y == 0)
    for (int i = threadIdx.x; i < zero_words; i += blockDim.x) zero[i] = 0u;
  const int HD = H * dh, npv = np / V;
  const T* Ws[4] = {Wq, Wk, Wv, Wr};
  const int c = blockIdx.y;
  for (int v = blockIdx.x * blockDim.x + threadIdx.x; v < npv; v += gridDim.x * blockDim.x) {
    const int n = v * V;
    const int m = n / HD, j = n - m * HD;
    U u;
    if (m < 4 && vec) {
      u = *reinterpret_cast<const U*>(Ws[m] + (size_t)c * HD + j);
    } else {
      T* e = reinterpret_cast<T*>(&u);
#pragma unroll
      for (int q = 0; q < V; ++q) {
        const int nq = n + q, mq = nq / HD;
        T v = from_f<T>(0.f);
        if (mq < 4) v = Ws[mq][(size_t)c * HD + nq - mq * HD];
        else if (nq - 4 * HD < H) v = wg[(size_t)c * H + nq - 4 * HD];
        e[q] = v;
      }
    }
    *reinterpret_cast<U*>(Wp + (size_t)c * np + n) = u;
  }
}

// Column sums of a [S][stride] partial array in a fixed order: block b owns
// columns 32 b .. 32 b + 31; warp w adds rows w, w + 32, w + 64, ... (lanes
// read 32 consecutive floats); then warp 0 adds the 32 warp sums in order.
// mode 0: out[i];  mode 1 (conv parameters, i = 5 c + t): t < 4 -> out[4 c + t], else out2[c].
__global__ void __launch_bounds__(1024) k_colsum(const ColsumJobs js) {
  pdl_enter();  // the previous kernel's outputs are visible from here on
  __shared__ float red[32][33];
  if ((int)blockIdx.x < js.sc.blocks) {  // the split-K sum of dW into its five outputs
    const ScatterJob& X = js.sc;
    const int HD = X.H * X.dh;
    const size_t total = (size_t)X.d * X.np;
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < total; i += (size_t)X.blocks * blockDim.x) {
      const int c = (int)(i / X.np), n = (int)(i % X.np);
      if (n >= 4 * HD + X.H) continue;
      float s = 0.f;
      for (int k = 0; k < X.S; ++k) s += X.part[(size_t)k * total + i];
      if (n < 4 * HD) {
        if (X.out[n / HD]) X.out[n / HD][(size_t)c * HD + n % HD] = s;
      } else if (X.out[4]) {
        X.out[4][(size_t)c * X.H + n - 4 * HD] = s;
      }
    }
    return;
  }
  // this block's job: the jobs' column blocks are laid out one after another
  int jb = blockIdx.x - js.sc.blocks, j = 0;
  while (j + 1 < js.n && jb >= (int)((js.j[j].n + 31) / 32)) jb -= (int)((js.j[j++].n + 31) / 32);
  const ColsumJob& J = js.j[j];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t i = (int64_t)jb * 32 + lane;
  float s = 0.f;
  if (i < J.n)
    for (int k = warp; k < J.S; k += 32) s += J.part[(int64_t)k * J.stride + i];
  red[warp][lane] = s;
  __syncthreads();
  if (warp == 0 && i < J.n) {
    float t = 0.f;
    for (int w = 0; w < 32; ++w) t += red[w][lane];
    if (J.mode == 0) {
      J.out[i] = t;
    } else {
      const int64_t c = i / 5, q = i % 5;
      if (q < 4) { if (J.out) J.out[c * 4 + q] = t; }
      else if (J.out2) J.out2[c] = t;
    }
  }
}



// ------------------------------------------------------------ diagnostic
// The bounded mbarrier wait of the tensor-core kernels, run out on purpose:
// one thread waits for a phase of a barrier that nothing arrives at, gives up
// after `polls` polls (a bounded loop; nothing faults or hangs) and reports
// it through the timeout bit of the error word, as the kernels do.
__global__ void k_diag_wait(int* err, unsigned polls) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int fail;
  const uint32_t b = smem_u32(&bar);
  if (threadIdx.x == 0) {
    mbar_init(b, 1);
    mbar_init_fence();
    fail = 0;
  }
  __syncthreads();
  if (threadIdx.x == 0 && !mbar_wait(b, 0, &fail, polls)) atomicOr(err, kErrTimeout);
}

}  // namespace

cudaError_t launch_diag_wait(int* err, unsigned polls, cudaStream_t st) {
  k_diag_wait<<<1, 32, 0, st>>>(err, polls);
  return cudaGetLastError();
}

cudaError_t launch_plan(const SeqDesc& s, int ntile, const int* tile_sizes, int32_t* const* prefixes,
                        int* err, cudaStream_t st) {
  k_plan<<<1, 1024, 0, st>>>(s, ntile, tile_sizes[0], ntile > 1 ? tile_sizes[1] : 1,
                             ntile > 2 ? tile_sizes[2] : 1, prefixes[0], ntile > 1 ? prefixes[1] : nullptr,
                             ntile > 2 ? prefixes[2] : nullptr, err);
  return cudaGetLastError();
}

cudaError_t launch_conv_fwd(const ConvArgs& a, bool f32, cudaStream_t st, int* tiled) {
  const bool tile = !f32 && conv_tile_ok(a, false);
  if (tiled) *tiled = tile ? 1 : 0;
  if (tile) return launch_conv_fwd_tile(a, st);
  const int V = f32 ? 4 : 8;
  const long long items = (long long)((a.T + RUN - 1) / RUN) * (a.d / V);
  const unsigned grid = (unsigned)((items + 255) / 256);
  if (f32) k_conv_fwd<float><<<grid, 256, 0, st>>>(a);
  else k_conv_fwd<bf16><<<grid, 256, 0, st>>>(a);
  return cudaGetLastError();
}

int conv_bwd_blocks(int T) { return std::max(1, std::min(1024, (T + 127) / 128)); }
int conv_bwd_parts_max(int T) { return std::max(conv_bwd_blocks(T), conv_tile_parts_max(T)); }

cudaError_t launch_conv_bwd(const ConvArgs& a, bool f32, int* nparts, cudaStream_t st, int* tiled) {
  const bool tile = !f32 && conv_tile_ok(a, true);
  if (tiled) *tiled = tile ? 1 : 0;
  if (tile) {
    *nparts = conv_tile_parts(a.T, a.d);
    return launch_conv_bwd_tile(a, *nparts, st);
  }
  const int nblk = *nparts = conv_bwd_blocks(a.T);
  const int V = f32 ? 4 : 8;
  const int unit = RUNB * BW_ROWGROUPS;
  const int rows = ((a.T + nblk - 1) / nblk + unit - 1) / unit * unit;
  const dim3 grid((a.d / V + 63) / 64, nblk);
  if (f32) k_conv_bwd<float><<<grid, 256, 0, st>>>(a, rows);
  else k_conv_bwd<bf16><<<grid, 256, 0, st>>>(a, rows);
  return cudaGetLastError();
}

cudaError_t launch_pack_weights(const void* const* W, const void* w_g, int d, int H, int dh, bool f32,
                                void* Wp, int np, void* zero, size_t zero_bytes, cudaStream_t st) {
  uint32_t* zw = static_cast<uint32_t*>(zero);
  const int zn = (int)(zero_bytes / 4);
  int vec = 1;
  for (int m = 0; m < 4; ++m) vec &= ((uintptr_t)W[m] & 15) == 0;
  const int npv = np / (f32 ? 4 : 8);
  const dim3 grid((unsigned)std::max(1, (npv + 255) / 256), (unsigned)std::max(1, d));
  if (f32)
    return launch_pdl(k_pack<float>, dim3(grid), dim3(256), 0, st, (const float*)W[0], (const float*)W[1],
                      (const float*)W[2], (const float*)W[3], (const float*)w_g, d, H, dh, (float*)Wp, np, vec, zw, zn);
  return launch_pdl(k_pack<bf16>, dim3(grid), dim3(256), 0, st, (const bf16*)W[0], (const bf16*)W[1],
                    (const bf16*)W[2], (const bf16*)W[3], (const bf16*)w_g, d, H, dh, (bf16*)Wp, np, vec, zw, zn);
}

cudaError_t launch_colsums(ColsumJobs js, cudaStream_t st) {
  js.sc.blocks = 0;
  if (js.sc.part) {
    const size_t n = (size_t)js.sc.d * js.sc.np;
    js.sc.blocks = (int)std::min<size_t>((n + 1023) / 1024, (size_t)sm_count() * 2);
  }
  int blocks = js.sc.blocks;
  for (int j = 0; j < js.n; ++j) blocks += (int)((js.j[j].n + 31) / 32);
  if (blocks <= 0) return cudaSuccess;
  return launch_pdl(k_colsum, dim3((unsigned)blocks), dim3(1024), 0, st, js);
}



}  // namespace gbla
