// Eq. 4 depthwise causal Conv1d (kernel 4) and its backward for bf16 rows,
// streamed through shared memory.
//
// A tile is CR = 32 rows x up to CW = 512 channels.  Its input rows plus a
// 3-row halo arrive by bulk copies (cp.async.bulk, completing on an mbarrier)
// into a ring of shared-memory stages, issued by warp 0 several tiles ahead,
// so the copies of later tiles are in flight while the block computes on the
// current one.  A block is persistent over the row tiles of one channel tile.
// In the forward a thread computes 4 rows x 8 channels of a tile (16-byte
// shared loads and global stores); in the backward 8 rows x 4 channels,
// sliding a 4-row window down x and dx~, and keeps its own parameter-gradient
// partials, so the backward needs no reduction inside the block.
//
// Per-row sequence structure (the first row of the sequence and the end of
// its valid rows) is folded into a 9-bit mask per tile row, computed by
// warp 1 when the tile's copies are issued.  The mask is the same for every
// thread, so the branch between the full-window path and the boundary path is
// uniform.
#include <algorithm>

#include "pdl.cuh"
#include "kernels.h"
#include "mbarrier.cuh"

namespace gbla {
namespace {

constexpr int CR = 32;           // rows per tile (one mask per lane of warp 1)
constexpr int CW = 512;          // channels per tile: 256 pairs
constexpr int CROWS = CR + 3;    // staged rows per tensor
constexpr int NTH = 512;         // thread = (pair tid % 256, row half tid / 256)
constexpr int HALF = CR / 2;
constexpr int FWD_ST = 4, BWD_ST = 3;
constexpr int GX_MAX = 256;      // backward: blocks per channel tile, at most

// Mask bits of tile row i (global row l):
//   bit t      (t = 0..3)  x[l - 3 + t] is a row of l's sequence, l valid
//   bit 4 + k  (k = 0..3)  dx~[l + k] is a valid row of l's sequence (bit 4: l valid)
//   bit 8                  l < T: the row is stored
constexpr uint32_t M_ROW = 1u << 8;
constexpr uint32_t M_VALID = 1u << 4;
constexpr uint32_t M_FULL = 0x1FFu;

template <int NT, int ST>
struct ConvSmem {
  static constexpr int TENSOR = CROWS * CW * 2;           // bytes of one staged tensor
  static constexpr int STAGE = NT * TENSOR;
  static constexpr int MASKS = ST * STAGE;                // uint32 [ST][CR]
  static constexpr int BARS = MASKS + ST * CR * 4;        // uint64 [ST]
  static constexpr int BYTES = BARS + ST * 8;
};
static_assert(ConvSmem<2, BWD_ST>::BYTES <= 227 * 1024, "backward stages exceed shared memory");
static_assert(ConvSmem<1, FWD_ST>::BYTES <= 227 * 1024, "forward stages exceed shared memory");

__device__ uint32_t row_mask(const SeqDesc& sd, int l) {
  if (l >= sd.T) return 0;
  SeqCursor cur(sd);
  cur.seek(l);
  uint32_t m = M_ROW;
  if (l < cur.vend) {
#pragma unroll
    for (int t = 0; t < 4; ++t)
      if (l - 3 + t >= cur.s0) m |= 1u << t;
#pragma unroll
    for (int k = 0; k < 4; ++k)
      if (l + k < cur.vend) m |= 1u << (4 + k);
  }
  return m;
}

__device__ __forceinline__ float2 ld2(const uint8_t* base, int row, int cw, int pr) {
  const uint32_t u = *reinterpret_cast<const uint32_t*>(base + ((size_t)row * cw + 2 * pr) * 2);
  return make_float2(__uint_as_float(u << 16), __uint_as_float(u & 0xFFFF0000u));
}
__device__ __forceinline__ void fma2(float2& acc, float2 w, float2 x) {
  acc.x = fmaf(w.x, x.x, acc.x);
  acc.y = fmaf(w.y, x.y, acc.y);
}

// Issues the bulk copies of rows [lo, hi) of src (row stride d, channels c0 ..
// c0 + cw) into smem rows starting at dst; warp 0, every lane.  Contiguous when
// the tile spans every channel.
__device__ __forceinline__ void copy_rows(uint32_t dst, const bf16* src, int lo, int hi, int d, int c0, int cw,
                                          uint32_t bar, int lane) {
  if (cw == d) {
    if (lane == 0) bulk_g2s(dst, src + (size_t)lo * d, (uint32_t)((hi - lo) * d * 2), bar);
  } else {
    for (int r = lo + lane; r < hi; r += 32)
      bulk_g2s(dst + (uint32_t)((r - lo) * cw * 2), src + (size_t)r * d + c0, (uint32_t)(cw * 2), bar);
  }
}

// The persistent tile loop of both directions: issue(j, stage) starts the
// copies (warp 0) and the masks (warp 1) of the block's j-th tile,
// compute(stage, j) consumes it.  False if a wait gave up (after letting the
// copies still in flight land).
template <int NT, int ST, typename Issue, typename Compute>
__device__ __forceinline__ bool tile_loop(int ntile, uint8_t* smem, Issue issue, Compute compute) {
  typedef ConvSmem<NT, ST> S;
  const int tid = threadIdx.x, warp = tid >> 5;
  const uint32_t bars = smem_u32(smem + S::BARS);
  if (tid == 0) {
    for (int s = 0; s < ST; ++s) mbar_init(bars + 8 * s, 1);
    mbar_init_fence();
  }
  __syncthreads();
  if (warp <= 1)
    for (int j = 0; j < ST - 1 && j < ntile; ++j) issue(j, j);
  int fail = 0, it = 0;
  for (; it < ntile; ++it) {
    if (__syncthreads_or(fail)) break;  // also: every thread is done with stage (it - 1) % ST
    const int jn = it + ST - 1;
    if (warp <= 1 && jn < ntile) issue(jn, jn % ST);
    const int st = it % ST;
    if (!mbar_wait_bounded(bars + 8 * st, (uint32_t)((it / ST) & 1))) {
      fail = 1;
      continue;
    }
    compute(st, it);
  }
  fail = __syncthreads_or(fail);
  if (fail && tid == 0) {  // bounded waits for the copies still in flight
    const int issued = min(ntile, it + ST - 1);
    for (int j = it - 1; j < issued; ++j) mbar_wait_bounded(bars + 8 * (j % ST), (uint32_t)((j / ST) & 1));
  }
  return !fail;
}

// x~[l, c] = b[c] + sum_t w[c, t] x[l - 3 + t, c]; taps before the sequence
// start read 0; padding rows get 0.  Thread (channel octet tid % 64, row
// quarter-group tid / 64) computes 4 rows x 8 channels of a tile from 7
// 16-byte shared loads and leaves them as 16-byte stores.
constexpr int FV = 8;                 // channels per thread (16 bytes of bf16)
constexpr int FRG = NTH / (CW / FV);  // row groups
constexpr int FRR = CR / FRG;         // rows per thread
static_assert(FRR == 4 && FRG * FRR == CR, "forward: 8 row groups of 4 rows");
__device__ __forceinline__ void unpack8f(const uint4& u, float* f) {
  f[0] = __uint_as_float(u.x << 16); f[1] = __uint_as_float(u.x & 0xFFFF0000u);
  f[2] = __uint_as_float(u.y << 16); f[3] = __uint_as_float(u.y & 0xFFFF0000u);
  f[4] = __uint_as_float(u.z << 16); f[5] = __uint_as_float(u.z & 0xFFFF0000u);
  f[6] = __uint_as_float(u.w << 16); f[7] = __uint_as_float(u.w & 0xFFFF0000u);
}
__global__ void __launch_bounds__(NTH, 1) k_conv_fwd_tile(const ConvArgs a, int gx) {
  pdl_enter();  // the previous kernel's outputs are visible from here on
  typedef ConvSmem<1, FWD_ST> S;
  extern __shared__ __align__(128) uint8_t smem[];
  if (a.err && *a.err) return;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int cg = tid % (CW / FV), rg = tid / (CW / FV);
  const int c0 = blockIdx.y * CW, cw = min(CW, a.d - c0);
  const int c = c0 + FV * cg;
  const bool act = FV * cg < cw;
  const int n_rt = (a.T + CR - 1) / CR;
  const int ntile = n_rt > (int)blockIdx.x ? (n_rt - 1 - (int)blockIdx.x) / gx + 1 : 0;
  const bf16* x = (const bf16*)a.x;
  bf16* xt = (bf16*)a.xt;
  uint32_t* masks = reinterpret_cast<uint32_t*>(smem + S::MASKS);
  const uint32_t bars = smem_u32(smem + S::BARS);

  float w[4][FV], bias[FV];
#pragma unroll
  for (int v = 0; v < FV; ++v) bias[v] = 0.f;
  if (act) {
    const bf16* wc = (const bf16*)a.w + (size_t)c * 4;  // [c][4 taps], 8 channels = 64 bytes
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      float f[8];
      unpack8f(*reinterpret_cast<const uint4*>(wc + 8 * q), f);  // channels 2q, 2q + 1
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        w[t][2 * q] = f[t];
        w[t][2 * q + 1] = f[4 + t];
      }
    }
    if (a.b) unpack8f(*reinterpret_cast<const uint4*>((const bf16*)a.b + c), bias);
  }

  auto issue = [&](int j, int st) {
    const int r0 = ((int)blockIdx.x + j * gx) * CR;
    if (warp == 0) {
      const int lo = max(0, r0 - 3), hi = min(a.T, r0 + CR);
      if (lane == 0) mbar_expect_tx(bars + 8 * st, (uint32_t)((hi - lo) * cw * 2));
      __syncwarp();
      copy_rows(smem_u32(smem + st * S::STAGE) + (uint32_t)((lo - (r0 - 3)) * cw * 2), x, lo, hi, a.d, c0, cw,
                bars + 8 * st, lane);
    } else {
      masks[st * CR + lane] = row_mask(a.seq, r0 + lane);
    }
  };
  auto compute = [&](int st, int j) {
    const int r0 = ((int)blockIdx.x + j * gx) * CR;
    const uint8_t* xs = smem + st * S::STAGE;  // smem row i + t holds x[r0 + i - 3 + t]
    const uint32_t* mk = masks + st * CR;
    if (!act) return;
    const int i0 = rg * FRR;
    float xv[FRR + 3][FV];
#pragma unroll
    for (int r = 0; r < FRR + 3; ++r)
      unpack8f(*reinterpret_cast<const uint4*>(xs + ((size_t)(i0 + r) * cw + FV * cg) * 2), xv[r]);
#pragma unroll
    for (int ii = 0; ii < FRR; ++ii) {
      const int i = i0 + ii;
      const uint32_t m = mk[i];
      if (!(m & M_ROW)) continue;
      float o[FV];
#pragma unroll
      for (int v = 0; v < FV; ++v) o[v] = 0.f;
      if (m & M_VALID) {
#pragma unroll
        for (int v = 0; v < FV; ++v) {
          float acc = bias[v];
          if (m & 1u) acc = fmaf(w[0][v], xv[ii][v], acc);
          if (m & 2u) acc = fmaf(w[1][v], xv[ii + 1][v], acc);
          if (m & 4u) acc = fmaf(w[2][v], xv[ii + 2][v], acc);
          o[v] = fmaf(w[3][v], xv[ii + 3][v], acc);
        }
      }
      *reinterpret_cast<uint4*>(xt + (size_t)(r0 + i) * a.d + c) =
          make_uint4(pack_bf16(o[0], o[1]), pack_bf16(o[2], o[3]), pack_bf16(o[4], o[5]), pack_bf16(o[6], o[7]));
    }
  };
  if (!tile_loop<1, FWD_ST>(ntile, smem, issue, compute) && tid == 0 && a.err_out)
    atomicOr(a.err_out, kErrTimeout);
}

// Backward, for rows l of a sequence (valid rows [s0, vend)):
//   dx[l]  = sum_k w[3 - k] dx~[l + k]   (terms with l + k < vend)
//   dw[t] += x[l - 3 + t] dx~[l]  (l - 3 + t >= s0);   db += dx~[l]
// Thread (channel quad tid % 128, row group tid / 128) of block (bx, channel
// tile) computes 8 rows x 4 channels of each tile, sliding a 4-row window of
// x and dx~ (8-byte shared loads), and writes its parameter partials to
// part[4 bx + row group][c][0..4].
constexpr int BV = 4;                 // channels per thread
constexpr int BRG = NTH / (CW / BV);  // row groups
constexpr int BRR = CR / BRG;         // rows per thread
static_assert(BRG == 4 && BRR == 8, "backward: 4 row groups of 8 rows");
__device__ __forceinline__ void unpack4f(const uint2& u, float* f) {
  f[0] = __uint_as_float(u.x << 16); f[1] = __uint_as_float(u.x & 0xFFFF0000u);
  f[2] = __uint_as_float(u.y << 16); f[3] = __uint_as_float(u.y & 0xFFFF0000u);
}
__global__ void __launch_bounds__(NTH, 1) k_conv_bwd_tile(const ConvArgs a, int gx) {
  pdl_enter();  // the previous kernel's outputs are visible from here on
  typedef ConvSmem<2, BWD_ST> S;
  extern __shared__ __align__(128) uint8_t smem[];
  if (a.err && *a.err) return;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int cq = tid % (CW / BV), rg = tid / (CW / BV);
  const int c0 = blockIdx.y * CW, cw = min(CW, a.d - c0);
  const int c = c0 + BV * cq;
  const bool act = BV * cq < cw;
  const int n_rt = (a.T + CR - 1) / CR;
  const int ntile = n_rt > (int)blockIdx.x ? (n_rt - 1 - (int)blockIdx.x) / gx + 1 : 0;
  const bf16* x = (const bf16*)a.x;
  const bf16* gx_ = (const bf16*)a.dxt;
  bf16* dx = (bf16*)a.dx;
  uint32_t* masks = reinterpret_cast<uint32_t*>(smem + S::MASKS);
  const uint32_t bars = smem_u32(smem + S::BARS);

  float w[4][BV];
  if (act) {
    const uint4* wc = reinterpret_cast<const uint4*>((const bf16*)a.w + (size_t)c * 4);  // [c][4 taps]
#pragma unroll
    for (int q = 0; q < 2; ++q) {  // channels c + 2q, c + 2q + 1
      float f[8];
      const uint4 u = wc[q];
      unpack4f(make_uint2(u.x, u.y), f);
      unpack4f(make_uint2(u.z, u.w), f + 4);
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        w[t][2 * q] = f[t];
        w[t][2 * q + 1] = f[4 + t];
      }
    }
  }
  float dw[4][BV], db[BV];
#pragma unroll
  for (int v = 0; v < BV; ++v) {
    db[v] = 0.f;
#pragma unroll
    for (int t = 0; t < 4; ++t) dw[t][v] = 0.f;
  }

  auto issue = [&](int j, int st) {
    const int r0 = ((int)blockIdx.x + j * gx) * CR;
    if (warp == 0) {
      const int xlo = max(0, r0 - 3), xhi = min(a.T, r0 + CR);
      const int ghi = min(a.T, r0 + CROWS);
      if (lane == 0) mbar_expect_tx(bars + 8 * st, (uint32_t)((xhi - xlo + ghi - r0) * cw * 2));
      __syncwarp();
      const uint32_t base = smem_u32(smem + st * S::STAGE);
      copy_rows(base + (uint32_t)((xlo - (r0 - 3)) * cw * 2), x, xlo, xhi, a.d, c0, cw, bars + 8 * st, lane);
      copy_rows(base + S::TENSOR, gx_, r0, ghi, a.d, c0, cw, bars + 8 * st, lane);
    } else {
      masks[st * CR + lane] = row_mask(a.seq, r0 + lane);
    }
  };
  auto compute = [&](int st, int j) {
    const int r0 = ((int)blockIdx.x + j * gx) * CR;
    const uint8_t* xs = smem + st * S::STAGE;  // row i + t: x[r0 + i - 3 + t]
    const uint8_t* gs = xs + S::TENSOR;        // row i + k: dx~[r0 + i + k]
    const uint32_t* mk = masks + st * CR;
    if (!act) return;
    const int i0 = rg * BRR;
    float xv[BRR + 3][BV], gv[BRR + 3][BV];  // rows i0 .. i0 + 10, loaded as the window slides
#pragma unroll
    for (int r = 0; r < 3; ++r) {
      unpack4f(*reinterpret_cast<const uint2*>(xs + ((size_t)(i0 + r) * cw + c - c0) * 2), xv[r]);
      unpack4f(*reinterpret_cast<const uint2*>(gs + ((size_t)(i0 + r) * cw + c - c0) * 2), gv[r]);
    }
#pragma unroll
    for (int ii = 0; ii < BRR; ++ii) {
      const int i = i0 + ii;
      unpack4f(*reinterpret_cast<const uint2*>(xs + ((size_t)(i + 3) * cw + c - c0) * 2), xv[ii + 3]);
      unpack4f(*reinterpret_cast<const uint2*>(gs + ((size_t)(i + 3) * cw + c - c0) * 2), gv[ii + 3]);
      const uint32_t m = mk[i];
      if (!(m & M_ROW)) continue;
      float o[BV];
#pragma unroll
      for (int v = 0; v < BV; ++v) o[v] = 0.f;
      if (m & M_VALID) {
#pragma unroll
        for (int v = 0; v < BV; ++v) {
          const float g0 = gv[ii][v];
          float acc = w[3][v] * g0;
          if (m & (M_VALID << 1)) acc = fmaf(w[2][v], gv[ii + 1][v], acc);
          if (m & (M_VALID << 2)) acc = fmaf(w[1][v], gv[ii + 2][v], acc);
          if (m & (M_VALID << 3)) acc = fmaf(w[0][v], gv[ii + 3][v], acc);
          o[v] = acc;
          if (m & 1u) dw[0][v] = fmaf(xv[ii][v], g0, dw[0][v]);
          if (m & 2u) dw[1][v] = fmaf(xv[ii + 1][v], g0, dw[1][v]);
          if (m & 4u) dw[2][v] = fmaf(xv[ii + 2][v], g0, dw[2][v]);
          dw[3][v] = fmaf(xv[ii + 3][v], g0, dw[3][v]);
          db[v] += g0;
        }
      }
      *reinterpret_cast<uint2*>(dx + (size_t)(r0 + i) * a.d + c) = make_uint2(pack_bf16(o[0], o[1]), pack_bf16(o[2], o[3]));
    }
  };
  if (!tile_loop<2, BWD_ST>(ntile, smem, issue, compute)) {
    if (tid == 0 && a.err_out) atomicOr(a.err_out, kErrTimeout);
    return;
  }
  if (act) {
    float* P = a.part + ((size_t)(BRG * blockIdx.x + rg) * a.d + c) * 5;
#pragma unroll
    for (int v = 0; v < BV; ++v) {
      P[5 * v + 0] = dw[0][v]; P[5 * v + 1] = dw[1][v]; P[5 * v + 2] = dw[2][v]; P[5 * v + 3] = dw[3][v];
      P[5 * v + 4] = db[v];
    }
  }
}

int conv_gx(int T, int d) {
  const int n_rt = (T + CR - 1) / CR, n_ct = (d + CW - 1) / CW;
  return std::max(1, std::min(std::min(n_rt, GX_MAX), std::max(1, sm_count() / n_ct)));
}

}  // namespace

bool conv_tile_ok(const ConvArgs& a, bool bwd) {
  auto al = [](const void* p) { return ((uintptr_t)p & 15) == 0; };
  return a.T > 0 && a.d % 8 == 0 && al(a.x) && al(a.w) && (bwd ? al(a.dxt) && al(a.dx) : al(a.xt)) &&
         (bwd || !a.b || al(a.b));  // the forward reads 8 biases at a time
}

int conv_tile_parts(int T, int d) { return BRG * conv_gx(T, d); }
int conv_tile_parts_max(int T) { return BRG * std::max(1, std::min((T + CR - 1) / CR, GX_MAX)); }

cudaError_t launch_conv_fwd_tile(const ConvArgs& a, cudaStream_t st) {
  typedef ConvSmem<1, FWD_ST> S;
  cudaError_t e = cudaFuncSetAttribute(k_conv_fwd_tile, cudaFuncAttributeMaxDynamicSharedMemorySize, S::BYTES);
  if (e != cudaSuccess) return e;
  const int n_rt = (a.T + CR - 1) / CR, n_ct = (a.d + CW - 1) / CW;
  const int gx = std::max(1, std::min(n_rt, std::max(1, sm_count() / n_ct)));
  return launch_pdl(k_conv_fwd_tile, dim3(gx, n_ct), dim3(NTH), S::BYTES, st, a, gx);
}

cudaError_t launch_conv_bwd_tile(const ConvArgs& a, int nparts, cudaStream_t st) {
  typedef ConvSmem<2, BWD_ST> S;
  if (nparts != conv_tile_parts(a.T, a.d)) return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(k_conv_bwd_tile, cudaFuncAttributeMaxDynamicSharedMemorySize, S::BYTES);
  if (e != cudaSuccess) return e;
  const int gx = nparts / BRG, n_ct = (a.d + CW - 1) / CW;
  return launch_pdl(k_conv_bwd_tile, dim3(gx, n_ct), dim3(NTH), S::BYTES, st, a, gx);
}

}  // namespace gbla
