// The gated core under LION's decay masks, in the bidirectional chunkwise
// form ("Linear Attention for Efficient Bidirectional Sequence Modeling"
// notes: mask construction M = M^F + M^B - I with M^F_ij = prod_{t=j+1..i}
// lambda_t, M^B_ij = prod_{t=i+1..j} lambda_t; the chunkwise parallel form,
// Theorem 3.2, where the whole sequence is available and only the chunk
// states cross chunks), with this layer's feature map phi = elu + 1 and key
// gate ("Gated Bidirectional Linear Attention for Generative Retrieval",
// Eq. 5):
//   o_i = sum_j M_ij g_j (phi(q_i) . phi(k_j)) [v_j | 1] , divided by its last entry.
//
// A sequence is cut into chunks of C = 128 rows (the tiles of `tiles`).  With
// A_i = sum_{t = chunk start .. i} log lambda_t inside chunk c and A_e its
// last row's value:
//   M_ij = exp(-|A_i - A_j|)                               (i, j in chunk c)
//   L^F_c = sum_{j in c} e^{A_e - A_j} g_j phi(k_j) [v_j | 1]^T,
//   L^B_c = sum_{j in c} e^{A_j} g_j phi(k_j) [v_j | 1]^T,   Lambda_c = e^{A_e}
//   H^F_0 = 0,  H^F_{c+1} = Lambda_c H^F_c + L^F_c        (chunks before c)
//   H^B_last = 0, H^B_{c-1} = Lambda_c H^B_c + L^B_c       (chunks after c)
// (phi(K) is formed once per chunk in shared memory; phi(Q) per warp in its
// fragments.)
//   num|den_i = sum_{j in c} M_ij g_j (phi(q_i).phi(k_j)) [v_j | 1]
//             + e^{A_i} phi(q_i)^T H^F_c + e^{A_e - A_i} phi(q_i)^T H^B_c.
// Three kernels: the chunks' local states (k_decay_states), the two scans per
// (sequence, head) (k_decay_scan), the outputs per chunk (k_decay_out).  The
// contractions run on tensor cores (mma.sync m16n8k16, bf16 operands, fp32
// accumulation); the scans and decays in fp32.  The chunk states L and the
// scanned states H pass between the kernels in bf16 (the rounding of the
// tensor-core operands they become).  d_h = 64, bf16 I/O.
#include <algorithm>

#include "common.cuh"
#include "kernels.h"
#include "pdl.cuh"

namespace gbla {
namespace {

constexpr int DD = 64;                  // d_h
constexpr int CC = 128;                 // rows per chunk
constexpr int CPR = DD / 8;             // 16-byte chunks in a row of 64 bf16
constexpr int TBYTES = CC * DD * 2;     // one [128 rows][64] bf16 tile, 16 KB
constexpr int SLD = state_ld(DD);       // chunk-state row (bf16): 64 S + z + pad (72)
constexpr int HLD = DD + 16;            // bf16 scan-state row: 64 S + z + pad (80)
constexpr unsigned FULLM = 0xffffffffu;

__device__ __forceinline__ float phi_dev(float x) { return x > 0.f ? x + 1.f : __expf(x); }
__device__ __forceinline__ uint32_t phi2(uint32_t v) { return pack_bf16(phi_dev(bf_lo(v)), phi_dev(bf_hi(v))); }
__device__ __forceinline__ uint32_t scale2(uint32_t v, float a, float b) {
  return pack_bf16(bf_lo(v) * a, bf_hi(v) * b);
}

// The chunk's rows, validity and the inclusive prefix A of log lambda over its
// valid rows (rows past them: lambda = 1, gate 0), by one 128-thread group
// (threads t < 128 of the CTA).  A lives in shared memory As[128].
struct Chunk {
  int b, nvalid, c0, n_in;  // sequence, its valid rows, first row of the chunk in it, rows of the chunk
  size_t rb;                // first row (global)
};
__device__ __forceinline__ bool chunk_at(const SeqDesc& s, const Tiling& t, int idx, Chunk& c) {
  int row0, tin;
  if (!map_tile(s, t, idx, c.b, row0, c.nvalid, tin)) return false;
  c.c0 = tin * CC;
  c.n_in = max(0, min(CC, c.nvalid - c.c0));
  c.rb = (size_t)row0 + c.c0;
  return true;
}
// Inclusive prefix over the 128 rows of the chunk, 4 warps x 32 (blockDim >= 128).
__device__ __forceinline__ void log_prefix(const float* lam, int64_t ldl, int h, const Chunk& c, float* As,
                                           float* wsum) {
  const int t = threadIdx.x;
  if (t < CC) {
    float x = t < c.n_in ? __logf(fmaxf(__ldg(lam + (c.rb + t) * ldl + h), 1e-30f)) : 0.f;
    const int lane = t & 31, w = t >> 5;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float y = __shfl_up_sync(FULLM, x, o);
      if (lane >= o) x += y;
    }
    if (lane == 31) wsum[w] = x;
    As[t] = x;
  }
  __syncthreads();
  if (t < CC) {
    float add = 0.f;
    for (int w = 0; w < (t >> 5); ++w) add += wsum[w];
    As[t] += add;
  }
  __syncthreads();
}

// cp.async of the chunk's rows of a [rows, ld] bf16 matrix (head h) into a
// swizzled [128][64] tile; rows past n_in are zero.
__device__ __forceinline__ void load_tile(uint32_t dst, const bf16* src, int64_t ld, int h, const Chunk& c) {
  for (int i = threadIdx.x; i < CC * CPR; i += blockDim.x) {
    const int r = i / CPR, ch = i % CPR;
    const bool ok = r < c.n_in;
    cp_async16(dst + swz<CPR>(r, ch), src + (c.rb + (ok ? r : 0)) * ld + (size_t)h * DD + ch * 8, ok ? 16 : 0);
  }
}

// ======================================================================
// k_decay_states: per (chunk, head), L^F and L^B (bf16 [64][72], z in column
// 64) and Lambda_c.  8 warps: warp (wm, kg) owns state rows e in
// [16 wm, 16 wm + 16) and the 16-row key steps kk = kg (mod 2).
// ======================================================================
__global__ void __launch_bounds__(256) k_decay_states(const DecayArgs a) {
  pdl_enter();
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ float As[CC], wF[CC], wB[CC], wsum[4];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (a.err && *a.err) return;
  Chunk c;
  if (!chunk_at(a.seq, a.tiles, blockIdx.x, c)) return;
  const int h = blockIdx.y, H = a.H;
  const uint32_t kb = smem_u32(smem), vb = kb + TBYTES;
  load_tile(kb, (const bf16*)a.k, a.ld, h, c);
  load_tile(vb, (const bf16*)a.v, a.ld, h, c);
  cp_async_commit();
  log_prefix(a.lam, a.ldg, h, c, As, wsum);
  const float Ae = c.n_in > 0 ? As[c.n_in - 1] : 0.f;
  if (tid < CC) {
    const float gj = tid < c.n_in ? __ldg(a.g + (c.rb + tid) * a.ldg + h) : 0.f;
    wF[tid] = gj * __expf(Ae - As[tid]);
    wB[tid] = gj * __expf(As[tid]);
  }
  cp_async_wait<0>();
  __syncthreads();

  const int wm = warp & 3, kg = warp >> 2;
  const int mi = lane >> 3, rr = lane & 7, t4 = lane & 3;
  const uint32_t one = (lane >> 2) == 0 ? 0x3F803F80u : 0u;  // B column of ones -> z
  float accF[9][4], accB[9][4];
#pragma unroll
  for (int n = 0; n < 9; ++n)
#pragma unroll
    for (int u = 0; u < 4; ++u) accF[n][u] = accB[n][u] = 0.f;
#pragma unroll 2
  for (int kk = kg; kk < CC / 16; kk += 2) {
    const int j0 = kk * 16;
    // A = phi(K)^T rows e (16 wm ..), k = rows j of the chunk
    uint32_t k0, k1, k2, k3;
    ldsm_x4_t(kb + swz<CPR>(j0 + ((mi >> 1) << 3) + rr, 2 * wm + (mi & 1)), k0, k1, k2, k3);
    k0 = phi2(k0); k1 = phi2(k1); k2 = phi2(k2); k3 = phi2(k3);
    float f[4], bw[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int j = j0 + 2 * t4 + (u & 1) + ((u >> 1) << 3);
      f[u] = wF[j];
      bw[u] = wB[j];
    }
    const uint32_t aF0 = scale2(k0, f[0], f[1]), aF1 = scale2(k1, f[0], f[1]);
    const uint32_t aF2 = scale2(k2, f[2], f[3]), aF3 = scale2(k3, f[2], f[3]);
    const uint32_t aB0 = scale2(k0, bw[0], bw[1]), aB1 = scale2(k1, bw[0], bw[1]);
    const uint32_t aB2 = scale2(k2, bw[2], bw[3]), aB3 = scale2(k3, bw[2], bw[3]);
#pragma unroll
    for (int np = 0; np < DD / 16; ++np) {
      uint32_t b0, b1, b2, b3;
      ldsm_x4_t(vb + swz<CPR>(j0 + ((mi & 1) << 3) + rr, 2 * np + (mi >> 1)), b0, b1, b2, b3);
      mma_bf16(accF[2 * np], aF0, aF1, aF2, aF3, b0, b1);
      mma_bf16(accF[2 * np + 1], aF0, aF1, aF2, aF3, b2, b3);
      mma_bf16(accB[2 * np], aB0, aB1, aB2, aB3, b0, b1);
      mma_bf16(accB[2 * np + 1], aB0, aB1, aB2, aB3, b2, b3);
    }
    mma_bf16(accF[8], aF0, aF1, aF2, aF3, one, one);
    mma_bf16(accB[8], aB0, aB1, aB2, aB3, one, one);
  }
  // the two key-step groups, summed in a fixed order through shared memory
  __syncthreads();  // the tiles are read
  float* red = reinterpret_cast<float*>(smem);  // [2 dirs][4 wm][9][4][32]
  if (kg == 1) {
#pragma unroll
    for (int n = 0; n < 9; ++n)
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        red[(((0 * 4 + wm) * 9 + n) * 4 + u) * 32 + lane] = accF[n][u];
        red[(((1 * 4 + wm) * 9 + n) * 4 + u) * 32 + lane] = accB[n][u];
      }
  }
  __syncthreads();
  if (kg == 0) {
    const size_t slot = (size_t)blockIdx.x * H + h;
    bf16* PF = a.LF + slot * DD * SLD;
    bf16* PB = a.LB + slot * DD * SLD;
    const int e = wm * 16 + (lane >> 2);
#pragma unroll
    for (int n = 0; n < 9; ++n) {
      float vF[4], vB[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        vF[u] = accF[n][u] + red[(((0 * 4 + wm) * 9 + n) * 4 + u) * 32 + lane];
        vB[u] = accB[n][u] + red[(((1 * 4 + wm) * 9 + n) * 4 + u) * 32 + lane];
      }
      const int f = n * 8 + 2 * t4;  // n = 8: column 64 holds z, 65..71 are zero
      const bool zc = n < 8 || t4 == 0;
      *reinterpret_cast<uint32_t*>(PF + e * SLD + f) = zc ? pack_bf16(vF[0], n < 8 ? vF[1] : 0.f) : 0u;
      *reinterpret_cast<uint32_t*>(PF + (e + 8) * SLD + f) = zc ? pack_bf16(vF[2], n < 8 ? vF[3] : 0.f) : 0u;
      *reinterpret_cast<uint32_t*>(PB + e * SLD + f) = zc ? pack_bf16(vB[0], n < 8 ? vB[1] : 0.f) : 0u;
      *reinterpret_cast<uint32_t*>(PB + (e + 8) * SLD + f) = zc ? pack_bf16(vB[2], n < 8 ? vB[3] : 0.f) : 0u;
    }
    if (tid == 0) a.Lam[slot] = __expf(Ae);
  }
}

// ======================================================================
// k_decay_scan: per (sequence, head), the forward and the backward scan over
// the sequence's chunks; writes the bf16 states H^F_c, H^B_c [64][80] that
// chunk c's outputs read.  Each thread owns the bf16 pairs i, i + 256, ... of
// the [64][72] chunk state (fp32 running sums); the next chunk's L loads under
// the current update.
// ======================================================================
__global__ void __launch_bounds__(256) k_decay_scan(const DecayArgs a) {
  pdl_enter();
  if (a.err && *a.err) return;
  const int b = blockIdx.x, h = blockIdx.y, H = a.H;
  int first, cnt;
  seq_tiles(a.seq, a.tiles, b, first, cnt);
  constexpr int NP = DD * SLD / 2;             // bf16 pairs of a state (SLD is even: no pair straddles a row)
  constexpr int PER = (NP + 255) / 256;        // 9
  for (int dir = 0; dir < 2; ++dir) {
    const uint32_t* L = reinterpret_cast<const uint32_t*>(dir == 0 ? a.LF : a.LB);
    bf16* Hs = dir == 0 ? a.HF : a.HB;
    float st[PER][2];
#pragma unroll
    for (int q = 0; q < PER; ++q) st[q][0] = st[q][1] = 0.f;
    for (int s = 0; s < cnt; ++s) {
      const int cidx = first + (dir == 0 ? s : cnt - 1 - s);
      const size_t slot = (size_t)cidx * H + h;
      uint32_t lv[PER];
#pragma unroll
      for (int q = 0; q < PER; ++q) {
        const int i = threadIdx.x + 256 * q;
        lv[q] = i < NP ? __ldcg(L + slot * NP + i) : 0u;
      }
      const float lam = __ldcg(a.Lam + slot);
      // the state this chunk reads: chunks before it (forward) or after it (backward)
#pragma unroll
      for (int q = 0; q < PER; ++q) {
        const int i = threadIdx.x + 256 * q;
        if (i < NP) {
          const int e = (2 * i) / SLD, f = (2 * i) % SLD;  // f even: columns f, f + 1
          *reinterpret_cast<uint32_t*>(Hs + slot * DD * HLD + (size_t)e * HLD + f) =
              pack_bf16(f <= DD ? st[q][0] : 0.f, f + 1 <= DD ? st[q][1] : 0.f);
          st[q][0] = fmaf(lam, st[q][0], bf_lo(lv[q]));
          st[q][1] = fmaf(lam, st[q][1], bf_hi(lv[q]));
        }
      }
      for (int i = threadIdx.x; i < DD * (HLD - SLD) / 2; i += 256) {
        const int e = i / ((HLD - SLD) / 2), f = SLD + 2 * (i % ((HLD - SLD) / 2));
        *reinterpret_cast<uint32_t*>(Hs + slot * DD * HLD + (size_t)e * HLD + f) = 0u;
      }
    }
  }
}

// ======================================================================
// k_decay_out: per (chunk, head), 8 warps x 16 rows.  Per warp: the decayed
// chunk attention over the keys in two halves of 64 (S = phi(Q) phi(K)^T,
// weights S e^{-|A_i - A_j|} g_j as the A operand of W [V | 1]), then the
// inter-chunk terms e^{A_i} phi(Q) H^F + e^{A_e - A_i} phi(Q) H^B into the
// same accumulator, and o = num / den.
// ======================================================================
constexpr int HST = HLD + 8;             // shared-memory row of a scan state (bf16; 176 B: ldmatrix without bank conflicts)
constexpr int OUT_SMEM = 3 * TBYTES + 2 * DD * HST * 2;
constexpr int STATES_SMEM = 2 * 4 * 9 * 4 * 32 * 4;  // the key-step reduction; >= the two 16 KB tiles
static_assert(STATES_SMEM >= 2 * TBYTES, "the tiles fit the states kernel's shared memory");

__global__ void __launch_bounds__(256, 2) k_decay_out(const DecayArgs a) {
  pdl_enter();
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ float As[CC], gs[CC], wsum[4];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (a.err && *a.err) return;
  Chunk c;
  if (!chunk_at(a.seq, a.tiles, blockIdx.x, c)) return;
  const int h = blockIdx.y, H = a.H;
  const uint32_t qb = smem_u32(smem), kb = qb + TBYTES, vb = kb + TBYTES;
  const uint32_t hf = vb + TBYTES, hbw = hf + DD * HST * 2;
  load_tile(qb, (const bf16*)a.q, a.ld, h, c);
  load_tile(kb, (const bf16*)a.k, a.ld, h, c);
  load_tile(vb, (const bf16*)a.v, a.ld, h, c);
  const size_t slot = (size_t)blockIdx.x * H + h;
  for (int i = tid; i < DD * (HLD / 8); i += 256) {  // the two scan states, rows of 80 bf16 (unswizzled, padded)
    const int e = i / (HLD / 8), ch = i % (HLD / 8);
    cp_async16(hf + (e * HST + ch * 8) * 2, a.HF + slot * DD * HLD + (size_t)e * HLD + ch * 8, 16);
    cp_async16(hbw + (e * HST + ch * 8) * 2, a.HB + slot * DD * HLD + (size_t)e * HLD + ch * 8, 16);
  }
  cp_async_commit();
  log_prefix(a.lam, a.ldg, h, c, As, wsum);
  if (tid < CC) gs[tid] = tid < c.n_in ? __ldg(a.g + (c.rb + tid) * a.ldg + h) : 0.f;
  cp_async_wait<0>();
  __syncthreads();
  if (c.n_in == 0) return;
  // phi(K) once, in place: every warp reads all the keys
  for (int i = tid; i < CC * CPR; i += 256) {
    uint4* p = reinterpret_cast<uint4*>(smem + TBYTES + swz<CPR>(i / CPR, i % CPR));
    const uint4 w = *p;
    *p = make_uint4(phi2(w.x), phi2(w.y), phi2(w.z), phi2(w.w));
  }
  __syncthreads();
  const float Ae = As[c.n_in - 1];

  const int mi = lane >> 3, rr = lane & 7, g8 = lane >> 2, t4 = lane & 3;
  const int r0 = warp * 16;                         // this warp's rows
  const int ia = r0 + g8, ib = ia + 8;              // the two rows of this lane
  const float Aa = As[ia], Ab = As[ib];
  const uint32_t one = g8 == 0 ? 0x3F803F80u : 0u;
  // phi(Q) fragments of the warp's 16 rows, 4 feature steps
  uint32_t qa[4][4];
#pragma unroll
  for (int ks = 0; ks < 4; ++ks) {
    ldsm_x4(qb + swz<CPR>(r0 + ((mi & 1) << 3) + rr, 2 * ks + (mi >> 1)), qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3]);
#pragma unroll
    for (int u = 0; u < 4; ++u) qa[ks][u] = phi2(qa[ks][u]);
  }
  float acc[9][4];
#pragma unroll
  for (int n = 0; n < 9; ++n)
#pragma unroll
    for (int u = 0; u < 4; ++u) acc[n][u] = 0.f;
  for (int half = 0; half < 2; ++half) {
    const int k0 = half * 64;
    if (k0 >= c.n_in) break;
    // S = phi(Q) phi(K)^T over keys k0 .. k0 + 63: 8 n-tiles of 8 keys
    float s[8][4];
#pragma unroll
    for (int n = 0; n < 8; ++n)
#pragma unroll
      for (int u = 0; u < 4; ++u) s[n][u] = 0.f;
#pragma unroll
    for (int ks = 0; ks < 4; ++ks)
#pragma unroll
      for (int np = 0; np < 4; ++np) {
        uint32_t b0, b1, b2, b3;
        ldsm_x4(kb + swz<CPR>(k0 + 16 * np + ((mi >> 1) << 3) + rr, 2 * ks + (mi & 1)), b0, b1, b2, b3);
        mma_bf16(s[2 * np], qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3], b0, b1);
        mma_bf16(s[2 * np + 1], qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3], b2, b3);
      }
    // decayed, gated weights, packed as the A operand of W [V | 1]
    uint32_t wa[4][4];
#pragma unroll
    for (int n = 0; n < 8; ++n) {
      const int j = k0 + 8 * n + 2 * t4;
      const float g0 = gs[j], g1 = gs[j + 1], A0 = As[j], A1 = As[j + 1];
      const float w0 = s[n][0] * g0 * __expf(-fabsf(Aa - A0)), w1 = s[n][1] * g1 * __expf(-fabsf(Aa - A1));
      const float w2 = s[n][2] * g0 * __expf(-fabsf(Ab - A0)), w3 = s[n][3] * g1 * __expf(-fabsf(Ab - A1));
      wa[n >> 1][(n & 1) * 2 + 0] = pack_bf16(w0, w1);
      wa[n >> 1][(n & 1) * 2 + 1] = pack_bf16(w2, w3);
    }
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
      const int j0 = k0 + 16 * kk;
#pragma unroll
      for (int np = 0; np < 4; ++np) {
        uint32_t b0, b1, b2, b3;
        ldsm_x4_t(vb + swz<CPR>(j0 + ((mi & 1) << 3) + rr, 2 * np + (mi >> 1)), b0, b1, b2, b3);
        mma_bf16(acc[2 * np], wa[kk][0], wa[kk][1], wa[kk][2], wa[kk][3], b0, b1);
        mma_bf16(acc[2 * np + 1], wa[kk][0], wa[kk][1], wa[kk][2], wa[kk][3], b2, b3);
      }
      mma_bf16(acc[8], wa[kk][0], wa[kk][1], wa[kk][2], wa[kk][3], one, one);
    }
  }
  // inter-chunk terms: the row-scaled phi(Q) against [S | z] of the scans
  const float sa[2] = {__expf(Aa), __expf(Ae - Aa)}, sb[2] = {__expf(Ab), __expf(Ae - Ab)};
#pragma unroll
  for (int dir = 0; dir < 2; ++dir) {
    const uint32_t hs = dir == 0 ? hf : hbw;
#pragma unroll
    for (int ks = 0; ks < 4; ++ks) {
      const float x = sa[dir], y = sb[dir];
      const uint32_t a0 = scale2(qa[ks][0], x, x), a1 = scale2(qa[ks][1], y, y);
      const uint32_t a2 = scale2(qa[ks][2], x, x), a3 = scale2(qa[ks][3], y, y);
      const int e0 = ks * 16;
#pragma unroll
      for (int np = 0; np < 5; ++np) {  // columns 0 .. 79 of [S | z | 0]: n-tiles 0 .. 8 (9 unused)
        uint32_t b0, b1, b2, b3;
        const int row = e0 + ((mi & 1) << 3) + rr, col = 16 * np + ((mi >> 1) << 3);
        ldsm_x4_t(hs + (row * HST + col) * 2, b0, b1, b2, b3);
        mma_bf16(acc[2 * np], a0, a1, a2, a3, b0, b1);
        if (np < 4) mma_bf16(acc[2 * np + 1], a0, a1, a2, a3, b2, b3);
      }
    }
  }
  // o = num / den (den in column 0 of n-tile 8, held by the t4 == 0 lanes)
  const float dena = __shfl_sync(FULLM, acc[8][0], lane & ~3), denb = __shfl_sync(FULLM, acc[8][2], lane & ~3);
  const bool va = ia < c.n_in, vb2 = ib < c.n_in;
  bf16* o = (bf16*)a.o;
#pragma unroll
  for (int n = 0; n < 8; ++n) {
    const int f = 8 * n + 2 * t4;
    if (va)
      *reinterpret_cast<uint32_t*>(o + (c.rb + ia) * a.ld + (size_t)h * DD + f) = pack_bf16(acc[n][0] / dena, acc[n][1] / dena);
    if (vb2)
      *reinterpret_cast<uint32_t*>(o + (c.rb + ib) * a.ld + (size_t)h * DD + f) = pack_bf16(acc[n][2] / denb, acc[n][3] / denb);
  }
  if (a.den && t4 == 0) {
    if (va) a.den[(c.rb + ia) * a.ldg + h] = dena;
    if (vb2) a.den[(c.rb + ib) * a.ldg + h] = denb;
  }
}

// Zero outputs of rows in no sequence (padding): the chunks never write them.
__global__ void k_decay_pad(const DecayArgs a) {
  const int64_t n = (int64_t)a.seq.T * a.H * DD;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t row = i / (a.H * DD);
    if (a.seq.mode != SEQ_PADDED) return;
    const int b = (int)(row / a.seq.L);
    if (row - (int64_t)b * a.seq.L >= a.seq.lens[b]) {
      ((bf16*)a.o)[row * a.ld + i % (a.H * DD)] = __float2bfloat16_rn(0.f);
      if (a.den && i % DD == 0) a.den[row * a.ldg + (i % (a.H * DD)) / DD] = 0.f;
    }
  }
}

}  // namespace

cudaError_t launch_decay_states(const DecayArgs& a, int n_chunks, cudaStream_t st) {
  if (a.dh != DD) return cudaErrorNotSupported;
  return launch_pdl(k_decay_states, dim3(n_chunks, a.H), dim3(256), STATES_SMEM, st, a);
}

cudaError_t launch_decay_scan(const DecayArgs& a, int n_seq, cudaStream_t st) {
  if (a.dh != DD) return cudaErrorNotSupported;
  return launch_pdl(k_decay_scan, dim3(n_seq, a.H), dim3(256), 0, st, a);
}

cudaError_t launch_decay_out(const DecayArgs& a, int n_chunks, cudaStream_t st) {
  if (a.dh != DD) return cudaErrorNotSupported;
  cudaError_t e = cudaFuncSetAttribute(k_decay_out, cudaFuncAttributeMaxDynamicSharedMemorySize, OUT_SMEM);
  if (e != cudaSuccess) return e;
  e = launch_pdl(k_decay_out, dim3(n_chunks, a.H), dim3(256), OUT_SMEM, st, a);
  if (e != cudaSuccess || a.seq.mode != SEQ_PADDED) return e;
  const long long n = (long long)a.seq.T * a.H * DD;
  k_decay_pad<<<(unsigned)std::min<long long>((n + 255) / 256, 4096), 256, 0, st>>>(a);
  return cudaGetLastError();
}

}  // namespace gbla
