// Readout of the bf16 layer (Eq. 5/6 fused with the RmsNorm gate of Eq. 7) on
// the 5th-generation tensor cores, for d_h = 64 and 128 with phi(q) stored by
// the projection epilogue:
//   o_i = S'^T phi(q_i) / (z . phi(q_i)) + c,   y_i = RmsNorm(o_i) gamma SiLU(r_i)
// (S' the centred state, c its centre; rs and 1/den saved for the backward).
//
// Core form (CORE = true, the core entry point of Eq. 5): q as given, o_i the
// output (no gate), den_i optionally stored.  The ring then holds q alone;
// the epilogue group that owns an MMA tile first rewrites its rows of the
// tile as phi(q) in place (one thread per row, den = z . phi(q) on the way),
// and the MMA waits for that rewrite instead of the copy.  o leaves through
// the same rows of the tile (phi(q) is no longer needed once the MMA is done).
//
// Persistent: one CTA per SM walks a contiguous range of (row tile, head)
// units, head-major, so that consecutive units mostly share a (sequence,
// head) and its state.  Roles:
//   producer warp    lane 0: TMA loads of the 128-row phi(q) and r boxes of
//                    each MMA tile (one box per 64 columns, 128-byte swizzle)
//                    into a ring (6 stages at d_h = 64, 2 at d_h = 128); the
//                    state S' (bf16) into one of two buffers when the
//                    (sequence, head) changes;
//   MMA warp         lane 0: O' = phi(Q) S' (M = 128, N = K = d_h) into the
//                    TMEM accumulator of the tile's epilogue group;
//   epilogue warps   groups of four warps (4 groups at d_h = 64, 2 at 128)
//                    taking MMA tiles in turn; one thread per row: den =
//                    z . phi(q) on the CUDA cores, o and the row's sum of
//                    squares, then y from a second read of the accumulator;
//                    16-byte stores.
// A ring stage is free once the MMA has read phi(q) and the epilogue group has
// read phi(q) and r (its empty barrier counts the MMA commit and four warps).
//
// Every mbarrier wait is bounded; after one gives up, the kernel finishes its
// loops without waiting, sets the timeout bit of the error word, waits
// (bounded) for its copies and MMAs, frees its TMEM and returns.
#include "pdl.cuh"
#include "kernels.h"
#include "tcgen05.cuh"

namespace gbla {
namespace {

constexpr int RT = 128;                  // rows per MMA tile
constexpr int TILE = RT * 128;           // one 64-column atom of a tile: [128 rows][64 bf16], 16 KB

// Shapes and shared-memory layout by head width D (64 or 128) and form.
template <int D, bool CORE>
struct RCfg {
  static constexpr int NH = D / 64;                 // 64-column atoms of a row
  static constexpr int RST = CORE ? (D == 64 ? 8 : 4) : (D == 64 ? 6 : 2);  // ring stages (phi(q) atoms | r atoms)
  static constexpr int NG = D == 64 ? 4 : 2;        // epilogue groups of 4 warps; MMA tile j goes to group j % NG
  static constexpr int STAGE = (CORE ? 1 : 2) * NH * TILE;
  static constexpr int SATOM = D * 128;             // one 64-column atom of S' [e][f]
  static constexpr int SBUF = NH * SATOM;
  static constexpr int EW = 4 * NG;                 // epilogue warps
  static constexpr int NTH = (EW + 2) * 32;
  static constexpr int O_ST = 0;
  static constexpr int O_S = O_ST + RST * STAGE;    // two S' buffers
  static constexpr int O_BAR = O_S + 2 * SBUF;
  // full[RST], empty[RST], sfull[2], sfree[2], accf[NG], acce[NG], drain, phi[RST] (core)
  static constexpr int NBAR = 3 * RST + 4 + 2 * NG + 1;
  static constexpr int O_CZ = O_BAR + 8 * NBAR;     // [group][2 buffers][c | z] fp32, gamma
  static constexpr int O_SLOT = O_CZ + 4 * (NG * 2 * 2 * D + D);
  static constexpr int O_FAIL = O_SLOT + 4;
  static constexpr int SMEM = O_FAIL + 4 + 1024;
  static constexpr int TMEM_COLS = NG * D;          // one D-column accumulator per group
  static_assert(SMEM <= 227 * 1024, "shared memory");
  static_assert(TMEM_COLS <= 512 && (TMEM_COLS & (TMEM_COLS - 1)) == 0, "TMEM allocation");
};

__device__ __forceinline__ uint32_t swz_off(int row, int chunk) {
  return (uint32_t)(row * 128 + ((chunk ^ (row & 7)) << 4));
}
// SiLU(x) = x sigmoid(x) = (x / 2) (1 + tanh(x / 2)), with the hardware tanh
// approximation (relative error about 2^-11, below the bf16 rounding of y).
__device__ __forceinline__ float silu_fast(float x) {
  const float h = 0.5f * x;
  float t;
  asm("tanh.approx.f32 %0, %1;" : "=f"(t) : "f"(h));
  return fmaf(h, t, h);
}
__device__ __forceinline__ void unpack8(const uint4& u, float* f) {
  f[0] = bf_lo(u.x); f[1] = bf_hi(u.x); f[2] = bf_lo(u.y); f[3] = bf_hi(u.y);
  f[4] = bf_lo(u.z); f[5] = bf_hi(u.z); f[6] = bf_lo(u.w); f[7] = bf_hi(u.w);
}

// One unit = (row tile of the readout tiling, head).  Every role decodes the
// same units in the same order.
struct Unit {
  int h, b, seqh, ntl;   // head, sequence, b H + h, MMA tiles (0: skip)
  int nrows, nval;       // rows of the tile's slot, valid rows
  size_t rb;             // first row
};
__device__ __forceinline__ Unit unit_at(const ReadoutArgs& a, int u, int n_units_per_head) {
  Unit x;
  x.h = u / n_units_per_head;
  const int ti = u - x.h * n_units_per_head;
  int row0, nvalid, tin;
  x.ntl = 0; x.b = 0; x.nrows = 0; x.nval = 0; x.rb = 0;
  if (!map_tile(a.seq, a.tiles, ti, x.b, row0, nvalid, tin)) { x.seqh = -1; return x; }
  const int R0 = tin * a.tiles.tile;
  x.nrows = max(0, min(a.tiles.tile, slot_rows(a.seq, nvalid) - R0));
  x.nval = max(0, min(x.nrows, nvalid - R0));
  x.rb = (size_t)row0 + R0;
  x.ntl = (x.nrows + RT - 1) / RT;
  x.seqh = x.b * a.H + x.h;
  return x;
}

template <int D, bool CORE>
__global__ void __launch_bounds__(RCfg<D, CORE>::NTH, 1)
    k_readout_tc(const ReadoutArgs a, const __grid_constant__ CUtensorMap tmP,
                 const __grid_constant__ CUtensorMap tmS, int roff, int n_units_per_head, int n_units) {
  using C = RCfg<D, CORE>;
  constexpr int NH = C::NH, RST = C::RST, NG = C::NG, STAGE = C::STAGE, SBUF = C::SBUF, EW = C::EW,
                NTH = C::NTH, O_ST = C::O_ST, O_S = C::O_S, O_BAR = C::O_BAR, O_CZ = C::O_CZ,
                O_SLOT = C::O_SLOT, O_FAIL = C::O_FAIL, TMEM_COLS = C::TMEM_COLS;
  if (threadIdx.x == 0) {  // the descriptors load while the previous kernel finishes
    tma_prefetch_map(&tmP);
    tma_prefetch_map(&tmS);
  }
  pdl_enter();  // the previous kernel's outputs are visible from here on
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_align1024(smem_raw);
  const uint32_t sbase = smem_u32(smem);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (a.err && *a.err) return;
  // this CTA's contiguous range of units
  const int u0 = (int)(((long long)n_units * blockIdx.x) / gridDim.x);
  const int u1 = (int)(((long long)n_units * (blockIdx.x + 1)) / gridDim.x);

  const uint32_t bar0 = sbase + O_BAR;
  auto FULL = [&](int s) { return bar0 + 8 * s; };
  auto EMPTY = [&](int s) { return bar0 + 8 * (RST + s); };
  auto SFULL = [&](int k) { return bar0 + 8 * (2 * RST + k); };
  auto SFREE = [&](int k) { return bar0 + 8 * (2 * RST + 2 + k); };
  auto ACCF = [&](int g) { return bar0 + 8 * (2 * RST + 4 + g); };
  auto ACCE = [&](int g) { return bar0 + 8 * (2 * RST + 4 + NG + g); };
  const uint32_t DRAIN = bar0 + 8 * (2 * RST + 4 + 2 * NG);
  auto PHI = [&](int s) { return bar0 + 8 * (2 * RST + 4 + 2 * NG + 1 + s); };  // core: phi(q) written
  float* cz = reinterpret_cast<float*>(smem + O_CZ);  // [group][2][c D | z D]
  float* gam = cz + NG * 2 * 2 * D;
  uint32_t* slot = reinterpret_cast<uint32_t*>(smem + O_SLOT);
  volatile int* fail = reinterpret_cast<volatile int*>(smem + O_FAIL);

  if (tid == 0) {
    for (int s = 0; s < RST; ++s) {
      mbar_init(FULL(s), 1);
      mbar_init(EMPTY(s), 1 + 4);  // the MMA commit + the four warps of the tile's group
      if (CORE) mbar_init(PHI(s), 4);  // the four warps of the tile's group
    }
    for (int k = 0; k < 2; ++k) {
      mbar_init(SFULL(k), 1);
      mbar_init(SFREE(k), 1);
    }
    for (int g = 0; g < NG; ++g) {
      mbar_init(ACCF(g), 1);
      mbar_init(ACCE(g), 4);  // the group's four warps
    }
    mbar_init(DRAIN, 1);
    mbar_init_fence();
    *fail = 0;
  }
  for (int f = tid; f < D; f += NTH) gam[f] = a.rms_w ? __bfloat162float(((const bf16*)a.rms_w)[f]) : 1.f;
  if (warp == EW + 1) tmem_alloc(smem_u32(slot), TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *slot;

  if (warp == EW) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int j = 0, k = -1, prev = -1;  // MMA tiles issued, state buffers used
      int last_s[RST];
#pragma unroll
      for (int s = 0; s < RST; ++s) last_s[s] = 0;
      for (int u = u0; u < u1 && !*fail; ++u) {
        const Unit x = unit_at(a, u, n_units_per_head);
        if (x.ntl == 0) continue;
        if (x.seqh != prev) {  // the state of a new (sequence, head)
          ++k;
          prev = x.seqh;
          const int pb = k & 1;
          if (k >= 2 && !mbar_wait(SFREE(pb), ((k >> 1) - 1) & 1, fail)) break;
          mbar_expect_tx(SFULL(pb), SBUF);
#pragma unroll
          for (int hf = 0; hf < NH; ++hf)
            tma_load_2d(sbase + O_S + pb * SBUF + hf * C::SATOM, &tmS, SFULL(pb), 64 * hf, x.seqh * D);
        }
        bool ok = true;
        for (int t = 0; t < x.ntl; ++t, ++j) {
          const int s = j % RST;
          if (j >= RST && !mbar_wait(EMPTY(s), ((j / RST) - 1) & 1, fail)) { ok = false; break; }
          const uint32_t st = sbase + O_ST + s * STAGE;
          const int y = (int)x.rb + t * RT;
          mbar_expect_tx(FULL(s), STAGE);
#pragma unroll
          for (int hf = 0; hf < NH; ++hf) {
            tma_load_2d(st + hf * TILE, &tmP, FULL(s), x.h * D + 64 * hf, y);
            if (!CORE) tma_load_2d(st + (NH + hf) * TILE, &tmP, FULL(s), roff + x.h * D + 64 * hf, y);
          }
          last_s[s] = j + 1;
        }
        if (!ok) break;
      }
      if (*fail)  // let the copies still in flight land
        for (int s = 0; s < RST; ++s)
          if (last_s[s] > 0)
            for (uint32_t it = 0; it < kPollLimit && !mbar_try_wait(FULL(s), (uint32_t)((last_s[s] - 1) / RST) & 1);
                 ++it) {
            }
    }
  } else if (warp == EW + 1) {
    // ---------------------------------------------------------- MMA issuer
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16(RT, D, false, true);
      int j = 0, k = -1, prev = -1;
      for (int u = u0; u < u1 && !*fail; ++u) {
        const Unit x = unit_at(a, u, n_units_per_head);
        if (x.ntl == 0) continue;
        if (x.seqh != prev) {
          if (k >= 0) tc_commit(SFREE(k & 1));  // the previous state's MMAs are all issued
          ++k;
          prev = x.seqh;
          if (!mbar_wait(SFULL(k & 1), (k >> 1) & 1, fail)) break;
        }
        const uint32_t sS = sbase + O_S + (k & 1) * SBUF;
        bool ok = true;
        for (int t = 0; t < x.ntl; ++t, ++j) {
          const int s = j % RST, ab = j % NG;
          if (!mbar_wait(CORE ? PHI(s) : FULL(s), (j / RST) & 1, fail)) { ok = false; break; }
          if (j >= NG && !mbar_wait(ACCE(ab), ((j / NG) - 1) & 1, fail)) { ok = false; break; }
          tc_fence_after();
          const uint32_t sq = sbase + O_ST + s * STAGE;
          // K = e.  A = phi(Q) K-major (atom kk / 4, +32 B per 16 e inside it);
          // B = S' N-major (16 e-rows = 2048 B; its 64-column atoms SATOM apart).
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk)
            tc_mma(tmem + ab * D, sdesc(sq + (kk >> 2) * TILE + 32 * (kk & 3), 16, 1024),
                   sdesc(sS + 2048 * kk, C::SATOM, 1024), idesc, kk > 0);
          tc_commit(ACCF(ab));
          tc_commit(EMPTY(s));
        }
        if (!ok) break;
      }
      if (k >= 0) tc_commit(SFREE(k & 1));
      tc_commit(DRAIN);  // completes once every MMA issued above has finished
      for (uint32_t it = 0; it < kPollLimit && !mbar_try_wait(DRAIN, 0); ++it) {
      }
    }
  } else {
    // ----------------------------------------------------------- epilogue
    const int grp = warp >> 2, wq = warp & 3;  // group, TMEM lane quarter
    const int i = wq * 32 + lane;              // tile row = TMEM lane
    const uint32_t tl = tmem + ((uint32_t)(wq * 32) << 16) + grp * D;
    bf16* out = (bf16*)a.out;
    float* czg = cz + grp * 2 * 2 * D;
    int j = 0, k = -1, prev = -1;
    for (int u = u0; u < u1; ++u) {
      const Unit x = unit_at(a, u, n_units_per_head);
      if (x.ntl == 0) continue;
      if (x.seqh != prev) {  // centre and z of the new (sequence, head), per group
        ++k;
        prev = x.seqh;
        // the buffer replaced here served the state before the previous one:
        // every thread of the group passed the barrier below for the previous
        // state, so none still reads it
        float* czb = czg + (k & 1) * 2 * D;
        for (int idx = i; idx < 2 * D; idx += 128) {
          const int e = idx & (D - 1);
          if (idx < D) czb[e] = a.center ? a.center[(size_t)x.seqh * D + e] : 0.f;
          else czb[D + e] = __bfloat162float(a.state_bf[((size_t)x.seqh * D + e) * state_bf_ld(D) + D]);
        }
        named_bar(1 + grp, 128);
      }
      const float* cb = czg + (k & 1) * 2 * D;
      const float* zb = cb + D;
      for (int t = 0; t < x.ntl; ++t, ++j) {
        if (j % NG != grp) continue;  // another group's tile
        const int s = j % RST;
        const uint8_t* sq = smem + O_ST + s * STAGE;
        uint8_t* sr = smem + O_ST + s * STAGE + NH * TILE;
        const int rel = t * RT + i;
        const bool valid = rel < x.nval, store = rel < x.nrows;
        if (CORE) {
          // phi(q) in place over this group's copy of q, den = z . phi(q) on the way
          mbar_wait(FULL(s), (j / RST) & 1, fail);
          float den = 0.f;
          uint8_t* sqw = smem + O_ST + s * STAGE;
#pragma unroll
          for (int c = 0; c < 8 * NH; ++c) {
            uint4* qp = reinterpret_cast<uint4*>(sqw + (c >> 3) * TILE + swz_off(i, c & 7));
            float qv[8];
            unpack8(*qp, qv);
            uint32_t w[4];
#pragma unroll
            for (int jj = 0; jj < 8; jj += 2) {
              const float p0 = phi_f(qv[jj]), p1 = phi_f(qv[jj + 1]);
              const uint32_t pk = pack_bf16(p0, p1);
              // den from the bf16 values the MMA multiplies with
              den = fmaf(bf_lo(pk), zb[8 * c + jj], den);
              den = fmaf(bf_hi(pk), zb[8 * c + jj + 1], den);
              w[jj / 2] = pk;
            }
            *qp = make_uint4(w[0], w[1], w[2], w[3]);
          }
          fence_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(PHI(s));
          const float inv = valid ? 1.f / den : 0.f;
          const float cv = valid ? 1.f : 0.f;
          mbar_wait(ACCF(grp), (j / NG) & 1, fail);
          tc_fence_after();
          // o = O'/den + c over phi(q) of this row, 32 columns at a time
#pragma unroll
          for (int hh = 0; hh < D / 32; ++hh) {
            uint32_t o[32];
            tmem_ld32(tl + 32 * hh, o);
            if (hh == D / 32 - 1) {  // the accumulator is read: hand it back
              tc_fence_before();
              __syncwarp();
              if (lane == 0) mbar_arrive(ACCE(grp));
            }
#pragma unroll
            for (int c = 0; c < 4; ++c) {
              const int cc = 4 * hh + c;
              uint32_t w[4];
#pragma unroll
              for (int jj = 0; jj < 8; jj += 2) {
                const int F = 8 * cc + jj;
                w[jj / 2] = pack_bf16(fmaf(__uint_as_float(o[8 * c + jj]), inv, cv * cb[F]),
                                      fmaf(__uint_as_float(o[8 * c + jj + 1]), inv, cv * cb[F + 1]));
              }
              *reinterpret_cast<uint4*>(sqw + (cc >> 3) * TILE + swz_off(i, cc & 7)) = make_uint4(w[0], w[1], w[2], w[3]);
            }
          }
          __syncwarp();
          {
            const int ch = lane & 7;
#pragma unroll
            for (int hf = 0; hf < NH; ++hf)
#pragma unroll
              for (int it = 0; it < 8; ++it) {
                const int rr = wq * 32 + 4 * it + (lane >> 3), rl = t * RT + rr;
                const uint4 v = *reinterpret_cast<const uint4*>(sqw + hf * TILE + swz_off(rr, ch));
                if (rl < x.nrows)
                  *reinterpret_cast<uint4*>(out + (x.rb + rl) * a.ldo + (size_t)x.h * D + 64 * hf + 8 * ch) = v;
              }
          }
          if (a.den && store) a.den[(x.rb + rel) * a.H + x.h] = valid ? den : 0.f;
          __syncwarp();
          if (lane == 0) mbar_arrive(EMPTY(s));
          continue;
        }
        mbar_wait(ACCF(grp), (j / NG) & 1, fail);
        tc_fence_after();
        // O' columns 0..31 load under den = z . phi(q) (the row's phi(q) in shared memory)
        uint32_t ob[2][32];
        tmem_ld32_async(tl, ob[0]);
        float den = 0.f;
#pragma unroll
        for (int c = 0; c < 8 * NH; ++c) {
          float qv[8];
          unpack8(*reinterpret_cast<const uint4*>(sq + (c >> 3) * TILE + swz_off(i, c & 7)), qv);
#pragma unroll
          for (int jj = 0; jj < 8; ++jj) den = fmaf(qv[jj], zb[8 * c + jj], den);
        }
        const float inv = valid ? 1.f / den : 0.f;
        const float cv = valid ? 1.f : 0.f;
        // o = O'/den + c and its sum of squares, 32 columns at a time, the next
        // 32 loading under the current ones
        float ss = 0.f;
#pragma unroll
        for (int q = 0; q < D / 32; ++q) {
          tmem_wait32(ob[q & 1]);
          if (q + 1 < D / 32) tmem_ld32_async(tl + 32 * (q + 1), ob[(q + 1) & 1]);
#pragma unroll
          for (int f = 0; f < 32; ++f) {
            const float v = fmaf(__uint_as_float(ob[q & 1][f]), inv, cv * cb[32 * q + f]);
            ss = fmaf(v, v, ss);
          }
        }
        const float rs = rsqrtf(ss * (1.f / D) + a.eps);
        // y = RMSNorm(o) * gamma * SiLU(r); O' is read again, 32 columns at a time
#pragma unroll
        for (int hh = 0; hh < D / 32; ++hh) {
          uint32_t o[32];
          tmem_ld32(tl + 32 * hh, o);
          if (hh == D / 32 - 1) {  // the accumulator is read: hand it back
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(ACCE(grp));
          }
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            const int cc = 4 * hh + c;  // 8-column chunk of the row
            uint8_t* rp = sr + (cc >> 3) * TILE + swz_off(i, cc & 7);
            float rv[8];
            unpack8(*reinterpret_cast<const uint4*>(rp), rv);
            uint32_t w[4];
#pragma unroll
            for (int jj = 0; jj < 8; jj += 2) {
              const int f = 8 * c + jj, F = 32 * hh + f;
              const float v0 = fmaf(__uint_as_float(o[f]), inv, cv * cb[F]);
              const float v1 = fmaf(__uint_as_float(o[f + 1]), inv, cv * cb[F + 1]);
              const float r0 = rv[jj], r1 = rv[jj + 1];
              const float y0 = v0 * rs * gam[F] * silu_fast(r0);
              const float y1 = v1 * rs * gam[F + 1] * silu_fast(r1);
              w[jj / 2] = pack_bf16(y0, y1);
            }
            // y over the r chunk just read (this lane's own row)
            *reinterpret_cast<uint4*>(rp) = make_uint4(w[0], w[1], w[2], w[3]);
          }
        }
        // the warp's 32 rows of y leave as whole 128-byte lines: eight lanes per line
        __syncwarp();
        {
          const int ch = lane & 7;
#pragma unroll
          for (int hf = 0; hf < NH; ++hf)
#pragma unroll
            for (int it = 0; it < 8; ++it) {
              const int rr = wq * 32 + 4 * it + (lane >> 3), rl = t * RT + rr;
              const uint4 v = *reinterpret_cast<const uint4*>(sr + hf * TILE + swz_off(rr, ch));
              if (rl < x.nrows)
                *reinterpret_cast<uint4*>(out + (x.rb + rl) * a.ldo + (size_t)x.h * D + 64 * hf + 8 * ch) = v;
            }
        }
        if (a.rsinv && store)
          *reinterpret_cast<float2*>(a.rsinv + 2 * ((x.rb + rel) * a.H + x.h)) = make_float2(valid ? rs : 0.f, inv);
        __syncwarp();
        if (lane == 0) mbar_arrive(EMPTY(s));
      }
    }
  }
  __syncwarp();  // single-lane roles rejoin their warps: the CTA barrier below is warp-aligned
  __syncthreads();
  const bool bad = *fail != 0;
  tc_fence_before();
  __syncthreads();
  if (warp == EW + 1) tmem_dealloc(tmem, TMEM_COLS);
  if (bad && tid == 0 && a.err_out) atomicOr(a.err_out, kErrTimeout);
}

template <int D, bool CORE>
cudaError_t launch_readout_tc_d(const ReadoutArgs& a, int n_tiles, long long roff, cudaStream_t st) {
  using C = RCfg<D, CORE>;
  CUtensorMap tmP, tmS;
  if (!make_map(&tmP, a.q, (uint64_t)a.ldq, (uint64_t)a.seq.T, (uint64_t)a.ldq, 64, RT, false) ||
      !make_map(&tmS, a.state_bf, (uint64_t)state_bf_ld(D), (uint64_t)a.seq.n_seq * a.H * D,
                (uint64_t)state_bf_ld(D), 64, D, false))
    return cudaErrorNotSupported;
  cudaError_t e = cudaFuncSetAttribute(k_readout_tc<D, CORE>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
  if (e != cudaSuccess) return e;
  const int n_units = n_tiles * a.H;
  const int grid = n_units < sm_count() ? n_units : sm_count();
  return launch_pdl(k_readout_tc<D, CORE>, dim3(grid), dim3(C::NTH), C::SMEM, st, a, tmP, tmS, (int)roff, n_tiles, n_units);
}

}  // namespace

cudaError_t launch_readout_tc(const ReadoutArgs& a, int n_tiles, cudaStream_t st) {
  auto al16 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; };
  const long long roff = ((const bf16*)a.r - (const bf16*)a.q);
  if ((a.dh != 64 && a.dh != 128) || !a.pre || a.ldr != a.ldq || roff < 0 || roff % 8 || !al16(a.q) ||
      !al16(a.out) || !al16(a.state_bf) || a.ldq % 8 || a.ldo % 8 || a.seq.T <= 0 || n_tiles <= 0 || a.den)
    return cudaErrorNotSupported;
  return a.dh == 64 ? launch_readout_tc_d<64, false>(a, n_tiles, roff, st)
                    : launch_readout_tc_d<128, false>(a, n_tiles, roff, st);
}

cudaError_t launch_readout_core_tc(const ReadoutArgs& a, int n_tiles, cudaStream_t st) {
  auto al16 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; };
  if ((a.dh != 64 && a.dh != 128) || a.pre || a.r || !al16(a.q) || !al16(a.out) || !al16(a.state_bf) ||
      a.ldq % 8 || a.ldo % 8 || a.seq.T <= 0 || n_tiles <= 0 || a.tiles.tile % RT)
    return cudaErrorNotSupported;
  return a.dh == 64 ? launch_readout_tc_d<64, true>(a, n_tiles, 0, st)
                    : launch_readout_tc_d<128, true>(a, n_tiles, 0, st);
}

}  // namespace gbla
