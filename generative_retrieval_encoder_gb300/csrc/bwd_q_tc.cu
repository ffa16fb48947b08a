// Query-side backward of the bf16 layer (Eq. 5-7) on the 5th-generation
// tensor cores, for d_h = 64 with phi(q) stored by the projection epilogue.
//
// Per 128-row tile of one head:
//   (a)  O' = phi(Q) S'                          tcgen05 -> TMEM cols 0..63
//   epilogue 1 (one thread per row and column range; rs and 1/den of each
//   row come from the training forward's readout):
//        o = O'/den + c,  u = o rs,  y = u gamma SiLU(r)   (RMSNorm gate, Eq. 7)
//        dr, dgamma (accumulated in TMEM cols 192..255), du = dy gamma SiLU(r),
//        m = mean(du u), do = rs (du - u m), dn = do / den,
//        dden = -(do . O'/den) / den = -rs (du . o' - m u . o') / den
//   (d)  dq~ = dn S'^T                           tcgen05 -> TMEM cols 64..127
//   (e)  [dS' | dz'] += [dn | dden]^T phi(Q)     tcgen05 -> TMEM cols 128..191
//   epilogue 2: dq = (dq~ + dden z) min(1, phi(q))   (phi' of elu + 1)
//
// Work split: the (128-row tile, head) units, head-major, are cut into one
// contiguous range per CTA (two CTAs per SM), so every SM gets the same number
// of tiles.  A run of units of one (sequence, head) inside a range is a
// segment: its [dS' | dz'] accumulates in TMEM and, at the segment's end,
// leaves as one partial, in slot p + blockIdx.x of the partial array (p =
// h n_seq + b: pairs in unit order, so the slot is unique).  The CTA whose
// partial completes a (sequence, head) sums its partials in slot order (a
// fixed order) and forms dz''; the CTA then loads the next segment's S' and
// goes on.  dgamma accumulates over the whole range.
//
// Nine warps.  Warps 0-7 compute: warp w reads TMEM lanes 32 (w % 4) .. + 31
// (tile rows) and the columns 32 (w / 4) .. + 31, in rounds of 16 columns (18
// warps an SM leave 96 registers a thread).  Warp 8 only issues: the TMA
// copies (two stages ahead) and the MMAs, each group once its inputs are
// complete: (d), (a) of the next tile and (e) once every compute warp has
// written dn, so (a) of the next tile runs under epilogue 2 of this one.  A
// compute warp that issued them would reach the row-sum exchange of the next
// tile last, every tile (an MMA issue takes 100+ cycles under this load), and
// hold up the other seven there.  Operand tiles are
// [128 rows][64 bf16] in the 128-byte swizzle shared by TMA and the MMA
// descriptors; the epilogue writes dn and dden into the dy and r tiles of the
// same stage (each thread owns its row's columns), which then serve as the A
// operand of (d) and (e).
//
// Core form (CORE = true, the core entry point's backward of Eq. 5): q and
// d_o as given, no gate: do = d_o, so
//   dn = d_o / den,   dden = -(d_o . O') / den^2,   den = z . phi(q),
// one pass sums z . phi(q) and d_o . O' over the row (exchanged like the
// layer's sums), a second writes dn.  The stage holds q and d_o (the third
// tile only carries dden for (e)).  phi(q) is written over q in shared memory
// one tile ahead, while the compute warps wait for (d) of the tile before, and
// (a) waits for that rewrite.  No dgamma.
//
// Every mbarrier wait is bounded; after one gives up, the kernel finishes its
// loops without waiting (uniform control flow, so no barrier is left
// waiting), sets the timeout bit of the error word, waits (bounded) for its
// copies and MMAs, frees its TMEM and returns.
#include "core_common.cuh"
#include "pdl.cuh"
#include "kernels.h"
#include "tcgen05.cuh"

namespace gbla {
namespace {

constexpr int QD = 64;               // d_h
constexpr int QT = 128;              // rows per tile (MMA M)
constexpr int TILE = QT * 128;       // [128 rows][64 bf16], 16 KB
constexpr int QST = 2;               // stages
constexpr int STAGE = 3 * TILE;      // phi(Q) | dy -> dn | r -> du, dden
constexpr int LD = state_ld(QD);     // partial / dstate row: 64 dS' + dz' + pad
constexpr int BLD = state_bf_ld(QD);  // bf16 state row

constexpr int O_S = 0;                       // S' [e][f] (8 KB)
constexpr int O_ST = O_S + 8192;             // stages (1024-aligned)
constexpr int O_BAR = O_ST + QST * STAGE;
constexpr int NBAR = 3 * QST + 4;            // full, empty, a_done, dn_ready, d_done, s_ready, phi (core)
constexpr int O_F = O_BAR + 8 * NBAR;        // gamma, centre, z (fp32), row exchange [3][2][128]
constexpr int O_SLOT = O_F + 4 * (3 * QD + 3 * 2 * QT);
constexpr int O_FAIL = O_SLOT + 4;
constexpr int O_LAST = O_FAIL + 4;
constexpr int SMEM = O_LAST + 12 + 1024;     // last-arrival flag, c0, count; alignment slack
constexpr int TMEM_COLS = 256;               // O' | dq~ | dS' | dgamma
static_assert(2 * (SMEM + 1024) <= 233472, "two CTAs per SM");
static_assert(QST == 2, "the issuing thread tracks two stages");
static_assert(QST * STAGE >= (QT + 4) * (QD + 1) * 4, "the stage memory holds the dgamma reduction");

constexpr int EW = 8;                 // compute warps
constexpr int NCT = EW * 32;          // compute threads
constexpr int NTH = NCT + 32;         // + the issuing warp
constexpr int CPT = QD / (EW / 4);    // columns per thread (32)
constexpr int RC = 16;                // columns per round: one 16-column TMEM load
constexpr int NR = CPT / RC;          // rounds
static_assert(NCT == 4 * QD, "the dgamma sum maps threads to (quarter, column)");

__device__ __forceinline__ uint32_t swz_off(int row, int chunk) {
  return (uint32_t)(row * 128 + ((chunk ^ (row & 7)) << 4));
}
__device__ __forceinline__ void unpack8(const uint4& u, float* f) {
  f[0] = bf_lo(u.x); f[1] = bf_hi(u.x); f[2] = bf_lo(u.y); f[3] = bf_hi(u.y);
  f[4] = bf_lo(u.z); f[5] = bf_hi(u.z); f[6] = bf_lo(u.w); f[7] = bf_hi(u.w);
}
// sigmoid(x) = (1 + tanh(x / 2)) / 2 with the hardware tanh approximation
// (relative error about 2^-11, far below the bf16 rounding of the outputs).
__device__ __forceinline__ float sigmoid_fast(float x) {
  float t;
  asm("tanh.approx.f32 %0, %1;" : "=f"(t) : "f"(0.5f * x));
  return fmaf(0.5f, t, 0.5f);
}

// One unit = (128-row tile, head): sub-tile `sub` of tile ti of a.tiles
// (whose tile is a multiple of 128 rows), head h.  u = h (n_tiles spt) + ti spt + sub.
struct QTile {
  int h, b, seqh;        // head, sequence, b H + h (-1: no rows)
  int nrows, nval;       // rows of the sequence slot in the tile, valid rows
  size_t rb;             // first row
};
__device__ __forceinline__ QTile qtile_at(const BwdQArgs& a, int u, int upt, int spt) {
  QTile x;
  x.h = u / upt;
  const int r = u - x.h * upt, ti = r / spt, sub = r - ti * spt;
  int row0, nvalid, tin;
  x.b = 0; x.nrows = 0; x.nval = 0; x.rb = 0; x.seqh = -1;
  if (!map_tile(a.seq, a.tiles, ti, x.b, row0, nvalid, tin)) return x;
  const int R0 = tin * a.tiles.tile + sub * QT;
  x.nrows = max(0, min(QT, slot_rows(a.seq, nvalid) - R0));
  if (x.nrows == 0) return x;
  x.nval = max(0, min(x.nrows, nvalid - R0));
  x.rb = (size_t)row0 + R0;
  x.seqh = x.b * a.H + x.h;
  return x;
}
// The next unit of [u, u1) with rows, from u on; u1 if none.
__device__ __forceinline__ int next_unit(const BwdQArgs& a, int u, int u1, int upt, int spt, QTile& x) {
  for (; u < u1; ++u) {
    x = qtile_at(a, u, upt, spt);
    if (x.seqh >= 0) return u;
  }
  x.seqh = -1;
  return u1;
}
// The CTA whose range [floor(N c / G), floor(N (c + 1) / G)) holds unit u.
__device__ __forceinline__ int cta_of(int u, int n_units, int grid) {
  return (int)((((long long)u + 1) * grid + n_units - 1) / n_units) - 1;
}

__device__ __forceinline__ void tmem_wait16(uint32_t (&r)[16]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
  tmem_tie16(r);
}

template <bool CORE>
__global__ void __launch_bounds__(NTH, 2)
    k_bwd_q_tc(const BwdQArgs a, const __grid_constant__ CUtensorMap tmP, const __grid_constant__ CUtensorMap tmY,
               int roff, int upt, int spt, int n_units) {
  if (threadIdx.x == NCT) {  // the descriptors load while the previous kernel finishes
    tma_prefetch_map(&tmP);
    tma_prefetch_map(&tmY);
  }
  pdl_enter();  // the previous kernel's outputs are visible from here on
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_align1024(smem_raw);
  const uint32_t sbase = smem_u32(smem);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (a.err && *a.err) return;
  const int H = a.H, G = gridDim.x, nseq = a.seq.n_seq;
  const int u0 = (int)(((long long)n_units * blockIdx.x) / G);
  const int u1 = (int)(((long long)n_units * (blockIdx.x + 1)) / G);
  QTile cur;
  int ucur = next_unit(a, u0, u1, upt, spt, cur);
  if (ucur >= u1) {  // no rows in this range: a zero dgamma partial
    if (!CORE)
      for (int f = tid; f < QD; f += NTH) a.gamma_part[(size_t)blockIdx.x * QD + f] = 0.f;
    return;
  }

  float* gam = reinterpret_cast<float*>(smem + O_F);
  float* cen = gam + QD;
  float* zf = cen + QD;
  float* xch = zf + QD;
  uint32_t* slot = reinterpret_cast<uint32_t*>(smem + O_SLOT);
  volatile int* fail = reinterpret_cast<volatile int*>(smem + O_FAIL);
  volatile int* lastf = reinterpret_cast<volatile int*>(smem + O_LAST);
  const uint32_t bar0 = sbase + O_BAR;
  const uint32_t A_DONE = bar0 + 8 * (2 * QST), DN_READY = A_DONE + 8, D_DONE = A_DONE + 16, S_READY = A_DONE + 24;
  auto FULL = [&](int s) { return bar0 + 8 * s; };
  auto PHI = [&](int s) { return bar0 + 8 * (2 * QST + 4 + s); };  // core: phi(q) written over q
  auto EMPTY = [&](int s) { return bar0 + 8 * (QST + s); };
  const bool issuer = tid == NCT;  // lane 0 of warp 8

  // ---------------------------------------------------------- copies (issuer)
  int issued[QST] = {0, 0};  // 1 + index of the last tile loaded into each stage
  int ld_k = 0, ld_u = ucur;  // the next tile to load: its index and unit
  QTile ld_x = cur;
  auto load_next = [&]() {
    const int s = ld_k % QST;
    const uint32_t st = sbase + O_ST + s * STAGE;
    const int y = (int)ld_x.rb;
    mbar_expect_tx(FULL(s), (CORE ? 2 : 3) * TILE);
    tma_load_2d(st, &tmP, FULL(s), ld_x.h * QD, y);
    tma_load_2d(st + TILE, &tmY, FULL(s), ld_x.h * QD, y);
    if (!CORE) tma_load_2d(st + 2 * TILE, &tmP, FULL(s), roff + ld_x.h * QD, y);
    issued[s] = ld_k + 1;
    ++ld_k;
    ld_u = next_unit(a, ld_u + 1, u1, upt, spt, ld_x);
  };
  if (issuer) {  // barriers, then the first two tiles' copies before anything else
    for (int s = 0; s < QST; ++s) {
      mbar_init(FULL(s), 1);
      mbar_init(EMPTY(s), EW + 1);  // (e) commit + one arrival per compute warp
    }
    mbar_init(A_DONE, 1);
    mbar_init(DN_READY, EW);
    mbar_init(D_DONE, 1);
    mbar_init(S_READY, EW);
    if (CORE)
      for (int s = 0; s < QST; ++s) mbar_init(PHI(s), EW);
    mbar_init_fence();
    *fail = 0;
    load_next();
    if (ld_u < u1) load_next();
  }
  // S' of (sequence, head) seqh into its swizzled rows e; fp32 centre and z (compute threads).
  auto load_state = [&](int seqh) {
    const bf16* sbf = a.state_bf + (size_t)seqh * QD * BLD;
    for (int i = tid; i < QD * 8; i += NCT) {
      const int e = i >> 3, c = i & 7;
      *reinterpret_cast<uint4*>(smem + O_S + swz_off(e, c)) = *reinterpret_cast<const uint4*>(sbf + e * BLD + c * 8);
    }
    for (int f = tid; f < QD; f += NCT) {
      cen[f] = a.center ? a.center[(size_t)seqh * QD + f] : 0.f;
      zf[f] = __bfloat162float(sbf[f * BLD + QD]);
    }
    fence_async_smem();
  };
  if (tid < NCT) {
    for (int f = tid; f < QD; f += NCT) gam[f] = a.rms_w ? __bfloat162float(((const bf16*)a.rms_w)[f]) : 1.f;
    load_state(cur.seqh);
  }
  if (warp == 0) tmem_alloc(smem_u32(slot), TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *slot;
  const uint32_t sS = sbase + O_S;

  if (warp == EW) {
    // ======================================================== issuing warp
    if (lane == 0) {
      // (a): K = e.  A = phi(Q) K-major (+32 B per 16 e); B = S' N-major (16 e-rows = 2048 B).
      auto issue_a = [&](int k) {
        if (!mbar_wait(CORE ? PHI(k % QST) : FULL(k % QST), (k / QST) & 1, fail)) return;
        tc_fence_after();
        const uint32_t sq = sbase + O_ST + (k % QST) * STAGE;
        const uint32_t id_a = idesc_bf16(QT, QD, false, true);
#pragma unroll
        for (int kk = 0; kk < QD / 16; ++kk)
          tc_mma(tmem, sdesc(sq + 32 * kk, 16, 1024), sdesc(sS + 2048 * kk, 8192, 1024), id_a, kk > 0);
        tc_commit(A_DONE);
      };
      QTile x = cur;
      int ux = ucur, k = 0, kseg = 0, nsr = 0;  // tile, first tile of its segment, S_READY phases seen
      while (true) {
        QTile nx;
        const int unx = next_unit(a, ux + 1, u1, upt, spt, nx);
        const bool has_next = unx < u1, same = has_next && nx.seqh == x.seqh;
        const int s = k % QST;
        if (k == kseg) {  // a segment's first tile: (a) once its S' is in shared memory
          if (k > 0) {
            mbar_wait(S_READY, nsr & 1, fail);
            ++nsr;
          }
          issue_a(k);
        }
        // (d), (a) of the next tile, (e) once every compute warp has written dn and dden
        if (mbar_wait(DN_READY, k & 1, fail)) {
          tc_fence_after();
          const uint32_t sq = sbase + O_ST + s * STAGE, sy = sq + TILE;
          // (d): K = f.  A = dn (the dy tile) K-major; B = S' K-major (rows e).
          const uint32_t id_d = idesc_bf16(QT, QD, false, false), id_e = idesc_bf16(QT, QD, true, true);
#pragma unroll
          for (int kk = 0; kk < QD / 16; ++kk)
            tc_mma(tmem + 64, sdesc(sy + 32 * kk, 16, 1024), sdesc(sS + 32 * kk, 16, 1024), id_d, kk > 0);
          tc_commit(D_DONE);
          // (a) of the next tile before (e): epilogue 2 and the next pass 1 wait
          // on (d) and (a); (e) only gates the reuse of this stage.  (Core: after
          // (e), since (a) waits for the rewrite of q the compute warps do next.)
          if (same && !CORE) issue_a(k + 1);
          // (e): K = rows.  A = [dn | dden ...] M-major, its two 64-wide halves the
          // dy and r tiles (one tile apart); B = phi(Q) N-major.
#pragma unroll
          for (int kk = 0; kk < QT / 16; ++kk)
            tc_mma(tmem + 128, sdesc(sy + 2048 * kk, TILE, 1024), sdesc(sq + 2048 * kk, 8192, 1024), id_e,
                   (k == kseg && kk == 0) ? 0u : 1u);
          tc_commit(EMPTY(s));
          if (same && CORE) issue_a(k + 1);
        }
        // the tile after next into this stage once it is free
        if (ld_k == k + QST && ld_u < u1 && mbar_wait(EMPTY(s), (k / QST) & 1, fail)) load_next();
        if (!has_next) break;
        if (!same) kseg = k + 1;
        x = nx;
        ux = unx;
        ++k;
      }
      if (*fail)  // let the copies still in flight land
        for (int s = 0; s < QST; ++s)
          if (issued[s] > 0)
            for (uint32_t it = 0; it < kPollLimit && !mbar_try_wait(FULL(s), (uint32_t)((issued[s] - 1) / QST) & 1);
                 ++it) {
            }
    }
    __syncwarp();
  } else {
    // ======================================================== compute warps
    const int q = warp & 3, part = warp >> 2;
    const int i = q * 32 + lane;  // tile row = TMEM lane
    const int f0 = part * CPT;
    const uint32_t tl = tmem + ((uint32_t)(q * 32) << 16);
    // rs and 1/den of this thread's row of a tile (0 on rows outside the sequence: u = dn = 0 there)
    auto rsinv_of = [&](const QTile& x) {
      return (!CORE && i < x.nval) ? __ldg(reinterpret_cast<const float2*>(a.rsinv + 2 * ((x.rb + i) * H + x.h)))
                                   : make_float2(0.f, 0.f);
    };
    // core: phi(q) over q in tile kt's stage, this thread's 32 columns of its row
    auto phi_rows = [&](int kt) {
      const int st = kt % QST;
      mbar_wait(FULL(st), (kt / QST) & 1, fail);
      uint8_t* tq = smem + O_ST + st * STAGE;
#pragma unroll
      for (int ch = 0; ch < CPT / 8; ++ch) {
        uint4* qp = reinterpret_cast<uint4*>(tq + swz_off(i, (f0 >> 3) + ch));
        float v[8];
        unpack8(*qp, v);
        *qp = make_uint4(pack_bf16(phi_f(v[0]), phi_f(v[1])), pack_bf16(phi_f(v[2]), phi_f(v[3])),
                         pack_bf16(phi_f(v[4]), phi_f(v[5])), pack_bf16(phi_f(v[6]), phi_f(v[7])));
      }
      fence_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(PHI(st));
    };
    float2 ri_cur = rsinv_of(cur);
    if (CORE) phi_rows(0);
    int k = 0;
    while (true) {
      QTile nxt;
      const int unxt = next_unit(a, ucur + 1, u1, upt, spt, nxt);
      const bool has_next = unxt < u1, same = has_next && nxt.seqh == cur.seqh;
      const float2 ri_next = has_next ? rsinv_of(nxt) : make_float2(0.f, 0.f);
      const int s = k % QST, h = cur.h;
      uint8_t* sq = smem + O_ST + s * STAGE;
      uint8_t* sy = sq + TILE;
      uint8_t* sr = sy + TILE;
      const bool store = i < cur.nrows;
      const size_t row = cur.rb + i;
      const float rs = ri_cur.x, inv = ri_cur.y;
      mbar_wait(A_DONE, k & 1, fail);
      tc_fence_after();
      float dden;
      if constexpr (CORE) {
        // z . phi(q) and d_o . O' over this thread's columns, in rounds of 16
        float dp = 0.f, D1 = 0.f;
#pragma unroll
        for (int rd = 0; rd < NR; ++rd) {
          const int fr = f0 + RC * rd;
          uint32_t o[RC];
          tmem_ld16(tl + fr, o);
#pragma unroll
          for (int ch = 0; ch < RC / 8; ++ch) {
            const int f = fr + 8 * ch, cc = f >> 3;
            float qv[8], yv[8];
            unpack8(*reinterpret_cast<const uint4*>(sq + swz_off(i, cc)), qv);
            unpack8(*reinterpret_cast<const uint4*>(sy + swz_off(i, cc)), yv);
#pragma unroll
            for (int jj = 0; jj < 8; ++jj) {
              dp = fmaf(qv[jj], zf[f + jj], dp);
              D1 = fmaf(yv[jj], __uint_as_float(o[8 * ch + jj]), D1);
            }
          }
        }
        // the row's two column ranges, added in a fixed order
        xch[(0 + part) * QT + i] = dp;
        xch[(2 + part) * QT + i] = D1;
        named_bar(1, NCT);
        const float den = xch[0 * QT + i] + xch[1 * QT + i];
        const float invd = i < cur.nval ? 1.f / den : 0.f;
        dden = -(xch[2 * QT + i] + xch[3 * QT + i]) * invd * invd;
        // dn = d_o / den -> the dy tile
#pragma unroll
        for (int ch = 0; ch < CPT / 8; ++ch) {
          const int cc = (f0 >> 3) + ch;
          uint4* yp = reinterpret_cast<uint4*>(sy + swz_off(i, cc));
          float yv[8];
          unpack8(*yp, yv);
          *yp = make_uint4(pack_bf16(yv[0] * invd, yv[1] * invd), pack_bf16(yv[2] * invd, yv[3] * invd),
                           pack_bf16(yv[4] * invd, yv[5] * invd), pack_bf16(yv[6] * invd, yv[7] * invd));
        }
        // dden in column 64 of [dn | dden] (first element of the third tile's row)
        if (part == 0) *reinterpret_cast<uint4*>(sr + swz_off(i, 0)) = make_uint4(pack_bf16(dden, 0.f), 0u, 0u, 0u);
      } else {
        // pass 1 in rounds of 16 columns: dr, dgamma, du (into the r tile);
        // sums m = du . u, D1 = du . o', D2 = u . o'.
        float m = 0.f, D1 = 0.f, D2 = 0.f;
  #pragma unroll
        for (int rd = 0; rd < NR; ++rd) {
          const int fr = f0 + RC * rd;
          uint32_t o[RC], g[RC];
          tmem_ld16_async(tl + fr, o);
          if (k > 0) {
            tmem_ld16_async(tl + 192 + fr, g);
            tmem_wait16(o);
            tmem_tie16(g);
          } else {
            tmem_wait16(o);
  #pragma unroll
            for (int j = 0; j < RC; ++j) g[j] = 0u;
          }
  #pragma unroll
          for (int ch = 0; ch < RC / 8; ++ch) {
            const int f = fr + 8 * ch, cc = f >> 3;
            float yv[8], rv[8];
            unpack8(*reinterpret_cast<const uint4*>(sy + swz_off(i, cc)), yv);
            unpack8(*reinterpret_cast<const uint4*>(sr + swz_off(i, cc)), rv);
            uint32_t dup[4], drp[4];
  #pragma unroll
            for (int j = 0; j < 8; j += 2) {
              float du2[2], dr2[2];
  #pragma unroll
              for (int w = 0; w < 2; ++w) {
                const int jj = j + w, kk = 8 * ch + jj;
                const float op = __uint_as_float(o[kk]) * inv;  // centred o'
                const float u = (op + cen[f + jj]) * rs;
                const float r = rv[jj], dy = yv[jj];
                const float sg = sigmoid_fast(r);
                const float av = r * sg;
                const float dyg = dy * gam[f + jj];
                du2[w] = dyg * av;
                g[kk] = __float_as_uint(fmaf(dy * av, u, __uint_as_float(g[kk])));
                dr2[w] = dyg * u * sg * fmaf(r, 1.f - sg, 1.f);
                m = fmaf(du2[w], u, m);
                D1 = fmaf(du2[w], op, D1);
                D2 = fmaf(u, op, D2);
              }
              dup[j / 2] = pack_bf16(du2[0], du2[1]);
              drp[j / 2] = pack_bf16(dr2[0], dr2[1]);
            }
            *reinterpret_cast<uint4*>(sr + swz_off(i, cc)) = make_uint4(dup[0], dup[1], dup[2], dup[3]);
            if (store)
              *reinterpret_cast<uint4*>((bf16*)a.dr + row * a.lddr + (size_t)h * QD + f) =
                  make_uint4(drp[0], drp[1], drp[2], drp[3]);
          }
          tmem_st16(tl + 192 + fr, g);
        }
        // the row's two column ranges, added in a fixed order
        xch[(0 + part) * QT + i] = m;
        xch[(2 + part) * QT + i] = D1;
        xch[(4 + part) * QT + i] = D2;
        named_bar(1, NCT);
        m = xch[0 * QT + i] + xch[1 * QT + i];
        D1 = xch[2 * QT + i] + xch[3 * QT + i];
        D2 = xch[4 * QT + i] + xch[5 * QT + i];
        m *= 1.f / QD;
        dden = -rs * fmaf(-m, D2, D1) * inv;
        // pass 2: dn = rs (du - u m) / den -> the dy tile
  #pragma unroll
        for (int rd = 0; rd < NR; ++rd) {
          const int fr = f0 + RC * rd;
          uint32_t o[RC];
          tmem_ld16(tl + fr, o);  // O' again
  #pragma unroll
          for (int ch = 0; ch < RC / 8; ++ch) {
            const int f = fr + 8 * ch, cc = f >> 3;
            float du[8];
            unpack8(*reinterpret_cast<const uint4*>(sr + swz_off(i, cc)), du);
            uint32_t dn[4];
  #pragma unroll
            for (int j = 0; j < 8; j += 2) {
              float d2[2];
  #pragma unroll
              for (int w = 0; w < 2; ++w) {
                const int jj = j + w;
                const float u = fmaf(__uint_as_float(o[8 * ch + jj]), inv, cen[f + jj]) * rs;
                d2[w] = rs * fmaf(-u, m, du[jj]) * inv;
              }
              dn[j / 2] = pack_bf16(d2[0], d2[1]);
            }
            *reinterpret_cast<uint4*>(sy + swz_off(i, cc)) = make_uint4(dn[0], dn[1], dn[2], dn[3]);
          }
        }
        // dden in column 64 of [dn | dden] (first element of the r tile's row);
        // that chunk's du was consumed above by this row's first column range.
        if (part == 0) *reinterpret_cast<uint4*>(sr + swz_off(i, 0)) = make_uint4(pack_bf16(dden, 0.f), 0u, 0u, 0u);
      }
      if (!CORE) tmem_st_wait();
      fence_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(DN_READY);
      if (CORE && has_next) phi_rows(k + 1);  // q of the next tile, while (d) runs
      // epilogue 2: dq = (dq~ + dden z) min(1, phi(q))
      mbar_wait(D_DONE, k & 1, fail);
      tc_fence_after();
#pragma unroll
      for (int rd = 0; rd < NR; ++rd) {
        const int fr = f0 + RC * rd;
        uint32_t o[RC];
        tmem_ld16(tl + 64 + fr, o);  // dq~
#pragma unroll
        for (int ch = 0; ch < RC / 8; ++ch) {
          const int f = fr + 8 * ch, cc = f >> 3;
          float qv[8];
          unpack8(*reinterpret_cast<const uint4*>(sq + swz_off(i, cc)), qv);
          uint32_t dq[4];
#pragma unroll
          for (int j = 0; j < 8; j += 2)
            dq[j / 2] = pack_bf16(fmaf(dden, zf[f + j], __uint_as_float(o[8 * ch + j])) * fminf(1.f, qv[j]),
                                  fmaf(dden, zf[f + j + 1], __uint_as_float(o[8 * ch + j + 1])) * fminf(1.f, qv[j + 1]));
          if (store)
            *reinterpret_cast<uint4*>((bf16*)a.dq + row * a.lddq + (size_t)h * QD + f) =
                make_uint4(dq[0], dq[1], dq[2], dq[3]);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(EMPTY(s));
      if (!same) {
        // The segment ends with tile k.  Once its stage's EMPTY phase completes,
        // every compute warp is past epilogue 2 and (e), the segment's last MMA,
        // has finished: [dS' | dz'] (TMEM lane f = column f of the state, column
        // 128 + e = row e) leaves as this CTA's partial of the pair.
        mbar_wait(EMPTY(s), (k / QST) & 1, fail);
        tc_fence_after();
        const int b = cur.b, p = h * nseq + b;
        {
          float* P = a.partial + (size_t)(p + blockIdx.x) * QD * LD;
#pragma unroll
          for (int rd = 0; rd < NR; ++rd) {
            uint32_t dsv[RC];
            tmem_ld16(tl + 128 + f0 + RC * rd, dsv);
            if (i < LD)
#pragma unroll
              for (int e = 0; e < RC; ++e)
                P[(size_t)(f0 + RC * rd + e) * LD + i] = i <= QD ? __uint_as_float(dsv[e]) : 0.f;
          }
        }
        tc_fence_before();
        __threadfence();
        named_bar(1, NCT);
        if (tid == 0) {  // the CTAs holding units of (b, h): c0 .. c0 + count - 1
          int first, cnt;
          seq_tiles(a.seq, a.tiles, b, first, cnt);
          const int U0 = h * upt + spt * first;
          int U1 = U0 + spt * cnt - 1;  // the pair's last unit with rows
          while (U1 > U0 && qtile_at(a, U1, upt, spt).seqh < 0) --U1;
          const int c0 = cta_of(U0, n_units, G), count = cta_of(U1, n_units, G) - c0 + 1;
          const bool last = atomicAdd(a.counters + (size_t)b * H + h, 1) == count - 1;
          lastf[0] = (last && !*fail) ? 1 : 0;
          lastf[1] = c0;
          lastf[2] = count;
        }
        named_bar(1, NCT);
        if (lastf[0]) {  // this partial completes (b, h): [dS | dz''] in slot order
          __threadfence();
          combine_state(a.partial, nullptr, p + lastf[1], lastf[2], 1, 0, QD, cur.seqh, false, a.dstate,
                        a.dstate_bf, nullptr, nullptr, nullptr, a.center, nullptr, NCT, 1);
        }
        if (!has_next) break;
        named_bar(1, NCT);  // every compute thread has read lastf
        load_state(nxt.seqh);
        tc_fence_before();
        named_bar(1, NCT);
        if (lane == 0) mbar_arrive(S_READY);  // the issuing warp may start (a) of the new segment
      }
      cur = nxt;
      ucur = unxt;
      ri_cur = ri_next;
      ++k;
    }
    __syncwarp();
  }
  __syncthreads();
  const bool bad = *fail != 0;

  // dgamma: per-lane sums in TMEM, reduced over the 128 lanes in a fixed order
  float* red = reinterpret_cast<float*>(smem + O_ST);  // [128][65]: the stages are free now
  if (!CORE && !bad && tid < NCT) {
    const int q = warp & 3, f0 = (warp >> 2) * CPT, i = q * 32 + lane;
#pragma unroll
    for (int rd = 0; rd < NR; ++rd) {
      uint32_t gv[RC];
      tmem_ld16(tmem + ((uint32_t)(q * 32) << 16) + 192 + f0 + RC * rd, gv);
#pragma unroll
      for (int j = 0; j < RC; ++j) red[i * (QD + 1) + f0 + RC * rd + j] = __uint_as_float(gv[j]);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, TMEM_COLS);
  if (bad) {
    if (tid == 0 && a.err_out) atomicOr(a.err_out, kErrTimeout);
    return;
  }
  if (CORE) return;
  float* red4 = red + QT * (QD + 1);
  if (tid < NCT) {
    const int f = tid & (QD - 1), qr = tid / QD;
    float v = 0.f;
    for (int r = qr * (QT / 4); r < (qr + 1) * (QT / 4); ++r) v += red[r * (QD + 1) + f];
    red4[qr * QD + f] = v;
  }
  __syncthreads();
  if (tid < QD)
    a.gamma_part[(size_t)blockIdx.x * QD + tid] = ((red4[tid] + red4[QD + tid]) + red4[2 * QD + tid]) + red4[3 * QD + tid];
}

}  // namespace

cudaError_t launch_bwd_q_tc(const BwdQArgs& a, int hd, int n_tiles, int* nparts, cudaStream_t st) {
  auto al16 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; };
  const bool core = !a.pre && !a.r && !a.rsinv && !a.rms_w && !a.dr && !a.gamma_part;
  const long long roff = core ? 0 : ((const bf16*)a.r - (const bf16*)a.q);
  if (a.dh != QD || hd % 8 || !al16(a.q) || !al16(a.dy) || !al16(a.dq) || !al16(a.partial) || a.ldq % 8 ||
      a.lddy % 8 || a.lddq % 8 || a.seq.T <= 0 || n_tiles <= 0 || a.tiles.tile % QT)
    return cudaErrorNotSupported;
  if (!core && (!a.pre || !a.rsinv || a.ldr != a.ldq || roff < 0 || roff % 8 || !al16(a.dr) || a.lddr % 8))
    return cudaErrorNotSupported;
  const int spt = a.tiles.tile / QT, upt = n_tiles * spt, n_units = upt * a.H;
  int grid = n_units < 2 * sm_count() ? n_units : 2 * sm_count();  // two CTAs per SM
  const int room = a.partial_slots - a.seq.n_seq * a.H;  // partial slots beyond one per (sequence, head)
  if (room < grid) grid = room;
  if (grid <= 0) return cudaErrorNotSupported;
  CUtensorMap tmP, tmY;
  // 128-byte L2 promotion: a box row is one head's 128 bytes; wider promotion
  // would fetch the neighbouring head's columns, which another CTA reads.
  if (!make_map(&tmP, a.q, (uint64_t)a.ldq, (uint64_t)a.seq.T, (uint64_t)a.ldq, 64, QT, false) ||
      !make_map(&tmY, a.dy, (uint64_t)a.lddy, (uint64_t)a.seq.T, (uint64_t)a.lddy, 64, QT, false))
    return cudaErrorNotSupported;
  auto kern = core ? k_bwd_q_tc<true> : k_bwd_q_tc<false>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, cudaSharedmemCarveoutMaxShared);
  if (e != cudaSuccess) return e;
  *nparts = grid;
  return launch_pdl(kern, dim3(grid), dim3(NTH), SMEM, st, a, tmP, tmY, (int)roff, upt, spt, n_units);
}

}  // namespace gbla
