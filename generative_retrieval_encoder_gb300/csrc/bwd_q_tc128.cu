// Query-side backward of the bf16 layer (Eq. 5-7) on the 5th-generation
// tensor cores, for d_h = 128 with phi(q) stored by the projection epilogue.
// The arithmetic is that of the d_h = 64 kernel (bwd_q_tc.cu); per 128-row
// tile of one head:
//   (a)  O' = phi(Q) S'                           tcgen05 -> TMEM cols 0..127
//   epilogue 1: the RMSNorm-gate backward (Eq. 7) row by row: dr, dgamma
//        (accumulated in TMEM cols 272..399), du = dy gamma SiLU(r),
//        m = mean(du u), dn = rs (du - u m) / den,
//        dden = -rs (du . O' - m u . O') / den^2
//   (d)  dq~ = dn S'^T                            tcgen05 -> TMEM cols 0..127 (O' is read by then)
//   (e)  [dS' | dz'] += phi(Q)^T [dn | dden]      tcgen05 -> TMEM cols 128..271
//   epilogue 2: dq = (dq~ + dden z) min(1, phi(q))
// (e) takes phi(Q) as the M-major A operand (M = the 128 state rows) and
// [dn | dden] as the N-major B operand with N = 144: its three 64-column
// atoms are the two atoms of the dy tile (dn) and the first atom of the r
// tile, whose column 0 holds dden; so TMEM lane e holds row e of dS' in
// columns 128..255 and dz'_e in column 256.
//
// Work split as in the d_h = 64 kernel: contiguous ranges of (128-row tile,
// head) units, one CTA per SM (the shared memory holds two 96 KB stages and
// the 32 KB state); runs of one (sequence, head) leave [dS' | dz'] as a
// partial in slot h n_seq + b + CTA, and the CTA completing a (sequence, head)
// combines its partials in slot order.  Sixteen warps: warp w reads TMEM
// lanes 32 (w % 4) .. + 31 (tile rows) and owns the 32 columns 32 (w / 4) ..
// + 31 of its row (half a swizzle atom); the four owners of a row exchange
// their row sums through TMEM columns 400..415.  Thread 0 issues the copies
// and the MMAs.  O' and dq~ share TMEM columns, so (a) of the next tile is
// issued once every warp has finished epilogue 2.
//
// Every mbarrier wait is bounded; after one gives up, the kernel finishes its
// loops without waiting, sets the timeout bit of the error word, waits
// (bounded) for its copies and MMAs, frees its TMEM and returns.
#include "core_common.cuh"
#include "pdl.cuh"
#include "kernels.h"
#include "tcgen05.cuh"

namespace gbla {
namespace {

constexpr int QD = 128;              // d_h
constexpr int QT = 128;              // rows per tile (MMA M)
constexpr int ATOM = QT * 128;       // one 64-column atom of a tile, 16 KB
constexpr int TILE = 2 * ATOM;       // [128 rows][128 bf16]
constexpr int QST = 2;               // stages
constexpr int STAGE = 3 * TILE;      // phi(Q) | dy -> dn | r -> du, dden
constexpr int SATOM = QD * 128;      // one 64-column atom of S' [e][f], 16 KB
constexpr int LD = state_ld(QD);     // partial / dstate row: 128 dS' + dz' + pad
constexpr int BLD = state_bf_ld(QD);  // bf16 state row

constexpr int O_S = 0;                       // S' (two atoms, 32 KB)
constexpr int O_ST = O_S + 2 * SATOM;        // stages (1024-aligned)
constexpr int O_BAR = O_ST + QST * STAGE;
constexpr int NBAR = 2 * QST + 4;            // full, empty, a_done, dn_ready, d_done, seg
constexpr int O_F = O_BAR + 8 * NBAR;        // gamma, centre, z (fp32)
constexpr int O_SLOT = O_F + 4 * 3 * QD;
constexpr int O_FAIL = O_SLOT + 4;
constexpr int O_LAST = O_FAIL + 4;
constexpr int SMEM = O_LAST + 12 + 1024;     // last-arrival flag, c0, count; alignment slack
constexpr int TMEM_COLS = 512;
constexpr int C_DS = 128, C_DG = 272, C_X = 400;  // TMEM columns: [dS' | dz'], dgamma, row-sum exchange (16)
static_assert(SMEM <= 227 * 1024, "shared memory");
static_assert(QST * STAGE >= QT * (QD + 1) * 4, "the stage memory holds the dgamma reduction");
static_assert(O_F % 16 == 0, "float4 reads of gamma, centre and z");

constexpr int EW = 16;                // warps
constexpr int NTH = EW * 32;
constexpr int NPART = EW / 4;         // owners of a row
constexpr int CPT = QD / NPART;       // columns per thread (32)
static_assert(CPT == 32, "a thread holds one 32-column TMEM load");

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
__device__ __forceinline__ void tmem_st4(uint32_t taddr, float a, float b, float c, float d) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x4.b32 [%0], {%1,%2,%3,%4};" ::"r"(taddr), "r"(__float_as_uint(a)),
               "r"(__float_as_uint(b)), "r"(__float_as_uint(c)), "r"(__float_as_uint(d))
               : "memory");
}

// One unit = (128-row tile, head): sub-tile `sub` of tile ti of a.tiles,
// head h.  u = h (n_tiles spt) + ti spt + sub.
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
__device__ __forceinline__ int next_unit(const BwdQArgs& a, int u, int u1, int upt, int spt, QTile& x) {
  for (; u < u1; ++u) {
    x = qtile_at(a, u, upt, spt);
    if (x.seqh >= 0) return u;
  }
  x.seqh = -1;
  return u1;
}
__device__ __forceinline__ int cta_of(int u, int n_units, int grid) {
  return (int)((((long long)u + 1) * grid + n_units - 1) / n_units) - 1;
}

__global__ void __launch_bounds__(NTH, 1)
    k_bwd_q_tc128(const BwdQArgs a, const __grid_constant__ CUtensorMap tmP, const __grid_constant__ CUtensorMap tmY,
                  int roff, int upt, int spt, int n_units) {
  if (threadIdx.x == 0) {  // the descriptors load while the previous kernel finishes
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
    for (int f = tid; f < QD; f += NTH) a.gamma_part[(size_t)blockIdx.x * QD + f] = 0.f;
    return;
  }

  float* gam = reinterpret_cast<float*>(smem + O_F);
  float* cen = gam + QD;
  float* zf = cen + QD;
  uint32_t* slot = reinterpret_cast<uint32_t*>(smem + O_SLOT);
  volatile int* fail = reinterpret_cast<volatile int*>(smem + O_FAIL);
  volatile int* lastf = reinterpret_cast<volatile int*>(smem + O_LAST);
  const uint32_t bar0 = sbase + O_BAR;
  const uint32_t A_DONE = bar0 + 8 * (2 * QST), DN_READY = A_DONE + 8, D_DONE = A_DONE + 16, SEG = A_DONE + 24;
  auto FULL = [&](int s) { return bar0 + 8 * s; };
  auto EMPTY = [&](int s) { return bar0 + 8 * (QST + s); };

  // ---------------------------------------------------------- thread 0: copies and MMAs
  const bool leader = tid == 0;
  int issued[QST] = {0, 0};  // 1 + index of the last tile loaded into each stage
  int ld_k = 0, ld_u = ucur;
  QTile ld_x = cur;
  auto load_next = [&]() {
    const int s = ld_k % QST;
    const uint32_t st = sbase + O_ST + s * STAGE;
    const int y = (int)ld_x.rb;
    mbar_expect_tx(FULL(s), 3 * TILE);
#pragma unroll
    for (int hf = 0; hf < 2; ++hf) {
      tma_load_2d(st + hf * ATOM, &tmP, FULL(s), ld_x.h * QD + 64 * hf, y);
      tma_load_2d(st + TILE + hf * ATOM, &tmY, FULL(s), ld_x.h * QD + 64 * hf, y);
      tma_load_2d(st + 2 * TILE + hf * ATOM, &tmP, FULL(s), roff + ld_x.h * QD + 64 * hf, y);
    }
    issued[s] = ld_k + 1;
    ++ld_k;
    ld_u = next_unit(a, ld_u + 1, u1, upt, spt, ld_x);
  };
  if (leader) {
    for (int s = 0; s < QST; ++s) {
      mbar_init(FULL(s), 1);
      mbar_init(EMPTY(s), EW + 1);  // (e) commit + one arrival per warp
    }
    mbar_init(A_DONE, 1);
    mbar_init(DN_READY, EW);
    mbar_init(D_DONE, 1);
    mbar_init(SEG, 1);
    mbar_init_fence();
    *fail = 0;
    load_next();
    if (ld_u < u1) load_next();
  }
  // S' of (sequence, head) seqh into its two swizzled atoms; fp32 centre and z.
  auto load_state = [&](int seqh) {
    const bf16* sbf = a.state_bf + (size_t)seqh * QD * BLD;
    for (int i = tid; i < QD * 16; i += NTH) {
      const int e = i >> 4, c = i & 15;
      *reinterpret_cast<uint4*>(smem + O_S + (c >> 3) * SATOM + swz_off(e, c & 7)) =
          *reinterpret_cast<const uint4*>(sbf + e * BLD + c * 8);
    }
    for (int f = tid; f < QD; f += NTH) {
      cen[f] = a.center ? a.center[(size_t)seqh * QD + f] : 0.f;
      zf[f] = __bfloat162float(sbf[f * BLD + QD]);
    }
    fence_async_smem();
  };
  for (int f = tid; f < QD; f += NTH) gam[f] = a.rms_w ? __bfloat162float(((const bf16*)a.rms_w)[f]) : 1.f;
  load_state(cur.seqh);
  if (warp == 0) tmem_alloc(smem_u32(slot), TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *slot;

  const int q = warp & 3, part = warp >> 2;
  const int i = q * 32 + lane;  // tile row = TMEM lane
  const int f0 = part * CPT;    // this thread's columns: half of atom part / 2 of each tile
  const int c0 = (part & 1) * 4;  // its first 8-column chunk inside that atom
  const uint32_t tl = tmem + ((uint32_t)(q * 32) << 16);
  {  // dgamma starts at zero
    uint32_t zero[32];
#pragma unroll
    for (int j = 0; j < 32; ++j) zero[j] = 0u;
    tmem_st32(tl + C_DG + f0, zero);
    tmem_st_wait();
  }

  const uint32_t sS = sbase + O_S;
  // (a): K = e.  A = phi(Q) K-major (atom kk / 4); B = S' N-major (atoms SATOM apart).
  auto issue_a = [&](int k) {
    if (!mbar_wait(FULL(k % QST), (k / QST) & 1, fail)) return;
    tc_fence_after();
    const uint32_t sq = sbase + O_ST + (k % QST) * STAGE;
    const uint32_t id_a = idesc_bf16(QT, QD, false, true);
#pragma unroll
    for (int kk = 0; kk < QD / 16; ++kk)
      tc_mma(tmem, sdesc(sq + (kk >> 2) * ATOM + 32 * (kk & 3), 16, 1024), sdesc(sS + 2048 * kk, SATOM, 1024), id_a,
             kk > 0);
    tc_commit(A_DONE);
  };
  // (d) and (e) of tile k, once every warp has written dn and dden.  first: k opens its segment.
  auto issue_de = [&](int k, bool first) {
    const int s = k % QST;
    const uint32_t sq = sbase + O_ST + s * STAGE, sy = sq + TILE;
    if (!mbar_wait(DN_READY, k & 1, fail)) return;
    tc_fence_after();
    // (d): K = f.  A = dn (the dy tile) K-major; B = S' K-major (rows e).
    const uint32_t id_d = idesc_bf16(QT, QD, false, false), id_e = idesc_bf16(QT, QD + 16, true, true);
#pragma unroll
    for (int kk = 0; kk < QD / 16; ++kk)
      tc_mma(tmem, sdesc(sy + (kk >> 2) * ATOM + 32 * (kk & 3), 16, 1024),
             sdesc(sS + (kk >> 2) * SATOM + 32 * (kk & 3), 16, 1024), id_d, kk > 0);
    tc_commit(D_DONE);
    // (e): K = rows.  A = phi(Q) M-major (its two atoms ATOM apart); B = [dn |
    // dden] N-major, N = 144: the dy tile's two atoms and the r tile's first.
#pragma unroll
    for (int kk = 0; kk < QT / 16; ++kk)
      tc_mma(tmem + C_DS, sdesc(sq + 2048 * kk, ATOM, 1024), sdesc(sy + 2048 * kk, ATOM, 1024), id_e,
             (first && kk == 0) ? 0u : 1u);
    tc_commit(EMPTY(s));
  };
  if (leader) issue_a(0);

  auto rsinv_of = [&](const QTile& x) {
    return i < x.nval ? __ldg(reinterpret_cast<const float2*>(a.rsinv + 2 * ((x.rb + i) * H + x.h)))
                      : make_float2(0.f, 0.f);
  };
  float2 ri_cur = rsinv_of(cur);
  int k = 0, kseg = 0, ns = 0;
  while (true) {
    QTile nxt;
    const int unxt = next_unit(a, ucur + 1, u1, upt, spt, nxt);
    const bool has_next = unxt < u1, same = has_next && nxt.seqh == cur.seqh;
    const float2 ri_next = has_next ? rsinv_of(nxt) : make_float2(0.f, 0.f);
    const int s = k % QST, h = cur.h;
    uint8_t* sq = smem + O_ST + s * STAGE + (part >> 1) * ATOM;  // the atom holding this thread's columns
    uint8_t* sy = sq + TILE;
    uint8_t* sr = sy + TILE;
    const bool store = i < cur.nrows;
    const size_t row = cur.rb + i;
    const float rs = ri_cur.x, inv = ri_cur.y;
    mbar_wait(A_DONE, k & 1, fail);
    tc_fence_after();
    // pass 1: dr, dgamma, du (into the r tile); sums m = du . u, D1 = du . o', D2 = u . o'.
    float m = 0.f, D1 = 0.f, D2 = 0.f;
    {
      uint32_t o[32], g[32];
      tmem_ld32_async(tl + f0, o);
      tmem_ld32_async(tl + C_DG + f0, g);
      tmem_wait32(o);
      tmem_tie32(g);
#pragma unroll
      for (int ch = 0; ch < 4; ++ch) {
        const int cc = c0 + ch, f = f0 + 8 * ch;
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
      tmem_st32(tl + C_DG + f0, g);
    }
    // the row's four owners add their sums in a fixed order, through TMEM
    tmem_st4(tl + C_X + 4 * part, m, D1, D2, 0.f);
    tmem_st_wait();
    tc_fence_before();
    named_bar(1, EW * 32);
    tc_fence_after();
    {
      uint32_t xv[16];
      tmem_ld16(tl + C_X, xv);
      m = (((__uint_as_float(xv[0]) + __uint_as_float(xv[4])) + __uint_as_float(xv[8])) + __uint_as_float(xv[12])) *
          (1.f / QD);
      D1 = ((__uint_as_float(xv[1]) + __uint_as_float(xv[5])) + __uint_as_float(xv[9])) + __uint_as_float(xv[13]);
      D2 = ((__uint_as_float(xv[2]) + __uint_as_float(xv[6])) + __uint_as_float(xv[10])) + __uint_as_float(xv[14]);
    }
    const float dden = -rs * fmaf(-m, D2, D1) * inv;
    // pass 2: dn = rs (du - u m) / den -> the dy tile
    {
      uint32_t o[32];
      tmem_ld32(tl + f0, o);
#pragma unroll
      for (int ch = 0; ch < 4; ++ch) {
        const int cc = c0 + ch, f = f0 + 8 * ch;
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
    // dden in column 128 of [dn | dden]: the first element of the r tile's
    // first atom (part 0, the owner of that chunk, consumed its du above)
    if (part == 0) *reinterpret_cast<uint4*>(sr + swz_off(i, 0)) = make_uint4(pack_bf16(dden, 0.f), 0u, 0u, 0u);
    tmem_st_wait();
    fence_async_smem();
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(DN_READY);
    if (leader) issue_de(k, k == kseg);
    __syncwarp();
    // epilogue 2: dq = (dq~ + dden z) min(1, phi(q))
    mbar_wait(D_DONE, k & 1, fail);
    tc_fence_after();
    {
      uint32_t o[32];
      tmem_ld32(tl + f0, o);  // dq~
#pragma unroll
      for (int ch = 0; ch < 4; ++ch) {
        const int cc = c0 + ch, f = f0 + 8 * ch;
        float qv[8];
        unpack8(*reinterpret_cast<const uint4*>(sq + swz_off(i, cc)), qv);
        uint32_t dq[4];
#pragma unroll
        for (int j = 0; j < 8; j += 2)
          dq[j / 2] = pack_bf16(fmaf(dden, zf[f + j], __uint_as_float(o[8 * ch + j])) * fminf(1.f, qv[j]),
                                fmaf(dden, zf[f + j + 1], __uint_as_float(o[8 * ch + j + 1])) * fminf(1.f, qv[j + 1]));
        if (store)
          *reinterpret_cast<uint4*>((bf16*)a.dq + row * a.lddq + (size_t)h * QD + f) = make_uint4(dq[0], dq[1], dq[2], dq[3]);
      }
    }
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(EMPTY(s));
    // every warp has read dq~ once EMPTY(s) completes: (a) of the next tile of
    // the segment may overwrite the columns, and the stage takes tile k + 2
    if (leader && mbar_wait(EMPTY(s), (k / QST) & 1, fail)) {
      if (same) issue_a(k + 1);
      if (ld_k == k + QST && ld_u < u1) load_next();
    }
    __syncwarp();
    if (!same) {
      // The segment ends with tile k: [dS' | dz'] (TMEM lane e = row e of the
      // state, columns 128 + f) leaves as this CTA's partial of the pair.
      if (leader) tc_commit(SEG);
      mbar_wait(SEG, ns & 1, fail);
      tc_fence_after();
      const int b = cur.b, p = h * nseq + b;
      {
        float* P = a.partial + (size_t)(p + blockIdx.x) * QD * LD + (size_t)i * LD;
        {
          uint32_t dsv[32];
          tmem_ld32(tl + C_DS + f0, dsv);
#pragma unroll
          for (int j = 0; j < 32; j += 4)
            *reinterpret_cast<float4*>(P + f0 + j) =
                make_float4(__uint_as_float(dsv[j]), __uint_as_float(dsv[j + 1]), __uint_as_float(dsv[j + 2]),
                            __uint_as_float(dsv[j + 3]));
        }
        uint32_t zv[8];
        tmem_ld8(tl + C_DS + QD, zv);  // dz' in column 128, then zero padding
        if (part == 3)
          *reinterpret_cast<float4*>(P + QD) = make_float4(__uint_as_float(zv[0]), 0.f, 0.f, 0.f);
        else if (part == 2)
          *reinterpret_cast<float4*>(P + QD + 4) = make_float4(0.f, 0.f, 0.f, 0.f);
      }
      tc_fence_before();
      __threadfence();
      __syncthreads();
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
      __syncthreads();
      if (lastf[0]) {  // this partial completes (b, h): [dS | dz''] in slot order
        __threadfence();
        combine_state(a.partial, nullptr, p + lastf[1], lastf[2], 1, 0, QD, cur.seqh, false, a.dstate,
                      a.dstate_bf, nullptr, nullptr, nullptr, a.center, nullptr);
      }
      ++ns;
      if (!has_next) break;
      load_state(nxt.seqh);  // every thread is done with tile k (the barriers above)
      tc_fence_before();
      __syncthreads();
      tc_fence_after();
      if (leader) issue_a(k + 1);
      kseg = k + 1;
    }
    cur = nxt;
    ucur = unxt;
    ri_cur = ri_next;
    ++k;
  }
  if (leader && *fail)  // let the copies still in flight land
    for (int s = 0; s < QST; ++s)
      if (issued[s] > 0)
        for (uint32_t it = 0; it < kPollLimit && !mbar_try_wait(FULL(s), (uint32_t)((issued[s] - 1) / QST) & 1);
             ++it) {
        }
  __syncwarp();  // single-lane roles rejoin their warps: the CTA barrier below is warp-aligned
  __syncthreads();
  const bool bad = *fail != 0;

  // dgamma: per-lane sums in TMEM, reduced over the 128 lanes in a fixed order
  float* red = reinterpret_cast<float*>(smem + O_ST);  // [128][129]: the stages are free now
  if (!bad) {
    uint32_t gv[32];
    tmem_ld32(tl + C_DG + f0, gv);
#pragma unroll
    for (int j = 0; j < 32; ++j) red[i * (QD + 1) + f0 + j] = __uint_as_float(gv[j]);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, TMEM_COLS);
  if (bad) {
    if (tid == 0 && a.err_out) atomicOr(a.err_out, kErrTimeout);
    return;
  }
  float* red2 = red + QT * (QD + 1);
  {  // four row quarters per column, then their sum: a fixed order
    const int f = tid & (QD - 1), qr = tid / QD;
    float v = 0.f;
    for (int r = qr * (QT / 4); r < (qr + 1) * (QT / 4); ++r) v += red[r * (QD + 1) + f];
    red2[qr * QD + f] = v;
  }
  __syncthreads();
  if (tid < QD)
    a.gamma_part[(size_t)blockIdx.x * QD + tid] = ((red2[tid] + red2[QD + tid]) + red2[2 * QD + tid]) + red2[3 * QD + tid];
}

}  // namespace

cudaError_t launch_bwd_q_tc128(const BwdQArgs& a, int hd, int n_tiles, int* nparts, cudaStream_t st) {
  auto al16 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; };
  const long long roff = ((const bf16*)a.r - (const bf16*)a.q);
  if (a.dh != QD || !a.pre || !a.rsinv || hd % 8 || a.ldr != a.ldq || roff < 0 || roff % 8 || !al16(a.q) ||
      !al16(a.dy) || !al16(a.dq) || !al16(a.dr) || !al16(a.partial) || a.ldq % 8 || a.lddy % 8 || a.lddq % 8 ||
      a.lddr % 8 || a.seq.T <= 0 || n_tiles <= 0 || a.tiles.tile % QT)
    return cudaErrorNotSupported;
  const int spt = a.tiles.tile / QT, upt = n_tiles * spt, n_units = upt * a.H;
  int grid = n_units < sm_count() ? n_units : sm_count();  // one CTA per SM
  const int room = a.partial_slots - a.seq.n_seq * a.H;  // partial slots beyond one per (sequence, head)
  if (room < grid) grid = room;
  if (grid <= 0) return cudaErrorNotSupported;
  CUtensorMap tmP, tmY;
  if (!make_map(&tmP, a.q, (uint64_t)a.ldq, (uint64_t)a.seq.T, (uint64_t)a.ldq, 64, QT, false) ||
      !make_map(&tmY, a.dy, (uint64_t)a.lddy, (uint64_t)a.seq.T, (uint64_t)a.lddy, 64, QT, false))
    return cudaErrorNotSupported;
  cudaError_t e = cudaFuncSetAttribute(k_bwd_q_tc128, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM);
  if (e != cudaSuccess) return e;
  *nparts = grid;
  return launch_pdl(k_bwd_q_tc128, dim3(grid), dim3(NTH), SMEM, st, a, tmP, tmY, (int)roff, upt, spt, n_units);
}

}  // namespace gbla
