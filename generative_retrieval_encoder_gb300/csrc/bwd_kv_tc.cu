// Key-side backward of the bf16 layer (Eq. 5/6) on the 5th-generation tensor
// cores, for d_h = 64 and 128 with phi(k) stored by the projection epilogue.  Per token
// j of a sequence and head, with [dS | dz''] the combined state gradient (dz''
// the centring-corrected z column):
//   dk~_j = bf16(dS) v_j + dz'',   dv_j = g_j dS^T phi(k_j),
//   dg_j = phi(k_j) . dk~_j,  dk_j = g_j dk~_j min(1, phi(k_j)),
//   ds_j = dg_j g_j (1 - g_j)  (sigmoid gate)   or   dg_j g_j  (softmax gate)
// (phi' of elu + 1 from the stored phi; ds is the gradient of the gate logit).
// Softmax gate: the stored gate holds the logits s_j and g_j = exp(s_j - m)
// with m the sequence's maximum logit from the forward combine; the softmax
// normaliser cancels in Eq. 5, so ds_j = dg_j g_j is the logit gradient.
//
// Persistent: one CTA per SM walks a contiguous range of (row tile, head)
// units, head-major, so that consecutive units mostly share a (sequence,
// head) and its [dS | dz''].  Roles:
//   producer warp    lane 0: TMA loads of the 128-row phi(k) and v boxes of
//                    each MMA tile (one box per 64 columns) into a ring (6
//                    stages at d_h = 64, 2 at 128); bf16 dS (128-byte swizzle)
//                    into one of two buffers when the (sequence, head) changes;
//   MMA warp         lane 0: D1 = V dS^T and D2 = phi(K) dS (M = 128,
//                    N = K = d_h) into the TMEM columns of the tile's group;
//   epilogue warps   groups of four warps (4 at d_h = 64, 2 at 128) taking MMA
//                    tiles in turn, one thread per row; dk and dv replace phi(k)
//                    and v in the consumed tiles and leave as whole 128-byte
//                    lines.
// The gate multiplies dv after the MMA, so both MMAs read the loaded tiles.
//
// Core form (CORE = true, the core entry point's backward of Eq. 5): k and v
// as given (two tensors), the gate's values, and dg_j itself out in fp32.  The
// epilogue group that owns an MMA tile first rewrites its rows of the k tile
// as phi(k) in place, and the MMAs wait for that rewrite instead of the copy.
//
// Every mbarrier wait is bounded; after one gives up, the kernel finishes its
// loops without waiting, sets the timeout bit of the error word, waits
// (bounded) for its copies and MMAs, frees its TMEM and returns.
#include "pdl.cuh"
#include "kernels.h"
#include "tcgen05.cuh"

namespace gbla {
namespace {

constexpr int KT = 128;                  // rows per MMA tile
constexpr int TILE = KT * 128;           // one 64-column atom of a tile: [128 rows][64 bf16], 16 KB

// Shapes and shared-memory layout by head width D (64 or 128).
template <int D, bool CORE>
struct KCfg {
  static constexpr int NH = D / 64;                 // 64-column atoms of a row
  static constexpr int KST = D == 64 ? 6 : 2;       // ring stages (phi(k) atoms | v atoms)
  static constexpr int NG = D == 64 ? 4 : 2;        // epilogue groups of 4 warps; MMA tile j goes to group j % NG
  static constexpr int STAGE = 2 * NH * TILE;
  static constexpr int SATOM = D * 128;             // one 64-column atom of dS [e][f]
  static constexpr int SBUF = NH * SATOM;
  static constexpr int EW = 4 * NG;
  static constexpr int NTH = (EW + 2) * 32;
  static constexpr int O_ST = 0;
  static constexpr int O_S = O_ST + KST * STAGE;    // two dS buffers
  static constexpr int O_BAR = O_S + 2 * SBUF;
  // full[KST], empty[KST], sfull[2], sfree[2], accf[NG], acce[NG], drain, phi[KST] (core)
  static constexpr int NBAR = 3 * KST + 4 + 2 * NG + 1;
  static constexpr int O_DZ = O_BAR + 8 * NBAR;     // [group][2 buffers][dz'' D] fp32
  static constexpr int O_RED = O_DZ + 4 * NG * 2 * D;  // [group][4 warps] ds sums
  static constexpr int O_M = O_RED + 4 * NG * 4;    // [group][2 buffers] maximum logit (softmax gate)
  static constexpr int O_SLOT = O_M + 4 * NG * 2;
  static constexpr int O_FAIL = O_SLOT + 4;
  static constexpr int SMEM = O_FAIL + 4 + 1024;
  static constexpr int TMEM_COLS = NG * 2 * D;      // per group: D1 | D2
  static_assert(SMEM <= 227 * 1024, "shared memory");
  static_assert(TMEM_COLS <= 512, "TMEM");
};

__device__ __forceinline__ uint32_t swz_off(int row, int chunk) {
  return (uint32_t)(row * 128 + ((chunk ^ (row & 7)) << 4));
}
__device__ __forceinline__ void unpack8(const uint4& u, float* f) {
  f[0] = bf_lo(u.x); f[1] = bf_hi(u.x); f[2] = bf_lo(u.y); f[3] = bf_hi(u.y);
  f[4] = bf_lo(u.z); f[5] = bf_hi(u.z); f[6] = bf_lo(u.w); f[7] = bf_hi(u.w);
}

struct Unit {
  int h, b, seqh, ntl, ti;
  int nrows, nval;
  size_t rb;
};
__device__ __forceinline__ Unit unit_at(const BwdKVArgs& a, int u, int n_units_per_head) {
  Unit x;
  x.h = u / n_units_per_head;
  x.ti = u - x.h * n_units_per_head;
  int row0, nvalid, tin;
  x.ntl = 0; x.b = 0; x.nrows = 0; x.nval = 0; x.rb = 0;
  if (!map_tile(a.seq, a.tiles, x.ti, x.b, row0, nvalid, tin)) { x.seqh = -1; return x; }
  const int R0 = tin * a.tiles.tile;
  x.nrows = max(0, min(a.tiles.tile, slot_rows(a.seq, nvalid) - R0));
  x.nval = max(0, min(x.nrows, nvalid - R0));
  x.rb = (size_t)row0 + R0;
  x.ntl = (x.nrows + KT - 1) / KT;
  x.seqh = x.b * a.H + x.h;
  return x;
}

template <int D, bool CORE>
__global__ void __launch_bounds__(KCfg<D, CORE>::NTH, 1)
    k_bwd_kv_tc(const BwdKVArgs a, const __grid_constant__ CUtensorMap tmP, const __grid_constant__ CUtensorMap tmV,
                const __grid_constant__ CUtensorMap tmS, int n_units_per_head, int n_units) {
  using C = KCfg<D, CORE>;
  constexpr int NH = C::NH, KST = C::KST, NG = C::NG, STAGE = C::STAGE, SBUF = C::SBUF, EW = C::EW,
                NTH = C::NTH, O_ST = C::O_ST, O_S = C::O_S, O_BAR = C::O_BAR, O_DZ = C::O_DZ, O_RED = C::O_RED,
                O_M = C::O_M, O_SLOT = C::O_SLOT, O_FAIL = C::O_FAIL, TMEM_COLS = C::TMEM_COLS;
  (void)NTH;
  if (threadIdx.x == 0) {  // the descriptors load while the previous kernel finishes
    tma_prefetch_map(&tmP);
    tma_prefetch_map(&tmV);
    tma_prefetch_map(&tmS);
  }
  pdl_enter();  // the previous kernel's outputs are visible from here on
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_align1024(smem_raw);
  const uint32_t sbase = smem_u32(smem);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (a.err && *a.err) return;
  const int u0 = (int)(((long long)n_units * blockIdx.x) / gridDim.x);
  const int u1 = (int)(((long long)n_units * (blockIdx.x + 1)) / gridDim.x);
  const int tiles_per_unit = a.tiles.tile / KT;  // db_g partial slots per unit

  const uint32_t bar0 = sbase + O_BAR;
  auto FULL = [&](int s) { return bar0 + 8 * s; };
  auto EMPTY = [&](int s) { return bar0 + 8 * (KST + s); };
  auto SFULL = [&](int k) { return bar0 + 8 * (2 * KST + k); };
  auto SFREE = [&](int k) { return bar0 + 8 * (2 * KST + 2 + k); };
  auto ACCF = [&](int g) { return bar0 + 8 * (2 * KST + 4 + g); };
  auto ACCE = [&](int g) { return bar0 + 8 * (2 * KST + 4 + NG + g); };
  const uint32_t DRAIN = bar0 + 8 * (2 * KST + 4 + 2 * NG);
  auto PHI = [&](int s) { return bar0 + 8 * (2 * KST + 4 + 2 * NG + 1 + s); };  // core: phi(k) written
  float* dzs = reinterpret_cast<float*>(smem + O_DZ);
  float* red = reinterpret_cast<float*>(smem + O_RED);
  float* mgs = reinterpret_cast<float*>(smem + O_M);
  const bool logits = a.gate_kind == GATE_LOGITS;
  uint32_t* slot = reinterpret_cast<uint32_t*>(smem + O_SLOT);
  volatile int* fail = reinterpret_cast<volatile int*>(smem + O_FAIL);

  if (tid == 0) {
    for (int s = 0; s < KST; ++s) {
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
      mbar_init(ACCE(g), 4);
    }
    mbar_init(DRAIN, 1);
    mbar_init_fence();
    *fail = 0;
  }
  if (warp == EW + 1) tmem_alloc(smem_u32(slot), TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *slot;

  if (warp == EW) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int j = 0, k = -1, prev = -1;
      int last_s[KST];
#pragma unroll
      for (int s = 0; s < KST; ++s) last_s[s] = 0;
      for (int u = u0; u < u1 && !*fail; ++u) {
        const Unit x = unit_at(a, u, n_units_per_head);
        if (x.ntl == 0) continue;
        if (x.seqh != prev) {
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
          const int s = j % KST;
          if (j >= KST && !mbar_wait(EMPTY(s), ((j / KST) - 1) & 1, fail)) { ok = false; break; }
          const uint32_t st = sbase + O_ST + s * STAGE;
          const int y = (int)x.rb + t * KT;
          mbar_expect_tx(FULL(s), STAGE);
#pragma unroll
          for (int hf = 0; hf < NH; ++hf) {
            tma_load_2d(st + hf * TILE, &tmP, FULL(s), x.h * D + 64 * hf, y);
            tma_load_2d(st + (NH + hf) * TILE, &tmV, FULL(s), x.h * D + 64 * hf, y);
          }
          last_s[s] = j + 1;
        }
        if (!ok) break;
      }
      if (*fail)
        for (int s = 0; s < KST; ++s)
          if (last_s[s] > 0)
            for (uint32_t it = 0; it < kPollLimit && !mbar_try_wait(FULL(s), (uint32_t)((last_s[s] - 1) / KST) & 1);
                 ++it) {
            }
    }
  } else if (warp == EW + 1) {
    // ---------------------------------------------------------- MMA issuer
    if (lane == 0) {
      const uint32_t id_k = idesc_bf16(KT, D, false, false), id_v = idesc_bf16(KT, D, false, true);
      int j = 0, k = -1, prev = -1;
      for (int u = u0; u < u1 && !*fail; ++u) {
        const Unit x = unit_at(a, u, n_units_per_head);
        if (x.ntl == 0) continue;
        if (x.seqh != prev) {
          if (k >= 0) tc_commit(SFREE(k & 1));
          ++k;
          prev = x.seqh;
          if (!mbar_wait(SFULL(k & 1), (k >> 1) & 1, fail)) break;
        }
        const uint32_t sS = sbase + O_S + (k & 1) * SBUF;
        bool ok = true;
        for (int t = 0; t < x.ntl; ++t, ++j) {
          const int s = j % KST, g = j % NG;
          if (!mbar_wait(CORE ? PHI(s) : FULL(s), (j / KST) & 1, fail)) { ok = false; break; }
          if (j >= NG && !mbar_wait(ACCE(g), ((j / NG) - 1) & 1, fail)) { ok = false; break; }
          tc_fence_after();
          const uint32_t sk = sbase + O_ST + s * STAGE, sv = sk + NH * TILE;
          const uint32_t d = tmem + g * 2 * D;
          // D1[j][e] = sum_f v[j][f] dS[e][f]: A = V K-major (atom kk / 4), B = dS
          // K-major (rows e; its K = f runs through the atoms SATOM apart).
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk)
            tc_mma(d, sdesc(sv + (kk >> 2) * TILE + 32 * (kk & 3), 16, 1024),
                   sdesc(sS + (kk >> 2) * C::SATOM + 32 * (kk & 3), 16, 1024), id_k, kk > 0);
          // D2[j][f] = sum_e phi(k)[j][e] dS[e][f]: A = phi(K) K-major (atom kk / 4),
          // B = dS N-major (16 e-rows = 2048 B; its 64-column atoms SATOM apart).
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk)
            tc_mma(d + D, sdesc(sk + (kk >> 2) * TILE + 32 * (kk & 3), 16, 1024),
                   sdesc(sS + 2048 * kk, C::SATOM, 1024), id_v, kk > 0);
          tc_commit(ACCF(g));
          tc_commit(EMPTY(s));
        }
        if (!ok) break;
      }
      if (k >= 0) tc_commit(SFREE(k & 1));
      tc_commit(DRAIN);
      for (uint32_t it = 0; it < kPollLimit && !mbar_try_wait(DRAIN, 0); ++it) {
      }
    }
  } else {
    // ----------------------------------------------------------- epilogue
    const int grp = warp >> 2, wq = warp & 3;
    const int i = wq * 32 + lane;
    const uint32_t tl = tmem + ((uint32_t)(wq * 32) << 16) + grp * 2 * D;
    float* dzg = dzs + grp * 2 * D;
    float* mg = mgs + grp * 2;
    int j = 0, k = -1, prev = -1;
    for (int u = u0; u < u1; ++u) {
      const Unit x = unit_at(a, u, n_units_per_head);
      if (x.ntl == 0) {
        // no rows: zero db_g partials of the unit (written by group 0)
        if (grp == 0 && wq == 0 && lane == 0 && a.bg_part)
          for (int t = 0; t < tiles_per_unit; ++t)
            a.bg_part[((size_t)x.ti * tiles_per_unit + t) * a.H + x.h] = 0.f;
        continue;
      }
      if (x.seqh != prev) {  // dz'' of the new (sequence, head), per group
        ++k;
        prev = x.seqh;
        // the buffer replaced here served the state before the previous one
        for (int e = i; e < D; e += 128) dzg[(k & 1) * D + e] = a.dstate[((size_t)x.seqh * D + e) * state_ld(D) + D];
        if (i == 0) mg[k & 1] = logits ? a.state_m[x.seqh] : 0.f;
        named_bar(1 + grp, 128);
      }
      const float* dz = dzg + (k & 1) * D;
      const float mseq = mg[k & 1];
      if (grp == 0 && wq == 0 && lane == 0 && a.bg_part)  // slots of MMA tiles the unit lacks
        for (int t = x.ntl; t < tiles_per_unit; ++t) a.bg_part[((size_t)x.ti * tiles_per_unit + t) * a.H + x.h] = 0.f;
      for (int t = 0; t < x.ntl; ++t, ++j) {
        if (j % NG != grp) continue;  // another group's tile
        const int s = j % KST;
        uint8_t* sk = smem + O_ST + s * STAGE;
        uint8_t* sv = sk + NH * TILE;
        const int rel = t * KT + i;
        const bool valid = rel < x.nval, store = rel < x.nrows;
        const size_t row = x.rb + rel;
        const float gin = valid ? __ldg(a.g + row * a.ldg + x.h) : 0.f;
        const float g = logits ? (valid ? __expf(gin - mseq) : 0.f) : gin;
        if (CORE) {  // phi(k) in place over this group's rows of the k tile
          mbar_wait(FULL(s), (j / KST) & 1, fail);
#pragma unroll
          for (int c = 0; c < 8 * NH; ++c) {
            uint4* kp = reinterpret_cast<uint4*>(sk + (c >> 3) * TILE + swz_off(i, c & 7));
            float kv[8];
            unpack8(*kp, kv);
            *kp = make_uint4(pack_bf16(phi_f(kv[0]), phi_f(kv[1])), pack_bf16(phi_f(kv[2]), phi_f(kv[3])),
                             pack_bf16(phi_f(kv[4]), phi_f(kv[5])), pack_bf16(phi_f(kv[6]), phi_f(kv[7])));
          }
          fence_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(PHI(s));
        }
        mbar_wait(ACCF(grp), (j / NG) & 1, fail);
        tc_fence_after();
        // dk~ = D1 + dz'', dg = phi(k) . dk~, dk = g dk~ min(1, phi(k)) -> the phi(k) row;
        // 32 accumulator columns at a time, the next 32 loading under the current ones
        float dg = 0.f;
        uint32_t ob[2][32];
        tmem_ld32_async(tl, ob[0]);
#pragma unroll
        for (int hh = 0; hh < D / 32; ++hh) {
          tmem_wait32(ob[hh & 1]);
          if (hh + 1 < D / 32) tmem_ld32_async(tl + 32 * (hh + 1), ob[(hh + 1) & 1]);
          const uint32_t* o = ob[hh & 1];
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            const int cc = 4 * hh + c;  // 8-column chunk of the row
            uint8_t* kp = sk + (cc >> 3) * TILE + swz_off(i, cc & 7);
            float kv[8];
            unpack8(*reinterpret_cast<const uint4*>(kp), kv);
            uint32_t w[4];
#pragma unroll
            for (int jj = 0; jj < 8; jj += 2) {
              const int f = 8 * c + jj, e = 32 * hh + f;
              const float d0 = __uint_as_float(o[f]) + dz[e], d1 = __uint_as_float(o[f + 1]) + dz[e + 1];
              dg = fmaf(kv[jj], d0, dg);
              dg = fmaf(kv[jj + 1], d1, dg);
              w[jj / 2] = pack_bf16(g * d0 * fminf(1.f, kv[jj]), g * d1 * fminf(1.f, kv[jj + 1]));
            }
            *reinterpret_cast<uint4*>(kp) = make_uint4(w[0], w[1], w[2], w[3]);
          }
        }
        // dv = g D2 -> the v row
        tmem_ld32_async(tl + D, ob[0]);
#pragma unroll
        for (int hh = 0; hh < D / 32; ++hh) {
          tmem_wait32(ob[hh & 1]);
          if (hh + 1 < D / 32) tmem_ld32_async(tl + D + 32 * (hh + 1), ob[(hh + 1) & 1]);
          const uint32_t* o = ob[hh & 1];
          if (hh == D / 32 - 1) {  // the accumulators are read: hand them back
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(ACCE(grp));
          }
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            const int cc = 4 * hh + c;
            uint32_t w[4];
#pragma unroll
            for (int jj = 0; jj < 8; jj += 2)
              w[jj / 2] = pack_bf16(g * __uint_as_float(o[8 * c + jj]), g * __uint_as_float(o[8 * c + jj + 1]));
            *reinterpret_cast<uint4*>(sv + (cc >> 3) * TILE + swz_off(i, cc & 7)) = make_uint4(w[0], w[1], w[2], w[3]);
          }
        }
        // the gate-logit gradient (core: dL/dg itself, fp32)
        const float ds = valid ? (CORE ? dg : logits ? dg * g : dg * g * (1.f - g)) : 0.f;
        if (store) {
          if (CORE)
            reinterpret_cast<float*>(a.ds)[row * a.ldds + x.h] = ds;
          else
            reinterpret_cast<bf16*>(a.ds)[row * a.ldds + x.h] = __float2bfloat16_rn(ds);
        }
        // the warp's 32 rows of dk and dv leave as whole 128-byte lines
        __syncwarp();
        {
          const int ch = lane & 7;
#pragma unroll
          for (int hf = 0; hf < NH; ++hf)
#pragma unroll
            for (int it = 0; it < 8; ++it) {
              const int rr = wq * 32 + 4 * it + (lane >> 3), rl = t * KT + rr;
              const uint4 vk = *reinterpret_cast<const uint4*>(sk + hf * TILE + swz_off(rr, ch));
              const uint4 vvv = *reinterpret_cast<const uint4*>(sv + hf * TILE + swz_off(rr, ch));
              if (rl < x.nrows) {
                *reinterpret_cast<uint4*>((bf16*)a.dk + (x.rb + rl) * a.lddk + (size_t)x.h * D + 64 * hf + 8 * ch) = vk;
                *reinterpret_cast<uint4*>((bf16*)a.dv + (x.rb + rl) * a.lddv + (size_t)x.h * D + 64 * hf + 8 * ch) = vvv;
              }
            }
        }
        // db_g partial of this MMA tile: the group's 128 rows, in a fixed order
        if (a.bg_part) {
          float v = ds;
          for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
          if (lane == 0) red[grp * 4 + wq] = v;
          named_bar(1 + grp, 128);
          if (wq == 0 && lane == 0)
            a.bg_part[((size_t)x.ti * tiles_per_unit + t) * a.H + x.h] =
                ((red[grp * 4] + red[grp * 4 + 1]) + red[grp * 4 + 2]) + red[grp * 4 + 3];
          named_bar(1 + grp, 128);
        }
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
cudaError_t launch_bwd_kv_tc_d(const BwdKVArgs& a, int n_tiles, int* nparts, cudaStream_t st) {
  using C = KCfg<D, CORE>;
  CUtensorMap tmP, tmV, tmS;
  if (!make_map(&tmP, a.k, (uint64_t)(a.H * D), (uint64_t)a.seq.T, (uint64_t)a.ldk, 64, KT, false) ||
      !make_map(&tmV, a.v, (uint64_t)(a.H * D), (uint64_t)a.seq.T, (uint64_t)a.ldv, 64, KT, false) ||
      !make_map(&tmS, a.dstate_bf, (uint64_t)state_bf_ld(D), (uint64_t)a.seq.n_seq * a.H * D,
                (uint64_t)state_bf_ld(D), 64, D, false))
    return cudaErrorNotSupported;
  cudaError_t e = cudaFuncSetAttribute(k_bwd_kv_tc<D, CORE>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
  if (e != cudaSuccess) return e;
  const int n_units = n_tiles * a.H;
  const int grid = n_units < sm_count() ? n_units : sm_count();
  *nparts = n_tiles * (a.tiles.tile / KT);
  return launch_pdl(k_bwd_kv_tc<D, CORE>, dim3(grid), dim3(C::NTH), C::SMEM, st, a, tmP, tmV, tmS, n_tiles, n_units);
}

}  // namespace

cudaError_t launch_bwd_kv_tc(const BwdKVArgs& a, int n_tiles, int* nparts, cudaStream_t st) {
  auto al16 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; };
  const bool sig = a.gate_kind == GATE_VALUES && a.gate_grad == GG_SIGMOID;
  const bool soft = a.gate_kind == GATE_LOGITS && a.gate_grad == GG_SOFTMAX && a.state_m;
  const bool core = !a.pre && a.gate_kind == GATE_VALUES && a.gate_grad == GG_DG && !a.bg_part;
  if ((a.dh != 64 && a.dh != 128) || !(a.pre ? (sig || soft) : core) || !al16(a.k) || !al16(a.v) ||
      !al16(a.dk) || !al16(a.dv) || !al16(a.dstate_bf) || a.ldk % 8 || a.ldv % 8 || a.lddk % 8 || a.lddv % 8 ||
      a.seq.T <= 0 || n_tiles <= 0 || a.tiles.tile % KT || a.zero_cols_to > a.zero_cols_from)
    return cudaErrorNotSupported;
  if (core)
    return a.dh == 64 ? launch_bwd_kv_tc_d<64, true>(a, n_tiles, nparts, st)
                      : launch_bwd_kv_tc_d<128, true>(a, n_tiles, nparts, st);
  return a.dh == 64 ? launch_bwd_kv_tc_d<64, false>(a, n_tiles, nparts, st)
                    : launch_bwd_kv_tc_d<128, false>(a, n_tiles, nparts, st);
}

}  // namespace gbla
