// bf16 GBLA state kernels (sm_103a): tensor-core (mma.sync m16n8k16, fp32
// accumulate) contractions of the d_h x d_h state, fed by cp.async pipelines
// of 16-byte loads into XOR-swizzled shared memory.
//
// "Gated Bidirectional Linear Attention for Generative Retrieval", section
// "Core method":
//   reduce : S = sum_j k~_j v_j^T, z = sum_j k~_j, k~_j = g_j phi(k_j)  (Eq. 5/6)
//            computed as K~^T [V | 1] per chunk of rows, then combined in a
//            fixed order by the last CTA of each (sequence, head).
//   readout: o_i = phi(q_i)^T [S | z] -> n_i / den_i                     (Eq. 5/6)
//            optionally fused with y = RmsNorm(o) gamma SiLU(r)          (Eq. 7)
//   bwd_q  : recompute o; RmsNorm-gate backward; dn = do/den,
//            dden = -(do.o)/den; dq~ = [dn | dden] [S | z]^T; dq = dq~ phi'(q);
//            [dS | dz] = sum_i phi(q_i) [dn_i | dden_i]^T (split-L + combine)
//   bwd_kv : dk~ = dS v + dz; dv = dS^T k~; dg = phi(k).dk~;
//            dk = g dk~ phi'(k); gate derivative.
#include "core_common.cuh"
#include "pdl.cuh"

namespace gbla {
namespace {

constexpr unsigned FULL = 0xffffffffu;

template <int DH>
struct Cfg {
  static constexpr int CPR = DH / 8;     // 16-byte chunks in a row of DH bf16
  static constexpr int NT = DH / 8 + 1;  // 8-wide n-tiles of [S | z]
  static constexpr int SPAD = DH + 24;   // smem row stride (elements) of [S | z | 0] copies
  static constexpr int BLD = DH + 16;    // global row stride of the bf16 state copy
};

__device__ __forceinline__ float silu_f(float x) { return x / (1.f + __expf(-x)); }

// Loads the bf16 [S | z | 0] copy of one (sequence, head) into smem rows of
// stride SPAD (padding makes the 8 rows that ldmatrix reads hit 8 bank groups).
template <int DH, int NTHR>
__device__ __forceinline__ void load_state_bf(bf16* Ss, const bf16* src) {
  using C = Cfg<DH>;
  for (int i = threadIdx.x; i < DH * (C::BLD / 8); i += NTHR) {
    const int e = i / (C::BLD / 8), c = i % (C::BLD / 8);
    cp_async16(smem_u32(Ss + e * C::SPAD + c * 8), src + (size_t)e * C::BLD + c * 8, 16);
  }
}

// A fragment of phi(rows) for the m16n8k16 "row" operand: 16 rows x 16
// columns starting at (r0, 16*ks) of a swizzled [rows][DH] tile.
template <int DH>
__device__ __forceinline__ void a_rows(uint32_t base, int r0, int ks, int lane, uint32_t (&a)[4]) {
  const int mi = lane >> 3, rr = lane & 7;
  ldsm_x4(base + swz<DH / 8>(r0 + ((mi & 1) << 3) + rr, 2 * ks + (mi >> 1)), a[0], a[1], a[2], a[3]);
}
__device__ __forceinline__ uint32_t phi2(uint32_t v) { return pack_bf16(phi_f(bf_lo(v)), phi_f(bf_hi(v))); }
// phi' from the raw value x, or (PRE) from the stored phi(x): phi' = min(1, phi).
template <bool PRE>
__device__ __forceinline__ float dphi_s(float x) { return PRE ? fminf(1.f, x) : dphi_f(x); }
// phi(x) from the raw value, or (PRE) the stored phi(x) itself.
template <bool PRE>
__device__ __forceinline__ float phik(float x) { return PRE ? x : phi_f(x); }

// =====================================================================
// reduce: per (chunk, head) CTA, 8 warps.  Warp (wm, kg) owns state rows
// e in [16 wm, 16 wm + 16) and the k-steps kk = kg (mod KS) of every tile.
// =====================================================================
template <int DH>
struct RedCfg {
  static constexpr int WM = DH / 16;
  static constexpr int KS = 8 / WM;
  static constexpr int TT = 64;
  static constexpr int STAGES = DH == 128 ? 3 : 4;
  static constexpr int TILE = TT * DH * 2;
  static constexpr int SMEM = STAGES * (2 * TILE + TT * 4);
};

// Resident CTAs per SM as their shared memory allows: three up to d_h = 64,
// two at d_h = 128 (at most 128 registers a thread; 129 left room for one).
template <int DH, bool PRE>
__global__ void __launch_bounds__(256, DH == 128 ? 2 : 3) k_reduce_bf16(const ReduceArgs a) {
  pdl_enter();  // the previous kernel's outputs are visible from here on
  using C = Cfg<DH>;
  using R = RedCfg<DH>;
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ float red8[8];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int wm = warp % R::WM, kg = warp / R::WM;
  if (a.err && *a.err) return;
  int b, row0, nvalid, cin;
  if (!map_tile(a.seq, a.chunks, blockIdx.x, b, row0, nvalid, cin)) return;
  const int h = blockIdx.y, H = a.H;
  const int CH = a.chunks.tile;
  const int c0 = cin * CH;
  const int n_in = max(0, min(CH, nvalid - c0));
  const int ntiles = (n_in + R::TT - 1) / R::TT;
  const bool logits = a.gate_kind == GATE_LOGITS;
  const size_t rbase = (size_t)row0 + c0;
  const bf16* kp = (const bf16*)a.k + rbase * a.ldk + (size_t)h * DH;
  const bf16* vp = (const bf16*)a.v + rbase * a.ldv + (size_t)h * DH;
  const float* gp = a.g + rbase * a.ldg + h;

  float mch = 0.f;
  if (logits) {  // chunk maximum of the logits: exp(s - mch) <= 1
    float m = -INFINITY;
    for (int i = tid; i < n_in; i += 256) m = fmaxf(m, gp[(size_t)i * a.ldg]);
    for (int o = 16; o; o >>= 1) m = fmaxf(m, __shfl_xor_sync(FULL, m, o));
    if (lane == 0) red8[warp] = m;
    __syncthreads();
    m = red8[0];
    for (int w = 1; w < 8; ++w) m = fmaxf(m, red8[w]);
    mch = m;
  }

  auto load = [&](int stage, int t) {
    const uint32_t kb = smem_u32(smem + stage * 2 * R::TILE), vb = kb + R::TILE;
    const uint32_t gb = smem_u32(smem + R::STAGES * 2 * R::TILE + stage * R::TT * 4);
    for (int i = tid; i < R::TT * C::CPR; i += 256) {
      const int r = i / C::CPR, c = i % C::CPR;
      const int tok = t * R::TT + r;
      const bool ok = tok < n_in;
      const size_t ro = ok ? (size_t)tok : 0;
      cp_async16(kb + swz<C::CPR>(r, c), kp + ro * a.ldk + c * 8, ok ? 16 : 0);
      cp_async16(vb + swz<C::CPR>(r, c), vp + ro * a.ldv + c * 8, ok ? 16 : 0);
    }
    for (int i = tid; i < R::TT; i += 256) {
      const int tok = t * R::TT + i;
      const bool ok = tok < n_in;
      cp_async4(gb + i * 4, gp + (ok ? (size_t)tok : 0) * a.ldg, ok ? 4 : 0);
    }
  };

  float acc[C::NT][4];
#pragma unroll
  for (int i = 0; i < C::NT; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;

#pragma unroll
  for (int s = 0; s < R::STAGES - 1; ++s) {
    if (s < ntiles) load(s, s);
    cp_async_commit();
  }
  const int mi = lane >> 3, rr = lane & 7, t4 = lane & 3;
  const uint32_t one = (lane >> 2) == 0 ? 0x3F803F80u : 0u;  // B column of ones -> z
  for (int t = 0; t < ntiles; ++t) {
    cp_async_wait<R::STAGES - 2>();
    __syncthreads();
    {
      const int tn = t + R::STAGES - 1;
      if (tn < ntiles) load(tn % R::STAGES, tn);
      cp_async_commit();
    }
    const int st = t % R::STAGES;
    const uint32_t kb = smem_u32(smem + st * 2 * R::TILE), vb = kb + R::TILE;
    const float* gs = reinterpret_cast<const float*>(smem + R::STAGES * 2 * R::TILE + st * R::TT * 4);
#pragma unroll
    for (int kk = kg; kk < R::TT / 16; kk += R::KS) {
      const int j0 = kk * 16;
      uint32_t a0, a1, a2, a3;
      ldsm_x4_t(kb + swz<C::CPR>(j0 + ((mi >> 1) << 3) + rr, 2 * wm + (mi & 1)), a0, a1, a2, a3);
      {  // k~ = g phi(k) on the A fragment (rows past the chunk have g = 0)
        float gv[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int j = j0 + 2 * t4 + (u & 1) + ((u >> 1) << 3);
          const float x = gs[j];
          gv[u] = (t * R::TT + j < n_in) ? (logits ? __expf(x - mch) : x) : 0.f;
        }
        a0 = pack_bf16(phik<PRE>(bf_lo(a0)) * gv[0], phik<PRE>(bf_hi(a0)) * gv[1]);
        a1 = pack_bf16(phik<PRE>(bf_lo(a1)) * gv[0], phik<PRE>(bf_hi(a1)) * gv[1]);
        a2 = pack_bf16(phik<PRE>(bf_lo(a2)) * gv[2], phik<PRE>(bf_hi(a2)) * gv[3]);
        a3 = pack_bf16(phik<PRE>(bf_lo(a3)) * gv[2], phik<PRE>(bf_hi(a3)) * gv[3]);
      }
#pragma unroll
      for (int np = 0; np < DH / 16; ++np) {
        uint32_t b0, b1, b2, b3;
        ldsm_x4_t(vb + swz<C::CPR>(j0 + ((mi & 1) << 3) + rr, 2 * np + (mi >> 1)), b0, b1, b2, b3);
        mma_bf16(acc[2 * np], a0, a1, a2, a3, b0, b1);
        mma_bf16(acc[2 * np + 1], a0, a1, a2, a3, b2, b3);
      }
      mma_bf16(acc[C::NT - 1], a0, a1, a2, a3, one, one);
    }
  }
  cp_async_wait<0>();
  __syncthreads();

  if (R::KS > 1) {  // fixed-order sum of the k-split groups
    float* red = reinterpret_cast<float*>(smem);
    if (kg > 0) {
#pragma unroll
      for (int nt = 0; nt < C::NT; ++nt)
#pragma unroll
        for (int u = 0; u < 4; ++u)
          red[((((kg - 1) * R::WM + wm) * C::NT + nt) * 4 + u) * 32 + lane] = acc[nt][u];
    }
    __syncthreads();
    if (kg == 0) {
      for (int g2 = 1; g2 < R::KS; ++g2)
#pragma unroll
        for (int nt = 0; nt < C::NT; ++nt)
#pragma unroll
          for (int u = 0; u < 4; ++u)
            acc[nt][u] += red[((((g2 - 1) * R::WM + wm) * C::NT + nt) * 4 + u) * 32 + lane];
    }
  }
  constexpr int LD = state_ld(DH);
  if (kg == 0) {
    float* P = a.partial + ((size_t)blockIdx.x * H + h) * DH * LD;
    const int e = wm * 16 + (lane >> 2);
#pragma unroll
    for (int nt = 0; nt < C::NT; ++nt) {
      const int f = nt * 8 + 2 * t4;
      *reinterpret_cast<float2*>(P + e * LD + f) = make_float2(acc[nt][0], acc[nt][1]);
      *reinterpret_cast<float2*>(P + (e + 8) * LD + f) = make_float2(acc[nt][2], acc[nt][3]);
    }
  }
  if (logits && tid == 0) a.partial_m[(size_t)blockIdx.x * H + h] = n_in > 0 ? mch : -INFINITY;
  int first, count;
  seq_tiles(a.seq, a.chunks, b, first, count);
  if (!arrive_last(a.counters + (size_t)b * H + h, count)) return;
  combine_state(a.partial, a.partial_m, first, count, H, h, DH, b * H + h, logits, a.state,
                a.state_bf, a.state_m, a.pub_state, a.center, nullptr, reinterpret_cast<float*>(smem));
  static_assert(R::SMEM >= DH * state_ld(DH) * 4, "the combine's staging buffer fits the tile memory");
}

// The centre c of the state (see combine_state) at the accumulator columns
// this lane holds: cols nt*8 + 2*(lane&3) and +1 of every n-tile.
template <int DH>
__device__ __forceinline__ void load_center_cols(const float* center, int seqh, int t4, float (&c)[DH / 8][2]) {
#pragma unroll
  for (int nt = 0; nt < DH / 8; ++nt) {
    c[nt][0] = center ? center[(size_t)seqh * DH + nt * 8 + 2 * t4] : 0.f;
    c[nt][1] = center ? center[(size_t)seqh * DH + nt * 8 + 2 * t4 + 1] : 0.f;
  }
}

// =====================================================================
// readout: per (row range of `tiles`, head) CTA -- the library passes its
// chunks (up to 2048 rows), so that one load of the state serves them all --
// 4 warps x 16 rows per 64-row sub-tile, double-buffered.  o = phi(q) [S | z]
// with the division in the epilogue.
// =====================================================================
template <int DH, bool NORM>
struct RdCfg {
  static constexpr int TT = 64;
  static constexpr int TILE = TT * DH * 2;
  static constexpr int SMEM = DH * Cfg<DH>::SPAD * 2 + 2 * TILE * (NORM ? 2 : 1);
};

template <int DH, bool NORM, bool PRE>
__global__ void __launch_bounds__(128) k_readout_bf16(const ReadoutArgs a) {
  using C = Cfg<DH>;
  using R = RdCfg<DH, NORM>;
  extern __shared__ __align__(128) uint8_t smem[];
  bf16* Ss = reinterpret_cast<bf16*>(smem);
  uint8_t* qt = smem + DH * C::SPAD * 2;
  uint8_t* rt = qt + 2 * R::TILE;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (a.err && *a.err) return;
  int b, row0, nvalid, tin;
  if (!map_tile(a.seq, a.tiles, blockIdx.x, b, row0, nvalid, tin)) return;
  const int h = blockIdx.y, H = a.H;
  const int R0 = tin * a.tiles.tile;
  const int nrows = min(a.tiles.tile, slot_rows(a.seq, nvalid) - R0);
  if (nrows <= 0) return;
  const int nval = max(0, min(nrows, nvalid - R0));
  const int nsub = (nrows + R::TT - 1) / R::TT;
  const size_t rb = (size_t)row0 + R0;
  const bf16* qp = (const bf16*)a.q + rb * a.ldq + (size_t)h * DH;
  const bf16* rp = NORM ? (const bf16*)a.r + rb * a.ldr + (size_t)h * DH : nullptr;
  bf16* op = (bf16*)a.out + rb * a.ldo + (size_t)h * DH;

  load_state_bf<DH, 128>(Ss, a.state_bf + (size_t)(b * H + h) * DH * C::BLD);
  auto load = [&](int buf, int s) {
    for (int i = tid; i < R::TT * C::CPR; i += 128) {
      const int r = i / C::CPR, c = i % C::CPR;
      const int tok = s * R::TT + r;
      const bool ok = tok < nval;
      const size_t ro = ok ? (size_t)tok : 0;
      cp_async16(smem_u32(qt + buf * R::TILE) + swz<C::CPR>(r, c), qp + ro * a.ldq + c * 8, ok ? 16 : 0);
      if (NORM)
        cp_async16(smem_u32(rt + buf * R::TILE) + swz<C::CPR>(r, c), rp + ro * a.ldr + c * 8, ok ? 16 : 0);
    }
  };
  load(0, 0);
  cp_async_commit();

  const int g = lane >> 2, t4 = lane & 3, mi = lane >> 3, rr = lane & 7;
  float gam[DH / 8][2], cen[DH / 8][2];
#pragma unroll
  for (int nt = 0; nt < DH / 8; ++nt) {
    gam[nt][0] = gam[nt][1] = 1.f;
    if (NORM && a.rms_w) {
      gam[nt][0] = __bfloat162float(((const bf16*)a.rms_w)[nt * 8 + 2 * t4]);
      gam[nt][1] = __bfloat162float(((const bf16*)a.rms_w)[nt * 8 + 2 * t4 + 1]);
    }
  }
  load_center_cols<DH>(a.center, b * H + h, t4, cen);
  const uint32_t sb = smem_u32(Ss);
  for (int s = 0; s < nsub; ++s) {
    if (s + 1 < nsub) load((s + 1) & 1, s + 1);
    cp_async_commit();
    cp_async_wait<1>();
    __syncthreads();
    const int buf = s & 1;
    const uint32_t qb = smem_u32(qt + buf * R::TILE);
    const int r0w = warp * 16;
    float acc[C::NT][4];
#pragma unroll
    for (int i = 0; i < C::NT; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;
#pragma unroll
    for (int ks = 0; ks < DH / 16; ++ks) {
      uint32_t af[4];
      a_rows<DH>(qb, r0w, ks, lane, af);
      if (!PRE) {  // PRE: the tile already holds phi(q)
#pragma unroll
        for (int u = 0; u < 4; ++u) af[u] = phi2(af[u]);
      }
      const uint32_t srow = sb + ((ks * 16 + ((mi & 1) << 3) + rr) * C::SPAD) * 2;
#pragma unroll
      for (int np = 0; np < DH / 16; ++np) {
        uint32_t b0, b1, b2, b3;
        ldsm_x4_t(srow + (2 * np + (mi >> 1)) * 16, b0, b1, b2, b3);
        mma_bf16(acc[2 * np], af[0], af[1], af[2], af[3], b0, b1);
        mma_bf16(acc[2 * np + 1], af[0], af[1], af[2], af[3], b2, b3);
      }
      uint32_t z0, z1, z2, z3;
      ldsm_x4_t(srow + (DH / 8 + (mi >> 1)) * 16, z0, z1, z2, z3);
      mma_bf16(acc[C::NT - 1], af[0], af[1], af[2], af[3], z0, z1);
    }
    const float den0 = __shfl_sync(FULL, acc[C::NT - 1][0], lane & ~3);
    const float den1 = __shfl_sync(FULL, acc[C::NT - 1][2], lane & ~3);
    const int ra = s * R::TT + r0w + g, rb2 = ra + 8;
    const bool va = ra < nval, vb = rb2 < nval;
    const float inv0 = va ? 1.f / den0 : 0.f, inv1 = vb ? 1.f / den1 : 0.f;
    const float c0 = va ? 1.f : 0.f, c1 = vb ? 1.f : 0.f;  // o = c + S'^T q~ / den on valid rows
    float o[DH / 8][4];
#pragma unroll
    for (int nt = 0; nt < DH / 8; ++nt) {
      o[nt][0] = acc[nt][0] * inv0 + c0 * cen[nt][0]; o[nt][1] = acc[nt][1] * inv0 + c0 * cen[nt][1];
      o[nt][2] = acc[nt][2] * inv1 + c1 * cen[nt][0]; o[nt][3] = acc[nt][3] * inv1 + c1 * cen[nt][1];
    }
    float rs0 = 1.f, rs1 = 1.f;
    if (NORM) {
      float ss0 = 0.f, ss1 = 0.f;
#pragma unroll
      for (int nt = 0; nt < DH / 8; ++nt) {
        ss0 += o[nt][0] * o[nt][0] + o[nt][1] * o[nt][1];
        ss1 += o[nt][2] * o[nt][2] + o[nt][3] * o[nt][3];
      }
      ss0 += __shfl_xor_sync(FULL, ss0, 1); ss0 += __shfl_xor_sync(FULL, ss0, 2);
      ss1 += __shfl_xor_sync(FULL, ss1, 1); ss1 += __shfl_xor_sync(FULL, ss1, 2);
      rs0 = rsqrtf(ss0 / DH + a.eps); rs1 = rsqrtf(ss1 / DH + a.eps);
      const uint8_t* rtb = rt + buf * R::TILE;
#pragma unroll
      for (int nt = 0; nt < DH / 8; ++nt) {
        const uint32_t rv0 = *reinterpret_cast<const uint32_t*>(rtb + swz<C::CPR>(r0w + g, nt) + t4 * 4);
        const uint32_t rv1 = *reinterpret_cast<const uint32_t*>(rtb + swz<C::CPR>(r0w + g + 8, nt) + t4 * 4);
        o[nt][0] *= rs0 * gam[nt][0] * silu_f(bf_lo(rv0));
        o[nt][1] *= rs0 * gam[nt][1] * silu_f(bf_hi(rv0));
        o[nt][2] *= rs1 * gam[nt][0] * silu_f(bf_lo(rv1));
        o[nt][3] *= rs1 * gam[nt][1] * silu_f(bf_hi(rv1));
      }
    }
    uint8_t* qtb = qt + buf * R::TILE;  // this warp's q rows are consumed: stage the output
#pragma unroll
    for (int nt = 0; nt < DH / 8; ++nt) {
      *reinterpret_cast<uint32_t*>(qtb + swz<C::CPR>(r0w + g, nt) + t4 * 4) = pack_bf16(o[nt][0], o[nt][1]);
      *reinterpret_cast<uint32_t*>(qtb + swz<C::CPR>(r0w + g + 8, nt) + t4 * 4) = pack_bf16(o[nt][2], o[nt][3]);
    }
    __syncwarp();
    for (int i = lane; i < 16 * C::CPR; i += 32) {
      const int row = r0w + i / C::CPR, c = i % C::CPR;
      const int rel = s * R::TT + row;
      if (rel < nrows)
        *reinterpret_cast<uint4*>(op + (size_t)rel * a.ldo + c * 8) =
            *reinterpret_cast<const uint4*>(qtb + swz<C::CPR>(row, c));
    }
    if (a.den && t4 == 0) {
      if (ra < nrows) a.den[(rb + ra) * H + h] = va ? den0 : 0.f;
      if (rb2 < nrows) a.den[(rb + rb2) * H + h] = vb ? den1 : 0.f;
    }
    if (NORM && a.rsinv && t4 == 0) {
      if (ra < nrows) *reinterpret_cast<float2*>(a.rsinv + 2 * ((rb + ra) * H + h)) = make_float2(va ? rs0 : 0.f, inv0);
      if (rb2 < nrows) *reinterpret_cast<float2*>(a.rsinv + 2 * ((rb + rb2) * H + h)) = make_float2(vb ? rs1 : 0.f, inv1);
    }
    __syncthreads();
  }
}

// =====================================================================
// bwd_q: per (chunk, head) CTA.  NW warps x 16 rows per tile.
// =====================================================================
template <int DH, bool NORM>
struct BqCfg {
  static constexpr int NW = DH == 128 ? 8 : 4;
  static constexpr int TT = NW * 16;
  static constexpr int WM = DH / 16;
  static constexpr int KS = NW / WM;
  static constexpr int STAGES = DH == 128 ? 1 : 2;
  static constexpr int TILE = TT * DH * 2;
  static constexpr int NIN = NORM ? 3 : 2;  // q, dy|d_o, [r]
  // d_h = 128: each thread's dgamma sums (d_h / 4 floats) live in shared
  // memory, [slot][thread], to keep registers for the accumulators
  static constexpr bool GSM = NORM && DH == 128;
  static constexpr int GSM_BYTES = GSM ? NW * 32 * (DH / 4) * 4 : 0;
  static constexpr int SMEM = DH * Cfg<DH>::SPAD * 2 + TT * Cfg<DH>::SPAD * 2 + STAGES * NIN * TILE + GSM_BYTES;
};

template <int DH, bool NORM, bool PRE>
__global__ void __launch_bounds__(BqCfg<DH, NORM>::NW * 32) k_bwd_q_bf16(const BwdQArgs a) {
  using C = Cfg<DH>;
  using R = BqCfg<DH, NORM>;
  constexpr int NTHR = R::NW * 32;
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ float gred[R::NW][DH];
  bf16* Ss = reinterpret_cast<bf16*>(smem);
  bf16* Dn = Ss + DH * C::SPAD;
  uint8_t* tiles = reinterpret_cast<uint8_t*>(Dn + R::TT * C::SPAD);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int wm = warp % R::WM, kg = warp / R::WM;
  if (a.err && *a.err) return;
  int b, row0, nvalid, cin;
  if (!map_tile(a.seq, a.chunks, blockIdx.x, b, row0, nvalid, cin)) {  // no chunk: a zero dgamma partial
    if (NORM)
      for (int f = tid; f < DH; f += NTHR) a.gamma_part[((size_t)blockIdx.x * a.H + blockIdx.y) * DH + f] = 0.f;
    return;
  }
  const int h = blockIdx.y, H = a.H;
  const int CH = a.chunks.tile;
  const int c0 = cin * CH;
  const int nrows = max(0, min(CH, slot_rows(a.seq, nvalid) - c0));
  const int nval = max(0, min(nrows, nvalid - c0));
  const int ntiles = (nrows + R::TT - 1) / R::TT;
  const size_t rb = (size_t)row0 + c0;
  const bf16* qp = (const bf16*)a.q + rb * a.ldq + (size_t)h * DH;
  const bf16* yp = (const bf16*)a.dy + rb * a.lddy + (size_t)h * DH;
  const bf16* rp = NORM ? (const bf16*)a.r + rb * a.ldr + (size_t)h * DH : nullptr;
  bf16* dqp = (bf16*)a.dq + rb * a.lddq + (size_t)h * DH;
  bf16* drp = NORM ? (bf16*)a.dr + rb * a.lddr + (size_t)h * DH : nullptr;

  load_state_bf<DH, NTHR>(Ss, a.state_bf + (size_t)(b * H + h) * DH * C::BLD);
  auto tile_ptr = [&](int stage, int which) { return tiles + (stage * R::NIN + which) * R::TILE; };
  auto load = [&](int stage, int t) {
    for (int i = tid; i < R::TT * C::CPR; i += NTHR) {
      const int r = i / C::CPR, c = i % C::CPR;
      const int tok = t * R::TT + r;
      const bool ok = tok < nval;
      const size_t ro = ok ? (size_t)tok : 0;
      const uint32_t o = swz<C::CPR>(r, c);
      cp_async16(smem_u32(tile_ptr(stage, 0)) + o, qp + ro * a.ldq + c * 8, ok ? 16 : 0);
      cp_async16(smem_u32(tile_ptr(stage, 1)) + o, yp + ro * a.lddy + c * 8, ok ? 16 : 0);
      if (NORM) cp_async16(smem_u32(tile_ptr(stage, 2)) + o, rp + ro * a.ldr + c * 8, ok ? 16 : 0);
    }
  };

  const int g = lane >> 2, t4 = lane & 3, mi = lane >> 3, rr = lane & 7;
  // gamma and the state centre live in shared memory (read as float2 at this
  // lane's columns) to keep registers for the accumulators.
  __shared__ __align__(16) float s_gam[DH];  // read as float2: needs 8-byte alignment
  __shared__ __align__(16) float s_cen[DH];
  for (int f = tid; f < DH; f += NTHR) {
    s_gam[f] = (NORM && a.rms_w) ? __bfloat162float(((const bf16*)a.rms_w)[f]) : 1.f;
    s_cen[f] = (NORM && a.center) ? a.center[(size_t)(b * H + h) * DH + f] : 0.f;
  }
  float gacc[R::GSM ? 1 : DH / 8][2];
  float* gsm = reinterpret_cast<float*>(tiles + R::STAGES * R::NIN * R::TILE) + tid;  // slot j at gsm[j * NTHR]
  if (R::GSM) {
#pragma unroll
    for (int j = 0; j < DH / 4; ++j) gsm[j * NTHR] = 0.f;
  } else {
#pragma unroll
    for (int nt = 0; nt < DH / 8; ++nt) gacc[nt][0] = gacc[nt][1] = 0.f;
  }
  float accS[C::NT][4];
#pragma unroll
  for (int i = 0; i < C::NT; ++i) accS[i][0] = accS[i][1] = accS[i][2] = accS[i][3] = 0.f;

  const uint32_t sb = smem_u32(Ss), dnb = smem_u32(Dn);
  // Tile t+1 is prefetched only after the barrier that ends every warp's use
  // of its buffer (tile t-1, read until the end of step (e)).
  if (ntiles > 0) load(0, 0);
  cp_async_commit();
  for (int t = 0; t < ntiles; ++t) {
    cp_async_wait<0>();
    __syncthreads();
    if (R::STAGES == 2) {
      if (t + 1 < ntiles) load((t + 1) & 1, t + 1);
      cp_async_commit();
    }
    const int st = R::STAGES == 2 ? (t & 1) : 0;
    const uint32_t qb = smem_u32(tile_ptr(st, 0));
    uint8_t* ytb = tile_ptr(st, 1);
    uint8_t* rtb = tile_ptr(st, 2);
    const int r0w = warp * 16;
    // (a) recompute n, den
    float acc[C::NT][4];
#pragma unroll
    for (int i = 0; i < C::NT; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;
#pragma unroll
    for (int ks = 0; ks < DH / 16; ++ks) {
      uint32_t af[4];
      a_rows<DH>(qb, r0w, ks, lane, af);
      if (!PRE) {  // PRE: the tile already holds phi(q)
#pragma unroll
        for (int u = 0; u < 4; ++u) af[u] = phi2(af[u]);
      }
      const uint32_t srow = sb + ((ks * 16 + ((mi & 1) << 3) + rr) * C::SPAD) * 2;
#pragma unroll
      for (int np = 0; np < DH / 16; ++np) {
        uint32_t b0, b1, b2, b3;
        ldsm_x4_t(srow + (2 * np + (mi >> 1)) * 16, b0, b1, b2, b3);
        mma_bf16(acc[2 * np], af[0], af[1], af[2], af[3], b0, b1);
        mma_bf16(acc[2 * np + 1], af[0], af[1], af[2], af[3], b2, b3);
      }
      uint32_t z0, z1, z2, z3;
      ldsm_x4_t(srow + (DH / 8 + (mi >> 1)) * 16, z0, z1, z2, z3);
      mma_bf16(acc[C::NT - 1], af[0], af[1], af[2], af[3], z0, z1);
    }
    const float den0 = __shfl_sync(FULL, acc[C::NT - 1][0], lane & ~3);
    const float den1 = __shfl_sync(FULL, acc[C::NT - 1][2], lane & ~3);
    const int ra = t * R::TT + r0w + g, rb2 = ra + 8;
    const bool va = ra < nval, vb = rb2 < nval;
    const float inv0 = va ? 1.f / den0 : 0.f, inv1 = vb ? 1.f / den1 : 0.f;
    // acc <- o' = S'^T q~ / den (centred); the full output is o = o' + c
#pragma unroll
    for (int nt = 0; nt < DH / 8; ++nt) {
      acc[nt][0] *= inv0; acc[nt][1] *= inv0; acc[nt][2] *= inv1; acc[nt][3] *= inv1;
    }
    const float cv[4] = {va ? 1.f : 0.f, va ? 1.f : 0.f, vb ? 1.f : 0.f, vb ? 1.f : 0.f};
    float dO[DH / 8][4];
    if (NORM) {
      float ss0 = 0.f, ss1 = 0.f;
#pragma unroll
      for (int nt = 0; nt < DH / 8; ++nt) {
        const float2 ce = *reinterpret_cast<const float2*>(s_cen + nt * 8 + 2 * t4);
        const float o0 = acc[nt][0] + cv[0] * ce.x, o1 = acc[nt][1] + cv[1] * ce.y;
        const float o2 = acc[nt][2] + cv[2] * ce.x, o3 = acc[nt][3] + cv[3] * ce.y;
        ss0 += o0 * o0 + o1 * o1;
        ss1 += o2 * o2 + o3 * o3;
      }
      ss0 += __shfl_xor_sync(FULL, ss0, 1); ss0 += __shfl_xor_sync(FULL, ss0, 2);
      ss1 += __shfl_xor_sync(FULL, ss1, 1); ss1 += __shfl_xor_sync(FULL, ss1, 2);
      const float rs0 = rsqrtf(ss0 / DH + a.eps), rs1 = rsqrtf(ss1 / DH + a.eps);
      float m0 = 0.f, m1 = 0.f;
      const float rsv[4] = {rs0, rs0, rs1, rs1};
#pragma unroll
      for (int nt = 0; nt < DH / 8; ++nt) {
        const uint32_t o0 = swz<C::CPR>(r0w + g, nt) + t4 * 4, o1 = swz<C::CPR>(r0w + g + 8, nt) + t4 * 4;
        const uint32_t rv0 = *reinterpret_cast<const uint32_t*>(rtb + o0);
        const uint32_t rv1 = *reinterpret_cast<const uint32_t*>(rtb + o1);
        const uint32_t yv0 = *reinterpret_cast<const uint32_t*>(ytb + o0);
        const uint32_t yv1 = *reinterpret_cast<const uint32_t*>(ytb + o1);
        const float rv[4] = {bf_lo(rv0), bf_hi(rv0), bf_lo(rv1), bf_hi(rv1)};
        const float yv[4] = {bf_lo(yv0), bf_hi(yv0), bf_lo(yv1), bf_hi(yv1)};
        float dr[4], gd[2] = {0.f, 0.f};
        const float2 gm2 = *reinterpret_cast<const float2*>(s_gam + nt * 8 + 2 * t4);
        const float2 ce2 = *reinterpret_cast<const float2*>(s_cen + nt * 8 + 2 * t4);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const float gm = (q & 1) ? gm2.y : gm2.x;
          const float sg = 1.f / (1.f + __expf(-rv[q]));
          const float av = rv[q] * sg;
          const float u = (acc[nt][q] + cv[q] * ((q & 1) ? ce2.y : ce2.x)) * rsv[q];
          gd[q & 1] += yv[q] * u * av;
          dr[q] = cv[q] * yv[q] * u * gm * sg * (1.f + rv[q] * (1.f - sg));
          dO[nt][q] = yv[q] * gm * av;  // du
          if (q < 2) m0 += dO[nt][q] * u; else m1 += dO[nt][q] * u;
        }
        if (R::GSM) {
          gsm[(2 * nt) * NTHR] += gd[0];
          gsm[(2 * nt + 1) * NTHR] += gd[1];
        } else {
          gacc[R::GSM ? 0 : nt][0] += gd[0];
          gacc[R::GSM ? 0 : nt][1] += gd[1];
        }
        // stage dr into this warp's r rows (consumed)
        *reinterpret_cast<uint32_t*>(rtb + o0) = pack_bf16(dr[0], dr[1]);
        *reinterpret_cast<uint32_t*>(rtb + o1) = pack_bf16(dr[2], dr[3]);
      }
      m0 += __shfl_xor_sync(FULL, m0, 1); m0 += __shfl_xor_sync(FULL, m0, 2);
      m1 += __shfl_xor_sync(FULL, m1, 1); m1 += __shfl_xor_sync(FULL, m1, 2);
      m0 /= DH; m1 /= DH;
      const float mv[4] = {m0, m0, m1, m1};
#pragma unroll
      for (int nt = 0; nt < DH / 8; ++nt) {
        const float2 ce2 = *reinterpret_cast<const float2*>(s_cen + nt * 8 + 2 * t4);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const float u = (acc[nt][q] + cv[q] * ((q & 1) ? ce2.y : ce2.x)) * rsv[q];
          dO[nt][q] = rsv[q] * (dO[nt][q] - u * mv[q]);
        }
      }
    } else {
#pragma unroll
      for (int nt = 0; nt < DH / 8; ++nt) {
        const uint32_t yv0 = *reinterpret_cast<const uint32_t*>(ytb + swz<C::CPR>(r0w + g, nt) + t4 * 4);
        const uint32_t yv1 = *reinterpret_cast<const uint32_t*>(ytb + swz<C::CPR>(r0w + g + 8, nt) + t4 * 4);
        dO[nt][0] = bf_lo(yv0); dO[nt][1] = bf_hi(yv0); dO[nt][2] = bf_lo(yv1); dO[nt][3] = bf_hi(yv1);
      }
    }
    // (c) dn = do / den, dden = -(do . o) / den
    float dot0 = 0.f, dot1 = 0.f;
#pragma unroll
    for (int nt = 0; nt < DH / 8; ++nt) {
      dot0 += dO[nt][0] * acc[nt][0] + dO[nt][1] * acc[nt][1];
      dot1 += dO[nt][2] * acc[nt][2] + dO[nt][3] * acc[nt][3];
    }
    dot0 += __shfl_xor_sync(FULL, dot0, 1); dot0 += __shfl_xor_sync(FULL, dot0, 2);
    dot1 += __shfl_xor_sync(FULL, dot1, 1); dot1 += __shfl_xor_sync(FULL, dot1, 2);
    const float dd0 = -dot0 * inv0, dd1 = -dot1 * inv1;
    uint32_t afr[DH / 16 + 1][4];
#pragma unroll
    for (int j = 0; j < DH / 16; ++j) {
      afr[j][0] = pack_bf16(dO[2 * j][0] * inv0, dO[2 * j][1] * inv0);
      afr[j][1] = pack_bf16(dO[2 * j][2] * inv1, dO[2 * j][3] * inv1);
      afr[j][2] = pack_bf16(dO[2 * j + 1][0] * inv0, dO[2 * j + 1][1] * inv0);
      afr[j][3] = pack_bf16(dO[2 * j + 1][2] * inv1, dO[2 * j + 1][3] * inv1);
    }
    afr[DH / 16][0] = pack_bf16(t4 == 0 ? dd0 : 0.f, 0.f);
    afr[DH / 16][1] = pack_bf16(t4 == 0 ? dd1 : 0.f, 0.f);
    afr[DH / 16][2] = 0u;
    afr[DH / 16][3] = 0u;
    // [dn | dden | 0] rows of this warp into Dn (for the dS contraction)
#pragma unroll
    for (int j = 0; j <= DH / 16; ++j) {
      bf16* d0 = Dn + (r0w + g) * C::SPAD + j * 16 + 2 * t4;
      bf16* d1 = Dn + (r0w + g + 8) * C::SPAD + j * 16 + 2 * t4;
      *reinterpret_cast<uint32_t*>(d0) = afr[j][0];
      *reinterpret_cast<uint32_t*>(d1) = afr[j][1];
      *reinterpret_cast<uint32_t*>(d0 + 8) = afr[j][2];
      *reinterpret_cast<uint32_t*>(d1 + 8) = afr[j][3];
    }
    // (d) dq~ = [dn | dden] [S | z]^T
    float accq[DH / 8][4];
#pragma unroll
    for (int i = 0; i < DH / 8; ++i) accq[i][0] = accq[i][1] = accq[i][2] = accq[i][3] = 0.f;
#pragma unroll
    for (int j = 0; j <= DH / 16; ++j) {
#pragma unroll
      for (int np = 0; np < DH / 16; ++np) {
        uint32_t b0, b1, b2, b3;
        ldsm_x4(sb + ((np * 16 + ((mi >> 1) << 3) + rr) * C::SPAD + (2 * j + (mi & 1)) * 8) * 2, b0, b1, b2, b3);
        mma_bf16(accq[2 * np], afr[j][0], afr[j][1], afr[j][2], afr[j][3], b0, b1);
        mma_bf16(accq[2 * np + 1], afr[j][0], afr[j][1], afr[j][2], afr[j][3], b2, b3);
      }
    }
    // dq = dq~ phi'(q); staged into this warp's dy rows (consumed)
    const uint8_t* qtb = tile_ptr(st, 0);
#pragma unroll
    for (int nt = 0; nt < DH / 8; ++nt) {
      const uint32_t o0 = swz<C::CPR>(r0w + g, nt) + t4 * 4, o1 = swz<C::CPR>(r0w + g + 8, nt) + t4 * 4;
      const uint32_t q0 = *reinterpret_cast<const uint32_t*>(qtb + o0);
      const uint32_t q1 = *reinterpret_cast<const uint32_t*>(qtb + o1);
      *reinterpret_cast<uint32_t*>(ytb + o0) =
          pack_bf16(va ? accq[nt][0] * dphi_s<PRE>(bf_lo(q0)) : 0.f, va ? accq[nt][1] * dphi_s<PRE>(bf_hi(q0)) : 0.f);
      *reinterpret_cast<uint32_t*>(ytb + o1) =
          pack_bf16(vb ? accq[nt][2] * dphi_s<PRE>(bf_lo(q1)) : 0.f, vb ? accq[nt][3] * dphi_s<PRE>(bf_hi(q1)) : 0.f);
    }
    __syncwarp();
    for (int i = lane; i < 16 * C::CPR; i += 32) {
      const int row = r0w + i / C::CPR, c = i % C::CPR;
      const int rel = t * R::TT + row;
      if (rel < nrows) {
        *reinterpret_cast<uint4*>(dqp + (size_t)rel * a.lddq + c * 8) =
            *reinterpret_cast<const uint4*>(ytb + swz<C::CPR>(row, c));
        if (NORM)
          *reinterpret_cast<uint4*>(drp + (size_t)rel * a.lddr + c * 8) =
              *reinterpret_cast<const uint4*>(rtb + swz<C::CPR>(row, c));
      }
    }
    __syncthreads();
    // (e) [dS | dz] += phi(Q)^T [dn | dden] over this tile's rows
#pragma unroll
    for (int kk = kg; kk < R::TT / 16; kk += R::KS) {
      const int j0 = kk * 16;
      uint32_t a0, a1, a2, a3;
      ldsm_x4_t(qb + swz<C::CPR>(j0 + ((mi >> 1) << 3) + rr, 2 * wm + (mi & 1)), a0, a1, a2, a3);
      if (!PRE) { a0 = phi2(a0); a1 = phi2(a1); a2 = phi2(a2); a3 = phi2(a3); }
      const uint32_t drow = dnb + ((j0 + ((mi & 1) << 3) + rr) * C::SPAD) * 2;
#pragma unroll
      for (int np = 0; np < DH / 16; ++np) {
        uint32_t b0, b1, b2, b3;
        ldsm_x4_t(drow + (2 * np + (mi >> 1)) * 16, b0, b1, b2, b3);
        mma_bf16(accS[2 * np], a0, a1, a2, a3, b0, b1);
        mma_bf16(accS[2 * np + 1], a0, a1, a2, a3, b2, b3);
      }
      uint32_t z0, z1, z2, z3;
      ldsm_x4_t(drow + (DH / 8 + (mi >> 1)) * 16, z0, z1, z2, z3);
      mma_bf16(accS[C::NT - 1], a0, a1, a2, a3, z0, z1);
    }
    if (R::STAGES == 1) {
      __syncthreads();
      if (t + 1 < ntiles) load(0, t + 1);
      cp_async_commit();
    }
  }
  cp_async_wait<0>();
  __syncthreads();

  // dgamma partial of this CTA (fixed-order reduction)
  if (NORM) {
#pragma unroll
    for (int nt = 0; nt < DH / 8; ++nt)
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        float v = R::GSM ? gsm[(2 * nt + q) * NTHR] : gacc[R::GSM ? 0 : nt][q];
        v += __shfl_xor_sync(FULL, v, 4);
        v += __shfl_xor_sync(FULL, v, 8);
        v += __shfl_xor_sync(FULL, v, 16);
        if (g == 0) gred[warp][nt * 8 + 2 * t4 + q] = v;
      }
    __syncthreads();
    for (int f = tid; f < DH; f += NTHR) {
      float v = 0.f;
      for (int w = 0; w < R::NW; ++w) v += gred[w][f];
      a.gamma_part[((size_t)blockIdx.x * H + h) * DH + f] = v;
    }
  }
  if (R::KS > 1) {
    float* red = reinterpret_cast<float*>(tiles);
    if (kg > 0) {
#pragma unroll
      for (int nt = 0; nt < C::NT; ++nt)
#pragma unroll
        for (int u = 0; u < 4; ++u)
          red[((((kg - 1) * R::WM + wm) * C::NT + nt) * 4 + u) * 32 + lane] = accS[nt][u];
    }
    __syncthreads();
    if (kg == 0) {
      for (int g2 = 1; g2 < R::KS; ++g2)
#pragma unroll
        for (int nt = 0; nt < C::NT; ++nt)
#pragma unroll
          for (int u = 0; u < 4; ++u)
            accS[nt][u] += red[((((g2 - 1) * R::WM + wm) * C::NT + nt) * 4 + u) * 32 + lane];
    }
  }
  constexpr int LD = state_ld(DH);
  if (kg == 0) {
    float* P = a.partial + ((size_t)blockIdx.x * H + h) * DH * LD;
    const int e = wm * 16 + g;
#pragma unroll
    for (int nt = 0; nt < C::NT; ++nt) {
      const int f = nt * 8 + 2 * t4;
      *reinterpret_cast<float2*>(P + e * LD + f) = make_float2(accS[nt][0], accS[nt][1]);
      *reinterpret_cast<float2*>(P + (e + 8) * LD + f) = make_float2(accS[nt][2], accS[nt][3]);
    }
  }
  int first, count;
  seq_tiles(a.seq, a.chunks, b, first, count);
  if (!arrive_last(a.counters + (size_t)b * H + h, count)) return;
  // stage the combined state in the tile memory where it fits (not for d_h = 128 without the norm inputs)
  constexpr bool kStage = R::STAGES * R::NIN * R::TILE >= DH * state_ld(DH) * 4;
  combine_state(a.partial, nullptr, first, count, H, h, DH, b * H + h, false, a.dstate, a.dstate_bf,
                nullptr, nullptr, nullptr, a.center, kStage ? reinterpret_cast<float*>(tiles) : nullptr);
}

// =====================================================================
// bwd_kv: per (row range of `tiles`, head) CTA (the library passes its
// chunks, as for the readout), 4 warps x 16 rows per 64-row sub-tile.
// =====================================================================
template <int DH>
struct BkvCfg {
  static constexpr int TT = 64;
  static constexpr int TILE = TT * DH * 2;
  static constexpr int SMEM = DH * Cfg<DH>::SPAD * 2 + 2 * (2 * TILE + TT * 4);
};

template <int DH, bool PRE>
__global__ void __launch_bounds__(128) k_bwd_kv_bf16(const BwdKVArgs a) {
  using C = Cfg<DH>;
  using R = BkvCfg<DH>;
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ float bred[4];
  bf16* Ss = reinterpret_cast<bf16*>(smem);
  uint8_t* tiles = smem + DH * C::SPAD * 2;
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
  const int nsub = (nrows + R::TT - 1) / R::TT;
  const size_t rb = (size_t)row0 + R0;
  const bf16* kp = (const bf16*)a.k + rb * a.ldk + (size_t)h * DH;
  const bf16* vp = (const bf16*)a.v + rb * a.ldv + (size_t)h * DH;
  const float* gp = a.g + rb * a.ldg + h;
  bf16* dkp = (bf16*)a.dk + rb * a.lddk + (size_t)h * DH;
  bf16* dvp = (bf16*)a.dv + rb * a.lddv + (size_t)h * DH;
  const bool logits = a.gate_kind == GATE_LOGITS;
  const float mseq = logits ? a.state_m[b * H + h] : 0.f;

  load_state_bf<DH, 128>(Ss, a.dstate_bf + (size_t)(b * H + h) * DH * C::BLD);
  // dz column in fp32: dz (uncentred forward state) or dz'' = dz' - bf16(dS) c
  // (centred forward state, see combine_state), so that dk~ = bf16(dS) v + dz
  // in both cases with the raw bf16 v as the tensor-core operand.
  __shared__ float s_dz[DH];
  for (int e = tid; e < DH; e += 128) s_dz[e] = a.dstate[((size_t)(b * H + h) * DH + e) * state_ld(DH) + DH];
  auto kt = [&](int buf) { return tiles + buf * (2 * R::TILE + R::TT * 4); };
  auto load = [&](int buf, int s) {
    const uint32_t kb = smem_u32(kt(buf)), vb = kb + R::TILE, gb = vb + R::TILE;
    for (int i = tid; i < R::TT * C::CPR; i += 128) {
      const int r = i / C::CPR, c = i % C::CPR;
      const int tok = s * R::TT + r;
      const bool ok = tok < nval;
      const size_t ro = ok ? (size_t)tok : 0;
      cp_async16(kb + swz<C::CPR>(r, c), kp + ro * a.ldk + c * 8, ok ? 16 : 0);
      cp_async16(vb + swz<C::CPR>(r, c), vp + ro * a.ldv + c * 8, ok ? 16 : 0);
    }
    for (int i = tid; i < R::TT; i += 128) {
      const int tok = s * R::TT + i;
      const bool ok = tok < nval;
      cp_async4(gb + i * 4, gp + (ok ? (size_t)tok : 0) * a.ldg, ok ? 4 : 0);
    }
  };
  load(0, 0);
  cp_async_commit();
  const int g = lane >> 2, t4 = lane & 3, mi = lane >> 3, rr = lane & 7;
  const uint32_t sb = smem_u32(Ss);
  float bsum = 0.f;
  for (int s = 0; s < nsub; ++s) {
    if (s + 1 < nsub) load((s + 1) & 1, s + 1);
    cp_async_commit();
    cp_async_wait<1>();
    __syncthreads();
    uint8_t* ktb = kt(s & 1);
    uint8_t* vtb = ktb + R::TILE;
    const float* gs = reinterpret_cast<const float*>(vtb + R::TILE);
    const uint32_t kb = smem_u32(ktb), vb = smem_u32(vtb);
    const int r0w = warp * 16;
    const int ra = s * R::TT + r0w + g, rb2 = ra + 8;
    const bool va = ra < nval, vb2 = rb2 < nval;
    float gr0 = gs[r0w + g], gr1 = gs[r0w + g + 8];
    if (logits) { gr0 = __expf(gr0 - mseq); gr1 = __expf(gr1 - mseq); }
    if (!va) gr0 = 0.f;
    if (!vb2) gr1 = 0.f;
    float acck[DH / 8][4], accv[DH / 8][4];
#pragma unroll
    for (int i = 0; i < DH / 8; ++i) {
      acck[i][0] = acck[i][1] = acck[i][2] = acck[i][3] = 0.f;
      accv[i][0] = accv[i][1] = accv[i][2] = accv[i][3] = 0.f;
    }
#pragma unroll
    for (int ks = 0; ks < DH / 16; ++ks) {
      uint32_t av[4], ak[4];
      a_rows<DH>(vb, r0w, ks, lane, av);
      a_rows<DH>(kb, r0w, ks, lane, ak);
      ak[0] = pack_bf16(phik<PRE>(bf_lo(ak[0])) * gr0, phik<PRE>(bf_hi(ak[0])) * gr0);
      ak[1] = pack_bf16(phik<PRE>(bf_lo(ak[1])) * gr1, phik<PRE>(bf_hi(ak[1])) * gr1);
      ak[2] = pack_bf16(phik<PRE>(bf_lo(ak[2])) * gr0, phik<PRE>(bf_hi(ak[2])) * gr0);
      ak[3] = pack_bf16(phik<PRE>(bf_lo(ak[3])) * gr1, phik<PRE>(bf_hi(ak[3])) * gr1);
#pragma unroll
      for (int np = 0; np < DH / 16; ++np) {
        uint32_t b0, b1, b2, b3;
        // dk~ = V dS^T : B[k=f][n=e] = dS[e][f] (non-transposed rows e)
        ldsm_x4(sb + ((np * 16 + ((mi >> 1) << 3) + rr) * C::SPAD + (2 * ks + (mi & 1)) * 8) * 2, b0, b1, b2, b3);
        mma_bf16(acck[2 * np], av[0], av[1], av[2], av[3], b0, b1);
        mma_bf16(acck[2 * np + 1], av[0], av[1], av[2], av[3], b2, b3);
        // dv = K~ dS : B[k=e][n=f] = dS[e][f] (transposed rows e)
        ldsm_x4_t(sb + ((ks * 16 + ((mi & 1) << 3) + rr) * C::SPAD + (2 * np + (mi >> 1)) * 8) * 2, b0, b1, b2, b3);
        mma_bf16(accv[2 * np], ak[0], ak[1], ak[2], ak[3], b0, b1);
        mma_bf16(accv[2 * np + 1], ak[0], ak[1], ak[2], ak[3], b2, b3);
      }
    }
    // epilogue
    float dg0 = 0.f, dg1 = 0.f;
    float kv[DH / 8][4];
#pragma unroll
    for (int nt = 0; nt < DH / 8; ++nt) {
      const int e = nt * 8 + 2 * t4;
      const float dz0 = s_dz[e], dz1 = s_dz[e + 1];
      acck[nt][0] += dz0; acck[nt][1] += dz1; acck[nt][2] += dz0; acck[nt][3] += dz1;
      const uint32_t k0 = *reinterpret_cast<const uint32_t*>(ktb + swz<C::CPR>(r0w + g, nt) + t4 * 4);
      const uint32_t k1 = *reinterpret_cast<const uint32_t*>(ktb + swz<C::CPR>(r0w + g + 8, nt) + t4 * 4);
      kv[nt][0] = bf_lo(k0); kv[nt][1] = bf_hi(k0); kv[nt][2] = bf_lo(k1); kv[nt][3] = bf_hi(k1);
      dg0 += phik<PRE>(kv[nt][0]) * acck[nt][0] + phik<PRE>(kv[nt][1]) * acck[nt][1];
      dg1 += phik<PRE>(kv[nt][2]) * acck[nt][2] + phik<PRE>(kv[nt][3]) * acck[nt][3];
    }
    dg0 += __shfl_xor_sync(FULL, dg0, 1); dg0 += __shfl_xor_sync(FULL, dg0, 2);
    dg1 += __shfl_xor_sync(FULL, dg1, 1); dg1 += __shfl_xor_sync(FULL, dg1, 2);
#pragma unroll
    for (int nt = 0; nt < DH / 8; ++nt) {
      const uint32_t o0 = swz<C::CPR>(r0w + g, nt) + t4 * 4, o1 = swz<C::CPR>(r0w + g + 8, nt) + t4 * 4;
      *reinterpret_cast<uint32_t*>(ktb + o0) =
          pack_bf16(gr0 * acck[nt][0] * dphi_s<PRE>(kv[nt][0]), gr0 * acck[nt][1] * dphi_s<PRE>(kv[nt][1]));
      *reinterpret_cast<uint32_t*>(ktb + o1) =
          pack_bf16(gr1 * acck[nt][2] * dphi_s<PRE>(kv[nt][2]), gr1 * acck[nt][3] * dphi_s<PRE>(kv[nt][3]));
      *reinterpret_cast<uint32_t*>(vtb + o0) = pack_bf16(accv[nt][0], accv[nt][1]);
      *reinterpret_cast<uint32_t*>(vtb + o1) = pack_bf16(accv[nt][2], accv[nt][3]);
    }
    __syncwarp();
    for (int i = lane; i < 16 * C::CPR; i += 32) {
      const int row = r0w + i / C::CPR, c = i % C::CPR;
      const int rel = s * R::TT + row;
      if (rel < nrows) {
        *reinterpret_cast<uint4*>(dkp + (size_t)rel * a.lddk + c * 8) =
            *reinterpret_cast<const uint4*>(ktb + swz<C::CPR>(row, c));
        *reinterpret_cast<uint4*>(dvp + (size_t)rel * a.lddv + c * 8) =
            *reinterpret_cast<const uint4*>(vtb + swz<C::CPR>(row, c));
      }
    }
    // gate gradient
    if (t4 == 0) {
      float o2[2];
      const float gv[2] = {gr0, gr1}, dgv[2] = {dg0, dg1};
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        if (a.gate_grad == GG_DG) o2[q] = dgv[q];
        else if (a.gate_grad == GG_SIGMOID) o2[q] = dgv[q] * gv[q] * (1.f - gv[q]);
        else o2[q] = gv[q] * dgv[q];
      }
      if (!va) o2[0] = 0.f;
      if (!vb2) o2[1] = 0.f;
      const int rows2[2] = {ra, rb2};
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        if (rows2[q] >= nrows) continue;
        const size_t idx = (rb + rows2[q]) * a.ldds + h;
        if (a.gate_grad == GG_DG) reinterpret_cast<float*>(a.ds)[idx] = o2[q];
        else reinterpret_cast<bf16*>(a.ds)[idx] = __float2bfloat16_rn(o2[q]);
        bsum += o2[q];
      }
    }
    if (h == 0 && a.zero_cols_to > a.zero_cols_from) {
      const int w = a.zero_cols_to - a.zero_cols_from;
      for (int i = lane; i < 16 * w; i += 32) {
        const int rel = s * R::TT + r0w + i / w;
        if (rel < nrows)
          reinterpret_cast<bf16*>(a.ds)[(rb + rel) * a.ldds + a.zero_cols_from + i % w] = __float2bfloat16_rn(0.f);
      }
    }
    __syncthreads();
  }
  if (a.bg_part) {
    for (int o = 16; o; o >>= 1) bsum += __shfl_xor_sync(FULL, bsum, o);
    if (lane == 0) bred[warp] = bsum;
    __syncthreads();
    if (tid == 0) a.bg_part[(size_t)blockIdx.x * H + h] = bred[0] + bred[1] + bred[2] + bred[3];
  }
}

template <typename K>
cudaError_t prep(K kernel, int smem) {
  return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
}

}  // namespace

// Dispatch on (d_h, norm, pre).  The feature-map-free ("pre") variants are
// built for the layer's sigmoid-gate path.
cudaError_t launch_reduce_bf16(const ReduceArgs& a, int grid_x, cudaStream_t st) {
  const dim3 grid(grid_x, a.H);
  cudaError_t e;
  switch (a.dh * 2 + (a.pre ? 1 : 0)) {
#define GBLA_CASE(D, P)                                                              \
  case D * 2 + P:                                                                    \
    if ((e = prep(k_reduce_bf16<D, P>, RedCfg<D>::SMEM)) != cudaSuccess) return e;   \
    return launch_pdl(k_reduce_bf16<D, P>, grid, dim3(256), RedCfg<D>::SMEM, st, a);
    GBLA_CASE(32, 0) GBLA_CASE(32, 1) GBLA_CASE(64, 0) GBLA_CASE(64, 1) GBLA_CASE(128, 0) GBLA_CASE(128, 1)
#undef GBLA_CASE
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

cudaError_t launch_readout_bf16(const ReadoutArgs& a, bool norm, int grid_x, cudaStream_t st) {
  const dim3 grid(grid_x, a.H);
  cudaError_t e;
  switch (a.dh * 4 + (norm ? 2 : 0) + (a.pre ? 1 : 0)) {
#define GBLA_CASE(D, N, P)                                                                      \
  case D * 4 + N * 2 + P:                                                                       \
    if ((e = prep(k_readout_bf16<D, N, P>, RdCfg<D, N>::SMEM)) != cudaSuccess) return e;        \
    k_readout_bf16<D, N, P><<<grid, 128, RdCfg<D, N>::SMEM, st>>>(a);                           \
    break;
    GBLA_CASE(32, 0, 0) GBLA_CASE(32, 1, 0) GBLA_CASE(64, 0, 0) GBLA_CASE(64, 1, 0) GBLA_CASE(128, 0, 0)
    GBLA_CASE(128, 1, 0) GBLA_CASE(32, 1, 1) GBLA_CASE(64, 1, 1) GBLA_CASE(128, 1, 1)
#undef GBLA_CASE
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

cudaError_t launch_bwd_q_bf16(const BwdQArgs& a, bool norm, int grid_x, cudaStream_t st) {
  const dim3 grid(grid_x, a.H);
  cudaError_t e;
  switch (a.dh * 4 + (norm ? 2 : 0) + (a.pre ? 1 : 0)) {
#define GBLA_CASE(D, N, P)                                                                          \
  case D * 4 + N * 2 + P:                                                                           \
    if ((e = prep(k_bwd_q_bf16<D, N, P>, BqCfg<D, N>::SMEM)) != cudaSuccess) return e;              \
    k_bwd_q_bf16<D, N, P><<<grid, BqCfg<D, N>::NW * 32, BqCfg<D, N>::SMEM, st>>>(a);                \
    break;
    GBLA_CASE(32, 0, 0) GBLA_CASE(32, 1, 0) GBLA_CASE(64, 0, 0) GBLA_CASE(64, 1, 0) GBLA_CASE(128, 0, 0)
    GBLA_CASE(128, 1, 0) GBLA_CASE(32, 1, 1) GBLA_CASE(64, 1, 1) GBLA_CASE(128, 1, 1)
#undef GBLA_CASE
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

cudaError_t launch_bwd_kv_bf16(const BwdKVArgs& a, int grid_x, cudaStream_t st) {
  const dim3 grid(grid_x, a.H);
  cudaError_t e;
  switch (a.dh * 2 + (a.pre ? 1 : 0)) {
#define GBLA_CASE(D, P)                                                            \
  case D * 2 + P:                                                                  \
    if ((e = prep(k_bwd_kv_bf16<D, P>, BkvCfg<D>::SMEM)) != cudaSuccess) return e; \
    k_bwd_kv_bf16<D, P><<<grid, 128, BkvCfg<D>::SMEM, st>>>(a);                    \
    break;
    GBLA_CASE(32, 0) GBLA_CASE(32, 1) GBLA_CASE(64, 0) GBLA_CASE(64, 1) GBLA_CASE(128, 0) GBLA_CASE(128, 1)
#undef GBLA_CASE
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

}  // namespace gbla
