// State reduction of the bf16 layer and core (Eq. 5/6, gate values) on the
// 5th-generation tensor cores, for d_h = 64:
//   [S | z] = sum_j k~_j [v_j | 1]^T,   k~_j = bf16(g_j phi(k_j))
// ("Gated Bidirectional Linear Attention for Generative Retrieval", section
// "Core method": the d_h x d_h state formed first, in the order of Eq. 3).  The
// gated key is rounded to bf16 as the tensor-core operand and z comes from the
// same rounded values through a column of ones.
//
// Work split: the (256-row tile, head) units, head-major, are cut into one
// contiguous range per CTA (one CTA per SM).  A run of units of one
// (sequence, head) inside a range is a segment: its [S | z]^T accumulates in
// one of two TMEM buffers (lane f = state column, lane 64 = z; column e =
// state row) and, at the segment's end, leaves as one partial, in slot
// p + blockIdx.x of the partial array (p = h n_seq + b: pairs in unit order, so
// the slot is unique).  The CTA whose partial completes a (sequence, head)
// sums the partials in slot order (a fixed order) and centres the state, with
// the arithmetic of combine_state.
//
// Roles, all walking the same units in the same order:
//   warp 12, lane 0  producer: TMA loads of the phi(k) and v boxes (128 rows x
//                    128 bytes, 128-byte swizzle; two of each per tile) into a
//                    3-stage ring, and the tile's descriptor (segment, segment
//                    end) into a small shared ring read by the MMA issuer;
//   warps 0-7        two transform groups of four warps, group g on rows
//                    128 g .. 128 g + 127 of every tile: each thread scales its
//                    row of phi(k) by its gate in shared memory
//                    (k~ = bf16(g phi(k)));
//   warp 13, lane 0  MMA issuer: D[f][e] += [V | 1]^T k~ with M = 128 (A
//                    M-major: the V tile, then a constant block whose first
//                    column is one, so that TMEM lane 64 holds z), N = 64 (the
//                    k~ tile, N-major), K = the tile's rows in 16-row steps; its
//                    commit frees the stage;
//   warps 8-11       drain group: at each segment end, the accumulator into
//                    the partial slot, the arrival count, and the combine when
//                    this partial completes its (sequence, head).  It never
//                    holds up the stream: the other accumulator serves the next
//                    segment meanwhile.
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

constexpr int KD = 64;                 // d_h
constexpr int KT = 128;                // rows per copy box (and per transform group)
constexpr int TT = 2 * KT;             // rows per tile (MMA K, in 16-row steps)
constexpr int TILE = KT * 128;         // [128 rows][64 bf16], 16 KB
constexpr int RST = 3;                 // ring stages: phi(k) rows 0-127 | 128-255, v rows 0-127 | 128-255
constexpr int STAGE = 4 * TILE;
constexpr int NG = 2;                  // transform groups of 4 warps
constexpr int W_DRAIN = 4 * NG;        // first warp of the drain group
constexpr int W_PROD = W_DRAIN + 4, W_MMA = W_PROD + 1;
constexpr int NTH = (W_MMA + 1) * 32;
constexpr int LD = state_ld(KD);       // partial row: 64 S + z + pad
constexpr int BLD = state_bf_ld(KD);   // bf16 state row

constexpr int O_ST = 0;
constexpr int O_ONE = O_ST + RST * STAGE;  // 16 rows x 128 B: logical column 0 is one, A's second atom
constexpr int O_SB = O_ONE + 2048;         // the combine's staging [64][LD] fp32, then the centre [64]
constexpr int SB = KD * LD * 4 + KD * 4;
constexpr int O_BAR = O_SB + SB;
// full[RST], scaled[RST], empty[RST], segf[2], sege[2], drain
constexpr int NBAR = 3 * RST + 5;
constexpr int O_DESC = O_BAR + 8 * NBAR;   // per stage: (sequence, head), segment end, halves
constexpr int O_MISC = O_DESC + 16 * RST;  // TMEM slot, fail, combine flag, first slot, count, pending
constexpr int SMEM = O_MISC + 48 + 1024;   // + alignment slack
constexpr int TMEM_COLS = 128;             // two 64-column accumulators
static_assert(SMEM <= 227 * 1024, "shared memory");
static_assert(O_ONE % 1024 == 0, "the constant block keeps the swizzle phase of a tile");

__device__ __forceinline__ uint32_t swz_off(int row, int chunk) {
  return (uint32_t)(row * 128 + ((chunk ^ (row & 7)) << 4));
}

// One unit = (256-row tile, head): sub-tile `sub` of tile ti of a.tiles,
// head h.  u = h (n_tiles spt) + ti spt + sub.
struct RTile {
  int h, b, seqh;   // head, sequence, b H + h (-1: no rows)
  int nval;         // valid rows in the tile (rows past them get gate 0)
  int halves;       // 128-row halves holding rows of the sequence slot (1 or 2)
  size_t rb;        // first row
};
__device__ __forceinline__ RTile rtile_at(const ReduceArgs& a, int u, int upt, int spt) {
  RTile x;
  x.h = u / upt;
  const int r = u - x.h * upt, ti = r / spt, sub = r - ti * spt;
  int row0, nvalid, tin;
  x.b = 0; x.nval = 0; x.rb = 0; x.seqh = -1; x.halves = 1;
  if (!map_tile(a.seq, a.tiles, ti, x.b, row0, nvalid, tin)) return x;
  const int R0 = tin * a.tiles.tile + sub * TT;
  // a tile without rows is no unit, except the first of an empty sequence:
  // its gates are all 0, so it leaves a zero partial and the state is zero
  const int rows = slot_rows(a.seq, nvalid);
  if (min(TT, rows - R0) <= 0 && !(rows == 0 && R0 == 0)) return x;
  x.halves = rows - R0 > KT ? 2 : 1;
  x.nval = max(0, min(TT, nvalid - R0));
  x.rb = (size_t)row0 + R0;
  x.seqh = x.b * a.H + x.h;
  return x;
}
// The next unit of [u, u1) with rows, from u on; u1 if none.
__device__ __forceinline__ int next_rtile(const ReduceArgs& a, int u, int u1, int upt, int spt, RTile& x) {
  for (; u < u1; ++u) {
    x = rtile_at(a, u, upt, spt);
    if (x.seqh >= 0) return u;
  }
  x.seqh = -1;
  return u1;
}
// The units with rows in [u0, u1).
__device__ __forceinline__ int n_tiles_cta(const ReduceArgs& a, int u0, int u1, int upt, int spt) {
  int n = 0;
  RTile x;
  for (int u = next_rtile(a, u0, u1, upt, spt, x); u < u1; u = next_rtile(a, u + 1, u1, upt, spt, x)) ++n;
  return n;
}
// The CTA whose range [floor(N c / G), floor(N (c + 1) / G)) holds unit u.
__device__ __forceinline__ int cta_of(int u, int n_units, int grid) {
  return (int)((((long long)u + 1) * grid + n_units - 1) / n_units) - 1;
}

// The state of one (sequence, head) from its partials in slots first ..
// first + count - 1, by NT threads (gt = thread index among them; bar = their
// named barrier, 0 for the whole CTA), with the arithmetic of combine_state in
// the same order: the partials summed in slot order; the public copy of
// [S | z]; the centre c_f = sum_e S[e][f] / sum_e z_e; S' = S - z c^T into the
// fp32 and bf16 states (z column kept).  combine_sum stages the sum in sb
// [64][LD]; combine_finish centres and writes it.  The partial loads of a
// thread are independent and issued together.
template <int NT>
__device__ void combine_sum(const ReduceArgs& a, int first, int count, int seqh, float* sb, int gt) {
  constexpr int N4 = KD * LD / 4;
  constexpr int PER = (N4 + NT - 1) / NT;
  const float4* __restrict__ P = reinterpret_cast<const float4*>(a.partial) + (size_t)first * N4;
  float4 acc[PER];
#pragma unroll
  for (int q = 0; q < PER; ++q) acc[q] = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int c = 0; c < count; ++c) {
    float4 v[PER];
#pragma unroll
    for (int q = 0; q < PER; ++q) {
      const int i = gt + q * NT;
      v[q] = i < N4 ? __ldcg(P + (size_t)c * N4 + i) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int q = 0; q < PER; ++q) {
      acc[q].x += v[q].x; acc[q].y += v[q].y; acc[q].z += v[q].z; acc[q].w += v[q].w;
    }
  }
#pragma unroll
  for (int q = 0; q < PER; ++q) {
    const int i = gt + q * NT;
    if (i >= N4) continue;
    reinterpret_cast<float4*>(sb)[i] = acc[q];
    if (a.pub_state) {
      const float v4[4] = {acc[q].x, acc[q].y, acc[q].z, acc[q].w};
#pragma unroll
      for (int w = 0; w < 4; ++w) {
        const int e = (4 * i + w) / LD, f = (4 * i + w) % LD;
        if (f <= KD) a.pub_state[((size_t)seqh * KD + e) * (KD + 1) + f] = v4[w];
      }
    }
  }
}
template <int NT>
__device__ void combine_finish(const ReduceArgs& a, int seqh, float* sb, float* cv, int gt, int bar) {
  constexpr int N4 = KD * LD / 4;
  if (a.center) {
    if (gt < KD) {
      float Z = 0.f, sf = 0.f;
#pragma unroll 16
      for (int e = 0; e < KD; ++e) Z += sb[e * LD + KD];
#pragma unroll 16
      for (int e = 0; e < KD; ++e) sf += sb[e * LD + gt];
      const float c = Z > 0.f ? sf / Z : 0.f;
      cv[gt] = c;
      a.center[(size_t)seqh * KD + gt] = c;
    }
    named_bar(bar, NT);
  }
  // S' = S - z c^T: LD = 72 floats a row, so a float4 never straddles a row
  float4* St = reinterpret_cast<float4*>(a.state + (size_t)seqh * KD * LD);
  for (int i = gt; i < N4; i += NT) {
    const int e = (4 * i) / LD, f = (4 * i) % LD;
    float4 v = reinterpret_cast<const float4*>(sb)[i];
    if (a.center && f < KD) {
      const float z = sb[e * LD + KD];
      v.x -= z * cv[f]; v.y -= z * cv[f + 1]; v.z -= z * cv[f + 2]; v.w -= z * cv[f + 3];
    }
    St[i] = v;
    if (a.state_bf)
      *reinterpret_cast<uint2*>(a.state_bf + ((size_t)seqh * KD + e) * BLD + f) =
          make_uint2(pack_bf16(v.x, v.y), pack_bf16(v.z, v.w));
  }
  if (a.state_bf)  // the row's last BLD - LD (= 8) columns
    for (int e = gt; e < KD; e += NT)
      *reinterpret_cast<uint4*>(a.state_bf + ((size_t)seqh * KD + e) * BLD + LD) = make_uint4(0u, 0u, 0u, 0u);
}
template <int NT>
__device__ void combine(const ReduceArgs& a, int first, int count, int seqh, float* sb, float* cv, int gt, int bar) {
  combine_sum<NT>(a, first, count, seqh, sb, gt);
  named_bar(bar, NT);
  combine_finish<NT>(a, seqh, sb, cv, gt, bar);
}
static_assert(LD % 4 == 0 && (BLD - LD) == 8 && BLD % 8 == 0, "vector stores of the state rows");

template <bool PRE>
__global__ void __launch_bounds__(NTH, 1)
    k_reduce_tc(const ReduceArgs a, const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                int upt, int spt, int n_units) {
  if (threadIdx.x == W_PROD * 32) {  // the descriptors load while the previous kernel finishes
    tma_prefetch_map(&tmK);
    tma_prefetch_map(&tmV);
  }
  pdl_enter();  // the previous kernel's outputs are visible from here on
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_align1024(smem_raw);
  const uint32_t sbase = smem_u32(smem);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (a.err && *a.err) return;
  const int G = gridDim.x, nseq = a.seq.n_seq;
  const int u0 = (int)(((long long)n_units * blockIdx.x) / G);
  const int u1 = (int)(((long long)n_units * (blockIdx.x + 1)) / G);
  {
    RTile x;
    if (next_rtile(a, u0, u1, upt, spt, x) >= u1) return;  // no rows in this range
  }
  uint32_t* slot = reinterpret_cast<uint32_t*>(smem + O_MISC);
  volatile int* fail = reinterpret_cast<volatile int*>(smem + O_MISC + 4);
  // combine flag, first slot, count, and the (sequence, head) whose combine waits for the end (-1: none)
  volatile int* gf = reinterpret_cast<volatile int*>(smem + O_MISC + 16);
  int* desc = reinterpret_cast<int*>(smem + O_DESC);  // [stage][seqh, segment end, halves, -]
  const uint32_t bar0 = sbase + O_BAR;
  auto FULL = [&](int s) { return bar0 + 8 * s; };
  auto SCALED = [&](int s) { return bar0 + 8 * (RST + s); };
  auto EMPTY = [&](int s) { return bar0 + 8 * (2 * RST + s); };
  auto SEGF = [&](int b) { return bar0 + 8 * (3 * RST + b); };
  auto SEGE = [&](int b) { return bar0 + 8 * (3 * RST + 2 + b); };
  const uint32_t DRAIN = bar0 + 8 * (3 * RST + 4);
  if (tid == 0) {
    for (int s = 0; s < RST; ++s) {
      mbar_init(FULL(s), 1);
      mbar_init(SCALED(s), 4 * NG);  // the eight transform warps
      mbar_init(EMPTY(s), 1);        // the MMA commit
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(SEGF(b), 1);
      mbar_init(SEGE(b), 1);
    }
    mbar_init(DRAIN, 1);
    mbar_init_fence();
    *fail = 0;
    gf[0] = 0;
    gf[3] = -1;
  }
  if (tid < 16)  // the constant block: row r holds (1, 0, ..., 0); swz_off places logical chunk c
#pragma unroll
    for (int c = 0; c < 8; ++c)
      *reinterpret_cast<uint4*>(smem + O_ONE + swz_off(tid, c)) = make_uint4(c == 0 ? pack_bf16(1.f, 0.f) : 0u, 0u, 0u, 0u);
  fence_async_smem();
  if (warp == 0) tmem_alloc(smem_u32(slot), TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *slot;

  if (warp == W_PROD) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int j = 0;
      int last_s[RST];
#pragma unroll
      for (int s = 0; s < RST; ++s) last_s[s] = 0;
      RTile x, y;
      int u = next_rtile(a, u0, u1, upt, spt, x);
      while (u < u1 && !*fail) {
        const int un = next_rtile(a, u + 1, u1, upt, spt, y);
        const int s = j % RST;
        if (j >= RST && !mbar_wait(EMPTY(s), ((j / RST) - 1) & 1, fail)) break;
        desc[4 * s + 0] = x.seqh;
        desc[4 * s + 1] = (un >= u1 || y.seqh != x.seqh) ? 1 : 0;
        desc[4 * s + 2] = x.halves;
        const uint32_t st = sbase + O_ST + s * STAGE;
        mbar_expect_tx(FULL(s), 2 * x.halves * TILE);
        for (int hf = 0; hf < x.halves; ++hf) {
          tma_load_2d(st + hf * TILE, &tmK, FULL(s), x.h * KD, (int)x.rb + hf * KT);
          tma_load_2d(st + (2 + hf) * TILE, &tmV, FULL(s), x.h * KD, (int)x.rb + hf * KT);
        }
        last_s[s] = j + 1;
        u = un;
        x = y;
        ++j;
      }
      if (*fail)  // let the copies still in flight land
        for (int s = 0; s < RST; ++s)
          if (last_s[s] > 0)
            for (uint32_t it = 0; it < kPollLimit && !mbar_try_wait(FULL(s), (uint32_t)((last_s[s] - 1) / RST) & 1);
                 ++it) {
            }
    }
  } else if (warp == W_MMA) {
    // ---------------------------------------------------------- MMA issuer
    if (lane == 0) {
      const uint32_t id = idesc_bf16(128, KD, true, true);
      int k = -1, prev = -1;
      const int nj = n_tiles_cta(a, u0, u1, upt, spt);
      for (int j = 0; j < nj && !*fail; ++j) {
        const int s = j % RST;
        if (!mbar_wait(SCALED(s), (j / RST) & 1, fail)) break;
        tc_fence_after();
        const int seqh = desc[4 * s + 0], last = desc[4 * s + 1], halves = desc[4 * s + 2];
        bool first = false;
        if (seqh != prev) {  // a new segment: its accumulator is drained by now
          ++k;
          prev = seqh;
          first = true;
          if (k >= 2 && !mbar_wait(SEGE(k & 1), ((k >> 1) - 1) & 1, fail)) break;
          tc_fence_after();
        }
        const uint32_t st = sbase + O_ST + s * STAGE;
        for (int kk = 0; kk < 8 * halves; ++kk) {
          // K step kk: rows 16 kk .. of the tile, in the half kk / 8.  A's
          // second 64-row atom is the constant block, the same 16 rows for
          // every step (rows 16 apart share the swizzle phase).
          const uint32_t off = (kk >> 3) * TILE + 2048 * (kk & 7);
          const uint32_t a0 = st + 2 * TILE + off;
          tc_mma(tmem + (k & 1) * KD, sdesc(a0, sbase + O_ONE - a0, 1024), sdesc(st + off, 8192, 1024), id,
                 (first && kk == 0) ? 0u : 1u);
        }
        tc_commit(EMPTY(s));
        if (last) tc_commit(SEGF(k & 1));
      }
      tc_commit(DRAIN);  // completes once every MMA issued above has finished
      for (uint32_t it = 0; it < kPollLimit && !mbar_try_wait(DRAIN, 0); ++it) {
      }
    }
  } else if (warp < W_DRAIN) {
    // ------------------------------------------------ transform groups
    const int grp = warp >> 2, wq = warp & 3;
    const int row = grp * KT + wq * 32 + lane;  // tile row
    auto gate_of = [&](const RTile& t) { return row < t.nval ? __ldg(a.g + (t.rb + row) * a.ldg + t.h) : 0.f; };
    // every tile; the gate of the next one loads under the current one
    int j = 0;
    RTile x;
    int u = next_rtile(a, u0, u1, upt, spt, x);
    float g = u < u1 ? gate_of(x) : 0.f;
    while (u < u1) {
      RTile xn;
      const int un = next_rtile(a, u + 1, u1, upt, spt, xn);
      const float gn = un < u1 ? gate_of(xn) : 0.f;
      const int s = j % RST;
      mbar_wait(FULL(s), (j / RST) & 1, fail);
      if (grp < x.halves) {  // k~ = bf16(g phi(k)) over this thread's row, in place
        uint8_t* sk = smem + O_ST + s * STAGE + grp * TILE;
        const int r = wq * 32 + lane;
        uint4 w4[8];
#pragma unroll
        for (int c = 0; c < 8; ++c) w4[c] = *reinterpret_cast<const uint4*>(sk + swz_off(r, c));
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          const uint32_t w[4] = {w4[c].x, w4[c].y, w4[c].z, w4[c].w};
          uint32_t o[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const float lo = PRE ? bf_lo(w[i]) : phi_f(bf_lo(w[i]));
            const float hi = PRE ? bf_hi(w[i]) : phi_f(bf_hi(w[i]));
            o[i] = pack_bf16(lo * g, hi * g);
          }
          *reinterpret_cast<uint4*>(sk + swz_off(r, c)) = make_uint4(o[0], o[1], o[2], o[3]);
        }
        fence_async_smem();
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(SCALED(s));
      x = xn;
      u = un;
      g = gn;
      ++j;
    }
  } else {
    // ------------------------------------------------------ drain group
    const int wq = warp & 3;
    const int row = wq * 32 + lane;  // TMEM lane
    float* sb = reinterpret_cast<float*>(smem + O_SB);
    int k = -1, prev = -1;
    RTile x, y;
    int u = next_rtile(a, u0, u1, upt, spt, x);
    while (u < u1) {
      const int un = next_rtile(a, u + 1, u1, upt, spt, y);
      const bool last = un >= u1 || y.seqh != x.seqh;
      if (x.seqh != prev) {
        ++k;
        prev = x.seqh;
      }
      if (last) {
        // segment k ends here: [S | z]^T (TMEM lane f = column f of the state,
        // lane 64 = z; column e = row e) is this CTA's partial of the pair
        mbar_wait(SEGF(k & 1), (k >> 1) & 1, fail);
        tc_fence_after();
        const int p = x.h * nseq + x.b;
        const uint32_t tl = tmem + ((uint32_t)(wq * 32) << 16) + (k & 1) * KD;
        if (row == 0) {  // the CTAs holding units of (b, h): c0 .. c0 + count - 1
          int first, cnt;
          seq_tiles(a.seq, a.tiles, x.b, first, cnt);
          const int U0 = x.h * upt + spt * first;
          int U1 = U0 + spt * max(cnt, 1) - 1;  // the pair's last unit with rows
          while (U1 > U0 && rtile_at(a, U1, upt, spt).seqh < 0) --U1;
          const int c0 = cta_of(U0, n_units, G), count = cta_of(U1, n_units, G) - c0 + 1;
          // every other CTA of the pair has left its partial already: this one
          // completes the pair straight from TMEM
          const int done = *reinterpret_cast<volatile int*>(a.counters + x.seqh);
          gf[0] = (done == count - 1 && !*fail) ? 2 : 0;
          gf[1] = p + c0;
          gf[2] = count;
        }
        named_bar(1, 128);
        if (gf[0] == 2) {
          __threadfence();
          // the sum over the pair's partials in slot order, this CTA's own
          // (slot p + blockIdx.x) from TMEM, into the staging
          const int first = gf[1], count = gf[2], q = p + blockIdx.x - first;
#pragma unroll
          for (int qq = 0; qq < 4; ++qq) {  // 16 state rows at a time
            uint32_t v[16];
            tmem_ld16(tl + 16 * qq, v);
            float acc[16];
#pragma unroll
            for (int e = 0; e < 16; ++e) acc[e] = 0.f;
            if (row < LD) {
              for (int c = 0; c < count; ++c) {
                if (c == q) {
#pragma unroll
                  for (int e = 0; e < 16; ++e) acc[e] += row <= KD ? __uint_as_float(v[e]) : 0.f;
                } else {
                  const float* Pc = a.partial + ((size_t)(first + c) * KD + 16 * qq) * LD + row;
                  float w[16];
#pragma unroll
                  for (int e = 0; e < 16; ++e) w[e] = __ldcg(Pc + (size_t)e * LD);
#pragma unroll
                  for (int e = 0; e < 16; ++e) acc[e] += w[e];
                }
              }
#pragma unroll
              for (int e = 0; e < 16; ++e) {
                const int E = 16 * qq + e;
                sb[E * LD + row] = acc[e];
                if (a.pub_state && row <= KD) a.pub_state[((size_t)x.seqh * KD + E) * (KD + 1) + row] = acc[e];
              }
            }
          }
          tc_fence_before();
          named_bar(1, 128);
          if (row == 0) {
            mbar_arrive(SEGE(k & 1));  // the accumulator is read
            atomicAdd(a.counters + x.seqh, 1);
          }
          combine_finish<128>(a, x.seqh, sb, sb + KD * LD, row, 1);
          named_bar(1, 128);  // the staging and the flags are free again
        } else {
          float* P = a.partial + (size_t)(p + blockIdx.x) * KD * LD;
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            uint32_t v[32];
            tmem_ld32(tl + 32 * hh, v);
            if (row < LD)
#pragma unroll
              for (int e = 0; e < 32; ++e) P[(size_t)(32 * hh + e) * LD + row] = row <= KD ? __uint_as_float(v[e]) : 0.f;
          }
          tc_fence_before();
          __threadfence();
          named_bar(1, 128);
          if (row == 0) {
            mbar_arrive(SEGE(k & 1));  // the accumulator is read
            const bool lastp = atomicAdd(a.counters + x.seqh, 1) == gf[2] - 1;
            gf[0] = (lastp && !*fail) ? 1 : 0;
          }
          named_bar(1, 128);
          if (gf[0]) {  // this partial completes (b, h)
            if (un >= u1) {  // the CTA's last segment: every warp combines it after the loops
              if (row == 0) gf[3] = x.seqh;
            } else {
              __threadfence();
              combine<128>(a, gf[1], gf[2], x.seqh, sb, sb + KD * LD, row, 1);
              named_bar(1, 128);  // the staging and the flags are free again
            }
          }
        }
      }
      u = un;
      x = y;
    }
  }
  __syncwarp();  // single-lane roles rejoin their warps: the CTA barrier below is warp-aligned
  __syncthreads();
  if (gf[0] == 1 && gf[3] >= 0 && !*fail) {
    __threadfence();
    combine<NTH>(a, gf[1], gf[2], gf[3], reinterpret_cast<float*>(smem + O_SB),
                 reinterpret_cast<float*>(smem + O_SB) + KD * LD, tid, 0);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, TMEM_COLS);
  if (*fail && tid == 0 && a.err_out) atomicOr(a.err_out, kErrTimeout);
}

}  // namespace

cudaError_t launch_reduce_tc(const ReduceArgs& a, int n_tiles, cudaStream_t st) {
  auto al16 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; };
  if (a.dh != KD || a.gate_kind != GATE_VALUES || !al16(a.k) || !al16(a.v) || !al16(a.partial) || a.ldk % 8 ||
      a.ldv % 8 || a.seq.T <= 0 || n_tiles <= 0 || a.tiles.tile % TT)
    return cudaErrorNotSupported;
  const int spt = a.tiles.tile / TT, upt = n_tiles * spt, n_units = upt * a.H;
  int grid = n_units < sm_count() ? n_units : sm_count();
  const int room = a.partial_slots - a.seq.n_seq * a.H;  // partial slots beyond one per (sequence, head)
  if (room < grid) grid = room;
  if (grid <= 0) return cudaErrorNotSupported;
  CUtensorMap tmK, tmV;
  const uint64_t hd = (uint64_t)a.H * KD;  // the heads' columns of a row
  // 128-byte L2 promotion: a box row is one head's 128 bytes
  if (!make_map(&tmK, a.k, hd, (uint64_t)a.seq.T, (uint64_t)a.ldk, 64, KT, false) ||
      !make_map(&tmV, a.v, hd, (uint64_t)a.seq.T, (uint64_t)a.ldv, 64, KT, false))
    return cudaErrorNotSupported;
  auto kern = a.pre ? k_reduce_tc<true> : k_reduce_tc<false>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM);
  if (e != cudaSuccess) return e;
  return launch_pdl(kern, dim3(grid), dim3(NTH), SMEM, st, a, tmK, tmV, upt, spt, n_units);
}

}  // namespace gbla
