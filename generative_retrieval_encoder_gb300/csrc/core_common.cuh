// Pieces shared by the fp32 and bf16 state kernels: the deterministic
// split-L combine of per-chunk partial states.
#pragma once

#include "kernels.h"

namespace gbla {

// Every CTA of a (sequence, head) calls this after writing its partial.  The
// CTA that arrives last (atomic ticket; no CTA ever waits) gets `true` and
// then owns the combine.  Counters are zeroed by the host before the launch.
__device__ __forceinline__ bool arrive_last(int* counter, int count) {
  __shared__ int s_last;
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) s_last = (atomicAdd(counter, 1) == count - 1);
  __syncthreads();
  const bool last = s_last != 0;
  if (last) __threadfence();
  return last;
}

// The threads that run a combine: the first n of the CTA (whole warps),
// synchronised by named barrier `id`; id 0 stands for the whole CTA.
struct Team {
  int n, id;
};
__device__ __forceinline__ void team_sync(const Team& t) {
  if (t.id == 0)
    __syncthreads();
  else
    asm volatile("bar.sync %0, %1;" ::"r"(t.id), "r"(t.n) : "memory");
}

// Dot products of length dh spread over a team of nt threads: `per` threads (a
// power of two, at most 32) share one, each summing every per-th term, and a
// butterfly of shuffles adds their sums (the same value in every lane of the
// group, since fp32 addition commutes).  Rows are visited in passes of
// nt / per; every thread of the team runs every pass, so the shuffles see
// whole warps (nt is a multiple of 32).  term(r, t) is the t-th term of row r;
// done(r, sum) is called by the group's first thread.
__device__ __forceinline__ int dot_split(int dh, int nt) {
  int per = 32;
  while (per > 1 && per * dh > nt) per >>= 1;
  return per;
}
template <class Term, class Done>
__device__ __forceinline__ void rows_dot(int rows, int dh, int nt, Term term, Done done) {
  const int per = dot_split(dh, nt), rpp = nt / per;
  const int j = threadIdx.x % per;
  for (int r0 = 0; r0 < rows; r0 += rpp) {
    const int r = r0 + threadIdx.x / per;
    const bool on = r < rows && (int)threadIdx.x < rpp * per;
    float acc = 0.f;
    if (on) {
#pragma unroll 8
      for (int t = j; t < dh; t += per) acc += term(r, t);
    }
    for (int o = per >> 1; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    if (on && j == 0) done(r, acc);
  }
}

// state[seqh] = sum over the sequence's chunks c = 0 .. count-1, in that
// order, of scale_c * partial[(first + c) * H + h].  scale_c = 1, or for
// softmax logits exp(m_c - m) with m the largest chunk maximum (the softmax
// normaliser cancels in Eq. 5, so only relative scales matter).
// Also writes the compact public copy [dh][dh+1] of [S | z] and m.
//
// Centering (center != null): for any constant vector c,
//   o_i = S^T q~_i / z.q~_i = c + (S - z c^T)^T q~_i / z.q~_i,
// so the kernels may work with S' = S - z c^T.  With c the k~-weighted mean
// of v, c_f = sum_e S[e][f] / sum_e z_e, S' holds only the spread of v around
// its mean; the differences that the backward takes (S - z o^T, dS v + dz)
// then no longer cancel in bf16 operands.  S' is formed here in fp32; c goes
// to center[seqh][dh].  Then `state` and the bf16 copy hold [S' | z | 0].
//
// Backward use (fwd_center != null, the combine of [dS | dz']): the key side
// computes dk~_j = dS (v_j - c) + dz'.  So that it can feed the exact bf16
// v_j to the tensor cores, the z column is replaced here, in fp32, by
// dz'' = dz' - bf16(dS) c, using the same bf16-rounded dS that the key side
// multiplies with: then bf16(dS) v_j + dz'' = bf16(dS) (v_j - c) + dz' exactly
// up to fp32 rounding, and no rounding of (v_j - c) enters the gate gradient
// (whose sum over a sequence cancels to ~1/sqrt(L) of its terms).
//
// sbuf (optional, 16-byte aligned shared memory of dh * state_ld(dh) floats):
// the combined state is staged there as well, so that the centring passes
// read shared memory instead of the global copy just written.
// team_n, team_id: the combine runs on the first team_n threads of the CTA,
// which meet at named barrier team_id (0: every thread, __syncthreads).
__device__ inline void combine_state(const float* partial, const float* partial_m, int first,
                                     int count, int H, int h, int dh, int seqh, bool logits,
                                     float* state, bf16* state_bf, float* state_m,
                                     float* pub_state, float* center = nullptr,
                                     const float* fwd_center = nullptr, float* sbuf = nullptr,
                                     int team_n = 0, int team_id = 0) {
  const Team team{team_n ? team_n : (int)blockDim.x, team_n ? team_id : 0};
  const int nt = team.n;
  const int LD = state_ld(dh);
  const int n = dh * LD;
  float m = 0.f;
  bool any = true;
  if (logits) {
    m = -INFINITY;
    for (int c = 0; c < count; ++c) m = fmaxf(m, __ldcg(partial_m + (size_t)(first + c) * H + h));
    any = m > -INFINITY;
    if (threadIdx.x == 0 && state_m) state_m[seqh] = any ? m : 0.f;
  }
  const float4* P = reinterpret_cast<const float4*>(partial);
  float4* S = reinterpret_cast<float4*>(state + (size_t)seqh * n);
  // Each thread sums PER float4s at a time, so that a partial's PER loads are
  // in flight together (the partials live in L2, whose latency the sum would
  // otherwise pay once per float4 and partial).
  constexpr int PER = 5;
  const int n4 = n / 4;
  for (int i0 = threadIdx.x; i0 < n4; i0 += PER * nt) {
    float4 acc[PER];
#pragma unroll
    for (int u = 0; u < PER; ++u) acc[u] = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int c = 0; c < count; ++c) {
      const float4* Pc = P + ((size_t)(first + c) * H + h) * n4;
      float4 p[PER];
#pragma unroll
      for (int u = 0; u < PER; ++u) {
        const int i = i0 + u * nt;
        p[u] = i < n4 ? __ldcg(Pc + i) : make_float4(0.f, 0.f, 0.f, 0.f);
      }
      float sc = 1.f;
      if (logits) {
        const float mc = __ldcg(partial_m + (size_t)(first + c) * H + h);
        sc = (any && mc > -INFINITY) ? __expf(mc - m) : 0.f;
      }
#pragma unroll
      for (int u = 0; u < PER; ++u) {
        acc[u].x += sc * p[u].x; acc[u].y += sc * p[u].y;
        acc[u].z += sc * p[u].z; acc[u].w += sc * p[u].w;
      }
    }
#pragma unroll
    for (int u = 0; u < PER; ++u) {
      const int i = i0 + u * nt;
      if (i >= n4) continue;
      S[i] = acc[u];
      if (sbuf) reinterpret_cast<float4*>(sbuf)[i] = acc[u];
      const float v4[4] = {acc[u].x, acc[u].y, acc[u].z, acc[u].w};
#pragma unroll
      for (int w = 0; w < 4; ++w) {
        const int e = (4 * i + w) / LD, f = (4 * i + w) % LD;
        if (state_bf && !center) state_bf[((size_t)seqh * dh + e) * state_bf_ld(dh) + f] = __float2bfloat16_rn(v4[w]);
        if (pub_state && f <= dh) pub_state[((size_t)seqh * dh + e) * (dh + 1) + f] = v4[w];
      }
    }
  }
  // the combined state as later passes read it: the staged copy, else the global one
  const float* Sr = sbuf ? sbuf : state + (size_t)seqh * n;
  if (fwd_center) {
    float* St = state + (size_t)seqh * n;
    team_sync(team);  // the team's state writes are visible to the whole team
    const float* c = fwd_center + (size_t)seqh * dh;
    rows_dot(
        dh, dh, nt, [&](int e, int f) { return __bfloat162float(__float2bfloat16_rn(Sr[e * LD + f])) * __ldg(c + f); },
        [&](int e, float dot) {
          const float acc = Sr[e * LD + dh] - dot;
          St[e * LD + dh] = acc;
          if (state_bf) state_bf[((size_t)seqh * dh + e) * state_bf_ld(dh) + dh] = __float2bfloat16_rn(acc);
        });
  }
  if (center) {
    __shared__ float cbuf[129];  // column sums of S, then sum_e z_e
    float* St = state + (size_t)seqh * n;
    team_sync(team);  // the team's state writes are visible to the whole team
    // column f < dh: sum_e S[e][f]; "column" dh: Z = sum_e z_e
    rows_dot(dh + 1, dh, nt, [&](int f, int e) { return Sr[e * LD + f]; }, [&](int f, float sum) { cbuf[f] = sum; });
    team_sync(team);
    const float Z = cbuf[dh];
    team_sync(team);  // every thread has read Z before cbuf[f] becomes c_f
    for (int f = threadIdx.x; f < dh; f += nt) {
      const float c = Z > 0.f ? cbuf[f] / Z : 0.f;
      cbuf[f] = c;
      center[(size_t)seqh * dh + f] = c;
    }
    team_sync(team);
    for (int i = threadIdx.x; i < n; i += nt) {
      const int e = i / LD, f = i % LD;
      float v = Sr[i];
      if (f < dh) {
        v -= Sr[e * LD + dh] * cbuf[f];
      }
      if (state_bf) state_bf[((size_t)seqh * dh + e) * state_bf_ld(dh) + f] = __float2bfloat16_rn(v);
      St[i] = v;  // the z column (f == dh), which other threads read, is left unchanged
    }
  }
  if (state_bf) {
    const int BLD = state_bf_ld(dh);
    for (int i = threadIdx.x; i < dh * (BLD - LD); i += nt) {
      const int e = i / (BLD - LD), f = LD + i % (BLD - LD);
      state_bf[((size_t)seqh * dh + e) * BLD + f] = __float2bfloat16_rn(0.f);
    }
  }
}

}  // namespace gbla
