// Shared device-side helpers of the GBLA kernels: sequence/tile mapping,
// bf16 packing, the phi feature map, and thin inline-PTX wrappers (cp.async,
// ldmatrix, mma.sync m16n8k16 bf16).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace gbla {

typedef __nv_bfloat16 bf16;

// ------------------------------------------------------------ sequence map
//
// A call's rows are split into sequences in one of three forms:
//   DENSE  : B slots of L rows, all valid
//   PADDED : B slots of L rows, the first lens[b] valid
//   VARLEN : sequence b is rows cu[b] .. cu[b+1]-1 of T rows
// Work is cut into fixed tiles of `tile` rows per sequence.  Dense/padded
// sequences all have ceil(L / tile) tiles (rows past the valid length are
// masked); varlen sequences have max(1, ceil(len / tile)) tiles, counted by
// a device-side prefix sum (plan kernel) so the host never reads cu_seqlens.
enum SeqMode { SEQ_DENSE = 0, SEQ_PADDED = 1, SEQ_VARLEN = 2 };

struct SeqDesc {
  int mode;
  int n_seq;
  int L;  // slot length (dense/padded) or T (varlen)
  int T;  // total rows
  const int32_t* lens;
  const int32_t* cu;
};

// Walks the rows of the sequences: for row l gives the first row s0 of its
// sequence, the end of its valid rows vend and the end of its slot send.
struct SeqCursor {
  const SeqDesc& s;
  int b, s0, vend, send;
  __device__ explicit SeqCursor(const SeqDesc& sd) : s(sd), b(0), s0(0), vend(0), send(0) {}
  __device__ void seek(int l) {
    if (s.mode != SEQ_VARLEN) {
      b = l / s.L;
      s0 = b * s.L;
      send = s0 + s.L;
      vend = s0 + (s.mode == SEQ_PADDED ? s.lens[b] : s.L);
    } else {
      int lo = 0, hi = s.n_seq - 1;  // last b with cu[b] <= l
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (s.cu[mid] <= l) lo = mid; else hi = mid - 1;
      }
      b = lo;
      while (b + 1 < s.n_seq && s.cu[b + 1] <= l) ++b;  // skip empty sequences
      s0 = s.cu[b];
      vend = send = s.cu[b + 1];
    }
  }
};

struct Tiling {
  int tile;               // rows per tile
  int per_seq;            // dense/padded: tiles per sequence
  const int32_t* prefix;  // varlen: [n_seq + 1] tile prefix (device)
};

// Maps a linear tile index to (sequence, first row of the sequence, number
// of valid rows of the sequence, tile index inside the sequence).  Returns
// false when the index lies past the last tile.
__device__ __forceinline__ bool map_tile(const SeqDesc& s, const Tiling& t, int idx, int& b,
                                         int& row0, int& nvalid, int& tin) {
  if (s.mode != SEQ_VARLEN) {
    b = idx / t.per_seq;
    if (b >= s.n_seq) return false;
    tin = idx - b * t.per_seq;
    row0 = b * s.L;
    nvalid = s.mode == SEQ_PADDED ? s.lens[b] : s.L;
    return true;
  }
  const int total = t.prefix[s.n_seq];
  if (idx >= total) return false;
  int lo = 0, hi = s.n_seq - 1;  // last b with prefix[b] <= idx
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (t.prefix[mid] <= idx) lo = mid; else hi = mid - 1;
  }
  b = lo;
  tin = idx - t.prefix[b];
  row0 = s.cu[b];
  nvalid = s.cu[b + 1] - s.cu[b];
  return true;
}

// Number of tiles of sequence b and the linear index of its first tile.
__device__ __forceinline__ void seq_tiles(const SeqDesc& s, const Tiling& t, int b, int& first,
                                          int& count) {
  if (s.mode != SEQ_VARLEN) {
    first = b * t.per_seq;
    count = t.per_seq;
  } else {
    first = t.prefix[b];
    count = t.prefix[b + 1] - t.prefix[b];
  }
}

// Rows of a sequence slot that tiles cover: L for dense/padded, len for varlen.
__device__ __forceinline__ int slot_rows(const SeqDesc& s, int nvalid) {
  return s.mode == SEQ_VARLEN ? nvalid : s.L;
}

// ------------------------------------------------------------ arithmetic

// phi(x) = elu(x) + 1 (alpha = 1): x + 1 for x > 0, e^x otherwise.
__device__ __forceinline__ float phi_f(float x) { return x > 0.f ? x + 1.f : __expf(x); }
// phi'(x): 1 for x > 0, e^x otherwise.
__device__ __forceinline__ float dphi_f(float x) { return x > 0.f ? 1.f : __expf(x); }

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}
__device__ __forceinline__ float bf_lo(uint32_t v) {
  return __uint_as_float(v << 16);
}
__device__ __forceinline__ float bf_hi(uint32_t v) {
  return __uint_as_float(v & 0xffff0000u);
}

template <typename T> __device__ __forceinline__ float to_f(T v);
template <> __device__ __forceinline__ float to_f<float>(float v) { return v; }
template <> __device__ __forceinline__ float to_f<bf16>(bf16 v) { return __bfloat162float(v); }
template <typename T> __device__ __forceinline__ T from_f(float v);
template <> __device__ __forceinline__ float from_f<float>(float v) { return v; }
template <> __device__ __forceinline__ bf16 from_f<bf16>(float v) { return __float2bfloat16_rn(v); }

// ------------------------------------------------------------ PTX wrappers

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// 16-byte global -> shared copy; bytes past src_bytes (0 or 16) are zero-filled.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, int src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src),
               "r"(src_bytes));
}
__device__ __forceinline__ void cp_async4(uint32_t dst, const void* src, int src_bytes) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;\n" ::"r"(dst), "l"(src),
               "r"(src_bytes));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::); }
template <int N> __device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N));
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                          uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

// D = A (16x16, row) * B (16x8, col) + D, bf16 inputs, fp32 accumulate.
__device__ __forceinline__ void mma_bf16(float* c, uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Byte offset of 16-byte chunk c of row r in a row-major bf16 tile with CPR
// chunks per row, XOR-swizzled so that ldmatrix (8 rows, one chunk column)
// touches 8 distinct bank groups.
template <int CPR>
__device__ __forceinline__ uint32_t swz(int r, int c) {
  int p;
  if (CPR >= 8) p = (c & ~7) | ((c ^ r) & 7);
  else if (CPR == 4) p = c ^ ((r >> 1) & 3);
  else p = c ^ ((r >> 2) & 1);
  return static_cast<uint32_t>(r * CPR * 16 + p * 16);
}

}  // namespace gbla
