// Device helpers shared by the libkvb kernels (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "kvb_internal.h"

namespace kvb {

constexpr unsigned kFull = 0xffffffffu;
constexpr int kMaxTok = 64 + 1;  // buffered tokens (capacity) + the current one

enum Variant { kPlain = 0, kGated = 1, kGatedDelta = 2 };

// ---------------------------------------------------------------- loads / stores
// The state is streamed once per step: read and written with the evict-first
// (".cs") policy so it does not push reusable data (buffer, q/k) out of L2.
__device__ __forceinline__ float4 ld_stream4(const float *p) {
  return __ldcs(reinterpret_cast<const float4 *>(p));
}
__device__ __forceinline__ void st_stream4(float *p, float4 v) {
  __stcs(reinterpret_cast<float4 *>(p), v);
}

// Four consecutive elements of a q/k/v row, widened to fp32.
__device__ __forceinline__ float4 ld4(const float *p) {
  return *reinterpret_cast<const float4 *>(p);
}
__device__ __forceinline__ float4 ld4(const __nv_bfloat16 *p) {
  uint2 raw = *reinterpret_cast<const uint2 *>(p);
  __nv_bfloat162 lo = *reinterpret_cast<__nv_bfloat162 *>(&raw.x);
  __nv_bfloat162 hi = *reinterpret_cast<__nv_bfloat162 *>(&raw.y);
  float2 a = __bfloat1622float2(lo), b = __bfloat1622float2(hi);
  return make_float4(a.x, a.y, b.x, b.y);
}
// Two consecutive elements, widened.
__device__ __forceinline__ float2 ld2(const float *p) {
  return *reinterpret_cast<const float2 *>(p);
}
__device__ __forceinline__ float2 ld2(const __nv_bfloat16 *p) {
  return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(p));
}

// Store four fp32 values into a row of the storage dtype.  Values stored here
// were read from the same dtype, so narrowing back is exact.
__device__ __forceinline__ void st4(float *p, float4 v) { *reinterpret_cast<float4 *>(p) = v; }
__device__ __forceinline__ void st4(__nv_bfloat16 *p, float4 v) {
  __nv_bfloat162 lo = __floats2bfloat162_rn(v.x, v.y);
  __nv_bfloat162 hi = __floats2bfloat162_rn(v.z, v.w);
  uint2 raw;
  raw.x = *reinterpret_cast<uint32_t *>(&lo);
  raw.y = *reinterpret_cast<uint32_t *>(&hi);
  *reinterpret_cast<uint2 *>(p) = raw;
}

__device__ __forceinline__ float to_float(float x) { return x; }
__device__ __forceinline__ float to_float(__nv_bfloat16 x) { return __bfloat162float(x); }

// Dot product of E consecutive fp32 values from two shared-memory rows.
template <int E>
__device__ __forceinline__ float dot_smem(const float *a, const float *b) {
  if constexpr (E == 4) {
    const float4 x = *reinterpret_cast<const float4 *>(a), y = *reinterpret_cast<const float4 *>(b);
    return x.x * y.x + x.y * y.y + x.z * y.z + x.w * y.w;
  } else {
    const float2 x = *reinterpret_cast<const float2 *>(a), y = *reinterpret_cast<const float2 *>(b);
    return x.x * y.x + x.y * y.y;
  }
}

__device__ __forceinline__ float4 f4(float a) { return make_float4(a, a, a, a); }
__device__ __forceinline__ void fma4(float4 &acc, float s, float4 x) {
  acc.x = fmaf(s, x.x, acc.x);
  acc.y = fmaf(s, x.y, acc.y);
  acc.z = fmaf(s, x.z, acc.z);
  acc.w = fmaf(s, x.w, acc.w);
}
__device__ __forceinline__ float4 add4(float4 a, float4 b) {
  return make_float4(a.x + b.x, a.y + b.y, a.z + b.z, a.w + b.w);
}
__device__ __forceinline__ float4 mul4(float s, float4 a) {
  return make_float4(s * a.x, s * a.y, s * a.z, s * a.w);
}

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) x += __shfl_xor_sync(kFull, x, off);
  return x;
}
// Sum over the 8 lanes that share (lane & 3): the row-split of the state tile.
__device__ __forceinline__ float rows_sum(float x) {
  x += __shfl_xor_sync(kFull, x, 4);
  x += __shfl_xor_sync(kFull, x, 8);
  x += __shfl_xor_sync(kFull, x, 16);
  return x;
}
__device__ __forceinline__ float4 rows_sum4(float4 v) {
  return make_float4(rows_sum(v.x), rows_sum(v.y), rows_sum(v.z), rows_sum(v.w));
}

// Sums of four per-lane values over the warp in 18 instructions instead of 40:
// lane L ends with the total of v[2 * ((L >> 4) & 1) + ((L >> 3) & 1)], so lanes
// 0, 8, 16, 24 hold the totals of v0, v1, v2, v3.
__device__ __forceinline__ float butterfly4(float v0, float v1, float v2, float v3, int lane) {
  const bool hi = lane & 16;
  float k0 = hi ? v2 : v0, k1 = hi ? v3 : v1;
  k0 += __shfl_xor_sync(kFull, hi ? v0 : v2, 16);
  k1 += __shfl_xor_sync(kFull, hi ? v1 : v3, 16);
  const bool b3 = lane & 8;
  float k = b3 ? k1 : k0;
  k += __shfl_xor_sync(kFull, b3 ? k0 : k1, 8);
  k += __shfl_xor_sync(kFull, k, 4);
  k += __shfl_xor_sync(kFull, k, 2);
  k += __shfl_xor_sync(kFull, k, 1);
  return k;
}
// Two values: lane L ends with the total of v[(L >> 4) & 1] (lanes 0 and 16).
__device__ __forceinline__ float butterfly2(float v0, float v1, int lane) {
  const bool hi = lane & 16;
  float k = hi ? v1 : v0;
  k += __shfl_xor_sync(kFull, hi ? v0 : v1, 16);
  k += __shfl_xor_sync(kFull, k, 8);
  k += __shfl_xor_sync(kFull, k, 4);
  k += __shfl_xor_sync(kFull, k, 2);
  k += __shfl_xor_sync(kFull, k, 1);
  return k;
}

// E consecutive elements of a key row, widened to fp32.
template <int E, typename KT>
__device__ __forceinline__ void load_row(const KT *p, float (&x)[E]) {
  if constexpr (E == 4) {
    const float4 v = ld4(p);
    x[0] = v.x; x[1] = v.y; x[2] = v.z; x[3] = v.w;
  } else {
    const float2 v = ld2(p);
    x[0] = v.x; x[1] = v.y;
  }
}

// E consecutive fp32 values from shared memory (one 64- or 128-bit load).
template <int E>
__device__ __forceinline__ void load_smem(const float *p, float (&x)[E]) {
  if constexpr (E == 4) {
    const float4 v = *reinterpret_cast<const float4 *>(p);
    x[0] = v.x; x[1] = v.y; x[2] = v.z; x[3] = v.w;
  } else {
    const float2 v = *reinterpret_cast<const float2 *>(p);
    x[0] = v.x; x[1] = v.y;
  }
}

// Record the first device-side error of a launch (never traps).
__device__ __forceinline__ void record_error(int32_t *err, int32_t kind, int32_t req, int32_t value) {
  if (atomicCAS(&err[0], 0, kind) == 0) {
    err[1] = req;
    err[2] = value;
  }
  atomicAdd(&err[3], 1);
}

// Global buffer row of token slot p of the request in row descriptor d, or -1
// if the block id is out of range (the error is recorded).  The first
// kRowBlocks blocks come with the descriptor; later ones from the block table.
__device__ __forceinline__ int buffer_row(const PoolView &P, const RowDesc &d, int p) {
  const int bi = P.bs_shift >= 0 ? p >> P.bs_shift : p / P.bs;
  const int blk = bi < kRowBlocks ? d.blk[bi] : P.table[(size_t)d.req * P.max_blocks + bi];
  if (blk < 0 || blk >= P.num_blocks) {
    record_error(P.err, kErrBlockRange, d.req, blk);
    return -1;
  }
  return blk * P.bs + (p - bi * P.bs);
}

// Row index of buffer row g (= block * block_size + slot) for one head, in a
// region laid out [block][heads][block_size][...]: within a block, each head's
// slots are contiguous, so a request's buffered tokens for one head form one
// contiguous run.
__device__ __forceinline__ size_t kv_row(const PoolView &P, int g, int head, int nheads) {
  const int blk = P.bs_shift >= 0 ? g >> P.bs_shift : g / P.bs, pos = g - blk * P.bs;
  return ((size_t)blk * nheads + head) * P.bs + pos;
}

// Inclusive prefix sums of the log-gates of `count` tokens, run by one warp.
// gate(i) supplies token i's log-gate; results go to A[0..count-1].
template <typename GateFn>
__device__ __forceinline__ void warp_prefix(int count, GateFn gate, float *A, int lane) {
  float carry = 0.f;
  for (int base = 0; base < count; base += 32) {
    int i = base + lane;
    float a = (i < count) ? gate(i) : 0.f;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      float y = __shfl_up_sync(kFull, a, off);
      if (lane >= off) a += y;
    }
    a += carry;
    if (i < count) A[i] = a;
    carry = __shfl_sync(kFull, a, 31);
  }
}

// One thread: ancestor sets of a draft tree (bit i = draft i; a draft counts as
// its own ancestor) and, when A is given, the drafts' log-gates (A[j] on entry)
// turned into cumulative values along each draft's path from A_root.
__device__ __forceinline__ void tree_walk(const int8_t *parent, int T, float A_root, float *A,
                                          unsigned long long *anc) {
  for (int j = 0; j < T; ++j) {
    int p = parent[j];
    if (p >= j || p < -1) p = -1;  // validated by the host; keeps every index in range
    anc[j] = (p < 0 ? 0ull : anc[p]) | (1ull << j);
    if (A) A[j] += p < 0 ? A_root : A[p];
  }
}

// n / d for a divisor prepared by make_fastdiv (0 <= n < 2^31).
__device__ __forceinline__ int fast_div(int n, FastDiv f) {
  return (int)((__umulhi((uint32_t)n, f.m) + (uint32_t)n) >> f.s);
}

// ------------------------------------------------------------------ tensor cores
// tf32 value of x, rounded to nearest (ties away): the operand form of
// mma.sync kind tf32, which reads the top 19 bits of a 32-bit register.
__device__ __forceinline__ uint32_t to_tf32(float x) {
  uint32_t r;
  asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
  return r;
}
// x = hi + lo with hi, lo tf32: a product of two such pairs, summed as
// hi*hi + hi*lo + lo*hi, keeps about 21 significant bits (fp32-like).
__device__ __forceinline__ void split_tf32(float x, uint32_t &hi, uint32_t &lo) {
  hi = to_tf32(x);
  lo = to_tf32(x - __uint_as_float(hi));
}
// d += a b for a 16x8 tile, k = 8, tf32 operands, fp32 accumulation.  Not
// volatile: the product has no side effects, so the compiler may interleave
// independent tiles.
__device__ __forceinline__ void mma_tf32(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
  asm(
      "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// The same product with the four accumulators of the tile given separately.
__device__ __forceinline__ void mma_tf32(float &d0, float &d1, float &d2, float &d3,
                                         const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm(
      "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d0), "+f"(d1), "+f"(d2), "+f"(d3)
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// ------------------------------------------------------------------ the fold's rank update
// The decode kernels hold a state tile in registers: lane (g = lane >> 2,
// t = lane & 3) of a warp owns rows RPT g .. RPT g + RPT - 1 and columns
// 4t .. 4t + 3 of the warp's 16 (s[j]: row RPT g + j).  A fold adds
// sum_{i<=n} k_i (w_i u_i)^T.  Read as mma.sync m16n8k8 tiles, the same
// registers are the accumulators when row r of row tile m is state row
// RPT (r mod 8) + 2m + r / 8 and column c of column tile h is column
// 4 (c / 2) + (c mod 2) + 2h: tile (m, h) holds s[2m] and s[2m + 1] (.x, .y for
// h = 0; .z, .w for h = 1), so no value moves between lanes.  The staged keys
// and values are stored in the matching orders (fold_kpos, fold_stage_u), so
// that each operand fragment is one 64-bit shared load; a staged row stride of
// 8 (mod 32) words keeps those loads free of bank conflicts.

// Position of state row `row` (0 .. 8 RPT - 1) within a staged key row.
template <int RPT>
__device__ __forceinline__ int fold_kpos(int row) {
  const int g = row / RPT, w = row - g * RPT;
  return (w >> 1) * 16 + 2 * g + (w & 1);
}
// State row held at position p of a staged key row (the inverse of fold_kpos).
template <int RPT>
__device__ __forceinline__ int fold_krow(int p) {
  return RPT * ((p & 15) >> 1) + 2 * (p >> 4) + (p & 1);
}
// Stage a lane's u values of columns 4t .. 4t + 3 of a 16-column block at p
// (column 4t of the staged row) in fold order: columns 4t, 4t + 2, 4t + 1, 4t + 3.
__device__ __forceinline__ void fold_stage_u(float *p, float4 u) {
  *reinterpret_cast<float4 *>(p) = make_float4(u.x, u.z, u.y, u.w);
}
// s += sum_{i<=n} k_i (w_i u_i)^T over this warp's tile, for staged key rows
// ks + i kst (fold_kpos order) and value rows us + i ust whose 16-column block
// of this warp starts at ublk (fold order), weights wt[i].  Ranks up to 4 use
// FMAs.  Larger ranks use the tensor cores, 8 tokens per k-step, with w_i u_i
// split into tf32 hi and lo parts (about 21 significant bits).  The keys are
// split too unless KEYS_TF32 (values that came from bf16 are exact in tf32).
// Tokens past n enter as zeros.
template <int RPT, bool KEYS_TF32>
__device__ __forceinline__ void fold_tile(float4 (&s)[RPT], const float *ks, int kst,
                                          const float *us, int ust, int ublk, const float *wt,
                                          int n, int lane) {
  const int g = lane >> 2, t = lane & 3;
  if (n < 4) {
    for (int i = 0; i <= n; ++i) {
      const float4 uu = *reinterpret_cast<const float4 *>(us + i * ust + ublk + 4 * t);
      const float w = wt[i];
      const float4 u = make_float4(w * uu.x, w * uu.z, w * uu.y, w * uu.w);
#pragma unroll
      for (int j = 0; j < RPT; j += 2) {
        const float2 k2 = *reinterpret_cast<const float2 *>(ks + i * kst + (j >> 1) * 16 + 2 * g);
        fma4(s[j], k2.x, u);
        fma4(s[j + 1], k2.y, u);
      }
    }
    return;
  }
  for (int kk = 0; kk <= n; kk += 8) {
    const int i0 = kk + t, i1 = i0 + 4;  // this lane's k rows t and t + 4
    float2 u0 = make_float2(0.f, 0.f), u1 = u0;
    float w0 = 0.f, w1 = 0.f;
    if (i0 <= n) {
      u0 = *reinterpret_cast<const float2 *>(us + i0 * ust + ublk + 2 * g);
      w0 = wt[i0];
    }
    if (i1 <= n) {
      u1 = *reinterpret_cast<const float2 *>(us + i1 * ust + ublk + 2 * g);
      w1 = wt[i1];
    }
    uint32_t bh0[2], bl0[2], bh1[2], bl1[2];  // column tiles 0 and 1: k rows t, t + 4
    split_tf32(w0 * u0.x, bh0[0], bl0[0]);
    split_tf32(w1 * u1.x, bh0[1], bl0[1]);
    split_tf32(w0 * u0.y, bh1[0], bl1[0]);
    split_tf32(w1 * u1.y, bh1[1], bl1[1]);
#pragma unroll
    for (int m = 0; m < RPT / 2; ++m) {
      float2 k0 = make_float2(0.f, 0.f), k1 = k0;
      if (i0 <= n) k0 = *reinterpret_cast<const float2 *>(ks + i0 * kst + m * 16 + 2 * g);
      if (i1 <= n) k1 = *reinterpret_cast<const float2 *>(ks + i1 * kst + m * 16 + 2 * g);
      float4 &r0 = s[2 * m], &r1 = s[2 * m + 1];
      if (KEYS_TF32) {
        const uint32_t a[4] = {__float_as_uint(k0.x), __float_as_uint(k0.y), __float_as_uint(k1.x),
                               __float_as_uint(k1.y)};
        mma_tf32(r0.x, r0.y, r1.x, r1.y, a, bh0[0], bh0[1]);
        mma_tf32(r0.z, r0.w, r1.z, r1.w, a, bh1[0], bh1[1]);
        mma_tf32(r0.x, r0.y, r1.x, r1.y, a, bl0[0], bl0[1]);
        mma_tf32(r0.z, r0.w, r1.z, r1.w, a, bl1[0], bl1[1]);
      } else {
        uint32_t a[4], al[4];
        split_tf32(k0.x, a[0], al[0]);
        split_tf32(k0.y, a[1], al[1]);
        split_tf32(k1.x, a[2], al[2]);
        split_tf32(k1.y, a[3], al[3]);
        mma_tf32(r0.x, r0.y, r1.x, r1.y, a, bh0[0], bh0[1]);
        mma_tf32(r0.z, r0.w, r1.z, r1.w, a, bh1[0], bh1[1]);
        mma_tf32(r0.x, r0.y, r1.x, r1.y, a, bl0[0], bl0[1]);
        mma_tf32(r0.z, r0.w, r1.z, r1.w, a, bl1[0], bl1[1]);
        mma_tf32(r0.x, r0.y, r1.x, r1.y, al, bh0[0], bh0[1]);
        mma_tf32(r0.z, r0.w, r1.z, r1.w, al, bh1[0], bh1[1]);
      }
    }
  }
}

}  // namespace kvb
