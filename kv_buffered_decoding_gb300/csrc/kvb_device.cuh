// Device helpers shared by the libkvb kernels (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "kvb_internal.h"

namespace kvb {

constexpr unsigned kFull = 0xffffffffu;
constexpr int kMaxTok = 64 + 1;  // buffered tokens (capacity) + the current one

enum Variant { kPlain = 0, kGated = 1, kGatedDelta = 2 };

// Tries of mbarrier.try_wait before a wait is declared lost (each try may
// suspend the thread for a while; data normally lands within microseconds).
constexpr uint32_t kSpinLimit = 1u << 22;

// ---------------------------------------------------------------- mbarrier + TMA bulk copy
__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}
// Bulk (non-tensor) asynchronous copy global -> shared, completing on `bar`.
// Both addresses 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes, uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// Wait for phase `parity` of `bar`, giving up after kSpinLimit tries.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *bar, uint32_t parity) {
  for (uint32_t i = 0; i < kSpinLimit; ++i)
    if (mbar_try_wait(bar, parity)) return true;
  return false;
}

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
  const int bi = p / P.bs;
  const int blk = bi < kRowBlocks ? d.blk[bi] : P.table[(size_t)d.req * P.max_blocks + bi];
  if (blk < 0 || blk >= P.num_blocks) {
    record_error(P.err, kErrBlockRange, d.req, blk);
    return -1;
  }
  return blk * P.bs + p % P.bs;
}

// Row index of buffer row g (= block * block_size + slot) for one head, in a
// region laid out [block][heads][block_size][...]: within a block, each head's
// slots are contiguous, so a request's buffered tokens for one head form one
// contiguous run.
__device__ __forceinline__ size_t kv_row(const PoolView &P, int g, int head, int nheads) {
  const int blk = g / P.bs, pos = g - blk * P.bs;
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

}  // namespace kvb
