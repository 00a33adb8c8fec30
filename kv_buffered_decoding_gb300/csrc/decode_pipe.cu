// Persistent, warp-specialized buffered decode for d_k = d_v = 128.
//
// Same computation as decode_kernel (decode.cu; "KVBuffer: IO-aware Serving
// for Linear Attention", Figure 1): per (request, value head) item, read the
// state tile S0 once, combine it with the buffered tokens, write o, append the
// token, and fold the buffer into S when it fills.  What changes is how the
// bytes move.  One CTA per SM walks a strided list of items.  A producer warp
// issues, for item k + NS, every transfer the item needs as TMA bulk copies
// (cp.async.bulk, completing on the stage's "full" mbarrier): the 64 KiB state
// tile, the token's q / k / v rows, its gate and beta rows, and the buffered
// keys, pseudo-values and gates, which the buffer layout keeps contiguous per
// head within a block.  Eight consumer warps compute item k from shared
// memory and release the stage on its "empty" mbarrier.  So HBM always has
// about NS - 1 state tiles in flight per SM, whatever the consumers are doing,
// and no consumer ever waits on a dependent global load.
//
// Every wait is bounded (kSpinLimit tries); a wait that runs out records
// kErrWaitTimeout in the pool's error word and the CTA winds down after making
// sure none of its bulk copies is still in flight.
#include <type_traits>

#include "kvb_device.cuh"

namespace kvb {

constexpr int kPipeD = 128;
constexpr int kPipeConsumers = 256;                 // 8 consumer warps
constexpr int kPipeThreads = kPipeConsumers + 32;   // + 1 producer warp
constexpr int kPipeMaxStages = 4;

// Byte offsets of one stage's buffers (each 128-byte aligned).
struct PipeStage {
  uint32_t s, q, kt, vt, lg, bt, kb, ub, gb, bytes;
};

__host__ __device__ inline uint32_t align128(uint32_t x) { return (x + 127u) & ~127u; }

__host__ __device__ inline PipeStage pipe_stage(int esz, int usz, int Hv, int nb, int bs) {
  PipeStage L;
  uint32_t o = 0;
  L.s = o;  o = align128(o + kPipeD * kPipeD * 4);
  L.q = o;  o = align128(o + kPipeD * esz);
  L.kt = o; o = align128(o + kPipeD * esz);
  L.vt = o; o = align128(o + kPipeD * esz);
  L.lg = o; o = align128(o + Hv * 4);
  L.bt = o; o = align128(o + Hv * 4);
  L.kb = o; o = align128(o + nb * kPipeD * esz);
  L.ub = o; o = align128(o + nb * kPipeD * usz);
  L.gb = o; o = align128(o + ((nb + bs - 1) / bs) * bs * 4);
  L.bytes = o;
  return L;
}

__device__ __forceinline__ void consumer_sync() { asm volatile("bar.sync 1, 256;" ::: "memory"); }
__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

template <typename KT>
__device__ __forceinline__ float4 lds4(const KT *p);
template <>
__device__ __forceinline__ float4 lds4<float>(const float *p) {
  return *reinterpret_cast<const float4 *>(p);
}
template <>
__device__ __forceinline__ float4 lds4<__nv_bfloat16>(const __nv_bfloat16 *p) {
  return ld4(p);
}

template <typename KT, int VARIANT, bool RECURRENT>
__global__ void __launch_bounds__(kPipeThreads, 1)
    decode_pipe_kernel(const PoolView P, const RowBatch rows, const TokenIO io, const int NS,
                       const int nb) {
  constexpr int D = kPipeD, RPT = D / 8;
  constexpr bool DELTA = VARIANT == kGatedDelta;
  using UT = typename std::conditional<DELTA, float, KT>::type;  // buffered u element type
  constexpr int esz = sizeof(KT), usz = sizeof(UT);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int group = P.Hv / P.Hk;
  const int total = rows.count * P.Hv;
  const PipeStage SL = pipe_stage(esz, usz, P.Hv, nb, P.bs);

  extern __shared__ __align__(128) unsigned char smem[];
  __shared__ __align__(8) uint64_t full[kPipeMaxStages], empty[kPipeMaxStages];
  __shared__ int valid[kPipeMaxStages];
  __shared__ float Acum[kMaxTok], wt[kMaxTok], sc[kMaxTok], cc[kMaxTok];
  __shared__ float e_t_s;
  __shared__ volatile int abort_flag;

  if (tid == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    abort_flag = 0;
  }
  __syncthreads();

  if (warp == kPipeConsumers / 32) {
    // ------------------------------------------------------------ producer
    if (lane != 0) return;
    int k = 0;
    for (;; ++k) {
      const int it = blockIdx.x + k * gridDim.x;
      if (it >= total || abort_flag) break;
      const int s = k % NS, round = k / NS;
      if (round > 0 && !mbar_wait_bounded(&empty[s], (round - 1) & 1)) {
        record_error(P.err, kErrWaitTimeout, -1, 1);
        abort_flag = 1;
        break;
      }
      const int row = it / P.Hv, h = it % P.Hv, hq = h / group;
      const RowDesc &d = rows.r[row];
      const size_t b = (size_t)rows.row0 + row;
      const int n = RECURRENT ? 0 : d.n;
      unsigned char *st = smem + (size_t)s * SL.bytes;
      // block ids of the buffered tokens' blocks; all checked before any copy
      const int nblk = (n + P.bs - 1) / P.bs;
      int ok = 1;
      for (int j = 0; j < nblk; ++j) {
        const int blk = j < kRowBlocks ? d.blk[j] : P.table[(size_t)d.req * P.max_blocks + j];
        if (blk < 0 || blk >= P.num_blocks) {
          record_error(P.err, kErrBlockRange, d.req, blk);
          ok = 0;
        }
      }
      valid[s] = ok;
      uint32_t bytes = 0;
      if (ok) {
        bytes = D * D * 4 + 3 * D * esz;
        if (VARIANT != kPlain && io.log_g) bytes += P.Hv * 4;
        if (DELTA) bytes += P.Hv * 4;
        bytes += n * D * esz + n * D * usz + nblk * P.bs * 4;
      }
      mbar_arrive_expect_tx(&full[s], bytes);  // also publishes valid[s]
      if (!ok) continue;
      const float *Sg = P.state + ((size_t)d.slot * P.Hv + h) * D * D;
#pragma unroll
      for (int c = 0; c < 4; ++c)
        bulk_g2s(st + SL.s + c * (D * D), Sg + c * (D * D / 4), D * D, &full[s]);
      bulk_g2s(st + SL.q, static_cast<const KT *>(io.q) + (b * P.Hk + hq) * D, D * esz, &full[s]);
      bulk_g2s(st + SL.kt, static_cast<const KT *>(io.k) + (b * P.Hk + hq) * D, D * esz, &full[s]);
      bulk_g2s(st + SL.vt, static_cast<const KT *>(io.v) + (b * P.Hv + h) * D, D * esz, &full[s]);
      if (VARIANT != kPlain && io.log_g) bulk_g2s(st + SL.lg, io.log_g + b * P.Hv, P.Hv * 4, &full[s]);
      if (DELTA) bulk_g2s(st + SL.bt, io.beta + b * P.Hv, P.Hv * 4, &full[s]);
      for (int j = 0; j < nblk; ++j) {
        const int blk = j < kRowBlocks ? d.blk[j] : P.table[(size_t)d.req * P.max_blocks + j];
        const int cnt = min(P.bs, n - j * P.bs);
        const size_t kr = ((size_t)blk * P.Hk + hq) * P.bs;  // first row of this head in the block
        const size_t vr = ((size_t)blk * P.Hv + h) * P.bs;
        bulk_g2s(st + SL.kb + (size_t)j * P.bs * D * esz, static_cast<const KT *>(P.kbuf) + kr * D,
                 cnt * D * esz, &full[s]);
        const UT *usrc = DELTA ? reinterpret_cast<const UT *>(P.ubuf)
                               : reinterpret_cast<const UT *>(P.vbuf);
        bulk_g2s(st + SL.ub + (size_t)j * P.bs * D * usz, usrc + vr * D, cnt * D * usz, &full[s]);
        bulk_g2s(st + SL.gb + (size_t)j * P.bs * 4, P.gbuf + vr, P.bs * 4, &full[s]);
      }
    }
    // leave no bulk copy in flight: wait for the last issued round of each stage
    for (int j = max(0, k - NS); j < k; ++j) mbar_wait_bounded(&full[j % NS], (j / NS) & 1);
    return;
  }

  // -------------------------------------------------------------- consumers
  const int rsub = lane >> 2, col0 = warp * 16 + (lane & 3) * 4;
  for (int k = 0;; ++k) {
    const int it = blockIdx.x + k * gridDim.x;
    if (it >= total) break;
    const int s = k % NS, round = k / NS;
    const bool got = mbar_wait_bounded(&full[s], round & 1);
    if (!got) {
      if (tid == 0) record_error(P.err, kErrWaitTimeout, -1, 2);
      abort_flag = 1;
    }
    consumer_sync();
    if (abort_flag) break;
    const unsigned char *st = smem + (size_t)s * SL.bytes;
    const int row = it / P.Hv, h = it % P.Hv, hq = h / group;
    const RowDesc &d = rows.r[row];
    const size_t b = (size_t)rows.row0 + row;
    const int n = RECURRENT ? 0 : d.n;
    const bool fold = RECURRENT || (d.flags & kFlagFlush);
    if (valid[s]) {
      const float *Ss = reinterpret_cast<const float *>(st + SL.s);
      const KT *qs = reinterpret_cast<const KT *>(st + SL.q);
      const KT *kts = reinterpret_cast<const KT *>(st + SL.kt);
      const KT *vts = reinterpret_cast<const KT *>(st + SL.vt);
      const KT *kb = reinterpret_cast<const KT *>(st + SL.kb);
      const UT *ub = reinterpret_cast<const UT *>(st + SL.ub);
      const float *gb = reinterpret_cast<const float *>(st + SL.gb);
      const float a_t = (VARIANT != kPlain && io.log_g) ? reinterpret_cast<const float *>(st + SL.lg)[h] : 0.f;
      const float beta_t = DELTA ? reinterpret_cast<const float *>(st + SL.bt)[h] : 0.f;
      const float scale = P.scale;

      // gate prefix sums and decay weights (warp 0); dot products (all warps)
      if (VARIANT != kPlain) {
        if (warp == 0) {
          warp_prefix(n + 1, [&](int i) { return i < n ? gb[i] : a_t; }, Acum, lane);
          __syncwarp();
          const float At = Acum[n];
          for (int i = lane; i <= n; i += 32) wt[i] = expf(At - Acum[i]);
          if (lane == 0) e_t_s = expf(At);
        }
      } else {
        for (int i = tid; i <= n; i += kPipeConsumers) wt[i] = 1.f;
        if (tid == 0) e_t_s = 1.f;
      }
      for (int i = warp; i <= n; i += kPipeConsumers / 32) {
        const KT *kp = (i < n) ? kb + (size_t)i * D : kts;
        const float4 kv = lds4<KT>(kp + lane * 4);
        const float4 qv = lds4<KT>(qs + lane * 4);
        float sq = scale * (qv.x * kv.x + qv.y * kv.y + qv.z * kv.z + qv.w * kv.w);
        float sk = 0.f;
        if (DELTA) {
          const float4 tv = lds4<KT>(kts + lane * 4);
          sk = tv.x * kv.x + tv.y * kv.y + tv.z * kv.z + tv.w * kv.w;
        }
        sq = warp_sum(sq);
        if (DELTA) sk = warp_sum(sk);
        if (lane == 0) {
          sc[i] = sq;
          cc[i] = sk;
        }
      }
      consumer_sync();

      // S0^T q (and S0^T k_t) over this thread's rows, reduced over the row lanes
      float4 aq = f4(0.f), ak = f4(0.f);
#pragma unroll
      for (int j = 0; j < RPT; ++j) {
        const int r = rsub + 8 * j;
        const float4 sv = *reinterpret_cast<const float4 *>(&Ss[r * D + col0]);
        fma4(aq, to_float(qs[r]), sv);
        if (DELTA) fma4(ak, to_float(kts[r]), sv);
      }
      aq = mul4(scale, rows_sum4(aq));
      if (DELTA) ak = rows_sum4(ak);

      // buffered tokens' terms, tokens split over the 8 row lanes
      float4 po = f4(0.f), pc = f4(0.f);
      for (int i = rsub; i < n; i += 8) {
        const float4 ui = lds4<UT>(ub + (size_t)i * D + col0);
        fma4(po, wt[i] * sc[i], ui);
        if (DELTA) fma4(pc, wt[i] * cc[i], ui);
      }
      po = rows_sum4(po);
      if (DELTA) pc = rows_sum4(pc);

      const float e_t = e_t_s;
      const float4 vt = lds4<KT>(vts + col0);
      float4 ut = vt;
      if (DELTA) {
        ut.x = beta_t * (vt.x - fmaf(e_t, ak.x, pc.x));
        ut.y = beta_t * (vt.y - fmaf(e_t, ak.y, pc.y));
        ut.z = beta_t * (vt.z - fmaf(e_t, ak.z, pc.z));
        ut.w = beta_t * (vt.w - fmaf(e_t, ak.w, pc.w));
      }
      float4 o = add4(mul4(e_t, aq), po);
      fma4(o, sc[n], ut);

      // append slot n of the request's buffer
      int g = -1;
      if (!RECURRENT) {
        const int bi = n / P.bs;
        const int blk = bi < kRowBlocks ? d.blk[bi] : P.table[(size_t)d.req * P.max_blocks + bi];
        if (blk >= 0 && blk < P.num_blocks) g = blk * P.bs + n % P.bs;
        else if (tid == 0) record_error(P.err, kErrBlockRange, d.req, blk);
      }
      if (rsub == 0) {
        __stcs(reinterpret_cast<float4 *>(io.o + (b * P.Hv + h) * D + col0), o);
        if (g >= 0) {
          st4(static_cast<KT *>(P.vbuf) + kv_row(P, g, h, P.Hv) * D + col0, vt);
          if (DELTA) st4(P.ubuf + kv_row(P, g, h, P.Hv) * D + col0, ut);
        }
      }
      if (g >= 0) {
        if (h % group == 0 && tid < D / 4)
          st4(static_cast<KT *>(P.kbuf) + kv_row(P, g, hq, P.Hk) * D + 4 * tid, lds4<KT>(kts + 4 * tid));
        if (tid == 0) {
          P.gbuf[kv_row(P, g, h, P.Hv)] = a_t;
          P.bbuf[kv_row(P, g, h, P.Hv)] = beta_t;
        }
      }

      // fold: S <- e^{A_t} S0 + sum_{i<n} e^{A_t-A_i} k_i u_i^T + k_t u_t^T
      if (fold) {
        float *Sg = P.state + ((size_t)d.slot * P.Hv + h) * D * D;
#pragma unroll 4
        for (int j = 0; j < RPT; ++j) {
          const int r = rsub + 8 * j;
          float4 sv = mul4(e_t, *reinterpret_cast<const float4 *>(&Ss[r * D + col0]));
          for (int i = 0; i < n; ++i)
            fma4(sv, wt[i] * to_float(kb[(size_t)i * D + r]), lds4<UT>(ub + (size_t)i * D + col0));
          fma4(sv, to_float(kts[r]), ut);
          st_stream4(Sg + r * D + col0, sv);
        }
      }
      if (!RECURRENT && h == 0 && tid == 0) P.dlen[d.req] = fold ? 0 : n + 1;
    }
    consumer_sync();  // every consumer is done with stage s and the scratch arrays
    if (tid == 0) mbar_arrive(&empty[s]);
  }
}

// ------------------------------------------------------------------ launcher
template <typename KT, int VARIANT, bool REC>
static cudaError_t run_pipe(const PoolView &P, const RowBatch &rows, const TokenIO &io, int NS,
                            int nb, size_t smem, int grid, cudaStream_t stream) {
  static size_t configured = 0;  // dynamic shared memory this instance is set up for
  if (smem > configured) {
    cudaError_t e = cudaFuncSetAttribute(decode_pipe_kernel<KT, VARIANT, REC>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    configured = smem;
  }
  decode_pipe_kernel<KT, VARIANT, REC><<<grid, kPipeThreads, smem, stream>>>(P, rows, io, NS, nb);
  return cudaGetLastError();
}

template <typename KT, int VARIANT>
static cudaError_t pipe_rec(const PoolView &P, const RowBatch &rows, const TokenIO &io, bool rec,
                            int NS, int nb, size_t smem, int grid, cudaStream_t s) {
  return rec ? run_pipe<KT, VARIANT, true>(P, rows, io, NS, nb, smem, grid, s)
             : run_pipe<KT, VARIANT, false>(P, rows, io, NS, nb, smem, grid, s);
}

template <typename KT>
static cudaError_t pipe_variant(const PoolView &P, const RowBatch &rows, const TokenIO &io,
                                int variant, bool rec, int NS, int nb, size_t smem, int grid,
                                cudaStream_t s) {
  switch (variant) {
    case kPlain: return pipe_rec<KT, kPlain>(P, rows, io, rec, NS, nb, smem, grid, s);
    case kGated: return pipe_rec<KT, kGated>(P, rows, io, rec, NS, nb, smem, grid, s);
    case kGatedDelta: return pipe_rec<KT, kGatedDelta>(P, rows, io, rec, NS, nb, smem, grid, s);
  }
  return kUnsupported;
}

static bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Launch the persistent kernel if it applies to this batch (all rows with a
// state, d = 128, bulk-copy alignment of every row it moves); otherwise return
// kUnsupported and let the caller use decode_kernel.
cudaError_t launch_decode_pipe(const PoolView &P, const RowBatch &rows, const TokenIO &io,
                               int variant, int dtype, int d, bool recurrent, int nmax,
                               cudaStream_t stream) {
  if (d != kPipeD || rows.count <= 0) return kUnsupported;
  if (P.Hv % 4 != 0 || P.bs % 4 != 0) return kUnsupported;
  if ((io.log_g && !aligned16(io.log_g)) || (io.beta && !aligned16(io.beta))) return kUnsupported;
  for (int i = 0; i < rows.count; ++i)
    if (rows.r[i].slot < 0) return kUnsupported;
  const int esz = dtype == 1 ? 2 : 4;
  const int usz = variant == kGatedDelta ? 4 : esz;
  const int nb = recurrent ? 0 : nmax;
  const PipeStage SL = pipe_stage(esz, usz, P.Hv, nb, P.bs);
  const size_t budget = 227 * 1024 - 2048;  // dynamic shared memory left after the static part
  int NS = (int)(budget / SL.bytes);
  if (NS > 3) NS = 3;
  if (NS < 2) return kUnsupported;
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  const int items = rows.count * P.Hv;
  const int grid = items < sms ? items : sms;
  const size_t smem = (size_t)NS * SL.bytes;
  if (dtype == 0) return pipe_variant<float>(P, rows, io, variant, recurrent, NS, nb, smem, grid, stream);
  if (dtype == 1)
    return pipe_variant<__nv_bfloat16>(P, rows, io, variant, recurrent, NS, nb, smem, grid, stream);
  return kUnsupported;
}

}  // namespace kvb
