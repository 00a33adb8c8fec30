// Buffered decode, recurrent decode (m = 0) and short-context decode kernels.
//
// KVBuffer ("KVBuffer: IO-aware Serving for Linear Attention", Figure 1):
// each decode step loads a request's state S0 together with its buffered KVs
// and computes the output; S0 is not written; when the buffer is full, all
// buffered KVs are folded into S0 and the state is written back to its slot.
// With S0 the state at the last fold, n tokens buffered since, and the current
// token t = n+1 (A_i = cumulative log-gate since the fold):
//   u_i = v_i                                                  plain / gated
//   u_t = beta_t (v_t - e^{A_t} S0^T k_t - sum_{i<=n} e^{A_t-A_i} (k_t.k_i) u_i)
//                                                              gated delta rule
//   o_t = e^{A_t} S0^T q_t + sum_{i<=t} e^{A_t-A_i} (q_t.k_i) u_i
//   fold:  S <- e^{A_t} S0 + sum_{i<=t} e^{A_t-A_i} k_i u_i^T
// which equals the per-token recurrence exactly (up to rounding).  A gated
// delta token's u is kept in the buffer (pseudo-value), so S0 is touched by two
// mat-vecs per step (S0^T q_t, S0^T k_t) whatever the buffer occupancy.
//
// Two CTAs of 128 threads per (batch row, value head) at d = 128, each owning 64
// state columns.  Warp w owns 16 of them; lane = 4*rsub + c owns columns
// 4c..4c+3 of rows 16*rsub .. 16*rsub+15, so every load of the state is a
// 64-byte segment of a row, the q / k operands of four rows come in one
// 128-bit shared load, and the reduction over rows is three xor-shuffles
// inside the warp.  The state tile stays in
// registers from its load to the fold, so S crosses HBM once per step (twice
// on a fold step, once in each direction).
#include <type_traits>

#include "kvb_device.cuh"

namespace kvb {

template <typename KT, int VARIANT, int D, bool RECURRENT, int NSPLIT>
__global__ void __launch_bounds__(2 * D / NSPLIT, 512 / (2 * D / NSPLIT))
    decode_kernel(const PoolView P, const RowBatch rows, const TokenIO io) {
  constexpr int DK = D, DV = D, NT = 2 * D / NSPLIT, NW = NT / 32, RPT = DK / 8, E = DK / 32;
  constexpr bool DELTA = VARIANT == kGatedDelta, GATED = VARIANT != kPlain;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int h = blockIdx.x / NSPLIT, part = blockIdx.x % NSPLIT;
  const int rsub = lane >> 2, row0 = rsub * RPT;  // this thread's rows: row0 .. row0 + RPT - 1
  const int col0 = part * (DV / NSPLIT) + warp * 16 + (lane & 3) * 4;
  const bool lead = part == 0;  // the column part that writes per-token keys and scalars
  const RowDesc d = rows.r[blockIdx.y];
  const size_t b = (size_t)rows.row0 + blockIdx.y;
  const int group = P.Hv / P.Hk;
  const int hq = h / group;
  const bool has_state = d.slot >= 0;
  const int n = RECURRENT ? 0 : d.n;
  const bool fold = RECURRENT || (d.flags & kFlagFlush);

  // staged rows of the folded tokens, in the orders of fold_tile (kvb_device.cuh)
  constexpr int KST = DK + 8, UST = DV + 8;
  extern __shared__ float4 dyn_smem[];
  float *ks = reinterpret_cast<float *>(dyn_smem);  // [lmax][KST] keys of folded tokens
  float *us = ks + (size_t)io.lmax * KST;           // [lmax][UST] their u
  __shared__ __align__(16) float qs[DK];
  __shared__ __align__(16) float kts[DK];
  __shared__ float wt[kMaxTok], sc[kMaxTok], cc[kMaxTok];
  __shared__ size_t koff[kMaxTok], voff[kMaxTok];  // key element offset; V/U/gate row
  __shared__ float e_t_s;
  __shared__ int bad;

  // 1. the state tile, into registers: the only large read, issued first
  float4 s[RPT];
  float *Sp = P.state + (has_state ? ((size_t)d.slot * P.Hv + h) * DK * DV : 0);
  if (has_state) {
#pragma unroll
    for (int j = 0; j < RPT; ++j) s[j] = ld_stream4(Sp + (row0 + j) * DV + col0);
  } else {
#pragma unroll
    for (int j = 0; j < RPT; ++j) s[j] = f4(0.f);
  }
  const float4 vt = ld4(static_cast<const KT *>(io.v) + (b * P.Hv + h) * DV + col0);
  float a_t = 0.f, beta_t = 0.f;
  if (GATED && io.log_g) a_t = io.log_g[b * P.Hv + h];
  if (DELTA) beta_t = io.beta[b * P.Hv + h];

  // 2. where tokens 0..n live (the only divisions by the block size); q, k to shared
  if (!RECURRENT && warp == 0) {
    int anybad = 0;
    for (int i = lane; i <= n; i += 32) {
      const int g = buffer_row(P, d, i);
      anybad |= (g < 0);
      if (g >= 0) {
        koff[i] = kv_row(P, g, hq, P.Hk) * DK;
        voff[i] = kv_row(P, g, h, P.Hv);
      }
    }
    anybad = __any_sync(kFull, anybad);
    if (lane == 0) bad = anybad;
  }
  const KT *qg = static_cast<const KT *>(io.q) + (b * P.Hk + hq) * DK;
  const KT *kg = static_cast<const KT *>(io.k) + (b * P.Hk + hq) * DK;
  for (int i = tid; i < DK; i += NT) {
    qs[i] = P.scale * to_float(qg[i]);
    kts[i] = to_float(kg[i]);
  }
  __syncthreads();
  if (!RECURRENT && bad) return;  // CTA-uniform

  // 3. issue every small load this thread needs after the mat-vec: the keys of its
  //    warp's first dot-product pass, its first buffered u, and (warp 0) the
  //    cumulative gates; their latency then overlaps the state tile's arrival
  const int p0 = 2 * warp, p1 = p0 + 1;
  float ka[E], kb[E];
#pragma unroll
  for (int e = 0; e < E; ++e) ka[e] = kb[e] = 0.f;
  if (p0 < n) load_row<E>(static_cast<const KT *>(P.kbuf) + koff[p0] + lane * E, ka);
  if (p1 < n) load_row<E>(static_cast<const KT *>(P.kbuf) + koff[p1] + lane * E, kb);
  float4 u_first = f4(0.f);
  if (!RECURRENT && rsub < n) {
    if (DELTA)
      u_first = ld4(P.ubuf + voff[rsub] * DV + col0);
    else
      u_first = ld4(static_cast<const KT *>(P.vbuf) + voff[rsub] * DV + col0);
  }
  float Ai0 = 0.f, Ai1 = 0.f;  // warp 0: cumulative gates of tokens lane, lane + 32
  if (GATED && warp == 0) {
    if (lane < n) Ai0 = P.gbuf[voff[lane]];
    if (lane + 32 < n) Ai1 = P.gbuf[voff[lane + 32]];
  }

  // 4. S0^T q_t (and S0^T k_t) over this thread's rows, operands four rows at a time
  float4 aq = f4(0.f), ak = f4(0.f);
  if (has_state) {
#pragma unroll
    for (int j = 0; j < RPT; j += 4) {
      const float4 q4 = *reinterpret_cast<const float4 *>(&qs[row0 + j]);
      fma4(aq, q4.x, s[j]);
      fma4(aq, q4.y, s[j + 1]);
      fma4(aq, q4.z, s[j + 2]);
      fma4(aq, q4.w, s[j + 3]);
      if (DELTA) {
        const float4 k4 = *reinterpret_cast<const float4 *>(&kts[row0 + j]);
        fma4(ak, k4.x, s[j]);
        fma4(ak, k4.y, s[j + 1]);
        fma4(ak, k4.z, s[j + 2]);
        fma4(ak, k4.w, s[j + 3]);
      }
    }
  }

  // 5. decay weights (warp 0): the buffer stores each token's cumulative log-gate
  //    since the last fold, so A_t = A_{n-1} + a_t and w_i = e^{A_t - A_i}
  float At = 0.f;
  if (GATED) {
    if (warp == 0) {
      const float A_prev = n > 0 ? __shfl_sync(kFull, n - 1 < 32 ? Ai0 : Ai1, (n - 1) & 31) : 0.f;
      At = A_prev + a_t;
      for (int i = lane; i <= n; i += 32) wt[i] = expf(At - (i < n ? (i < 32 ? Ai0 : Ai1) : At));
      if (lane == 0) e_t_s = expf(At);
    }
  } else {
    for (int i = tid; i <= n; i += NT) wt[i] = 1.f;
    if (tid == 0) e_t_s = 1.f;
  }
  //    dot products q.k_i (and k_t.k_i), two tokens per warp pass, one butterfly
  //    reduction for all of a pass's sums; the first pass's keys are already loaded
  for (int i0 = p0; i0 <= n; i0 += 2 * NW) {
    const int i1 = i0 + 1;
    float qv[E], tv[E];
    load_smem<E>(qs + lane * E, qv);
    load_smem<E>(kts + lane * E, tv);
    if (i0 != p0) {
      if (i0 < n) load_row<E>(static_cast<const KT *>(P.kbuf) + koff[i0] + lane * E, ka);
      if (i1 < n) load_row<E>(static_cast<const KT *>(P.kbuf) + koff[i1] + lane * E, kb);
    }
    if (i0 == n) {
#pragma unroll
      for (int e = 0; e < E; ++e) ka[e] = tv[e];
    }
    if (i1 >= n) {
#pragma unroll
      for (int e = 0; e < E; ++e) kb[e] = (i1 == n) ? tv[e] : 0.f;
    }
    float qa = 0.f, qb = 0.f, ta = 0.f, tb = 0.f;
#pragma unroll
    for (int e = 0; e < E; ++e) {
      qa = fmaf(qv[e], ka[e], qa);
      qb = fmaf(qv[e], kb[e], qb);
      if (DELTA) {
        ta = fmaf(tv[e], ka[e], ta);
        tb = fmaf(tv[e], kb[e], tb);
      }
    }
    if (DELTA) {
      const float r = butterfly4(qa, ta, qb, tb, lane);  // lanes 0, 8, 16, 24
      const int which = lane >> 3;
      if ((lane & 7) == 0) {
        if (which == 0) sc[i0] = r;
        else if (which == 1) cc[i0] = r;
        else if (i1 <= n) (which == 2 ? sc : cc)[i1] = r;
      }
    } else {
      const float r = butterfly2(qa, qb, lane);  // lanes 0, 16
      if (lane == 0) sc[i0] = r;
      else if (lane == 16 && i1 <= n) sc[i1] = r;
    }
    if (fold) {
#pragma unroll
      for (int e = 0; e < E; ++e) {
        const int kp = fold_kpos<RPT>(lane * E + e);
        ks[i0 * KST + kp] = ka[e];
        if (i1 <= n) ks[i1 * KST + kp] = kb[e];
      }
    }
  }
  __syncthreads();

  // 6. add this lane's share of the buffered tokens' terms, then one reduction over
  //    the 8 row lanes for both: o_part = e^{A_t} S0^T q + sum_i w_i (q.k_i) u_i
  const float e_t = e_t_s;
  float4 po = mul4(e_t, aq), pc = mul4(e_t, ak);
  for (int i = rsub; i < n; i += 8) {
    float4 ui = u_first;
    if (i != rsub) {
      if (DELTA)
        ui = ld4(P.ubuf + voff[i] * DV + col0);
      else
        ui = ld4(static_cast<const KT *>(P.vbuf) + voff[i] * DV + col0);
    }
    const float w = wt[i];
    fma4(po, w * sc[i], ui);
    if (DELTA) fma4(pc, w * cc[i], ui);
    if (fold) fold_stage_u(&us[i * UST + col0], ui);
  }
  po = rows_sum4(po);
  if (DELTA) pc = rows_sum4(pc);

  float4 ut = vt;
  if (DELTA) {
    ut.x = beta_t * (vt.x - pc.x);
    ut.y = beta_t * (vt.y - pc.y);
    ut.z = beta_t * (vt.z - pc.z);
    ut.w = beta_t * (vt.w - pc.w);
  }
  fma4(po, sc[n], ut);
  if (rsub == 0) {
    __stcs(reinterpret_cast<float4 *>(io.o + (b * P.Hv + h) * DV + col0), po);
    if (!RECURRENT) {
      st4(static_cast<KT *>(P.vbuf) + voff[n] * DV + col0, vt);
      if (DELTA) st4(P.ubuf + voff[n] * DV + col0, ut);
    }
    if (fold) fold_stage_u(&us[n * UST + col0], ut);
  }
  if (!RECURRENT && lead) {
    if (h % group == 0)
      for (int i = tid; i < DK / 4; i += NT)
        st4(static_cast<KT *>(P.kbuf) + koff[n] + 4 * i, *reinterpret_cast<const float4 *>(&kts[4 * i]));
    if (tid == 0) {
      P.gbuf[voff[n]] = At;  // cumulative since the last fold (0 for the plain variant)
      P.bbuf[voff[n]] = beta_t;
    }
  }

  // 7. fold: S <- e^{A_t} S0 + sum_{i<=n} k_i (w_i u_i)^T, a rank-(n+1) update of the
  //    register tile (on the tensor cores above rank 4), written back once
  if (fold && has_state) {
    __syncthreads();
#pragma unroll
    for (int j = 0; j < RPT; ++j) s[j] = mul4(e_t, s[j]);
    fold_tile<RPT, std::is_same<KT, __nv_bfloat16>::value>(s, ks, KST, us, UST, col0 - 4 * (lane & 3),
                                                            wt, n, lane);
#pragma unroll
    for (int j = 0; j < RPT; ++j) st_stream4(Sp + (row0 + j) * DV + col0, s[j]);
  }
  if (!RECURRENT && h == 0 && lead && tid == 0) P.dlen[d.req] = fold ? 0 : n + 1;
}

// Device-side lengths after an accept that folds nothing.
__global__ void set_lengths_kernel(const PoolView P, const RowBatch rows) {
  for (int i = threadIdx.x; i < rows.count; i += blockDim.x) P.dlen[rows.r[i].req] = rows.r[i].n;
}

// 128-bit copy, one tile of kCopyU x 256 16-byte words per CTA: every thread
// issues its kCopyU loads before its stores, and the grid covers the whole
// buffer (no grid-stride loop), so CTAs retire and are replaced continuously.
// On GB300 this reads 7.0 TB/s against 6.3-6.5 TB/s for grid-stride forms with
// a persistent grid (the HBM bandwidth probe).
constexpr int kCopyU = 4;
__global__ void __launch_bounds__(256) copy_probe_kernel(const float4 *__restrict__ src,
                                                         float4 *__restrict__ dst, size_t n16) {
  const size_t base = (size_t)blockIdx.x * (kCopyU * 256) + threadIdx.x;
  float4 x[kCopyU];
#pragma unroll
  for (int u = 0; u < kCopyU; ++u)
    if (base + u * 256 < n16) x[u] = src[base + u * 256];
#pragma unroll
  for (int u = 0; u < kCopyU; ++u)
    if (base + u * 256 < n16) dst[base + u * 256] = x[u];
}

// ------------------------------------------------------------------ launchers
// Column parts per (row, head) for d = 128: two 128-thread CTAs per head keep
// four CTAs resident per SM, so one CTA's serial phases (buffer lookups, dot
// products, barriers, stores) overlap the state loads of the others.
#ifndef KVB_DECODE_SPLIT
#define KVB_DECODE_SPLIT 2
#endif

template <typename KT, int VARIANT, int D, bool REC>
static cudaError_t run_decode(const PoolView &P, const RowBatch &rows, const TokenIO &io,
                              cudaStream_t stream) {
  constexpr int NS = (D == 128) ? KVB_DECODE_SPLIT : 1;
  const size_t smem = (size_t)io.lmax * 2 * (D + 8) * sizeof(float);
  cudaError_t e = ensure_smem((const void *)decode_kernel<KT, VARIANT, D, REC, NS>, smem);
  if (e != cudaSuccess) return e;
  dim3 grid(P.Hv * NS, rows.count);
  decode_kernel<KT, VARIANT, D, REC, NS><<<grid, 2 * D / NS, smem, stream>>>(P, rows, io);
  return cudaGetLastError();
}

template <typename KT, int VARIANT, int D>
static cudaError_t pick_rec(const PoolView &P, const RowBatch &rows, const TokenIO &io, bool rec,
                            cudaStream_t s) {
  return rec ? run_decode<KT, VARIANT, D, true>(P, rows, io, s)
             : run_decode<KT, VARIANT, D, false>(P, rows, io, s);
}

template <typename KT, int VARIANT>
static cudaError_t pick_d(const PoolView &P, const RowBatch &rows, const TokenIO &io, int d,
                          bool rec, cudaStream_t s) {
  if (d == 128) return pick_rec<KT, VARIANT, 128>(P, rows, io, rec, s);
  if (d == 64) return pick_rec<KT, VARIANT, 64>(P, rows, io, rec, s);
  return kUnsupported;
}

template <typename KT>
static cudaError_t pick_variant(const PoolView &P, const RowBatch &rows, const TokenIO &io,
                                int variant, int d, bool rec, cudaStream_t s) {
  switch (variant) {
    case kPlain: return pick_d<KT, kPlain>(P, rows, io, d, rec, s);
    case kGated: return pick_d<KT, kGated>(P, rows, io, d, rec, s);
    case kGatedDelta: return pick_d<KT, kGatedDelta>(P, rows, io, d, rec, s);
  }
  return kUnsupported;
}

cudaError_t launch_decode(const PoolView &P, const RowBatch &rows, const TokenIO &io, int variant,
                          int dtype, int d, bool recurrent, int flush_len, int nmax,
                          cudaStream_t stream) {
  if (rows.count <= 0) return cudaSuccess;
  if (!recurrent && d == 128 && nmax <= kStageTok &&
      decode_stream_pays(rows.count * P.Hv, variant, dtype))
    return launch_decode_stream(P, rows, io, variant, dtype, stream);
  TokenIO io2 = io;
  io2.lmax = flush_len;
  if (dtype == 0) return pick_variant<float>(P, rows, io2, variant, d, recurrent, stream);
  if (dtype == 1) return pick_variant<__nv_bfloat16>(P, rows, io2, variant, d, recurrent, stream);
  return kUnsupported;
}

cudaError_t launch_set_lengths(const PoolView &P, const RowBatch &rows, cudaStream_t stream) {
  if (rows.count <= 0) return cudaSuccess;
  set_lengths_kernel<<<1, 256, 0, stream>>>(P, rows);
  return cudaGetLastError();
}

cudaError_t launch_copy_probe(const void *src, void *dst, size_t bytes, cudaStream_t stream) {
  const size_t n16 = bytes / 16;
  const size_t tiles = (n16 + kCopyU * 256 - 1) / (kCopyU * 256);
  if (tiles > 0x7fffffffull) return cudaErrorInvalidValue;
  copy_probe_kernel<<<(unsigned)tiles, 256, 0, stream>>>(static_cast<const float4 *>(src),
                                                          static_cast<float4 *>(dst), n16);
  return cudaGetLastError();
}

}  // namespace kvb
