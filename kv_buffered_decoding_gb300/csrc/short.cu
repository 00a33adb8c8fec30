// Short-context decode: outputs computed from the buffered keys and values
// alone, with no state (KVBuffer, "KVBuffer: IO-aware Serving for Linear
// Attention", abstract and "If this is right" section: short-context requests
// skip state creation and update entirely).  With S = 0 the decode formula
// reduces to attention over the buffer with decay weights:
//   u_t = v_t                                                 plain / gated
//   u_t = beta_t (v_t - sum_{i<t} e^{A_t-A_i} (k_t.k_i) u_i)   gated delta rule
//   o_t = sum_{i<t} e^{A_t-A_i} (q_t.k_i) u_i + (q_t.k_t) u_t
// One CTA of four warps per (batch row, value head).  Every buffered token's
// key, u (or v) and gate, and the current token's q, k, v, gate and beta, reach
// shared memory in one cp.async burst, so the row pays one memory round trip
// instead of one per chunk of tokens.  bf16 pools at d = 128 then run the sums
// on the tensor cores: short_tc_kernel (plain and gated: scores and the output
// sum both as mma.sync passes) and short_mma_kernel (delta rule: the scores as
// an mma.sync pass, the sums with FMAs).  short_kernel (fp32 pools, d = 64):
// warp w takes tokens w, w+4, w+8, ..., reduces each group's dot products with
// one butterfly, and accumulates e^{A_t-A_i} s_i u_i for its lane's columns;
// the four warps' partial sums are added once through shared memory.
#include <type_traits>

#include "kvb_device.cuh"

namespace kvb {

__device__ __forceinline__ void scp16(void *smem, const void *gmem) {
  const unsigned s = static_cast<unsigned>(__cvta_generic_to_shared(smem));
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(s), "l"(gmem) : "memory");
}
__device__ __forceinline__ void scp4(void *smem, const void *gmem) {
  const unsigned s = static_cast<unsigned>(__cvta_generic_to_shared(smem));
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;\n" ::"r"(s), "l"(gmem) : "memory");
}

// Shared-memory bytes for rows holding up to `nmax` buffered tokens.
template <typename KT, int VARIANT, int D>
constexpr size_t short_smem(int nmax) {
  constexpr size_t usz = VARIANT == kGatedDelta ? sizeof(float) : sizeof(KT);
  return (size_t)nmax * D * (sizeof(KT) + usz) + (size_t)((nmax + 3) & ~3) * sizeof(float);
}

template <typename KT, int VARIANT, int D>
__global__ void __launch_bounds__(128) short_kernel(const PoolView P,
                                                     const __grid_constant__ RowBatch rows,
                                                     const TokenIO io) {
  constexpr int NT = 128, NW = 4, E = D / 32;
  constexpr bool DELTA = VARIANT == kGatedDelta, GATED = VARIANT != kPlain;
  using UT = typename std::conditional<DELTA, float, KT>::type;  // stored u (or v)
  constexpr int C = DELTA ? 2 : 4;  // tokens per butterfly (four sums)
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int h = blockIdx.x;
  const RowDesc &d = rows.r[blockIdx.y];
  const size_t b = (size_t)rows.row0 + blockIdx.y;
  const int group = P.Hv / P.Hk;
  const int hq = h / group;
  const int n = d.n;  // buffered tokens; the current token goes to slot n
  const int nmax = io.lmax;

  extern __shared__ float4 dyn_smem[];
  KT *ks = reinterpret_cast<KT *>(dyn_smem);                     // [nmax][D] keys
  UT *usm = reinterpret_cast<UT *>(ks + (size_t)nmax * D);        // [nmax][D] u / v
  float *As = reinterpret_cast<float *>(usm + (size_t)nmax * D);  // [nmax] gates
  __shared__ __align__(16) KT qraw[D];  // the current token's q, k, v (raw)
  __shared__ __align__(16) KT kraw[D];
  __shared__ __align__(16) KT vraw[D];
  __shared__ float gate2[2];  // its log-gate and beta
  __shared__ __align__(16) float part_o[NW][D];
  __shared__ __align__(16) float part_c[NW][D];
  __shared__ size_t koff[kMaxTok], voff[kMaxTok];
  __shared__ float s_t_s;
  __shared__ int bad;

  // 1. where tokens 0..n live (warp 0)
  if (warp == 0) {
    int anybad = 0;
    for (int i = lane; i <= n; i += 32) {
      const int g = buffer_row(P, d, i);
      anybad |= (g < 0);
      if (g >= 0) {
        koff[i] = kv_row(P, g, hq, P.Hk) * D;
        voff[i] = kv_row(P, g, h, P.Hv);
      }
    }
    anybad = __any_sync(kFull, anybad);
    if (lane == 0) bad = anybad;
  }
  if (tid == 32) {
    if (!(GATED && io.log_g)) gate2[0] = 0.f;
    if (!DELTA) gate2[1] = 0.f;
  }
  __syncthreads();
  if (bad) return;  // CTA-uniform

  // 2. the current token's q, k, v, gate and beta, and every buffered token's key,
  //    u / v and gate, into shared memory in one burst
  {
    constexpr int KP = D * (int)sizeof(KT) / 16, UP = D * (int)sizeof(UT) / 16;
    constexpr int KE = 16 / (int)sizeof(KT), UE = 16 / (int)sizeof(UT);
    const KT *qg = static_cast<const KT *>(io.q) + (b * P.Hk + hq) * D;
    const KT *kg = static_cast<const KT *>(io.k) + (b * P.Hk + hq) * D;
    const KT *vg = static_cast<const KT *>(io.v) + (b * P.Hv + h) * D;
    for (int c = tid; c < 3 * KP; c += NT) {
      const int part = c / KP, p = c - part * KP;
      scp16((part == 0 ? qraw : part == 1 ? kraw : vraw) + p * KE,
            (part == 0 ? qg : part == 1 ? kg : vg) + p * KE);
    }
    if (tid == 0 && GATED && io.log_g) scp4(&gate2[0], io.log_g + b * P.Hv + h);
    if (tid == 1 && DELTA) scp4(&gate2[1], io.beta + b * P.Hv + h);
    for (int c = tid; c < n * KP; c += NT) {
      const int i = c / KP, p = c - i * KP;
      scp16(ks + (size_t)i * D + p * KE, static_cast<const KT *>(P.kbuf) + koff[i] + p * KE);
    }
    const UT *ub = DELTA ? reinterpret_cast<const UT *>(P.ubuf) : static_cast<const UT *>(P.vbuf);
    for (int c = tid; c < n * UP; c += NT) {
      const int i = c / UP, p = c - i * UP;
      scp16(usm + (size_t)i * D + p * UE, ub + voff[i] * D + p * UE);
    }
    if (GATED)
      for (int i = tid; i < n; i += NT) scp4(As + i, P.gbuf + voff[i]);
    asm volatile("cp.async.commit_group;\n" ::: "memory");
    asm volatile("cp.async.wait_group 0;\n" ::: "memory");
  }
  __syncthreads();

  const float a_t = gate2[0], beta_t = gate2[1];
  const float A_t = (GATED && n > 0 ? As[n - 1] : 0.f) + a_t;
  float qv[E], tv[E];
  load_row<E>(qraw + lane * E, qv);
#pragma unroll
  for (int e = 0; e < E; ++e) qv[e] *= P.scale;
  load_row<E>(kraw + lane * E, tv);
  if (warp == 0) {
    float st = 0.f;
#pragma unroll
    for (int e = 0; e < E; ++e) st = fmaf(qv[e], tv[e], st);
    st = warp_sum(st);
    if (lane == 0) s_t_s = st;
  }

  // 3. this warp's buffered tokens (w, w + 4, ...), C per butterfly
  float po[E], pc[E];
#pragma unroll
  for (int e = 0; e < E; ++e) po[e] = pc[e] = 0.f;
  for (int i0 = warp; i0 < n; i0 += NW * C) {
    float kc[C][E], uc[C][E], ac[C];
#pragma unroll
    for (int x = 0; x < C; ++x) {
      const int i = i0 + NW * x;
      if (i < n) {
        load_row<E>(ks + (size_t)i * D + lane * E, kc[x]);
        load_row<E>(usm + (size_t)i * D + lane * E, uc[x]);
        ac[x] = GATED ? As[i] : 0.f;
      } else {
#pragma unroll
        for (int e = 0; e < E; ++e) kc[x][e] = uc[x][e] = 0.f;
        ac[x] = A_t;
      }
    }
    float sums[4];
#pragma unroll
    for (int x = 0; x < C; ++x) {
      float sq = 0.f, sk = 0.f;
#pragma unroll
      for (int e = 0; e < E; ++e) {
        sq = fmaf(qv[e], kc[x][e], sq);
        if (DELTA) sk = fmaf(tv[e], kc[x][e], sk);
      }
      if (DELTA) {
        sums[2 * x] = sq;
        sums[2 * x + 1] = sk;
      } else {
        sums[x] = sq;
      }
    }
    const float r = butterfly4(sums[0], sums[1], sums[2], sums[3], lane);
    const float tot[4] = {__shfl_sync(kFull, r, 0), __shfl_sync(kFull, r, 8),
                          __shfl_sync(kFull, r, 16), __shfl_sync(kFull, r, 24)};
#pragma unroll
    for (int x = 0; x < C; ++x) {
      const float w = GATED ? expf(A_t - ac[x]) : 1.f;
      const float ws = w * (DELTA ? tot[2 * x] : tot[x]);
      const float wc = DELTA ? w * tot[2 * x + 1] : 0.f;
#pragma unroll
      for (int e = 0; e < E; ++e) {
        po[e] = fmaf(ws, uc[x][e], po[e]);
        if (DELTA) pc[e] = fmaf(wc, uc[x][e], pc[e]);
      }
    }
  }
#pragma unroll
  for (int e = 0; e < E; ++e) {
    part_o[warp][lane * E + e] = po[e];
    part_c[warp][lane * E + e] = pc[e];
  }
  __syncthreads();

  // 4. one thread per column: the current token's u and the output; append
  for (int c = tid; c < D; c += NT) {
    float o = 0.f, pcs = 0.f;
#pragma unroll
    for (int w = 0; w < NW; ++w) {
      o += part_o[w][c];
      if (DELTA) pcs += part_c[w][c];
    }
    const float vt = to_float(vraw[c]);
    float ut = vt;
    if (DELTA) ut = beta_t * (vt - pcs);
    o = fmaf(s_t_s, ut, o);
    io.o[(b * P.Hv + h) * D + c] = o;
    static_cast<KT *>(P.vbuf)[voff[n] * D + c] = vraw[c];
    if (DELTA) P.ubuf[voff[n] * D + c] = ut;
  }
  if (h % group == 0) {
    constexpr int KP = D * (int)sizeof(KT) / 16, KE = 16 / (int)sizeof(KT);
    for (int c = tid; c < KP; c += NT)
      *reinterpret_cast<uint4 *>(static_cast<KT *>(P.kbuf) + koff[n] + c * KE) =
          *reinterpret_cast<const uint4 *>(kraw + c * KE);
  }
  if (tid == 0) {
    P.gbuf[voff[n]] = GATED ? A_t : 0.f;  // cumulative
    P.bbuf[voff[n]] = beta_t;
    if (h == 0) P.dlen[d.req] = n + 1;
  }
}

// ------------------------------------------------------------------ tensor-core scores
// bf16 pools at d = 128.  Same arithmetic; the score dots of every buffered
// token and the current one (q.k_i, and k_t.k_i for the delta rule) are one
// pass of mma.sync.m16n8k16 (bf16 in, fp32 accumulate, exact products): A holds
// q in row 0 and k_t in row 1 (the other rows zero), B the chunk's keys (tokens
// 0..n-1 buffered, token n the current one), warp w the key tiles w, w+4, ...
// The lanes holding a token's dots turn them into its decay-weighted scores
// (one e^{A_t-A_i} per token instead of one per lane), and the warps then
// accumulate sum_i ws_i u_i (and sum_i wc_i u_i) over their tokens with FMAs.
constexpr int kSXS = 128 + 8;  // bf16 key row stride (272 B): fragment loads hit distinct banks

__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], uint32_t a0, uint32_t a2, uint32_t b0,
                                               uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(0u), "r"(a2), "r"(0u), "r"(b0), "r"(b1));
}

template <int VARIANT>
constexpr size_t short_mma_smem(int nmax) {
  constexpr size_t usz = VARIANT == kGatedDelta ? sizeof(float) : sizeof(__nv_bfloat16);
  return (size_t)((nmax + 1 + 7) & ~7) * kSXS * 2 + (size_t)nmax * 128 * usz +
         (size_t)((nmax + 3) & ~3) * sizeof(float);
}

template <int VARIANT>
__global__ void __launch_bounds__(128) short_mma_kernel(const PoolView P,
                                                         const __grid_constant__ RowBatch rows,
                                                         const TokenIO io) {
  using KT = __nv_bfloat16;
  constexpr int D = 128, NT = 128, NW = 4, E = D / 32, XS = kSXS;
  constexpr bool DELTA = VARIANT == kGatedDelta, GATED = VARIANT != kPlain;
  using UT = typename std::conditional<DELTA, float, KT>::type;  // stored u (or v)
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = lane >> 2, t = lane & 3;
  const int h = blockIdx.x;
  const RowDesc &d = rows.r[blockIdx.y];
  const size_t b = (size_t)rows.row0 + blockIdx.y;
  const int group = P.Hv / P.Hk;
  const int hq = h / group;
  const int n = d.n;  // buffered tokens; the current token goes to slot n
  const int nmax = io.lmax;

  extern __shared__ float4 dyn_smem[];
  KT *Kr = reinterpret_cast<KT *>(dyn_smem);  // [tiles * 8][XS] keys; row n = k_t
  UT *usm = reinterpret_cast<UT *>(Kr + (size_t)((nmax + 1 + 7) & ~7) * XS);  // [nmax][D]
  float *As = reinterpret_cast<float *>(usm + (size_t)nmax * D);              // [nmax] gates
  __shared__ __align__(16) KT qraw[D];  // the current token's q and v (raw)
  __shared__ __align__(16) KT vraw[D];
  __shared__ float gate2[2];  // its log-gate and beta
  __shared__ float ws[kMaxTok], wc[kMaxTok];  // decay-weighted scores per buffered token
  __shared__ __align__(16) float part_o[NW][D];
  __shared__ __align__(16) float part_c[NW][D];
  __shared__ size_t koff[kMaxTok], voff[kMaxTok];
  __shared__ float s_t_s;
  __shared__ int bad;

  // 1. where tokens 0..n live (warp 0)
  if (warp == 0) {
    int anybad = 0;
    for (int i = lane; i <= n; i += 32) {
      const int gr = buffer_row(P, d, i);
      anybad |= (gr < 0);
      if (gr >= 0) {
        koff[i] = kv_row(P, gr, hq, P.Hk) * D;
        voff[i] = kv_row(P, gr, h, P.Hv);
      }
    }
    anybad = __any_sync(kFull, anybad);
    if (lane == 0) bad = anybad;
  }
  if (tid == 32) {
    if (!(GATED && io.log_g)) gate2[0] = 0.f;
    if (!DELTA) gate2[1] = 0.f;
  }
  __syncthreads();
  if (bad) return;  // CTA-uniform

  // 2. the current token's q, k, v, gate and beta, and every buffered token's key,
  //    u / v and gate, in one burst
  {
    const KT *qg = static_cast<const KT *>(io.q) + (b * P.Hk + hq) * D;
    const KT *kg = static_cast<const KT *>(io.k) + (b * P.Hk + hq) * D;
    const KT *vg = static_cast<const KT *>(io.v) + (b * P.Hv + h) * D;
    for (int c = tid; c < 3 * 16; c += NT) {
      const int part = c >> 4, p = c & 15;
      KT *dst = part == 0 ? qraw : part == 1 ? Kr + (size_t)n * XS : vraw;
      scp16(dst + p * 8, (part == 0 ? qg : part == 1 ? kg : vg) + p * 8);
    }
    if (tid == 0 && GATED && io.log_g) scp4(&gate2[0], io.log_g + b * P.Hv + h);
    if (tid == 1 && DELTA) scp4(&gate2[1], io.beta + b * P.Hv + h);
    for (int c = tid; c < n * 16; c += NT) {
      const int i = c >> 4, p = c & 15;
      scp16(Kr + (size_t)i * XS + p * 8, static_cast<const KT *>(P.kbuf) + koff[i] + p * 8);
    }
    constexpr int UP = D * (int)sizeof(UT) / 16, UE = 16 / (int)sizeof(UT);
    const UT *ub = DELTA ? reinterpret_cast<const UT *>(P.ubuf) : static_cast<const UT *>(P.vbuf);
    for (int c = tid; c < n * UP; c += NT) {
      const int i = c / UP, p = c - i * UP;
      scp16(usm + (size_t)i * D + p * UE, ub + voff[i] * D + p * UE);
    }
    if (GATED)
      for (int i = tid; i < n; i += NT) scp4(As + i, P.gbuf + voff[i]);
    asm volatile("cp.async.commit_group;\n" ::: "memory");
    asm volatile("cp.async.wait_group 0;\n" ::: "memory");
  }
  __syncthreads();

  const float a_t = gate2[0], beta_t = gate2[1];
  const float A_t = (GATED && n > 0 ? As[n - 1] : 0.f) + a_t;

  // 3. score dots on the tensor cores; each token's weighted scores
  {
    const KT *arow = g == 0 ? qraw : Kr + (size_t)n * XS;  // row 0: q; row 1: k_t
    const bool has_a = g == 0 || (DELTA && g == 1);
    uint32_t af[8][2];
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
      af[ks][0] = has_a ? *reinterpret_cast<const uint32_t *>(arow + 16 * ks + 2 * t) : 0u;
      af[ks][1] = has_a ? *reinterpret_cast<const uint32_t *>(arow + 16 * ks + 2 * t + 8) : 0u;
    }
    const int tiles = (n + 1 + 7) >> 3;
    for (int tile = warp; tile < tiles; tile += NW) {
      float acc[4] = {0.f, 0.f, 0.f, 0.f};
      const KT *kr = Kr + (size_t)(tile * 8 + g) * XS;
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
        const uint32_t b0 = *reinterpret_cast<const uint32_t *>(kr + 16 * ks + 2 * t);
        const uint32_t b1 = *reinterpret_cast<const uint32_t *>(kr + 16 * ks + 2 * t + 8);
        mma_bf16_16816(acc, af[ks][0], af[ks][1], b0, b1);
      }
      // row g of D: tokens tile*8 + 2t and + 1 (rows 8..15 are zero)
      if (g < 2) {
#pragma unroll
        for (int x = 0; x < 2; ++x) {
          const int i = tile * 8 + 2 * t + x;
          if (i < n) {
            const float w = GATED ? expf(A_t - As[i]) : 1.f;
            if (g == 0) ws[i] = P.scale * w * acc[x];
            else wc[i] = w * acc[x];
          } else if (i == n && g == 0) {
            s_t_s = P.scale * acc[x];
          }
        }
      }
    }
  }
  __syncthreads();

  // 4. this warp's buffered tokens (w, w + 4, ...): partial o (and the delta rule's
  //    correction) for the lane's E columns
  {
    float po[E], pc[E];
#pragma unroll
    for (int e = 0; e < E; ++e) po[e] = pc[e] = 0.f;
#pragma unroll 4
    for (int i = warp; i < n; i += NW) {
      float u[E];
      load_row<E>(usm + (size_t)i * D + lane * E, u);
      const float a = ws[i];
      const float cc = DELTA ? wc[i] : 0.f;
#pragma unroll
      for (int e = 0; e < E; ++e) {
        po[e] = fmaf(a, u[e], po[e]);
        if (DELTA) pc[e] = fmaf(cc, u[e], pc[e]);
      }
    }
#pragma unroll
    for (int e = 0; e < E; ++e) {
      part_o[warp][lane * E + e] = po[e];
      part_c[warp][lane * E + e] = pc[e];
    }
  }
  __syncthreads();

  // 5. one thread per column: the current token's u and the output; append
  {
    const int c = tid;
    float o = 0.f, pcs = 0.f;
#pragma unroll
    for (int w = 0; w < NW; ++w) {
      o += part_o[w][c];
      if (DELTA) pcs += part_c[w][c];
    }
    const float vt = to_float(vraw[c]);
    float ut = vt;
    if (DELTA) ut = beta_t * (vt - pcs);
    o = fmaf(s_t_s, ut, o);
    io.o[(b * P.Hv + h) * D + c] = o;
    static_cast<KT *>(P.vbuf)[voff[n] * D + c] = vraw[c];
    if (DELTA) P.ubuf[voff[n] * D + c] = ut;
  }
  if (h % group == 0)
    for (int c = tid; c < 16; c += NT)
      *reinterpret_cast<uint4 *>(static_cast<KT *>(P.kbuf) + koff[n] + c * 8) =
          *reinterpret_cast<const uint4 *>(Kr + (size_t)n * XS + c * 8);
  if (tid == 0) {
    P.gbuf[voff[n]] = GATED ? A_t : 0.f;  // cumulative
    P.bbuf[voff[n]] = beta_t;
    if (h == 0) P.dlen[d.req] = n + 1;
  }
}

// ------------------------------------------------------------------ tensor-core output
// bf16 pools at d = 128 without the delta rule (u = v): one CTA of four warps
// per (batch row, value head), both sums on the tensor cores.  The chunk
// (tokens 0..n-1 buffered, token n the current one) arrives by 16-byte cp.async
// copies in swizzled rows (below).  The score dots q.k_i are one mma.sync pass with the
// keys as A (16 tokens per tile, fragments by ldmatrix; warp w: tiles w, w + 4)
// and q as column 0 of B; the lanes holding a token's dot form its weight
// w_i = scale e^{A_t-A_i} q.k_i and store it as bf16 hi and lo parts (w = hi +
// lo to about 16 significant bits).  The output is a second pass,
// o^T = V^T [w_hi w_lo], with V^T as A read from the row-major value rows by
// ldmatrix.trans and the two weight columns as B; warp w owns output columns
// 32w .. 32w + 31, so no partial sums cross warps.  The products' M and K run
// in steps of 16 tokens: the value rows are padded to a multiple of 16 (the
// padded rows zeroed, their weights 0); the key rows are not, and a score tile
// that runs past them reads value rows, whose dots are discarded.  Key and
// value rows are 256 bytes with their 16-byte chunks XOR-swizzled on the low
// three bits of the row (chunk c of row r at c ^ (r & 7)), so the eight rows of
// an ldmatrix read hit distinct banks without padding.  At up to 44 buffered
// tokens a CTA then needs under 24.9 KB, and nine CTAs fit on an SM: a batch
// of 256 rows x 16 heads is three full waves instead of three and a third.
struct ShortTcLayout {
  uint32_t kr, vr, as, ws, koff, voff, qrow, bytes;
};
__host__ __device__ inline ShortTcLayout short_tc_layout(int nmax) {
  const uint32_t LP = (uint32_t)(nmax + 1 + 15) & ~15u;
  ShortTcLayout l;
  l.kr = 0;                           // [nmax + 1][128] bf16 keys (row n: k_t)
  l.vr = l.kr + (nmax + 1) * 256;     // [LP][128] bf16 values (row n: v_t)
  l.as = l.vr + LP * 256;             // [LP] cumulative log-gates
  l.ws = l.as + LP * 4;               // [LP] weights, bf16 hi parts then [LP] lo parts
  l.koff = l.ws + LP * 4;             // [LP] key rows
  l.voff = l.koff + LP * 4;           // [LP] value rows
  l.qrow = l.voff + LP * 4;           // q (bf16)
  l.bytes = l.qrow + 128 * 2;
  return l;
}
// Byte offset of 16-byte chunk c of row r in a region of swizzled 256-byte rows.
__device__ __forceinline__ uint32_t swz(int r, int c) {
  return (uint32_t)(r * 256 + ((c ^ (r & 7)) << 4));
}

__device__ __forceinline__ void mma_bf16_full(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                              uint32_t a3, uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
template <int VARIANT>
__global__ void __launch_bounds__(128, 9) short_tc_kernel(const PoolView P,
                                                        const __grid_constant__ RowBatch rows,
                                                        const TokenIO io, FastDiv hv_div) {
  static_assert(VARIANT != kGatedDelta, "the delta rule keeps short_mma_kernel");
  using KT = __nv_bfloat16;
  constexpr int D = 128, NW = 4;
  constexpr bool GATED = VARIANT != kPlain;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = lane >> 2, t = lane & 3;
  const int u = blockIdx.x;
  const int y = fast_div(u, hv_div), h = u - y * P.Hv;
  const RowDesc &d = rows.r[y];
  const size_t b = (size_t)rows.row0 + y;
  const int group = P.Hv / P.Hk, hq = h / group;
  const int n = d.n, L = n + 1;  // buffered tokens; the current token goes to slot n
  const ShortTcLayout lay = short_tc_layout(io.lmax);
  const int LP = (io.lmax + 1 + 15) & ~15;

  extern __shared__ __align__(16) uint8_t sm[];
  uint8_t *Kr = sm + lay.kr;  // swizzled rows (swz)
  uint8_t *Vr = sm + lay.vr;
  float *As = reinterpret_cast<float *>(sm + lay.as);
  KT *whi = reinterpret_cast<KT *>(sm + lay.ws);
  KT *wlo = whi + LP;
  // buffer rows of the tokens (a pool's rows are far fewer than 2^32: 256 bytes each)
  uint32_t *krow = reinterpret_cast<uint32_t *>(sm + lay.koff);
  uint32_t *vrow = reinterpret_cast<uint32_t *>(sm + lay.voff);
  KT *qs = reinterpret_cast<KT *>(sm + lay.qrow);

  // 1. where tokens 0..n live (one thread per token)
  int bad = 0;
  if (tid < L) {
    const int gr = buffer_row(P, d, tid);
    bad = gr < 0;
    krow[tid] = gr >= 0 ? (uint32_t)kv_row(P, gr, hq, P.Hk) : 0u;
    vrow[tid] = gr >= 0 ? (uint32_t)kv_row(P, gr, h, P.Hv) : 0u;
  }
  if (__syncthreads_or(bad)) return;  // recorded in the error word; CTA-uniform

  // 2. the chunk in one burst: buffered keys, values and gates; the current
  //    token's q, k (row n) and v (row n)
  const KT *kb = static_cast<const KT *>(P.kbuf);
  const KT *vb = static_cast<const KT *>(P.vbuf);
  // first group: what the score pass needs (keys, q, gates); second: the values,
  // still in flight while the scores are formed
  for (int c = tid; c < n * 16; c += 128) {
    const int i = c >> 4, p = c & 15;
    scp16(Kr + swz(i, p), kb + (size_t)krow[i] * D + p * 8);
  }
  if (tid < 32) {
    const int p = tid & 15;
    if (tid < 16) scp16(qs + p * 8, static_cast<const KT *>(io.q) + (b * P.Hk + hq) * D + p * 8);
    else scp16(Kr + swz(n, p), static_cast<const KT *>(io.k) + (b * P.Hk + hq) * D + p * 8);
  }
  if (GATED && tid >= 64 && tid - 64 < n) scp4(As + tid - 64, P.gbuf + vrow[tid - 64]);
  asm volatile("cp.async.commit_group;\n" ::: "memory");
  for (int c = tid; c < n * 16; c += 128) {
    const int i = c >> 4, p = c & 15;
    scp16(Vr + swz(i, p), vb + (size_t)vrow[i] * D + p * 8);
  }
  if (tid >= 32 && tid < 48) {
    const int p = tid & 15;
    scp16(Vr + swz(n, p), static_cast<const KT *>(io.v) + (b * P.Hv + h) * D + p * 8);
  }
  asm volatile("cp.async.commit_group;\n" ::: "memory");
  // meanwhile: zero the padded value rows (the output product reads them) and
  // the padded tokens' weights
  for (int c = tid; c < (LP - L) * 16; c += 128)
    *reinterpret_cast<uint4 *>(Vr + (L + (c >> 4)) * 256 + (c & 15) * 16) = make_uint4(0u, 0u, 0u, 0u);
  if (tid >= L && tid < LP) whi[tid] = wlo[tid] = __float2bfloat16_rn(0.f);
  const float a_t = GATED && io.log_g ? io.log_g[b * P.Hv + h] : 0.f;
  asm volatile("cp.async.wait_group 1;\n" ::: "memory");  // keys, q and gates
  __syncthreads();
  const float A_t = (GATED && n > 0 ? As[n - 1] : 0.f) + a_t;

  // 3. score dots q.k_i of tokens 0..n: A = the keys (16 tokens per tile, by
  //    ldmatrix; warp w: tiles w, w + 4), B = q in column 0.  Lanes t == 0 hold
  //    tokens 16 mt + g and + 8 and write their weights w_i (token n: A_n = A_t)
  //    as bf16 hi and lo parts, w = hi + lo to about 16 significant bits
  {
    uint32_t bq[8][2];
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
      bq[ks][0] = g == 0 ? *reinterpret_cast<const uint32_t *>(qs + 16 * ks + 2 * t) : 0u;
      bq[ks][1] = g == 0 ? *reinterpret_cast<const uint32_t *>(qs + 16 * ks + 2 * t + 8) : 0u;
    }
    const int mtiles = (L + 15) >> 4;
    // lane l addresses row l & 15 of a tile (row & 7 == l & 7) and chunk 2 ks + (l >> 4)
    const uint32_t kaddr = static_cast<uint32_t>(__cvta_generic_to_shared(Kr)) +
                           (uint32_t)((lane & 15) * 256);
    const int xr = lane & 7, ch = lane >> 4;
    for (int mt = warp; mt < mtiles; mt += NW) {
      // two accumulator chains (even and odd k-steps) halve the dependent MMA chain
      float acc[4] = {0.f, 0.f, 0.f, 0.f}, acc2[4] = {0.f, 0.f, 0.f, 0.f};
      const uint32_t ka = kaddr + (uint32_t)(mt * 16 * 256);
#pragma unroll
      for (int ks = 0; ks < 8; ks += 2) {
        uint32_t a0, a1, a2, a3, c0, c1, c2, c3;
        asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                     : "=r"(a0), "=r"(a1), "=r"(a2), "=r"(a3)
                     : "r"(ka + (uint32_t)(((2 * ks + ch) ^ xr) << 4)));
        asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                     : "=r"(c0), "=r"(c1), "=r"(c2), "=r"(c3)
                     : "r"(ka + (uint32_t)(((2 * ks + 2 + ch) ^ xr) << 4)));
        mma_bf16_full(acc, a0, a1, a2, a3, bq[ks][0], bq[ks][1]);
        mma_bf16_full(acc2, c0, c1, c2, c3, bq[ks + 1][0], bq[ks + 1][1]);
      }
#pragma unroll
      for (int x = 0; x < 4; ++x) acc[x] += acc2[x];
      if (t == 0) {
#pragma unroll
        for (int x = 0; x < 2; ++x) {
          const int i = 16 * mt + g + 8 * x;
          if (i < L) {
            const float Ai = i < n ? As[i] : A_t;
            const float w = P.scale * (GATED ? expf(A_t - Ai) : 1.f) * acc[2 * x];
            const KT hi = __float2bfloat16_rn(w);
            whi[i] = hi;
            wlo[i] = __float2bfloat16_rn(w - __bfloat162float(hi));
          }
        }
      }
    }
  }
  asm volatile("cp.async.wait_group 0;\n" ::: "memory");  // the values
  __syncthreads();

  // 4. o^T = V^T w for this warp's 32 columns (two tiles of 16): A = V^T by
  //    ldmatrix.trans from the row-major value rows, B = the weights (column 0:
  //    hi parts, column 1: lo parts, the others zero)
  float oc[2][4];
#pragma unroll
  for (int mt = 0; mt < 2; ++mt) oc[mt][0] = oc[mt][1] = oc[mt][2] = oc[mt][3] = 0.f;
  // lane l addresses row (l & 7) + 8 (l >> 4) of a 16-token step (row & 7 == l & 7)
  // and chunk 4 w + ((l >> 3) & 1) + 2 mt
  const uint32_t vaddr = static_cast<uint32_t>(__cvta_generic_to_shared(Vr)) +
                         (uint32_t)(((lane & 7) + ((lane >> 4) << 3)) * 256);
  const int vch = 4 * warp + ((lane >> 3) & 1), vx = lane & 7;
  const uint32_t vo0 = (uint32_t)((vch ^ vx) << 4), vo1 = (uint32_t)(((vch + 2) ^ vx) << 4);
  const KT *wsrc = g == 0 ? whi : wlo;
  for (int kk = 0; kk < LP / 16; ++kk) {
    const uint32_t b0 = g < 2 ? *reinterpret_cast<const uint32_t *>(wsrc + 16 * kk + 2 * t) : 0u;
    const uint32_t b1 = g < 2 ? *reinterpret_cast<const uint32_t *>(wsrc + 16 * kk + 2 * t + 8) : 0u;
    const uint32_t va = vaddr + (uint32_t)(16 * kk * 256);
#pragma unroll
    for (int mt = 0; mt < 2; ++mt) {
      uint32_t a0, a1, a2, a3;
      asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                   : "=r"(a0), "=r"(a1), "=r"(a2), "=r"(a3) : "r"(va + (mt ? vo1 : vo0)));
      mma_bf16_full(oc[mt], a0, a1, a2, a3, b0, b1);
    }
  }

  // 5. the output (lanes t == 0: hi + lo sums of columns 32w + 16mt + g and + 8)
  //    and the current token's buffer entry
  if (t == 0) {
    float *orow = io.o + (b * P.Hv + h) * D + 32 * warp + g;
#pragma unroll
    for (int mt = 0; mt < 2; ++mt) {
      __stcs(orow + 16 * mt, oc[mt][0] + oc[mt][1]);
      __stcs(orow + 16 * mt + 8, oc[mt][2] + oc[mt][3]);
    }
  }
  if (tid < 16) {
    *reinterpret_cast<uint4 *>(static_cast<KT *>(P.vbuf) + (size_t)vrow[n] * D + tid * 8) =
        *reinterpret_cast<const uint4 *>(Vr + swz(n, tid));
  } else if (tid < 32 && h % group == 0) {
    *reinterpret_cast<uint4 *>(static_cast<KT *>(P.kbuf) + (size_t)krow[n] * D + (tid - 16) * 8) =
        *reinterpret_cast<const uint4 *>(Kr + swz(n, tid - 16));
  } else if (tid == 32) {
    P.gbuf[vrow[n]] = GATED ? A_t : 0.f;  // cumulative
    P.bbuf[vrow[n]] = 0.f;
    if (h == 0) P.dlen[d.req] = n + 1;
  }
}

template <int VARIANT>
static cudaError_t run_short_tc(const PoolView &P, const RowBatch &rows, const TokenIO &io,
                                cudaStream_t s) {
  const size_t smem = short_tc_layout(io.lmax).bytes;
  cudaError_t e = ensure_smem((const void *)short_tc_kernel<VARIANT>, smem);
  if (e != cudaSuccess) return e;
  short_tc_kernel<VARIANT><<<rows.count * P.Hv, 128, smem, s>>>(P, rows, io,
                                                                 make_fastdiv((uint32_t)P.Hv));
  return cudaGetLastError();
}

template <int VARIANT>
static cudaError_t run_short_mma(const PoolView &P, const RowBatch &rows, const TokenIO &io,
                                 cudaStream_t s) {
  cudaError_t e = ensure_smem((const void *)short_mma_kernel<VARIANT>,
                              short_mma_smem<VARIANT>(io.lmax));
  if (e != cudaSuccess) return e;
  dim3 grid(P.Hv, rows.count);
  short_mma_kernel<VARIANT><<<grid, 128, short_mma_smem<VARIANT>(io.lmax), s>>>(P, rows, io);
  return cudaGetLastError();
}

template <typename KT, int VARIANT, int D>
static cudaError_t run_short(const PoolView &P, const RowBatch &rows, const TokenIO &io,
                             cudaStream_t s) {
  cudaError_t e = ensure_smem((const void *)short_kernel<KT, VARIANT, D>,
                              short_smem<KT, VARIANT, D>(io.lmax));
  if (e != cudaSuccess) return e;
  dim3 grid(P.Hv, rows.count);
  short_kernel<KT, VARIANT, D><<<grid, 128, short_smem<KT, VARIANT, D>(io.lmax), s>>>(P, rows, io);
  return cudaGetLastError();
}

template <typename KT, int VARIANT>
static cudaError_t short_d(const PoolView &P, const RowBatch &rows, const TokenIO &io, int d,
                           cudaStream_t s) {
  if (d == 128) return run_short<KT, VARIANT, 128>(P, rows, io, s);
  if (d == 64) return run_short<KT, VARIANT, 64>(P, rows, io, s);
  return kUnsupported;
}

template <typename KT>
static cudaError_t short_variant(const PoolView &P, const RowBatch &rows, const TokenIO &io,
                                 int variant, int d, cudaStream_t s) {
  switch (variant) {
    case kPlain: return short_d<KT, kPlain>(P, rows, io, d, s);
    case kGated: return short_d<KT, kGated>(P, rows, io, d, s);
    case kGatedDelta: return short_d<KT, kGatedDelta>(P, rows, io, d, s);
  }
  return kUnsupported;
}

cudaError_t launch_short(const PoolView &P, const RowBatch &rows, const TokenIO &io, int variant,
                         int dtype, int d, cudaStream_t stream) {
  if (rows.count <= 0) return cudaSuccess;
  if (dtype == 1 && d == 128) {
    switch (variant) {
      case kPlain: return run_short_tc<kPlain>(P, rows, io, stream);
      case kGated: return run_short_tc<kGated>(P, rows, io, stream);
      case kGatedDelta: return run_short_mma<kGatedDelta>(P, rows, io, stream);
    }
  }
  if (dtype == 0) return short_variant<float>(P, rows, io, variant, d, stream);
  if (dtype == 1) return short_variant<__nv_bfloat16>(P, rows, io, variant, d, stream);
  return kUnsupported;
}

}  // namespace kvb
