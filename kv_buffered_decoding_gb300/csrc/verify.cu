// Parallel verification of T speculative draft tokens against one state.
//
// KVBuffer ("KVBuffer: IO-aware Serving for Linear Attention", Figure 2): the
// baseline keeps a temporary state per draft token; KVBuffer instead appends
// the drafts' KVs to the buffer and computes every draft's output from the
// same state S0 plus the buffer, storing no temporary state.  With n tokens
// buffered since the last fold and drafts at chunk positions n+1..n+T
// (A = cumulative log-gate over the chunk):
//   y_j = S0^T q_j,  z_j = S0^T k_j                 (2T mat-vecs, one pass over S0)
//   u_j = beta_j (v_j - e^{A_j} z_j - sum_{l<j} e^{A_j-A_l} (k_j.k_l) u_l)
//                                  gated delta: forward substitution over the
//                                  chunk, i.e. the UT transform of the block
//   o_j = e^{A_j} y_j + sum_{l<=j} e^{A_j-A_l} (q_j.k_l) u_l
// The drafts' K, V, u, gates go to buffer slots n..n+T-1; kvb_accept later
// keeps a prefix of them by length alone.
//
// bf16 pools at d = 128 run on the fifth-generation tensor cores
// (verify_tc.cu) when the chunk and draft count fit that kernel; the rest run
// here: verify_mma_kernel (bf16, d = 128: the mat-vecs and score dots as
// mma.sync passes) and verify_kernel (fp32 pools, d = 64), described next.
//
// Two CTAs of 128 threads per (batch row, value head) at d = 128, with the
// decode kernel's layout: warp w owns 16 state columns, each lane 16
// consecutive rows of four of them, and the tile stays in registers.  The 2T
// mat-vecs run eight vectors at a time (four drafts' S0^T q and S0^T k) and
// are reduced over the row lanes by one three-level transpose-reduction; the
// score dot products use butterfly reductions; the forward substitution is
// done per lane for its four columns without any cross-lane reduction.
#include <type_traits>

#include "kvb_device.cuh"

namespace kvb {

// Sum eight per-lane float4 vectors over the three row-lane bits (lane bits 4,
// 3, 2): on return, the lane whose row-lane index is r (lane >> 2) holds the
// total of vector r.  28 shuffles instead of 96 for eight separate reductions.
__device__ __forceinline__ float4 shfl_xor4(float4 v, int off) {
  return make_float4(__shfl_xor_sync(kFull, v.x, off), __shfl_xor_sync(kFull, v.y, off),
                     __shfl_xor_sync(kFull, v.z, off), __shfl_xor_sync(kFull, v.w, off));
}
__device__ __forceinline__ float4 reduce8_rows(const float4 (&acc)[8], int lane) {
  const bool b4 = lane & 16, b3 = lane & 8, b2 = lane & 4;
  float4 k1[4], k2[2];
#pragma unroll
  for (int x = 0; x < 4; ++x)
    k1[x] = add4(b4 ? acc[4 + x] : acc[x], shfl_xor4(b4 ? acc[x] : acc[4 + x], 16));
#pragma unroll
  for (int x = 0; x < 2; ++x)
    k2[x] = add4(b3 ? k1[2 + x] : k1[x], shfl_xor4(b3 ? k1[x] : k1[2 + x], 8));
  return add4(b2 ? k2[1] : k2[0], shfl_xor4(b2 ? k2[0] : k2[1], 4));
}

// Pair p of the chunk's score table, in order of draft j then token l <= n + j.
__device__ __forceinline__ void pair_jl(int p, int n, int &j, int &l) {
  j = 0;
  while (p > n + j) {
    p -= n + j + 1;
    ++j;
  }
  l = p;
}

template <typename KT, int VARIANT, int D, int NSPLIT, bool TREE>
__global__ void __launch_bounds__(2 * D / NSPLIT, 512 / (2 * D / NSPLIT))
    verify_kernel(const PoolView P, const RowBatch rows, const TokenIO io,
                  const __grid_constant__ TreeArg<TREE> tree) {
  constexpr int DK = D, DV = D, NT = 2 * D / NSPLIT, NW = NT / 32, RPT = DK / 8, E = DK / 32;
  constexpr int CW = DV / NSPLIT;  // columns of this CTA
  constexpr bool DELTA = VARIANT == kGatedDelta, GATED = VARIANT != kPlain;
  constexpr int DG = DELTA ? 4 : 8;  // drafts per group of eight mat-vec vectors
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int h = blockIdx.x / NSPLIT, part = blockIdx.x % NSPLIT;
  const int rsub = lane >> 2, row0 = rsub * RPT;
  const int colL = warp * 16 + (lane & 3) * 4, col0 = part * CW + colL;
  const bool lead = part == 0;
  const RowDesc d = rows.r[blockIdx.y];
  const size_t b = (size_t)rows.row0 + blockIdx.y;
  const int group = P.Hv / P.Hk;
  const int hq = h / group;
  const bool has_state = d.slot >= 0;
  const int n = d.n, T = io.T, L = n + T;
  const int LM = io.lmax;  // >= L for every row of the launch

  // shared: ks[LM][DK] keys of the chunk; qs[T][DK] scaled draft queries; and for
  // this CTA's columns: us[LM][CW] u's of the chunk, yq/yk[T][CW] mat-vecs,
  // vs[T][CW] draft values; sw/cw[T][LM] decay-weighted scores; Acum[LM]; bt[T];
  // koff/voff[LM]
  extern __shared__ float4 dyn_smem[];
  float *ks = reinterpret_cast<float *>(dyn_smem);
  float *qs = ks + (size_t)LM * DK;
  float *us = qs + (size_t)T * DK;
  float *yq = us + (size_t)LM * CW;
  float *yk = yq + (size_t)T * CW;
  float *vs = yk + (size_t)T * CW;
  float *sw = vs + (size_t)T * CW;
  float *cw = sw + (size_t)T * LM;
  float *Acum = cw + (size_t)T * LM;
  float *bt = Acum + ((LM + 1) & ~1);                                // even counts keep
  size_t *koff = reinterpret_cast<size_t *>(bt + ((T + 1) & ~1));  // koff 8-byte aligned
  size_t *voff = koff + LM;
  __shared__ int bad;
  __shared__ unsigned long long anc[KVB_MAX_DRAFTS];  // draft trees: ancestor sets

  // 1. the state tile, into registers
  float4 s[RPT];
  const float *Sp = P.state + (has_state ? ((size_t)d.slot * P.Hv + h) * DK * DV : 0);
  if (has_state) {
#pragma unroll
    for (int j = 0; j < RPT; ++j) s[j] = ld_stream4(Sp + (row0 + j) * DV + col0);
  } else {
#pragma unroll
    for (int j = 0; j < RPT; ++j) s[j] = f4(0.f);
  }

  // 2. where the chunk's tokens live; draft queries, keys, values, betas to shared
  if (warp == 0) {
    int anybad = 0;
    for (int i = lane; i < L; i += 32) {
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
  const KT *qg = static_cast<const KT *>(io.q) + b * T * P.Hk * DK;
  const KT *kg = static_cast<const KT *>(io.k) + b * T * P.Hk * DK;
  for (int idx = tid; idx < T * (DK / 4); idx += NT) {
    const int j = idx / (DK / 4), c = (idx % (DK / 4)) * 4;
    const size_t src = ((size_t)j * P.Hk + hq) * DK + c;
    *reinterpret_cast<float4 *>(&qs[j * DK + c]) = mul4(P.scale, ld4(qg + src));
    *reinterpret_cast<float4 *>(&ks[(n + j) * DK + c]) = ld4(kg + src);
  }
  const KT *vg = static_cast<const KT *>(io.v) + b * T * P.Hv * DV;
  for (int idx = tid; idx < T * (CW / 4); idx += NT) {
    const int j = idx / (CW / 4), c = (idx % (CW / 4)) * 4;
    *reinterpret_cast<float4 *>(&vs[j * CW + c]) =
        ld4(vg + ((size_t)j * P.Hv + h) * DV + part * CW + c);
  }
  if (DELTA)
    for (int j = tid; j < T; j += NT) bt[j] = io.beta[(b * T + j) * P.Hv + h];
  __syncthreads();
  if (bad) return;  // CTA-uniform

  // 3. cumulative log-gates of the chunk (warp 0): stored for the buffered tokens,
  //    continued over the drafts.  Buffered keys and u's to shared (all threads).
  if (GATED) {
    if (warp == 0) {
      const float *lg = io.log_g;
      for (int i = lane; i < n; i += 32) Acum[i] = P.gbuf[voff[i]];
      const float A_prev = n > 0 ? P.gbuf[voff[n - 1]] : 0.f;
      if constexpr (TREE) {  // cumulative along each draft's path
        for (int j = lane; j < T; j += 32) Acum[n + j] = lg ? lg[(b * T + j) * P.Hv + h] : 0.f;
        __syncwarp();
        if (lane == 0) tree_walk(tree.p[blockIdx.y], T, A_prev, Acum + n, anc);
      } else {
        warp_prefix(
            T, [&](int j) { return lg ? lg[(b * T + j) * P.Hv + h] : 0.f; }, Acum + n, lane);
        __syncwarp();
        for (int j = lane; j < T; j += 32) Acum[n + j] += A_prev;
      }
    }
  } else {
    for (int i = tid; i < L; i += NT) Acum[i] = 0.f;
    if constexpr (TREE) {
      if (tid == 0) tree_walk(tree.p[blockIdx.y], T, 0.f, nullptr, anc);
    }
  }
  for (int idx = tid; idx < n * (DK / 4); idx += NT) {
    const int i = idx / (DK / 4), c = (idx % (DK / 4)) * 4;
    *reinterpret_cast<float4 *>(&ks[i * DK + c]) =
        ld4(static_cast<const KT *>(P.kbuf) + koff[i] + c);
  }
  for (int idx = tid; idx < n * (CW / 4); idx += NT) {
    const int i = idx / (CW / 4), c = (idx % (CW / 4)) * 4;
    float4 u;
    if (DELTA)
      u = ld4(P.ubuf + voff[i] * DV + part * CW + c);
    else
      u = ld4(static_cast<const KT *>(P.vbuf) + voff[i] * DV + part * CW + c);
    *reinterpret_cast<float4 *>(&us[i * CW + c]) = u;
  }
  __syncthreads();

  // 4. decay-weighted scores, two (draft, token) pairs per warp pass:
  //    sw[j][l] = e^{A_{n+j}-A_l} q_j.k_l (l <= n+j); cw[j][l] = e^{A_{n+j}-A_l} k_{n+j}.k_l (l < n+j)
  const int npairs = T * (n + 1) + T * (T - 1) / 2;
  for (int p0 = 2 * warp; p0 < npairs; p0 += 2 * NW) {
    int ja, la, jb = 0, lb = 0;
    pair_jl(p0, n, ja, la);
    const bool has_b = p0 + 1 < npairs;
    if (has_b) pair_jl(p0 + 1, n, jb, lb);
    float q0[E], k0[E], x0[E], q1[E], k1[E], x1[E];
    load_smem<E>(qs + ja * DK + lane * E, q0);
    load_smem<E>(ks + (n + ja) * DK + lane * E, k0);
    load_smem<E>(ks + la * DK + lane * E, x0);
    load_smem<E>(qs + jb * DK + lane * E, q1);
    load_smem<E>(ks + (n + jb) * DK + lane * E, k1);
    load_smem<E>(ks + lb * DK + lane * E, x1);
    float qa = 0.f, ka = 0.f, qb = 0.f, kb = 0.f;
#pragma unroll
    for (int e = 0; e < E; ++e) {
      qa = fmaf(q0[e], x0[e], qa);
      qb = fmaf(q1[e], x1[e], qb);
      if (DELTA) {
        ka = fmaf(k0[e], x0[e], ka);
        kb = fmaf(k1[e], x1[e], kb);
      }
    }
    float r;
    int which;
    if (DELTA) {
      r = butterfly4(qa, ka, qb, kb, lane);
      which = lane >> 3;  // 0: q a, 1: k a, 2: q b, 3: k b
    } else {
      r = butterfly2(qa, qb, lane);
      which = (lane >> 4) * 2;  // 0: q a, 2: q b
    }
    if ((lane & 7) == 0 && (DELTA || (lane & 15) == 0)) {
      const bool second = which >= 2;
      if (!second || has_b) {
        const int j = second ? jb : ja, l = second ? lb : la;
        // draft trees: a draft sees the buffer and its own path only
        const bool on_path = !TREE || l < n || ((anc[j] >> (l - n)) & 1ull);
        const float w = GATED && on_path ? expf(Acum[n + j] - Acum[l]) : 1.f;
        if ((which & 1) == 0)
          sw[j * LM + l] = on_path ? w * r : 0.f;
        else
          cw[j * LM + l] = (on_path && l < n + j) ? w * r : 0.f;
      }
    }
  }

  // 5. mat-vecs from the register tile, eight vectors at a time
  for (int g0 = 0; g0 < T; g0 += DG) {
    float4 acc[8];
#pragma unroll
    for (int x = 0; x < 8; ++x) acc[x] = f4(0.f);
    if (has_state) {
#pragma unroll
      for (int jj = 0; jj < RPT; jj += 4) {
#pragma unroll
        for (int x = 0; x < DG; ++x) {
          const int j = g0 + x < T ? g0 + x : T - 1;  // duplicates past T are not stored
          const float4 q4 = *reinterpret_cast<const float4 *>(&qs[j * DK + row0 + jj]);
          fma4(acc[x], q4.x, s[jj]);
          fma4(acc[x], q4.y, s[jj + 1]);
          fma4(acc[x], q4.z, s[jj + 2]);
          fma4(acc[x], q4.w, s[jj + 3]);
          if (DELTA) {
            const float4 k4 = *reinterpret_cast<const float4 *>(&ks[(n + j) * DK + row0 + jj]);
            fma4(acc[4 + x], k4.x, s[jj]);
            fma4(acc[4 + x], k4.y, s[jj + 1]);
            fma4(acc[4 + x], k4.z, s[jj + 2]);
            fma4(acc[4 + x], k4.w, s[jj + 3]);
          }
        }
      }
    }
    const float4 tot = reduce8_rows(acc, lane);  // vector rsub of this group
    const int x = DELTA ? (rsub & 3) : rsub;
    if (g0 + x < T) {
      float *dst = (DELTA && rsub >= 4) ? yk : yq;
      *reinterpret_cast<float4 *>(&dst[(g0 + x) * CW + colL]) = tot;
    }
  }
  __syncthreads();

  // 6. per draft, in order: u (forward substitution for the delta rule) and o,
  //    for this lane's four columns; every row lane computes the same values
  for (int j = 0; j < T; ++j) {
    const int t = n + j;  // chunk position of this draft
    const float e_j = GATED ? expf(Acum[t]) : 1.f;
    float4 po = mul4(e_j, *reinterpret_cast<const float4 *>(&yq[j * CW + colL]));
    float4 pc = f4(0.f);
    if (DELTA) pc = mul4(e_j, *reinterpret_cast<const float4 *>(&yk[j * CW + colL]));
    for (int l = 0; l < t; ++l) {
      const float4 u = *reinterpret_cast<const float4 *>(&us[l * CW + colL]);
      fma4(po, sw[j * LM + l], u);
      if (DELTA) fma4(pc, cw[j * LM + l], u);
    }
    const float4 vt = *reinterpret_cast<const float4 *>(&vs[j * CW + colL]);
    float4 ut = vt;
    if (DELTA) {
      const float bj = bt[j];
      ut.x = bj * (vt.x - pc.x);
      ut.y = bj * (vt.y - pc.y);
      ut.z = bj * (vt.z - pc.z);
      ut.w = bj * (vt.w - pc.w);
    }
    fma4(po, sw[j * LM + t], ut);
    if (rsub == 0) {
      __stcs(reinterpret_cast<float4 *>(io.o + ((b * T + j) * P.Hv + h) * DV + col0), po);
      *reinterpret_cast<float4 *>(&us[t * CW + colL]) = ut;
      st4(static_cast<KT *>(P.vbuf) + voff[t] * DV + col0, vt);
      if (DELTA) st4(P.ubuf + voff[t] * DV + col0, ut);
    }
    __syncwarp();  // u of this draft visible to the warp's other lanes
  }

  // 7. drafts' keys, cumulative gates and betas into the buffer
  if (lead) {
    if (h % group == 0)
      for (int idx = tid; idx < T * (DK / 4); idx += NT) {
        const int j = idx / (DK / 4), c = (idx % (DK / 4)) * 4;
        st4(static_cast<KT *>(P.kbuf) + koff[n + j] + c,
            *reinterpret_cast<const float4 *>(&ks[(n + j) * DK + c]));
      }
    for (int j = tid; j < T; j += NT) {
      P.gbuf[voff[n + j]] = Acum[n + j];  // cumulative since the last fold
      P.bbuf[voff[n + j]] = DELTA ? bt[j] : 0.f;
    }
  }
}

// ------------------------------------------------------------------ tensor-core verify
// bf16 pools at d = 128.  One CTA of four warps per (batch row, value head):
//  0. each lane starts streaming its first quarter of state rows into registers,
//     and warp 0 locates the chunk's tokens;
//  1. every small operand (draft q, k, v, betas, log-gates; buffered keys, u / v
//     and cumulative gates) reaches shared memory in one cp.async burst, raw;
//  2. the 2T mat-vecs and every score dot product are one pass of tensor-core
//     products over d_k: Y^T = X^T [S0 | K^T], X = [q_0..q_{T-1}, k_0..k_{T-1}]
//     (d_k x V, V = 2T for the delta rule, T otherwise, padded to 16) and K the
//     chunk's keys (buffered, then drafts).  Warp w owns state columns
//     32w..32w+31 and the key tiles w, w+4; each k-step of 8 is one
//     mma.sync.m16n8k8 per n-tile (tf32 in, fp32 accumulate).  A lane (g, t)
//     holds rows 8ks+t and 8ks+t+4 of its state columns 32w+4g..+3 (two
//     coalesced 128-bit loads); element i of each is the B fragment of state
//     n-tile i, so no data moves between lanes.  The state is rounded to tf32
//     (cvt.rna, relative error <= 2^-11 per element); q and k are bf16 and exact
//     in tf32, so the score dots are exact products with fp32 sums;
//  3. decay weights e^{A_j - A_l} on the scores (one entry per thread);
//  4. per draft, in order, one column per thread: u (the forward substitution of
//     the delta rule) and o;
//  5. the drafts' entries go to the buffer.
// The fp32 path and d = 64 keep verify_kernel.

__device__ __forceinline__ void vcp16(void *smem, const void *gmem) {
  const unsigned s = static_cast<unsigned>(__cvta_generic_to_shared(smem));
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(s), "l"(gmem) : "memory");
}
__device__ __forceinline__ void vcp4(void *smem, const void *gmem) {
  const unsigned s = static_cast<unsigned>(__cvta_generic_to_shared(smem));
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;\n" ::"r"(s), "l"(gmem) : "memory");
}
// bf16 -> the fp32 (and tf32) bit pattern of the same value
__device__ __forceinline__ uint32_t bf_bits(__nv_bfloat16 x) {
  return (uint32_t)__bfloat16_as_ushort(x) << 16;
}

constexpr int kVXS = 128 + 8;  // bf16 row stride of the staged vectors and keys (272 B)
constexpr int kVMaxTiles = 8;  // key tiles of 8 (two per warp): chunks of up to 64 tokens

// Byte offsets of the verify CTA's shared-memory arrays (16-byte aligned each).
struct VLayout {
  size_t xr, kr, us, vs, y, sc, sw, cw, acum, lg, bt, koff, voff, total;
};
__host__ __device__ inline VLayout verify_layout(int variant, int T, int LM) {
  const bool delta = variant == kGatedDelta;
  const size_t V = delta ? 2 * T : T, VP = (V + 15) / 16 * 16, LP = (LM + 7) / 8 * 8;
  auto up = [](size_t x) { return (x + 15) & ~(size_t)15; };
  VLayout l;
  l.xr = 0;
  l.kr = l.xr + up(VP * kVXS * 2);
  l.us = l.kr + up(LP * kVXS * 2);
  l.vs = l.us + up((size_t)LM * 128 * (delta ? 4 : 2));
  l.y = l.vs + (delta ? up((size_t)T * 128 * 2) : 0);
  l.sc = l.y + up(V * 128 * 4);
  l.sw = l.sc + up(V * LP * 4);
  l.cw = l.sw + up((size_t)T * LM * 4);
  l.acum = l.cw + (delta ? up((size_t)T * LM * 4) : 0);
  l.lg = l.acum + up((size_t)LM * 4);
  l.bt = l.lg + up((size_t)T * 4);
  l.koff = l.bt + up((size_t)T * 4);
  l.voff = l.koff + up((size_t)LM * 8);
  l.total = l.voff + up((size_t)LM * 8);
  return l;
}

template <int VARIANT, bool TREE>
__global__ void __launch_bounds__(128, 4)
    verify_mma_kernel(const PoolView P, const __grid_constant__ RowBatch rows, const TokenIO io,
                      const __grid_constant__ TreeArg<TREE> tree) {
  using KT = __nv_bfloat16;
  constexpr int D = 128, DK = D, DV = D, NT = 128, XS = kVXS;
  constexpr bool DELTA = VARIANT == kGatedDelta, GATED = VARIANT != kPlain;
  using UT = typename std::conditional<DELTA, float, KT>::type;  // stored u (or v)
  constexpr int UE = 16 / (int)sizeof(UT), UC = DV / UE;        // per 16-byte chunk, per row
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = lane >> 2, t = lane & 3;
  const int h = blockIdx.x;
  const RowDesc &d = rows.r[blockIdx.y];
  const size_t b = (size_t)rows.row0 + blockIdx.y;
  const int group = P.Hv / P.Hk;
  const int hq = h / group;
  const bool has_state = d.slot >= 0;
  const int n = d.n, T = io.T, L = n + T;
  const int LM = io.lmax;  // >= L for every row of the launch
  const int V = DELTA ? 2 * T : T, MT = (V + 15) / 16, LP = (LM + 7) / 8 * 8, NS = LP / 8;

  extern __shared__ float4 dyn_smem[];
  const VLayout lay = verify_layout(VARIANT, T, LM);
  char *base = reinterpret_cast<char *>(dyn_smem);
  KT *Xr = reinterpret_cast<KT *>(base + lay.xr);     // [VP][XS] vectors, raw
  KT *Kr = reinterpret_cast<KT *>(base + lay.kr);     // [LP][XS] chunk keys, raw
  UT *us = reinterpret_cast<UT *>(base + lay.us);     // [LM][DV] chunk u's (or v's)
  KT *vs = reinterpret_cast<KT *>(base + lay.vs);     // [T][DV] draft values (delta rule)
  float *Y = reinterpret_cast<float *>(base + lay.y);  // [V][DV] mat-vecs
  float *Sc = reinterpret_cast<float *>(base + lay.sc);  // [V][LP] dot products
  float *sw = reinterpret_cast<float *>(base + lay.sw);  // [T][LM] weighted q.k
  float *cw = reinterpret_cast<float *>(base + lay.cw);  // [T][LM] weighted k.k
  float *Acum = reinterpret_cast<float *>(base + lay.acum);
  float *lgr = reinterpret_cast<float *>(base + lay.lg);
  float *bt = reinterpret_cast<float *>(base + lay.bt);
  size_t *koff = reinterpret_cast<size_t *>(base + lay.koff);
  size_t *voff = reinterpret_cast<size_t *>(base + lay.voff);
  __shared__ int bad;
  __shared__ unsigned long long anc[KVB_MAX_DRAFTS];  // draft trees: ancestor sets

  const float *Sp = P.state + (has_state ? ((size_t)d.slot * P.Hv + h) * DK * DV : 0);
  const int cbase = warp * 32 + 4 * g;  // this lane's four state columns
  // rows 32q + 8i + t and + 4 (i = 0..3) of this lane's columns: quarter q of its rows
  float4 snx[8];
  auto load_quarter = [&](int q) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int r0 = q * 32 + i * 8 + t;
      snx[2 * i] = ld_stream4(Sp + (size_t)r0 * DV + cbase);
      snx[2 * i + 1] = ld_stream4(Sp + (size_t)(r0 + 4) * DV + cbase);
    }
  };
  if (has_state) load_quarter(0);

  // 0. where the chunk's tokens live
  if (warp == 0) {
    int anybad = 0;
    for (int i = lane; i < L; i += 32) {
      const int gr = buffer_row(P, d, i);
      anybad |= (gr < 0);
      if (gr >= 0) {
        koff[i] = kv_row(P, gr, hq, P.Hk) * DK;
        voff[i] = kv_row(P, gr, h, P.Hv);
      }
    }
    anybad = __any_sync(kFull, anybad);
    if (lane == 0) bad = anybad;
  }
  __syncthreads();
  if (bad) return;  // CTA-uniform

  // 1. the small operands, raw, in one burst
  {
    const KT *qg = static_cast<const KT *>(io.q) + b * T * P.Hk * DK;
    const KT *kg = static_cast<const KT *>(io.k) + b * T * P.Hk * DK;
    const KT *vg = static_cast<const KT *>(io.v) + b * T * P.Hv * DV;
    for (int c = tid; c < V * 16; c += NT) {  // q_j, then k_j (delta rule)
      const int m = c >> 4, p = c & 15;
      const KT *src = m < T ? qg + ((size_t)m * P.Hk + hq) * DK
                            : kg + ((size_t)(m - T) * P.Hk + hq) * DK;
      vcp16(Xr + m * XS + p * 8, src + p * 8);
    }
    for (int c = tid; c < L * 16; c += NT) {  // the chunk's keys: buffered, then drafts
      const int i = c >> 4, p = c & 15;
      const KT *src = i < n ? static_cast<const KT *>(P.kbuf) + koff[i]
                            : kg + ((size_t)(i - n) * P.Hk + hq) * DK;
      vcp16(Kr + i * XS + p * 8, src + p * 8);
    }
    // buffered u's (delta rule) or v's; without the delta rule the drafts' v's follow
    const int urows = DELTA ? n : L;
    const UT *ub = DELTA ? reinterpret_cast<const UT *>(P.ubuf) : static_cast<const UT *>(P.vbuf);
    for (int c = tid; c < urows * UC; c += NT) {
      const int i = c / UC, p = c - i * UC;
      const UT *src = i < n ? ub + voff[i] * DV
                            : reinterpret_cast<const UT *>(vg + ((size_t)(i - n) * P.Hv + h) * DV);
      vcp16(us + (size_t)i * DV + p * UE, src + p * UE);
    }
    if (DELTA)
      for (int c = tid; c < T * 16; c += NT) {
        const int j = c >> 4, p = c & 15;
        vcp16(vs + j * DV + p * 8, vg + ((size_t)j * P.Hv + h) * DV + p * 8);
      }
    if (GATED) {
      for (int i = tid; i < n; i += NT) vcp4(Acum + i, P.gbuf + voff[i]);
      if (io.log_g)
        for (int j = tid; j < T; j += NT) vcp4(lgr + j, io.log_g + (b * T + j) * P.Hv + h);
    }
    if (DELTA)
      for (int j = tid; j < T; j += NT) vcp4(bt + j, io.beta + (b * T + j) * P.Hv + h);
    asm volatile("cp.async.commit_group;\n" ::: "memory");
    asm volatile("cp.async.wait_group 0;\n" ::: "memory");
  }
  __syncthreads();

  // cumulative gates of the drafts (warp 0; along each draft's path for trees)
  if (GATED) {
    if (warp == 0) {
      const float A_prev = n > 0 ? Acum[n - 1] : 0.f;
      const bool lg = io.log_g != nullptr;
      if constexpr (TREE) {
        for (int j = lane; j < T; j += 32) Acum[n + j] = lg ? lgr[j] : 0.f;
        __syncwarp();
        if (lane == 0) tree_walk(tree.p[blockIdx.y], T, A_prev, Acum + n, anc);
      } else {
        warp_prefix(T, [&](int j) { return lg ? lgr[j] : 0.f; }, Acum + n, lane);
        __syncwarp();
        for (int j = lane; j < T; j += 32) Acum[n + j] += A_prev;
      }
    }
  } else {
    for (int i = tid; i < L; i += NT) Acum[i] = 0.f;
    if constexpr (TREE) {
      if (tid == 0) tree_walk(tree.p[blockIdx.y], T, 0.f, nullptr, anc);
    }
  }

  // 2. mat-vecs and score dots on the tensor cores
  const int ntile = warp < NS ? (warp + 4 < NS ? 2 : 1) : 0;  // this warp's key tiles
  for (int mt = 0; mt < MT; ++mt) {
    float acc[4][4], sacc[2][4];
#pragma unroll
    for (int i = 0; i < 4; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;
#pragma unroll
    for (int i = 0; i < 2; ++i) sacc[i][0] = sacc[i][1] = sacc[i][2] = sacc[i][3] = 0.f;
    const KT *xa = Xr + (mt * 16 + g) * XS;
    const KT *xb = xa + 8 * XS;
    if (mt > 0 && has_state) load_quarter(0);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      float4 cur[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) cur[i] = snx[i];
      if (q < 3 && has_state) load_quarter(q + 1);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int k0 = q * 32 + i * 8;
        const uint32_t a[4] = {bf_bits(xa[k0 + t]), bf_bits(xb[k0 + t]), bf_bits(xa[k0 + t + 4]),
                               bf_bits(xb[k0 + t + 4])};
        if (has_state) {
          const float4 s0 = cur[2 * i], s1 = cur[2 * i + 1];
          mma_tf32(acc[0], a, to_tf32(s0.x), to_tf32(s1.x));
          mma_tf32(acc[1], a, to_tf32(s0.y), to_tf32(s1.y));
          mma_tf32(acc[2], a, to_tf32(s0.z), to_tf32(s1.z));
          mma_tf32(acc[3], a, to_tf32(s0.w), to_tf32(s1.w));
        }
        if (ntile > 0) {
          const KT *kr = Kr + (warp * 8 + g) * XS + k0;
          mma_tf32(sacc[0], a, bf_bits(kr[t]), bf_bits(kr[t + 4]));
        }
        if (ntile > 1) {
          const KT *kr = Kr + ((warp + 4) * 8 + g) * XS + k0;
          mma_tf32(sacc[1], a, bf_bits(kr[t]), bf_bits(kr[t + 4]));
        }
      }
    }
    // state n-tile i: D[m][p] is vector m at column warp*32 + 4p + i
    const int m0 = mt * 16 + g, m1 = m0 + 8;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int c0 = warp * 32 + 8 * t + i, c1 = c0 + 4;
      if (m0 < V) {
        Y[m0 * DV + c0] = acc[i][0];
        Y[m0 * DV + c1] = acc[i][1];
      }
      if (m1 < V) {
        Y[m1 * DV + c0] = acc[i][2];
        Y[m1 * DV + c1] = acc[i][3];
      }
    }
    // key tile s: D[m][p] is vector m against key 8s + p
#pragma unroll
    for (int x = 0; x < 2; ++x)
      if (x < ntile) {
        const int l0 = (warp + 4 * x) * 8 + 2 * t;
        if (m0 < V) {
          Sc[m0 * LP + l0] = sacc[x][0];
          Sc[m0 * LP + l0 + 1] = sacc[x][1];
        }
        if (m1 < V) {
          Sc[m1 * LP + l0] = sacc[x][2];
          Sc[m1 * LP + l0 + 1] = sacc[x][3];
        }
      }
  }
  __syncthreads();

  // 3. decay-weighted scores; a tree draft sees the buffer and its own path only
  for (int idx = tid; idx < T * LM; idx += NT) {
    const int j = idx / LM, l = idx - j * LM;
    float wq = 0.f, wk = 0.f;
    if (l <= n + j) {
      const bool on_path = !TREE || l < n || ((anc[j] >> (l - n)) & 1ull);
      if (on_path) {
        const float w = GATED ? expf(Acum[n + j] - Acum[l]) : 1.f;
        wq = w * P.scale * Sc[j * LP + l];
        if (DELTA && l < n + j) wk = w * Sc[(T + j) * LP + l];
      }
    }
    sw[idx] = wq;
    if (DELTA) cw[idx] = wk;
  }
  __syncthreads();

  // 4. per draft, in order, one column per thread: u (forward substitution for the
  //    delta rule) and o
  const int c = tid;
  for (int j = 0; j < T; ++j) {
    const int tpos = n + j;
    const float e_j = GATED ? expf(Acum[tpos]) : 1.f;
    float po = e_j * P.scale * Y[j * DV + c];
    float pc = DELTA ? e_j * Y[(T + j) * DV + c] : 0.f;
    for (int l = 0; l < tpos; ++l) {
      const float u = to_float(us[l * DV + c]);
      po = fmaf(sw[j * LM + l], u, po);
      if (DELTA) pc = fmaf(cw[j * LM + l], u, pc);
    }
    float ut;
    if constexpr (DELTA) {
      ut = bt[j] * (to_float(vs[j * DV + c]) - pc);
      us[tpos * DV + c] = ut;  // read later only by this thread
    } else {
      ut = to_float(us[tpos * DV + c]);
    }
    po = fmaf(sw[j * LM + tpos], ut, po);
    __stcs(io.o + ((b * T + j) * P.Hv + h) * DV + c, po);
  }
  __syncthreads();

  // 5. drafts into the buffer: values and u's, keys (one value head per q/k head),
  //    cumulative gates, betas
  for (int idx = tid; idx < T * 16; idx += NT) {
    const int j = idx >> 4, p = idx & 15;
    const KT *src = DELTA ? vs + j * DV : reinterpret_cast<const KT *>(us) + (size_t)(n + j) * DV;
    *reinterpret_cast<uint4 *>(static_cast<KT *>(P.vbuf) + voff[n + j] * DV + p * 8) =
        *reinterpret_cast<const uint4 *>(src + p * 8);
  }
  if (DELTA)
    for (int idx = tid; idx < T * 32; idx += NT) {
      const int j = idx >> 5, p = idx & 31;
      *reinterpret_cast<float4 *>(P.ubuf + voff[n + j] * DV + p * 4) =
          *reinterpret_cast<const float4 *>(reinterpret_cast<const float *>(us) +
                                            (size_t)(n + j) * DV + p * 4);
    }
  if (h % group == 0)
    for (int idx = tid; idx < T * 16; idx += NT) {
      const int j = idx >> 4, p = idx & 15;
      *reinterpret_cast<uint4 *>(static_cast<KT *>(P.kbuf) + koff[n + j] + p * 8) =
          *reinterpret_cast<const uint4 *>(Kr + (n + j) * XS + p * 8);
    }
  for (int j = tid; j < T; j += NT) {
    P.gbuf[voff[n + j]] = Acum[n + j];
    P.bbuf[voff[n + j]] = DELTA ? bt[j] : 0.f;
  }
}

static size_t verify_mma_smem(int variant, int T, int LM) {
  return verify_layout(variant, T, LM).total;
}

template <int VARIANT, bool TREE>
static cudaError_t run_verify_mma(const PoolView &P, const RowBatch &rows, const TokenIO &io,
                                  const TreeArg<TREE> &tree, cudaStream_t stream) {
  const size_t smem = verify_mma_smem(VARIANT, io.T, io.lmax);
  cudaError_t e = ensure_smem((const void *)verify_mma_kernel<VARIANT, TREE>, smem);
  if (e != cudaSuccess) return e;
  dim3 grid(P.Hv, rows.count);
  verify_mma_kernel<VARIANT, TREE><<<grid, 128, smem, stream>>>(P, rows, io, tree);
  return cudaGetLastError();
}

// ------------------------------------------------------------------ launcher
static size_t verify_smem(int d, int split, int T, int LM) {
  const size_t cw = d / split;
  const size_t floats = (size_t)LM * d + (size_t)T * d + (size_t)LM * cw + 3 * (size_t)T * cw +
                        2 * (size_t)T * LM + ((LM + 1) & ~1) + ((T + 1) & ~1);
  return floats * sizeof(float) + 2 * (size_t)LM * sizeof(size_t);
}

template <typename KT, int VARIANT, int D, bool TREE>
static cudaError_t run_verify(const PoolView &P, const RowBatch &rows, const TokenIO &io,
                              const TreeArg<TREE> &tree, cudaStream_t stream) {
  constexpr int NS = D == 128 ? 2 : 1;
  const size_t smem = verify_smem(D, NS, io.T, io.lmax);
  cudaError_t e = ensure_smem((const void *)verify_kernel<KT, VARIANT, D, NS, TREE>, smem);
  if (e != cudaSuccess) return e;
  dim3 grid(P.Hv * NS, rows.count);
  verify_kernel<KT, VARIANT, D, NS, TREE><<<grid, 2 * D / NS, smem, stream>>>(P, rows, io, tree);
  return cudaGetLastError();
}

template <typename KT, int VARIANT, bool TREE>
static cudaError_t verify_d(const PoolView &P, const RowBatch &rows, const TokenIO &io, int d,
                            const TreeArg<TREE> &tree, cudaStream_t s) {
  if (d == 128) return run_verify<KT, VARIANT, 128, TREE>(P, rows, io, tree, s);
  if (d == 64) return run_verify<KT, VARIANT, 64, TREE>(P, rows, io, tree, s);
  return kUnsupported;
}

template <typename KT, bool TREE>
static cudaError_t verify_variant(const PoolView &P, const RowBatch &rows, const TokenIO &io,
                                  int variant, int d, const TreeArg<TREE> &tree, cudaStream_t s) {
  switch (variant) {
    case kPlain: return verify_d<KT, kPlain, TREE>(P, rows, io, d, tree, s);
    case kGated: return verify_d<KT, kGated, TREE>(P, rows, io, d, tree, s);
    case kGatedDelta: return verify_d<KT, kGatedDelta, TREE>(P, rows, io, d, tree, s);
  }
  return kUnsupported;
}

template <bool TREE>
static cudaError_t verify_dispatch(const PoolView &P, const RowBatch &rows, const TokenIO &io,
                                   int variant, int dtype, int d, const TreeArg<TREE> &tree,
                                   const StateMap *smap, cudaStream_t stream) {
  if (dtype == 0) return verify_variant<float, TREE>(P, rows, io, variant, d, tree, stream);
  if (dtype == 1) {
    // tcgen05 path (state by TMA, mat-vecs on the fifth-generation tensor cores)
    if (d == 128 && smap && verify_tc_fits(variant, io.T, io.lmax))
      return launch_verify_tc<TREE>(P, rows, io, variant, tree, *smap, stream);
    // tensor-core path for bf16 pools at d = 128 when its shared memory fits
    if (d == 128 && io.lmax <= 8 * kVMaxTiles &&
        verify_mma_smem(variant, io.T, io.lmax) <= 227 * 1024 - 1024) {
      switch (variant) {
        case kPlain: return run_verify_mma<kPlain, TREE>(P, rows, io, tree, stream);
        case kGated: return run_verify_mma<kGated, TREE>(P, rows, io, tree, stream);
        case kGatedDelta: return run_verify_mma<kGatedDelta, TREE>(P, rows, io, tree, stream);
      }
    }
    return verify_variant<__nv_bfloat16, TREE>(P, rows, io, variant, d, tree, stream);
  }
  return kUnsupported;
}

cudaError_t launch_verify(const PoolView &P, const RowBatch &rows, const TokenIO &io, int variant,
                          int dtype, int d, int max_len, cudaStream_t stream,
                          const TreeArg<true> *tree, const StateMap *smap) {
  if (rows.count <= 0) return cudaSuccess;
  TokenIO io2 = io;
  io2.lmax = max_len;
  if (tree) {
    if (rows.count > kTreeRows) return kUnsupported;
    return verify_dispatch<true>(P, rows, io2, variant, dtype, d, *tree, smap, stream);
  }
  return verify_dispatch<false>(P, rows, io2, variant, dtype, d, TreeArg<false>{}, smap, stream);
}

// ------------------------------------------------------------------ tree accept
// Compaction after a draft tree is accepted: the accepted path's entries (key,
// value, pseudo-value, cumulative gate, beta) move to the front of the draft
// slots in path order.  Path positions are visited in order with a barrier in
// between: the entry read at position l (slot n + path[l], path[l] >= l) is
// never one written before it, and a slot written at l is read only at an
// earlier position.  One CTA per (row, value head); the key rows of a q/k head
// are moved by its first value head.
template <typename KT>
__global__ void __launch_bounds__(128)
    tree_compact_kernel(const PoolView P, const RowBatch rows,
                        const __grid_constant__ TreeArg<true> path, int D, int delta) {
  const RowDesc d = rows.r[blockIdx.y];
  const int h = blockIdx.x, group = P.Hv / P.Hk, hq = h / group;
  const int n = d.n, len = d.flags;
  KT *kb = static_cast<KT *>(P.kbuf);
  KT *vb = static_cast<KT *>(P.vbuf);
  for (int l = 0; l < len; ++l) {
    const int src = path.p[blockIdx.y][l];
    if (src == l) continue;  // uniform over the CTA
    const int gs = buffer_row(P, d, n + src), gd = buffer_row(P, d, n + l);
    if (gs < 0 || gd < 0) return;  // uniform; recorded in the error word
    const size_t vs = kv_row(P, gs, h, P.Hv), vd = kv_row(P, gd, h, P.Hv);
    for (int c = threadIdx.x; c < D; c += blockDim.x) vb[vd * D + c] = vb[vs * D + c];
    if (delta)
      for (int c = threadIdx.x; c < D; c += blockDim.x) P.ubuf[vd * D + c] = P.ubuf[vs * D + c];
    if (threadIdx.x == 0) {
      P.gbuf[vd] = P.gbuf[vs];
      P.bbuf[vd] = P.bbuf[vs];
    }
    if (h % group == 0) {
      const size_t ks = kv_row(P, gs, hq, P.Hk) * D, kd = kv_row(P, gd, hq, P.Hk) * D;
      for (int c = threadIdx.x; c < D; c += blockDim.x) kb[kd + c] = kb[ks + c];
    }
    __syncthreads();
  }
}

cudaError_t launch_tree_compact(const PoolView &P, const RowBatch &rows,
                                const TreeArg<true> &path, int variant, int dtype, int d,
                                cudaStream_t stream) {
  if (rows.count <= 0) return cudaSuccess;
  if (rows.count > kTreeRows) return kUnsupported;
  dim3 grid(P.Hv, rows.count);
  const int delta = variant == kGatedDelta;
  if (dtype == 0)
    tree_compact_kernel<float><<<grid, 128, 0, stream>>>(P, rows, path, d, delta);
  else if (dtype == 1)
    tree_compact_kernel<__nv_bfloat16><<<grid, 128, 0, stream>>>(P, rows, path, d, delta);
  else
    return kUnsupported;
  return cudaGetLastError();
}

}  // namespace kvb
