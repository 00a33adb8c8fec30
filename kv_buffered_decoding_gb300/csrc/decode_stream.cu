// Buffered decode as a persistent, software-pipelined kernel (d = 128).
//
// The arithmetic is the one of decode_kernel (decode.cu; "KVBuffer: IO-aware
// Serving for Linear Attention", Figure 1): o_t = e^{A_t} S0^T q_t +
// sum_{i<=t} e^{A_t-A_i} (q_t.k_i) u_i with the gated-delta pseudo-value u_t,
// and a fold S <- e^{A_t} S0 + sum_i e^{A_t-A_i} k_i u_i^T when the buffer fills.
// What changes is how the bytes move.  A work unit is one (row, value head):
// two 32 KB column halves of S0 plus the token's q/k/v and up to kStageTok
// buffered tokens.  Each CTA walks units c, c + G, c + 2G, ... (G = resident
// CTAs).  Once a half's tile has moved from shared memory into registers,
// cp.async brings the next tile (the unit's second half, or the next unit's
// first half with all its small operands: q, k_t, v_t, buffered keys,
// pseudo-values, cumulative gates) into the freed buffer while the half
// computes.  HBM then streams without gaps, instead of idling
// while every resident CTA of an SM computes.  The tile is stored with its
// 16-byte chunks XOR-swizzled on row bit 4, so the per-thread reads (16 rows x
// 4 columns) are free of bank conflicts.
#include <type_traits>

#include "kvb_device.cuh"

namespace kvb {
namespace {

constexpr int kD = 128, kCW = 64;       // head dim; state columns per item
constexpr int kTileF4 = kD * kCW / 4;   // float4 chunks of a tile (2048)
constexpr int kStreamThreads = 128;

// A folding unit of a bf16 pool runs its rank update on the tensor cores
// (fold_tile, kvb_device.cuh) from rows restaged in that routine's orders: the
// keys of tokens 0..n over all state rows, and the current half's u.  fp32
// pools keep FMAs (their restaged rows would cost a resident CTA per SM).
constexpr int kFoldKS = kD + 8, kFoldUS = kCW + 8;  // staged row strides (floats)
template <typename KT>
constexpr bool kFoldOnTc = std::is_same<KT, __nv_bfloat16>::value;
template <typename KT>
constexpr size_t fold_stage_bytes() {
  return kFoldOnTc<KT> ? (size_t)(kStageTok + 1) * (kFoldKS + kFoldUS) * sizeof(float) : 0;
}

// The small operands of one head (double-buffered); the state tile has a
// single buffer, refilled as soon as a tile has moved into registers.
template <typename KT>
struct alignas(16) Stage {
  KT q[kD], k[kD], v[kD];               // current token's q, k, v (raw)
  KT keys[kStageTok][kD];               // buffered keys (raw)
  float uv[kStageTok][kD];              // buffered u (gated delta) / v rows
  float A[kStageTok];                   // buffered cumulative log-gates
  float a_t, beta_t;
  size_t koff[kStageTok + 1], voff[kStageTok + 1];  // tokens 0..n (n: this token's slot)
  int bad;
};

__device__ __forceinline__ int tile_slot(int r, int ch) { return r * 16 + (ch ^ (((r >> 4) & 1) << 2)); }

__device__ __forceinline__ void cp16(void *smem, const void *gmem) {
  const unsigned s = static_cast<unsigned>(__cvta_generic_to_shared(smem));
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(s), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp4(void *smem, const void *gmem) {
  const unsigned s = static_cast<unsigned>(__cvta_generic_to_shared(smem));
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;\n" ::"r"(s), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
__device__ __forceinline__ void cp_wait_all() { asm volatile("cp.async.wait_group 0;\n" ::: "memory"); }

// Four consecutive raw values as floats (fp32: one 16-byte load; bf16: 8 bytes).
__device__ __forceinline__ float4 raw4(const float *p) { return *reinterpret_cast<const float4 *>(p); }
__device__ __forceinline__ float4 raw4(const __nv_bfloat16 *p) {
  const uint2 w = *reinterpret_cast<const uint2 *>(p);
  return make_float4(__uint_as_float(w.x << 16), __uint_as_float(w.x & 0xffff0000u),
                     __uint_as_float(w.y << 16), __uint_as_float(w.y & 0xffff0000u));
}

// A work unit is one (row, value head); its two 64-column halves of the state
// pass through the tile buffer one after the other, and everything that does
// not depend on the columns (staging of q, k, v and the buffered tokens, the
// score dot products, the decay weights) is done once per unit.
template <typename KT, int VARIANT>
__global__ void __launch_bounds__(kStreamThreads, 4)
    decode_stream_kernel(const PoolView P, const __grid_constant__ RowBatch rows, const TokenIO io,
                         int units, FastDiv hv_div) {
  constexpr bool DELTA = VARIANT == kGatedDelta, GATED = VARIANT != kPlain;
  constexpr int RPT = 16, E = kD / 32;
  constexpr int VEC = 16 / (int)sizeof(KT);  // elements per 16-byte copy
  constexpr int NQ = kD / VEC;               // 16-byte chunks of q, k, v or a key
  constexpr int NU = DELTA ? kD / 4 : kD / VEC;  // chunks of a buffered u / v row
  using St = Stage<KT>;
  extern __shared__ float4 dyn_smem[];
  float4 *tile = dyn_smem;                                // [kTileF4] swizzled
  St *stages = reinterpret_cast<St *>(dyn_smem + kTileF4);  // [2]
  float *fks = reinterpret_cast<float *>(stages + 2);       // [kStageTok + 1][kFoldKS] (bf16 pools)
  float *fus = fks + (kStageTok + 1) * kFoldKS;             // [kStageTok + 1][kFoldUS]
  __shared__ __align__(16) float qs[kD], kts[kD];
  __shared__ float wt[kStageTok + 1], sc[kStageTok + 1], cc[kStageTok + 1];
  __shared__ float e_t_s, At_s;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int rsub = lane >> 2, row0 = rsub * RPT;
  const int chunk = warp * 4 + (lane & 3);  // this thread's float4 column chunk in a half
  const int colL = chunk * 4;               // ... as a column within the half
  const int group = P.Hv / P.Hk;

  // one half of unit u's state tile into the tile buffer (no commit)
  auto issue_tile = [&](int u, int part) {
    const int y = fast_div(u, hv_div), h = u - y * P.Hv;
    const float *Sp = P.state + ((size_t)rows.r[y].slot * P.Hv + h) * kD * kD + part * kCW;
    for (int i = tid; i < kTileF4; i += kStreamThreads) {
      const int r = i >> 4, ch = i & 15;
      cp16(&tile[tile_slot(r, ch)], Sp + (size_t)r * kD + ch * 4);
    }
  };
  // unit u's small operands into stages[st] (no commit)
  auto issue_small = [&](int u, int st) {
    St &S = stages[st];
    const int y = fast_div(u, hv_div), h = u - y * P.Hv;
    const RowDesc &d = rows.r[y];
    const size_t b = (size_t)rows.row0 + y;
    const int hq = h / group, n = d.n;
    // dealt round-robin over the warps (warp i of every CTA runs on scheduler i)
    const KT *qg = static_cast<const KT *>(io.q) + (b * P.Hk + hq) * kD;
    const KT *kg = static_cast<const KT *>(io.k) + (b * P.Hk + hq) * kD;
    const KT *vg = static_cast<const KT *>(io.v) + (b * P.Hv + h) * kD;
    constexpr int NSMALL = 3 * NQ + 2;
    for (int t = (tid & 31) * 4 + warp; t < NSMALL; t += kStreamThreads) {
      if (t < NQ) {
        cp16(&S.q[t * VEC], qg + t * VEC);
      } else if (t < 2 * NQ) {
        cp16(&S.k[(t - NQ) * VEC], kg + (t - NQ) * VEC);
      } else if (t < 3 * NQ) {
        cp16(&S.v[(t - 2 * NQ) * VEC], vg + (t - 2 * NQ) * VEC);
      } else if (t == 3 * NQ) {
        if (GATED && io.log_g) cp4(&S.a_t, io.log_g + b * P.Hv + h);
        else S.a_t = 0.f;
      } else {
        if (DELTA) cp4(&S.beta_t, io.beta + b * P.Hv + h);
        else S.beta_t = 0.f;
      }
    }
    // buffered tokens: every warp finds where tokens 0..n live (lane i: token i);
    // keys are copied by warps 0-1, u / v rows by warps 2-3, gates by warp 3
    size_t ko = 0, vo = 0;
    int anybad = 0;
    if (lane <= n) {
      const int g = buffer_row(P, d, lane);
      anybad = g < 0;
      if (g >= 0) {
        ko = kv_row(P, g, hq, P.Hk) * kD;
        vo = kv_row(P, g, h, P.Hv);
      }
    }
    anybad = __any_sync(kFull, anybad);
    if (warp == 3) {
      if (lane <= n) {
        S.koff[lane] = ko;
        S.voff[lane] = vo;
      }
      if (lane == 0) S.bad = anybad;
    }
    if (!anybad) {
      const int l2 = (warp & 1) * 32 + lane;  // lane among the two warps of a task
      // (uniform trip counts: every lane of the warp takes part in each shuffle)
      if (warp < 2) {
        const KT *kb = static_cast<const KT *>(P.kbuf);
        for (int c0 = 0; c0 < n * NQ; c0 += 64) {
          const int c = c0 + l2;
          const bool ok = c < n * NQ;
          const int i = ok ? c / NQ : 0, p = c - i * NQ;
          const size_t off = __shfl_sync(kFull, ko, i);
          if (ok) cp16(&S.keys[i][p * VEC], kb + off + p * VEC);
        }
      } else {
        for (int c0 = 0; c0 < n * NU; c0 += 64) {
          const int c = c0 + l2;
          const bool ok = c < n * NU;
          const int i = ok ? c / NU : 0, p = c - i * NU;
          const size_t row = __shfl_sync(kFull, vo, i) * kD;
          if (!ok) continue;
          if (DELTA)
            cp16(&S.uv[i][p * 4], P.ubuf + row + p * 4);
          else  // raw values fill the first half of the row; widened when read
            cp16(reinterpret_cast<KT *>(S.uv[i]) + p * VEC,
                 static_cast<const KT *>(P.vbuf) + row + p * VEC);
        }
        if (GATED && warp == 3 && lane < n) cp4(&S.A[lane], P.gbuf + vo);
      }
    }
  };
  auto tile_to_regs = [&](float4 (&s)[RPT]) {
#pragma unroll
    for (int j = 0; j < RPT; ++j) s[j] = tile[tile_slot(row0 + j, chunk)];
  };

  // one half of the unit's columns: outputs, appends and (on a fold) the state
  auto half = [&](float4 (&s)[RPT], const St &S, int part, int y, int h) {
    const bool lead = part == 0;
    const RowDesc &d = rows.r[y];
    const size_t b = (size_t)rows.row0 + y;
    const int n = d.n;
    const bool fold = (d.flags & kFlagFlush) != 0;
    const int col0 = part * kCW + colL;  // this thread's column within the head

    // S0^T q_t and S0^T k_t over this thread's rows
    float4 aq = f4(0.f), ak = f4(0.f);
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

    // first half only: decay weights w_i = e^{A_t - A_i} (warp 1) and the dot
    // products q.k_i, k_t.k_i, two tokens per warp pass, one butterfly each
    if (lead) {
      const float At = GATED ? At_s : 0.f;
      if (warp == 1) {
        for (int i = lane; i <= n; i += 32) wt[i] = GATED ? expf(At - (i < n ? S.A[i] : At)) : 1.f;
        if (lane == 0) e_t_s = GATED ? expf(At) : 1.f;
      }
      for (int i0 = 2 * warp; i0 <= n; i0 += 8) {
        const int i1 = i0 + 1;
        float qv[E], tv[E], ka[E], kb[E];
        load_smem<E>(qs + lane * E, qv);
        load_smem<E>(kts + lane * E, tv);
        if (i0 < n) {
          const float4 r4 = raw4(&S.keys[i0][lane * E]);
          ka[0] = r4.x; ka[1] = r4.y; ka[2] = r4.z; ka[3] = r4.w;
        } else {
#pragma unroll
          for (int e = 0; e < E; ++e) ka[e] = tv[e];
        }
        if (i1 < n) {
          const float4 r4 = raw4(&S.keys[i1][lane * E]);
          kb[0] = r4.x; kb[1] = r4.y; kb[2] = r4.z; kb[3] = r4.w;
        } else {
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
      }
      __syncthreads();
    }

    // this lane's share of the buffered terms, one reduction over the row lanes
    const float e_t = e_t_s;
    float4 po = mul4(e_t, aq), pc = mul4(e_t, ak);
    for (int i = rsub; i < n; i += 8) {
      const float4 ui = DELTA ? *reinterpret_cast<const float4 *>(&S.uv[i][col0])
                              : raw4(reinterpret_cast<const KT *>(S.uv[i]) + col0);
      const float w = wt[i];
      fma4(po, w * sc[i], ui);
      if (DELTA) fma4(pc, w * cc[i], ui);
    }
    po = rows_sum4(po);
    if (DELTA) pc = rows_sum4(pc);
    const float4 vt = raw4(&S.v[col0]);
    float4 ut = vt;
    if (DELTA) {
      const float bt = S.beta_t;
      ut.x = bt * (vt.x - pc.x);
      ut.y = bt * (vt.y - pc.y);
      ut.z = bt * (vt.z - pc.z);
      ut.w = bt * (vt.w - pc.w);
    }
    fma4(po, sc[n], ut);
    if (rsub == 0) {
      __stcs(reinterpret_cast<float4 *>(io.o + (b * P.Hv + h) * kD + col0), po);
      st4(static_cast<KT *>(P.vbuf) + S.voff[n] * kD + col0, vt);
      if (DELTA) st4(P.ubuf + S.voff[n] * kD + col0, ut);
    }
    if (lead) {
      if (h % group == 0 && warp == 2)  // 32 lanes x 4 elements of k_t
        st4(static_cast<KT *>(P.kbuf) + S.koff[n] + 4 * lane,
            *reinterpret_cast<const float4 *>(&kts[4 * lane]));
      if (tid == 0) {
        P.gbuf[S.voff[n]] = GATED ? At_s : 0.f;  // cumulative since the last fold
        P.bbuf[S.voff[n]] = S.beta_t;
      }
    }

    // fold: S <- e^{A_t} S0 + sum_{i<=n} k_i (w_i u_i)^T, written back once
    if (fold && kFoldOnTc<KT>) {
#pragma unroll
      for (int j = 0; j < RPT; ++j) s[j] = mul4(e_t, s[j]);
      // restage the unit's keys (first half; they serve both) and this half's u,
      // then the rank-(n+1) update (CTA-uniform: the whole CTA works on one unit)
      if (lead)
        for (int c = tid; c < (n + 1) * kD; c += kStreamThreads) {
          const int i = c >> 7, p = c & (kD - 1), r = fold_krow<RPT>(p);
          fks[i * kFoldKS + p] = i < n ? to_float(S.keys[i][r]) : kts[r];
        }
      for (int i = rsub; i <= n; i += 8)
        fold_stage_u(&fus[i * kFoldUS + colL],
                     i < n ? (DELTA ? *reinterpret_cast<const float4 *>(&S.uv[i][col0])
                                    : raw4(reinterpret_cast<const KT *>(S.uv[i]) + col0))
                           : ut);
      __syncthreads();
      fold_tile<RPT, true>(s, fks, kFoldKS, fus, kFoldUS, 16 * warp, wt, n, lane);
      float *Sp = P.state + ((size_t)d.slot * P.Hv + h) * kD * kD;
#pragma unroll
      for (int j = 0; j < RPT; ++j) st_stream4(Sp + (size_t)(row0 + j) * kD + col0, s[j]);
    } else if (fold) {
#pragma unroll
      for (int j = 0; j < RPT; ++j) s[j] = mul4(e_t, s[j]);
      for (int i = 0; i <= n; ++i) {
        const float4 u = i < n ? mul4(wt[i], DELTA ? *reinterpret_cast<const float4 *>(&S.uv[i][col0])
                                                   : raw4(reinterpret_cast<const KT *>(S.uv[i]) + col0))
                               : ut;
#pragma unroll
        for (int j = 0; j < RPT; j += 4) {
          const float4 k4 = i < n ? raw4(&S.keys[i][row0 + j])
                                  : *reinterpret_cast<const float4 *>(&kts[row0 + j]);
          fma4(s[j], k4.x, u);
          fma4(s[j + 1], k4.y, u);
          fma4(s[j + 2], k4.z, u);
          fma4(s[j + 3], k4.w, u);
        }
      }
      float *Sp = P.state + ((size_t)d.slot * P.Hv + h) * kD * kD;
#pragma unroll
      for (int j = 0; j < RPT; ++j) st_stream4(Sp + (size_t)(row0 + j) * kD + col0, s[j]);
    }
    if (h == 0 && !lead && tid == 0) P.dlen[d.req] = fold ? 0 : n + 1;
  };

  int u = blockIdx.x, st = 0;
  if (u < units) {
    issue_tile(u, 0);
    issue_small(u, 0);
    cp_commit();
  }
  for (; u < units; u += gridDim.x, st ^= 1) {
    const int y = fast_div(u, hv_div), h = u - y * P.Hv;
    const St &S = stages[st];
    float4 s[RPT];
    // first half: its tile and the unit's small operands are staged
    cp_wait_all();
    __syncthreads();  // also: every thread is done with the previous unit
    const bool bad = S.bad != 0;  // CTA-uniform; the error is recorded
    tile_to_regs(s);
    qs[tid] = P.scale * to_float(S.q[tid]);
    kts[tid] = to_float(S.k[tid]);
    if (GATED && tid == 0) {
      const int n = rows.r[y].n;
      At_s = (n > 0 && !bad ? S.A[n - 1] : 0.f) + S.a_t;
    }
    __syncthreads();  // the tile buffer is free
    issue_tile(u, 1);
    cp_commit();
    if (!bad) half(s, S, 0, y, h);
    // second half
    cp_wait_all();
    __syncthreads();
    tile_to_regs(s);
    __syncthreads();  // the tile buffer is free; the other small stage is unused
    if (u + (int)gridDim.x < units) {
      issue_tile(u + gridDim.x, 0);
      issue_small(u + gridDim.x, st ^ 1);
      cp_commit();
    }
    if (!bad) half(s, S, 1, y, h);
  }
}

// ------------------------------------------------------------------ flush
// The standalone fold (kvb_flush, and kvb_accept when the buffer fills) with the
// same streaming: S <- e^{A_L} S0 + sum_{i<=L} e^{A_L-A_i} k_i u_i^T for the L
// buffered tokens (L <= kStageTok), each unit's two column halves passing
// through the tile buffer while the staged keys, u / v rows and gates of the
// next unit arrive.  Rows flagged kFlagFromZero start from S = 0.
template <typename KT>
struct alignas(16) FStage {
  KT keys[kStageTok][kD];   // buffered keys (raw)
  float uv[kStageTok][kD];  // buffered u (gated delta) / v rows
  float A[kStageTok];       // buffered cumulative log-gates
  int bad;
};

template <typename KT, int VARIANT>
__global__ void __launch_bounds__(kStreamThreads, 4)
    flush_stream_kernel(const PoolView P, const __grid_constant__ RowBatch rows, int units,
                        FastDiv hv_div) {
  constexpr bool DELTA = VARIANT == kGatedDelta, GATED = VARIANT != kPlain;
  constexpr int RPT = 16;
  constexpr int VEC = 16 / (int)sizeof(KT);
  constexpr int NQ = kD / VEC;
  constexpr int NU = DELTA ? kD / 4 : kD / VEC;
  using St = FStage<KT>;
  extern __shared__ float4 dyn_smem[];
  float4 *tile = dyn_smem;
  St *stages = reinterpret_cast<St *>(dyn_smem + kTileF4);
  float *fks = reinterpret_cast<float *>(stages + 2);  // [kStageTok + 1][kFoldKS] (bf16 pools)
  float *fus = fks + (kStageTok + 1) * kFoldKS;        // [kStageTok + 1][kFoldUS]
  __shared__ float wt[kStageTok];

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int rsub = lane >> 2, row0 = rsub * RPT;
  const int chunk = warp * 4 + (lane & 3), colL = chunk * 4;
  const int group = P.Hv / P.Hk;

  auto issue_tile = [&](int u, int part) {
    const int y = fast_div(u, hv_div), h = u - y * P.Hv;
    const float *Sp = P.state + ((size_t)rows.r[y].slot * P.Hv + h) * kD * kD + part * kCW;
    for (int i = tid; i < kTileF4; i += kStreamThreads) {
      const int r = i >> 4, ch = i & 15;
      cp16(&tile[tile_slot(r, ch)], Sp + (size_t)r * kD + ch * 4);
    }
  };
  auto issue_small = [&](int u, int st) {
    St &S = stages[st];
    const int y = fast_div(u, hv_div), h = u - y * P.Hv;
    const RowDesc &d = rows.r[y];
    const int hq = h / group, L = d.n;
    size_t ko = 0, vo = 0;
    int anybad = 0;
    if (lane < L) {
      const int g = buffer_row(P, d, lane);
      anybad = g < 0;
      if (g >= 0) {
        ko = kv_row(P, g, hq, P.Hk) * kD;
        vo = kv_row(P, g, h, P.Hv);
      }
    }
    anybad = __any_sync(kFull, anybad);
    if (warp == 3 && lane == 0) S.bad = anybad;
    if (!anybad) {
      const int l2 = (warp & 1) * 32 + lane;
      if (warp < 2) {
        const KT *kb = static_cast<const KT *>(P.kbuf);
        for (int c0 = 0; c0 < L * NQ; c0 += 64) {
          const int c = c0 + l2;
          const bool ok = c < L * NQ;
          const int i = ok ? c / NQ : 0, p = c - i * NQ;
          const size_t off = __shfl_sync(kFull, ko, i);
          if (ok) cp16(&S.keys[i][p * VEC], kb + off + p * VEC);
        }
      } else {
        for (int c0 = 0; c0 < L * NU; c0 += 64) {
          const int c = c0 + l2;
          const bool ok = c < L * NU;
          const int i = ok ? c / NU : 0, p = c - i * NU;
          const size_t row = __shfl_sync(kFull, vo, i) * kD;
          if (!ok) continue;
          if (DELTA)
            cp16(&S.uv[i][p * 4], P.ubuf + row + p * 4);
          else
            cp16(reinterpret_cast<KT *>(S.uv[i]) + p * VEC, static_cast<const KT *>(P.vbuf) + row + p * VEC);
        }
        if (GATED && warp == 3 && lane < L) cp4(&S.A[lane], P.gbuf + vo);
      }
    }
  };
  // the unit's state half, scaled by e^{A_L} (zero for rows that start from S = 0)
  auto tile_to_regs = [&](float4 (&s)[RPT], bool zero, float eL) {
#pragma unroll
    for (int j = 0; j < RPT; ++j) s[j] = zero ? f4(0.f) : mul4(eL, tile[tile_slot(row0 + j, chunk)]);
  };
  auto fold_half = [&](float4 (&s)[RPT], const St &S, int part, int y, int h) {
    const RowDesc &d = rows.r[y];
    const int L = d.n, col0 = part * kCW + colL;
    if constexpr (kFoldOnTc<KT>) {
      // restage the unit's keys (first half; they serve both) and this half's u,
      // then the rank-L update (CTA-uniform: the whole CTA works on one unit)
      if (part == 0)
        for (int c = tid; c < L * kD; c += kStreamThreads) {
          const int i = c >> 7, p = c & (kD - 1);
          fks[i * kFoldKS + p] = to_float(S.keys[i][fold_krow<RPT>(p)]);
        }
      for (int i = rsub; i < L; i += 8)
        fold_stage_u(&fus[i * kFoldUS + colL],
                     DELTA ? *reinterpret_cast<const float4 *>(&S.uv[i][col0])
                           : raw4(reinterpret_cast<const KT *>(S.uv[i]) + col0));
      __syncthreads();
      fold_tile<RPT, true>(s, fks, kFoldKS, fus, kFoldUS, 16 * warp, wt, L - 1, lane);
    } else {
      for (int i = 0; i < L; ++i) {
        const float4 u = mul4(wt[i], DELTA ? *reinterpret_cast<const float4 *>(&S.uv[i][col0])
                                           : raw4(reinterpret_cast<const KT *>(S.uv[i]) + col0));
#pragma unroll
        for (int j = 0; j < RPT; j += 4) {
          const float4 k4 = raw4(&S.keys[i][row0 + j]);
          fma4(s[j], k4.x, u);
          fma4(s[j + 1], k4.y, u);
          fma4(s[j + 2], k4.z, u);
          fma4(s[j + 3], k4.w, u);
        }
      }
    }
    float *Sp = P.state + ((size_t)d.slot * P.Hv + h) * kD * kD;
#pragma unroll
    for (int j = 0; j < RPT; ++j) st_stream4(Sp + (size_t)(row0 + j) * kD + col0, s[j]);
  };

  int u = blockIdx.x, st = 0;
  if (u < units) {
    issue_tile(u, 0);
    issue_small(u, 0);
    cp_commit();
  }
  for (; u < units; u += gridDim.x, st ^= 1) {
    const int y = fast_div(u, hv_div), h = u - y * P.Hv;
    const St &S = stages[st];
    float4 s[RPT];
    cp_wait_all();
    __syncthreads();  // first half and the unit's tokens staged; previous unit done
    const bool bad = S.bad != 0, zero = (rows.r[y].flags & kFlagFromZero) != 0;
    const int L = rows.r[y].n;
    const float AL = GATED && L > 0 && !bad ? S.A[L - 1] : 0.f;
    const float eL = GATED ? expf(AL) : 1.f;
    if (warp == 1 && lane < L) wt[lane] = GATED && !bad ? expf(AL - S.A[lane]) : 1.f;
    tile_to_regs(s, zero, eL);
    __syncthreads();  // the tile buffer is free; weights ready
    issue_tile(u, 1);
    cp_commit();
    if (!bad) fold_half(s, S, 0, y, h);
    cp_wait_all();
    __syncthreads();
    tile_to_regs(s, zero, eL);
    __syncthreads();
    if (u + (int)gridDim.x < units) {
      issue_tile(u + gridDim.x, 0);
      issue_small(u + gridDim.x, st ^ 1);
      cp_commit();
    }
    if (!bad) {
      fold_half(s, S, 1, y, h);
      if (h == 0 && tid == 0) P.dlen[rows.r[y].req] = 0;
    }
  }
}

// Resident CTAs of the kernel on the current device (its persistent grid).
template <typename KT, int VARIANT>
int flush_ctas() {
  constexpr size_t smem = kTileF4 * sizeof(float4) + 2 * sizeof(FStage<KT>) + fold_stage_bytes<KT>();
  int ctas = 0;
  return resident_ctas((const void *)flush_stream_kernel<KT, VARIANT>, kStreamThreads, smem,
                       &ctas) == cudaSuccess ? ctas : 0;
}

template <typename KT, int VARIANT>
cudaError_t run_flush_stream(const PoolView &P, const RowBatch &rows, cudaStream_t stream) {
  constexpr size_t smem = kTileF4 * sizeof(float4) + 2 * sizeof(FStage<KT>) + fold_stage_bytes<KT>();
  const int cap = flush_ctas<KT, VARIANT>();
  if (cap <= 0) return kUnsupported;
  const int units = rows.count * P.Hv;
  const int grid = units < cap ? units : cap;
  flush_stream_kernel<KT, VARIANT><<<grid, kStreamThreads, smem, stream>>>(
      P, rows, units, make_fastdiv((uint32_t)P.Hv));
  return cudaGetLastError();
}

template <typename KT>
int fctas_for(int variant) {
  switch (variant) {
    case kPlain: return flush_ctas<KT, kPlain>();
    case kGated: return flush_ctas<KT, kGated>();
    case kGatedDelta: return flush_ctas<KT, kGatedDelta>();
  }
  return 0;
}

// Resident CTAs of the kernel on the current device (its persistent grid).
template <typename KT, int VARIANT>
int stream_ctas() {
  constexpr size_t smem = kTileF4 * sizeof(float4) + 2 * sizeof(Stage<KT>) + fold_stage_bytes<KT>();
  int ctas = 0;
  return resident_ctas((const void *)decode_stream_kernel<KT, VARIANT>, kStreamThreads, smem,
                       &ctas) == cudaSuccess ? ctas : 0;
}

template <typename KT, int VARIANT>
cudaError_t run_stream(const PoolView &P, const RowBatch &rows, const TokenIO &io,
                       cudaStream_t stream) {
  constexpr size_t smem = kTileF4 * sizeof(float4) + 2 * sizeof(Stage<KT>) + fold_stage_bytes<KT>();
  const int cap = stream_ctas<KT, VARIANT>();
  if (cap <= 0) return kUnsupported;
  const int units = rows.count * P.Hv;
  const int grid = units < cap ? units : cap;
  decode_stream_kernel<KT, VARIANT><<<grid, kStreamThreads, smem, stream>>>(
      P, rows, io, units, make_fastdiv((uint32_t)P.Hv));
  return cudaGetLastError();
}

template <typename KT>
int ctas_for(int variant) {
  switch (variant) {
    case kPlain: return stream_ctas<KT, kPlain>();
    case kGated: return stream_ctas<KT, kGated>();
    case kGatedDelta: return stream_ctas<KT, kGatedDelta>();
  }
  return 0;
}

}  // namespace

bool flush_stream_pays(int units, int variant, int dtype) {
  const int cap = dtype == 1 ? fctas_for<__nv_bfloat16>(variant)
                             : dtype == 0 ? fctas_for<float>(variant) : 0;
  return cap > 0 && units >= 8 * cap;
}

cudaError_t launch_flush_stream(const PoolView &P, const RowBatch &rows, int variant, int dtype,
                                cudaStream_t stream) {
  if (rows.count <= 0) return cudaSuccess;
  if (dtype == 1) {
    switch (variant) {
      case kPlain: return run_flush_stream<__nv_bfloat16, kPlain>(P, rows, stream);
      case kGated: return run_flush_stream<__nv_bfloat16, kGated>(P, rows, stream);
      case kGatedDelta: return run_flush_stream<__nv_bfloat16, kGatedDelta>(P, rows, stream);
    }
  } else if (dtype == 0) {
    switch (variant) {
      case kPlain: return run_flush_stream<float, kPlain>(P, rows, stream);
      case kGated: return run_flush_stream<float, kGated>(P, rows, stream);
      case kGatedDelta: return run_flush_stream<float, kGatedDelta>(P, rows, stream);
    }
  }
  return kUnsupported;
}

bool decode_stream_pays(int units, int variant, int dtype) {
  // each resident CTA should get at least 8 units: fewer leave its pipeline
  // prologue and the last partial round of units unamortized
  const int cap = dtype == 1 ? ctas_for<__nv_bfloat16>(variant)
                             : dtype == 0 ? ctas_for<float>(variant) : 0;
  return cap > 0 && units >= 8 * cap;
}

cudaError_t launch_decode_stream(const PoolView &P, const RowBatch &rows, const TokenIO &io,
                                 int variant, int dtype, cudaStream_t stream) {
  if (rows.count <= 0) return cudaSuccess;
  if (dtype == 1) {
    switch (variant) {
      case kPlain: return run_stream<__nv_bfloat16, kPlain>(P, rows, io, stream);
      case kGated: return run_stream<__nv_bfloat16, kGated>(P, rows, io, stream);
      case kGatedDelta: return run_stream<__nv_bfloat16, kGatedDelta>(P, rows, io, stream);
    }
  } else if (dtype == 0) {
    switch (variant) {
      case kPlain: return run_stream<float, kPlain>(P, rows, io, stream);
      case kGated: return run_stream<float, kGated>(P, rows, io, stream);
      case kGatedDelta: return run_stream<float, kGatedDelta>(P, rows, io, stream);
    }
  }
  return kUnsupported;
}

}  // namespace kvb
