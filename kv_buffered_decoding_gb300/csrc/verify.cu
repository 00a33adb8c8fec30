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
// One CTA per (batch row, value head), the same thread layout as decode: warp
// w owns 16 state columns, lanes split rows by 8; the state tile stays in
// registers while the drafts are processed four at a time.
#include "kvb_device.cuh"

namespace kvb {

template <typename KT, int VARIANT, int D>
__global__ void __launch_bounds__(2 * D)
    verify_kernel(const PoolView P, const RowBatch rows, const TokenIO io) {
  constexpr int DK = D, DV = D, NT = 2 * D, RPT = DK / 8, E = DK / 32;
  constexpr bool DELTA = VARIANT == kGatedDelta;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int rsub = lane >> 2, col0 = warp * 16 + (lane & 3) * 4;
  const int h = blockIdx.x;
  const RowDesc d = rows.r[blockIdx.y];
  const size_t b = (size_t)rows.row0 + blockIdx.y;
  const int group = P.Hv / P.Hk;
  const int hq = h / group;
  const bool has_state = d.slot >= 0;
  const int n = d.n, T = io.T, L = n + T;
  const int LM = io.lmax;  // >= L for every row of the launch

  // shared layout (dynamic): ks[LM][DK] keys of the chunk, us[LM][DV] u of the
  // chunk, qs[T][DK] scaled draft queries, yq[T][DV], yk[T][DV] mat-vecs,
  // sw[T][LM], cw[T][LM] decay-weighted scores, Acum[LM], grow[LM]
  extern __shared__ float4 dyn_smem[];
  float *ks = reinterpret_cast<float *>(dyn_smem);
  float *us = ks + (size_t)LM * DK;
  float *qs = us + (size_t)LM * DV;
  float *yq = qs + (size_t)T * DK;
  float *yk = yq + (size_t)T * DV;
  float *sw = yk + (size_t)T * DV;
  float *cw = sw + (size_t)T * LM;
  float *Acum = cw + (size_t)T * LM;
  int *grow = reinterpret_cast<int *>(Acum + LM);
  __shared__ int bad;

  float4 s[RPT];
  const float *Sp = P.state + (has_state ? ((size_t)d.slot * P.Hv + h) * DK * DV : 0);
  if (has_state) {
#pragma unroll
    for (int j = 0; j < RPT; ++j) s[j] = ld_stream4(Sp + (rsub + 8 * j) * DV + col0);
  } else {
#pragma unroll
    for (int j = 0; j < RPT; ++j) s[j] = f4(0.f);
  }

  if (warp == 0) {
    int anybad = 0;
    for (int i = lane; i < L; i += 32) {
      const int g = buffer_row(P, d, i);
      grow[i] = g;
      anybad |= (g < 0);
    }
    anybad = __any_sync(kFull, anybad);
    if (lane == 0) bad = anybad;
  }
  // draft queries and keys (fp32, queries scaled)
  const KT *qg = static_cast<const KT *>(io.q) + b * T * P.Hk * DK;
  const KT *kg = static_cast<const KT *>(io.k) + b * T * P.Hk * DK;
  for (int idx = tid; idx < T * DK; idx += NT) {
    const int j = idx / DK, c = idx % DK;
    const size_t src = ((size_t)j * P.Hk + hq) * DK + c;
    qs[idx] = P.scale * to_float(qg[src]);
    ks[(size_t)(n + j) * DK + c] = to_float(kg[src]);
  }
  __syncthreads();
  if (bad) return;

  // cumulative log-gates over the chunk (warp 0): the buffer stores them for its
  // tokens; the drafts continue the sum.  Buffered keys and u to shared (others).
  if (VARIANT != kPlain) {
    if (warp == 0) {
      const float *lg = io.log_g;
      for (int i = lane; i < n; i += 32) Acum[i] = P.gbuf[kv_row(P, grow[i], h, P.Hv)];
      const float A_prev = n > 0 ? P.gbuf[kv_row(P, grow[n - 1], h, P.Hv)] : 0.f;
      warp_prefix(
          T, [&](int j) { return lg ? lg[(b * T + j) * P.Hv + h] : 0.f; }, Acum + n, lane);
      __syncwarp();
      for (int j = lane; j < T; j += 32) Acum[n + j] += A_prev;
    }
  } else {
    for (int i = tid; i < L; i += NT) Acum[i] = 0.f;
  }
  {
    // every thread helps stage the n buffered tokens; warp 0 joins after its scan
    for (int idx = tid; idx < n * (DK / 4); idx += NT) {
      const int i = idx / (DK / 4), c = (idx % (DK / 4)) * 4;
      *reinterpret_cast<float4 *>(&ks[(size_t)i * DK + c]) =
          ld4(static_cast<const KT *>(P.kbuf) + kv_row(P, grow[i], hq, P.Hk) * DK + c);
    }
    for (int idx = tid; idx < n * (DV / 4); idx += NT) {
      const int i = idx / (DV / 4), c = (idx % (DV / 4)) * 4;
      float4 u;
      if (DELTA)
        u = ld4(P.ubuf + kv_row(P, grow[i], h, P.Hv) * DV + c);
      else
        u = ld4(static_cast<const KT *>(P.vbuf) + kv_row(P, grow[i], h, P.Hv) * DV + c);
      *reinterpret_cast<float4 *>(&us[(size_t)i * DV + c]) = u;
    }
  }
  __syncthreads();

  // decay-weighted scores: sw[j][l] = e^{A_{n+j}-A_l} q_j.k_l (l <= n+j),
  // cw[j][l] = e^{A_{n+j}-A_l} k_{n+j}.k_l (l < n+j); one warp per pair
  const int npairs = T * L;
  for (int p = warp; p < npairs; p += NT / 32) {
    const int j = p / L, l = p % L;
    if (l > n + j) continue;  // warp-uniform
    const float *kl = &ks[(size_t)l * DK];
    const float *qj = &qs[(size_t)j * DK];
    const float *kj = &ks[(size_t)(n + j) * DK];
    float sq = dot_smem<E>(qj + lane * E, kl + lane * E);
    float sk = DELTA ? dot_smem<E>(kj + lane * E, kl + lane * E) : 0.f;
    sq = warp_sum(sq);
    if (DELTA) sk = warp_sum(sk);
    if (lane == 0) {
      const float w = (VARIANT != kPlain) ? expf(Acum[n + j] - Acum[l]) : 1.f;
      sw[j * LM + l] = w * sq;
      cw[j * LM + l] = (l < n + j) ? w * sk : 0.f;
    }
  }

  // mat-vecs, drafts four at a time, straight from the register-resident tile
  for (int j0 = 0; j0 < T; j0 += 4) {
    float4 aq[4], ak[4];
#pragma unroll
    for (int x = 0; x < 4; ++x) aq[x] = ak[x] = f4(0.f);
    if (has_state) {
#pragma unroll
      for (int jr = 0; jr < RPT; ++jr) {
        const int r = rsub + 8 * jr;
#pragma unroll
        for (int x = 0; x < 4; ++x) {
          if (j0 + x < T) {
            fma4(aq[x], qs[(size_t)(j0 + x) * DK + r], s[jr]);
            if (DELTA) fma4(ak[x], ks[(size_t)(n + j0 + x) * DK + r], s[jr]);
          }
        }
      }
#pragma unroll
      for (int x = 0; x < 4; ++x) {
        aq[x] = rows_sum4(aq[x]);
        if (DELTA) ak[x] = rows_sum4(ak[x]);
      }
    }
    if (rsub == 0) {
#pragma unroll
      for (int x = 0; x < 4; ++x) {
        if (j0 + x < T) {
          *reinterpret_cast<float4 *>(&yq[(size_t)(j0 + x) * DV + col0]) = aq[x];
          if (DELTA) *reinterpret_cast<float4 *>(&yk[(size_t)(j0 + x) * DV + col0]) = ak[x];
        }
      }
    }
  }
  __syncthreads();

  // per draft, in order: u_j (forward substitution for the delta rule), o_j
  const KT *vg = static_cast<const KT *>(io.v) + b * T * P.Hv * DV;
  for (int j = 0; j < T; ++j) {
    const int t = n + j;  // chunk position of this draft
    float4 po = f4(0.f), pc = f4(0.f);
    for (int l = rsub; l < t; l += 8) {
      const float4 u = *reinterpret_cast<const float4 *>(&us[(size_t)l * DV + col0]);
      fma4(po, sw[j * LM + l], u);
      if (DELTA) fma4(pc, cw[j * LM + l], u);
    }
    po = rows_sum4(po);
    if (DELTA) pc = rows_sum4(pc);
    const float e_j = (VARIANT != kPlain) ? expf(Acum[t]) : 1.f;
    const float4 vt = ld4(vg + ((size_t)j * P.Hv + h) * DV + col0);
    float4 ut = vt;
    if (DELTA) {
      const float bj = io.beta[(b * T + j) * P.Hv + h];
      const float4 z = *reinterpret_cast<const float4 *>(&yk[(size_t)j * DV + col0]);
      ut.x = bj * (vt.x - fmaf(e_j, z.x, pc.x));
      ut.y = bj * (vt.y - fmaf(e_j, z.y, pc.y));
      ut.z = bj * (vt.z - fmaf(e_j, z.z, pc.z));
      ut.w = bj * (vt.w - fmaf(e_j, z.w, pc.w));
    }
    const float4 y = *reinterpret_cast<const float4 *>(&yq[(size_t)j * DV + col0]);
    float4 o = add4(mul4(e_j, y), po);
    fma4(o, sw[j * LM + t], ut);
    if (rsub == 0) {
      __stcs(reinterpret_cast<float4 *>(io.o + ((b * T + j) * P.Hv + h) * DV + col0), o);
      *reinterpret_cast<float4 *>(&us[(size_t)t * DV + col0]) = ut;
      const size_t g = grow[t];
      st4(static_cast<KT *>(P.vbuf) + kv_row(P, (int)g, h, P.Hv) * DV + col0, vt);
      if (DELTA) st4(P.ubuf + kv_row(P, (int)g, h, P.Hv) * DV + col0, ut);
    }
    __syncwarp();  // u_t of this warp's columns visible to its other lanes
  }

  // drafts' keys and gates into the buffer
  for (int idx = tid; idx < T * (DK / 4); idx += NT) {
    const int j = idx / (DK / 4), c = (idx % (DK / 4)) * 4;
    if (h % group == 0)
      st4(static_cast<KT *>(P.kbuf) + kv_row(P, grow[n + j], hq, P.Hk) * DK + c,
          *reinterpret_cast<const float4 *>(&ks[(size_t)(n + j) * DK + c]));
  }
  for (int j = tid; j < T; j += NT) {
    const size_t g = grow[n + j];
    P.gbuf[kv_row(P, (int)g, h, P.Hv)] = Acum[n + j];  // cumulative since the last fold
    P.bbuf[kv_row(P, (int)g, h, P.Hv)] = DELTA ? io.beta[(b * T + j) * P.Hv + h] : 0.f;
  }
}

// ------------------------------------------------------------------ launcher
static size_t verify_smem(int d, int T, int LM) {
  return sizeof(float) * ((size_t)LM * d * 2 + (size_t)T * d * 3 + (size_t)T * LM * 2 + LM) +
         sizeof(int) * (size_t)LM;
}

template <typename KT, int VARIANT, int D>
static cudaError_t run_verify(const PoolView &P, const RowBatch &rows, const TokenIO &io,
                              cudaStream_t stream) {
  static bool configured = false;
  if (!configured) {
    const size_t most = verify_smem(D, kMaxTok - 1, kMaxTok - 1);
    cudaError_t e = cudaFuncSetAttribute(verify_kernel<KT, VARIANT, D>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)most);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  const size_t smem = verify_smem(D, io.T, io.lmax);
  dim3 grid(P.Hv, rows.count);
  verify_kernel<KT, VARIANT, D><<<grid, 2 * D, smem, stream>>>(P, rows, io);
  return cudaGetLastError();
}

template <typename KT, int VARIANT>
static cudaError_t verify_d(const PoolView &P, const RowBatch &rows, const TokenIO &io, int d,
                            cudaStream_t s) {
  if (d == 128) return run_verify<KT, VARIANT, 128>(P, rows, io, s);
  if (d == 64) return run_verify<KT, VARIANT, 64>(P, rows, io, s);
  return kUnsupported;
}

template <typename KT>
static cudaError_t verify_variant(const PoolView &P, const RowBatch &rows, const TokenIO &io,
                                  int variant, int d, cudaStream_t s) {
  switch (variant) {
    case kPlain: return verify_d<KT, kPlain>(P, rows, io, d, s);
    case kGated: return verify_d<KT, kGated>(P, rows, io, d, s);
    case kGatedDelta: return verify_d<KT, kGatedDelta>(P, rows, io, d, s);
  }
  return kUnsupported;
}

cudaError_t launch_verify(const PoolView &P, const RowBatch &rows, const TokenIO &io, int variant,
                          int dtype, int d, int max_len, cudaStream_t stream) {
  if (rows.count <= 0) return cudaSuccess;
  TokenIO io2 = io;
  io2.lmax = max_len;
  if (dtype == 0) return verify_variant<float>(P, rows, io2, variant, d, stream);
  if (dtype == 1) return verify_variant<__nv_bfloat16>(P, rows, io2, variant, d, stream);
  return kUnsupported;
}

}  // namespace kvb
