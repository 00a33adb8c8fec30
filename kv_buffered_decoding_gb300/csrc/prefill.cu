// Chunked prefill: build a request's state from its prompt, C = 64 tokens at a
// time, on the tensor cores.
//
// This is the step before the decode hot path ("KVBuffer: IO-aware Serving
// for Linear Attention", abstract: chunkwise computation of linear attention;
// the delta-rule chunk form with the UT transform is the one of the gated
// delta networks it serves).  Within a chunk of tokens 0..C-1 with cumulative
// log-gates A_i (inclusive, restarting at 0 each chunk) and the state S at
// the chunk start (d_k x d_v):
//   u_i = beta_i (v_i - e^{A_i} S^T k_i - sum_{j<i} e^{A_i-A_j} (k_i.k_j) u_j)   (delta rule)
//   u_i = v_i                                                                   (plain, gated)
//   o_i = e^{A_i} S^T q_i + sum_{j<=i} e^{A_i-A_j} (q_i.k_j) u_j
//   S  <- e^{A_{C-1}} S + sum_j e^{A_{C-1}-A_j} k_j u_j^T
// which is the per-token recurrence exactly (up to rounding), the same
// algebra as a buffer of C tokens folded into the state.  In matrix form the
// chunk is five products: Y = [Q; K] S, the two C x C Gram matrices Q K^T and
// K K^T, the unit lower-triangular solve (I + Mk) U = R (forward
// substitution; the UT transform), O += Mq U, and S += K^T diag(w) U.
//
// One CTA of 8 warps per (request, value head) walks the chunks in order.
// Shared memory holds the state (fp32), the chunk's q/k/v (double-buffered
// with cp.async when the inputs are bf16), U and one C x C buffer with both
// masked Gram matrices (Mk strictly below the diagonal, Mq transposed above
// it).  All products run as mma.sync m16n8k8 with tf32 operands and fp32
// accumulation; operands that are not exact in tf32 (the state, U, the Gram
// matrices, fp32 inputs) are split into hi + lo tf32 parts (three products
// per pair, about 21 significant bits), so the result keeps fp32-like
// accuracy.  bf16 inputs are exact in tf32 and take one part.
#include "kvb_device.cuh"

namespace kvb {
namespace {

constexpr int kChunk = 64;
constexpr int kPrefillThreads = 256;

template <typename KT, int D>
struct PrefillShape {
  static constexpr int C = kChunk;
  static constexpr bool BF16 = sizeof(KT) == 2;
  static constexpr int STAGES = BF16 ? 2 : 1;
  static constexpr int LDI = BF16 ? D + 8 : D + 4;  // input rows, elements (16-byte multiple)
  // fp32 rows of S, U and the Gram buffer: a stride of 8 banks (mod 32) makes
  // the fragment loads (lane g -> column, lane t -> row) conflict-free
  static constexpr int LDS = D + 8;
  static constexpr int LDX = C + 8;
  static constexpr size_t S_OFF = 0;
  static constexpr size_t U_OFF = S_OFF + (size_t)D * LDS * 4;
  static constexpr size_t X_OFF = U_OFF + (size_t)C * LDS * 4;
  static constexpr size_t IN_OFF = X_OFF + (size_t)C * LDX * 4;
  static constexpr size_t IN_TILE = (size_t)C * LDI * sizeof(KT);  // one of q, k, v
  static constexpr size_t G_OFF = IN_OFF + STAGES * 3 * IN_TILE;   // [STAGES][2][C] log-gate, beta
  static constexpr size_t A_OFF = G_OFF + (size_t)STAGES * 2 * C * 4;  // A, e^A, w: [3][C]
  static constexpr size_t BYTES = A_OFF + 3 * C * 4;
  static_assert(IN_OFF % 16 == 0 && IN_TILE % 16 == 0 && G_OFF % 16 == 0, "16-byte staging");
  static_assert(BYTES <= 227 * 1024, "fits one CTA's shared memory");
};

__device__ __forceinline__ void cp_async16(void *smem, const void *gmem, bool valid) {
  const unsigned s = static_cast<unsigned>(__cvta_generic_to_shared(smem));
  const int n = valid ? 16 : 0;  // 0: fill with zeros, read nothing
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(s), "l"(gmem), "r"(n)
               : "memory");
}
__device__ __forceinline__ void cp_async4(void *smem, const void *gmem, bool valid) {
  const unsigned s = static_cast<unsigned>(__cvta_generic_to_shared(smem));
  const int n = valid ? 4 : 0;
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;\n" ::"r"(s), "l"(gmem), "r"(n)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}

// One tf32 operand value in (hi, lo) form; exact sources leave lo unused.
template <bool EXACT>
__device__ __forceinline__ void operand(float x, uint32_t &hi, uint32_t &lo) {
  if (EXACT) {
    hi = __float_as_uint(x);
    lo = 0u;
  } else {
    split_tf32(x, hi, lo);
  }
}

// The two halves of d += a b with a, b in (hi, lo) form: the small cross
// terms first, then hi * hi.  Callers issue the first half for every tile of
// a step before the second, so consecutive products use different
// accumulators.
template <bool AX, bool BX>
__device__ __forceinline__ void mma_small(float (&d)[4], const uint32_t (&ah)[4],
                                          const uint32_t (&al)[4], const uint32_t (&bh)[2],
                                          const uint32_t (&bl)[2]) {
  if (!BX) mma_tf32(d, ah, bl[0], bl[1]);
  if (!AX) mma_tf32(d, al, bh[0], bh[1]);
}
__device__ __forceinline__ void mma_big(float (&d)[4], const uint32_t (&ah)[4],
                                        const uint32_t (&bh)[2]) {
  mma_tf32(d, ah, bh[0], bh[1]);
}

// A fragment (16 x 8, row-major source): rows r0+g, r0+g+8; columns c0+t, c0+t+4.
template <bool EXACT, typename T>
__device__ __forceinline__ void load_a(const T *src, int ld, int r0, int c0, int g, int t,
                                       uint32_t (&hi)[4], uint32_t (&lo)[4]) {
  operand<EXACT>(to_float(src[(r0 + g) * ld + c0 + t]), hi[0], lo[0]);
  operand<EXACT>(to_float(src[(r0 + g + 8) * ld + c0 + t]), hi[1], lo[1]);
  operand<EXACT>(to_float(src[(r0 + g) * ld + c0 + t + 4]), hi[2], lo[2]);
  operand<EXACT>(to_float(src[(r0 + g + 8) * ld + c0 + t + 4]), hi[3], lo[3]);
}

// A fragment of a transposed source: element (m, k) = src[k][m].
template <bool EXACT, typename T>
__device__ __forceinline__ void load_at(const T *src, int ld, int m0, int k0, int g, int t,
                                        uint32_t (&hi)[4], uint32_t (&lo)[4]) {
  operand<EXACT>(to_float(src[(k0 + t) * ld + m0 + g]), hi[0], lo[0]);
  operand<EXACT>(to_float(src[(k0 + t) * ld + m0 + g + 8]), hi[1], lo[1]);
  operand<EXACT>(to_float(src[(k0 + t + 4) * ld + m0 + g]), hi[2], lo[2]);
  operand<EXACT>(to_float(src[(k0 + t + 4) * ld + m0 + g + 8]), hi[3], lo[3]);
}

// Masked Gram rows 16 mt .. 16 mt + 15 against the chunk's keys, n-tiles nst ..
// nst + GNT - 1 (tiles wholly above the diagonal are skipped).  KK: Mk[i][j] =
// beta_i e^{A_i-A_j} k_i.k_j for j < i, stored at X[i][j]; otherwise Mq[i][j] =
// scale e^{A_i-A_j} q_i.k_j for j <= i, stored transposed at X[j][i+1].
template <bool XIN, bool KK, int GNT, int D, int LDI, int LDX, typename KT>
__device__ __forceinline__ void gram_rows(const KT *asrc, const KT *ks, int mt, int nst,
                                          const float *Acum, const float *bs, float scale,
                                          float *Xs, int g, int t) {
  float acc[GNT][4];
#pragma unroll
  for (int n = 0; n < GNT; ++n) acc[n][0] = acc[n][1] = acc[n][2] = acc[n][3] = 0.f;
#pragma unroll 2
  for (int k0 = 0; k0 < D; k0 += 8) {
    uint32_t ah[4], al[4], bh[GNT][2], bl[GNT][2];
    load_a<XIN>(asrc, LDI, 16 * mt, k0, g, t, ah, al);
#pragma unroll
    for (int n = 0; n < GNT; ++n) {
      const int row = 8 * (nst + n) + g;
      operand<XIN>(to_float(ks[row * LDI + k0 + t]), bh[n][0], bl[n][0]);
      operand<XIN>(to_float(ks[row * LDI + k0 + t + 4]), bh[n][1], bl[n][1]);
    }
#pragma unroll
    for (int n = 0; n < GNT; ++n)
      if (nst + n <= 2 * mt + 1) mma_small<XIN, XIN>(acc[n], ah, al, bh[n], bl[n]);
#pragma unroll
    for (int n = 0; n < GNT; ++n)
      if (nst + n <= 2 * mt + 1) mma_big(acc[n], ah, bh[n]);
  }
#pragma unroll
  for (int n = 0; n < GNT; ++n) {
    const int nt = nst + n;
    if (nt > 2 * mt + 1) continue;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int i = 16 * mt + g + (e >> 1) * 8, j = 8 * nt + 2 * t + (e & 1);
      if (KK) {
        if (j < i) Xs[i * LDX + j] = bs[i] * expf(Acum[i] - Acum[j]) * acc[n][e];
      } else {
        if (j <= i) Xs[j * LDX + i + 1] = scale * expf(Acum[i] - Acum[j]) * acc[n][e];
      }
    }
  }
}

template <typename KT, int VARIANT, int D>
__global__ void __launch_bounds__(kPrefillThreads, 1)
    prefill_kernel(const PoolView P, const RowBatch rows, const TokenIO io) {
  using Sh = PrefillShape<KT, D>;
  constexpr int C = Sh::C, LDI = Sh::LDI, LDS = Sh::LDS, LDX = Sh::LDX, STAGES = Sh::STAGES;
  constexpr bool DELTA = VARIANT == kGatedDelta, GATED = VARIANT != kPlain;
  constexpr bool XIN = Sh::BF16;  // q, k, v exact in tf32
  constexpr int NW3 = D / 32;     // n-tiles per warp in Y and O
  constexpr int MT = DELTA ? 4 : 2;  // m-tiles per warp in Y and O
  constexpr int MT6 = D / 16;  // m-tiles (state rows) per warp in the state update
  constexpr int NPW = D / 64;  // n-tiles (state columns) per warp in the state update

  extern __shared__ float4 dyn_smem[];
  char *sm = reinterpret_cast<char *>(dyn_smem);
  float *Ss = reinterpret_cast<float *>(sm + Sh::S_OFF);  // [D][LDS] state
  float *Us = reinterpret_cast<float *>(sm + Sh::U_OFF);  // [C][LDS] R, then U (delta rule)
  float *Xs = reinterpret_cast<float *>(sm + Sh::X_OFF);  // [C][LDX] Mk below, Mq^T above
  KT *In = reinterpret_cast<KT *>(sm + Sh::IN_OFF);      // [STAGES][q, k, v][C][LDI]
  float *Gr = reinterpret_cast<float *>(sm + Sh::G_OFF);  // [STAGES][log-gate, beta][C]
  float *Acum = reinterpret_cast<float *>(sm + Sh::A_OFF);
  float *eA = Acum + C;  // e^{A_i}
  float *wL = eA + C;    // e^{A_{C-1} - A_i}

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = lane >> 2, t = lane & 3;
  const int h = blockIdx.x;
  const RowDesc d = rows.r[blockIdx.y];
  const size_t b = (size_t)rows.row0 + blockIdx.y;
  const int hq = h / (P.Hv / P.Hk);
  const int L = d.n;
  const bool from_zero = (d.flags & kFlagFromZero) != 0;
  if (L == 0 && !from_zero) return;  // nothing to do: the state stays as it is
  const int Tp = io.T;
  const int nchunks = (L + C - 1) / C;
  float *Sg = P.state + ((size_t)d.slot * P.Hv + h) * D * D;

  for (int idx = tid; idx < D * D / 4; idx += kPrefillThreads) {
    const int r = idx / (D / 4), c4 = (idx % (D / 4)) * 4;
    const float4 v = from_zero ? f4(0.f) : ld_stream4(Sg + (size_t)r * D + c4);
    *reinterpret_cast<float4 *>(&Ss[r * LDS + c4]) = v;
  }

  const KT *qg = static_cast<const KT *>(io.q);
  const KT *kg = static_cast<const KT *>(io.k);
  const KT *vg = static_cast<const KT *>(io.v);
  // stage the chunk's q, k, v rows (zero past the prompt) and its gates
  auto issue = [&](int c) {
    const int s = c % STAGES, t0 = c * C;
    KT *qs = In + (size_t)(s * 3 + 0) * C * LDI;
    KT *ks = In + (size_t)(s * 3 + 1) * C * LDI;
    KT *vs = In + (size_t)(s * 3 + 2) * C * LDI;
    constexpr int VEC = 16 / (int)sizeof(KT), PER_ROW = D / VEC;
    for (int idx = tid; idx < C * PER_ROW; idx += kPrefillThreads) {
      const int i = idx / PER_ROW, p = (idx % PER_ROW) * VEC;
      const bool ok = t0 + i < L;
      const size_t tok = b * Tp + (ok ? t0 + i : L - 1);
      cp_async16(qs + i * LDI + p, qg + (tok * P.Hk + hq) * D + p, ok);
      cp_async16(ks + i * LDI + p, kg + (tok * P.Hk + hq) * D + p, ok);
      cp_async16(vs + i * LDI + p, vg + (tok * P.Hv + h) * D + p, ok);
    }
    if (tid < C) {
      const bool ok = t0 + tid < L;
      const size_t tok = b * Tp + (ok ? t0 + tid : L - 1);
      float *gs = Gr + (size_t)s * 2 * C;
      if (GATED) cp_async4(gs + tid, io.log_g + tok * P.Hv + h, ok);
      if (DELTA) cp_async4(gs + C + tid, io.beta + tok * P.Hv + h, ok);
    }
    cp_async_commit();
  };

  if (nchunks > 0) issue(0);
  for (int c = 0; c < nchunks; ++c) {
    const int s = c % STAGES, t0 = c * C;
    __syncthreads();  // the previous chunk is done with every buffer
    if (STAGES == 2) {
      if (c + 1 < nchunks) {
        issue(c + 1);
        cp_async_wait<1>();
      } else {
        cp_async_wait<0>();
      }
    } else {
      if (c > 0) issue(c);
      cp_async_wait<0>();
    }
    __syncthreads();
    const KT *qs = In + (size_t)(s * 3 + 0) * C * LDI;
    const KT *ks = In + (size_t)(s * 3 + 1) * C * LDI;
    const KT *vs = In + (size_t)(s * 3 + 2) * C * LDI;
    const float *gs = Gr + (size_t)s * 2 * C;
    const float *bs = gs + C;

    // cumulative log-gates, e^{A_i}, fold weights (warp 0)
    if (warp == 0) {
      float a0 = GATED ? gs[lane] : 0.f, a1 = GATED ? gs[lane + 32] : 0.f;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const float y0 = __shfl_up_sync(kFull, a0, off), y1 = __shfl_up_sync(kFull, a1, off);
        if (lane >= off) {
          a0 += y0;
          a1 += y1;
        }
      }
      a1 += __shfl_sync(kFull, a0, 31);
      const float AL = __shfl_sync(kFull, a1, 31);
      Acum[lane] = a0;
      Acum[lane + 32] = a1;
      eA[lane] = expf(a0);
      eA[lane + 32] = expf(a1);
      wL[lane] = expf(AL - a0);
      wL[lane + 32] = expf(AL - a1);
    }
    __syncthreads();

    // Gram matrix needed first: Mk for the delta rule, else Mq (all warps).  No
    // barrier after it: Y below neither reads nor writes X.
    gram_rows<XIN, DELTA, 4, D, LDI, LDX>(DELTA ? ks : qs, ks, warp >> 1, (warp & 1) * 4, Acum, bs,
                                          P.scale, Xs, g, t);

    // Y = [Q; K] S.  Q rows stay in registers as the output accumulator
    // (e^{A_i} scale q_i^T S); K rows become R_i = beta_i (v_i - e^{A_i} S^T k_i).
    const bool qwarp = !DELTA || warp < 4;
    const int mb = DELTA ? 0 : (warp >> 2) * 2;  // first m-tile (16 rows) of this warp
    const int nb = (warp & 3) * NW3;            // first n-tile (8 columns)
    float y[MT][NW3][4];
    {
      const KT *asrc = qwarp ? qs : ks;
#pragma unroll
      for (int m = 0; m < MT; ++m)
#pragma unroll
        for (int n = 0; n < NW3; ++n) y[m][n][0] = y[m][n][1] = y[m][n][2] = y[m][n][3] = 0.f;
#pragma unroll 2
      for (int k0 = 0; k0 < D; k0 += 8) {
        uint32_t bh[NW3][2], bl[NW3][2];
#pragma unroll
        for (int n = 0; n < NW3; ++n) {
          const int col = 8 * (nb + n) + g;
          split_tf32(Ss[(k0 + t) * LDS + col], bh[n][0], bl[n][0]);
          split_tf32(Ss[(k0 + t + 4) * LDS + col], bh[n][1], bl[n][1]);
        }
#pragma unroll
        for (int m = 0; m < MT; ++m) {
          uint32_t ah[4], al[4];
          load_a<XIN>(asrc, LDI, 16 * (mb + m), k0, g, t, ah, al);
#pragma unroll
          for (int n = 0; n < NW3; ++n) mma_small<XIN, false>(y[m][n], ah, al, bh[n], bl[n]);
#pragma unroll
          for (int n = 0; n < NW3; ++n) mma_big(y[m][n], ah, bh[n]);
        }
      }
#pragma unroll
      for (int m = 0; m < MT; ++m)
#pragma unroll
        for (int n = 0; n < NW3; ++n)
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int i = 16 * (mb + m) + g + (e >> 1) * 8, col = 8 * (nb + n) + 2 * t + (e & 1);
            if (qwarp) {
              y[m][n][e] *= P.scale * eA[i];
            } else {
              Us[i * LDS + col] = bs[i] * (to_float(vs[i * LDI + col]) - eA[i] * y[m][n][e]);
            }
          }
    }
    __syncthreads();

    // Delta rule: (I + Mk) U = R by forward substitution, one column per thread
    // of warps 4..7, while warps 0..3 build Mq (above the diagonal of X, apart
    // from the Mk entries the substitution reads).
    if (DELTA && warp < 4)
      gram_rows<XIN, false, 8, D, LDI, LDX>(qs, ks, warp, 0, Acum, bs, P.scale, Xs, g, t);
    if (DELTA && tid >= 128 && tid - 128 < D) {
      const int col = tid - 128;
      float u[C];
#pragma unroll
      for (int i = 0; i < C; ++i) u[i] = Us[i * LDS + col];
#pragma unroll
      for (int i = 1; i < C; ++i) {
        float s0 = 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f;
#pragma unroll
        for (int j = 0; j + 3 < i; j += 4) {
          const float4 x = *reinterpret_cast<const float4 *>(&Xs[i * LDX + j]);
          s0 = fmaf(x.x, u[j], s0);
          s1 = fmaf(x.y, u[j + 1], s1);
          s2 = fmaf(x.z, u[j + 2], s2);
          s3 = fmaf(x.w, u[j + 3], s3);
        }
#pragma unroll
        for (int j = i & ~3; j < i; ++j) s0 = fmaf(Xs[i * LDX + j], u[j], s0);
        u[i] -= (s0 + s1) + (s2 + s3);
      }
#pragma unroll
      for (int i = 0; i < C; ++i) Us[i * LDS + col] = u[i];
    }
    if (DELTA) __syncthreads();

    // O = e^{A} Y_q + Mq U for the prompt tokens of this chunk
    if (qwarp) {
      constexpr bool BX = !DELTA && XIN;  // U = V, exact when bf16
#pragma unroll 1
      for (int k0 = 0; k0 < C; k0 += 8) {
        uint32_t bh[NW3][2], bl[NW3][2];
#pragma unroll
        for (int n = 0; n < NW3; ++n) {
          const int col = 8 * (nb + n) + g;
          if (DELTA) {
            split_tf32(Us[(k0 + t) * LDS + col], bh[n][0], bl[n][0]);
            split_tf32(Us[(k0 + t + 4) * LDS + col], bh[n][1], bl[n][1]);
          } else {
            operand<BX>(to_float(vs[(k0 + t) * LDI + col]), bh[n][0], bl[n][0]);
            operand<BX>(to_float(vs[(k0 + t + 4) * LDI + col]), bh[n][1], bl[n][1]);
          }
        }
#pragma unroll
        for (int m = 0; m < MT; ++m) {
          const int r0 = 16 * (mb + m);
          if (k0 > r0 + 15) continue;  // Mq is zero above the diagonal
          uint32_t ah[4], al[4];
          const int ra = r0 + g, rb = r0 + g + 8, ka = k0 + t, kb = k0 + t + 4;
          split_tf32(ka <= ra ? Xs[ka * LDX + ra + 1] : 0.f, ah[0], al[0]);
          split_tf32(ka <= rb ? Xs[ka * LDX + rb + 1] : 0.f, ah[1], al[1]);
          split_tf32(kb <= ra ? Xs[kb * LDX + ra + 1] : 0.f, ah[2], al[2]);
          split_tf32(kb <= rb ? Xs[kb * LDX + rb + 1] : 0.f, ah[3], al[3]);
#pragma unroll
          for (int n = 0; n < NW3; ++n) mma_small<false, BX>(y[m][n], ah, al, bh[n], bl[n]);
#pragma unroll
          for (int n = 0; n < NW3; ++n) mma_big(y[m][n], ah, bh[n]);
        }
      }
#pragma unroll
      for (int m = 0; m < MT; ++m)
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          const int i = 16 * (mb + m) + g + 8 * half;
          if (t0 + i >= L) continue;
          float *orow = io.o + ((b * Tp + t0 + i) * P.Hv + h) * D;
#pragma unroll
          for (int n = 0; n < NW3; ++n)
            __stcs(reinterpret_cast<float2 *>(orow + 8 * (nb + n) + 2 * t),
                   make_float2(y[m][n][2 * half], y[m][n][2 * half + 1]));
        }
    }

    // S <- e^{A_{C-1}} S + K^T diag(w) U (no barrier: O and this step only read
    // U).  Warp w owns state columns 8 (NPW w) .. 8 (NPW w + NPW) - 1 over all
    // rows, so each w_i u_i is split into tf32 parts once.
    {
      const int nst = warp * NPW;
      const float eL = eA[C - 1];
      float acc[MT6][NPW][4];
#pragma unroll
      for (int m = 0; m < MT6; ++m)
#pragma unroll
        for (int n = 0; n < NPW; ++n) {
          const int col = 8 * (nst + n) + 2 * t;
          const float2 lo = *reinterpret_cast<const float2 *>(&Ss[(16 * m + g) * LDS + col]);
          const float2 hi = *reinterpret_cast<const float2 *>(&Ss[(16 * m + g + 8) * LDS + col]);
          acc[m][n][0] = eL * lo.x;
          acc[m][n][1] = eL * lo.y;
          acc[m][n][2] = eL * hi.x;
          acc[m][n][3] = eL * hi.y;
        }
#pragma unroll 1
      for (int k0 = 0; k0 < C; k0 += 8) {
        const float w0 = wL[k0 + t], w1 = wL[k0 + t + 4];
        uint32_t bh[NPW][2], bl[NPW][2];
#pragma unroll
        for (int n = 0; n < NPW; ++n) {
          const int col = 8 * (nst + n) + g;
          float u0, u1;
          if (DELTA) {
            u0 = Us[(k0 + t) * LDS + col];
            u1 = Us[(k0 + t + 4) * LDS + col];
          } else {
            u0 = to_float(vs[(k0 + t) * LDI + col]);
            u1 = to_float(vs[(k0 + t + 4) * LDI + col]);
          }
          split_tf32(w0 * u0, bh[n][0], bl[n][0]);
          split_tf32(w1 * u1, bh[n][1], bl[n][1]);
        }
#pragma unroll
        for (int m = 0; m < MT6; ++m) {
          uint32_t ah[4], al[4];
          load_at<XIN>(ks, LDI, 16 * m, k0, g, t, ah, al);
#pragma unroll
          for (int n = 0; n < NPW; ++n) mma_small<XIN, false>(acc[m][n], ah, al, bh[n], bl[n]);
#pragma unroll
          for (int n = 0; n < NPW; ++n) mma_big(acc[m][n], ah, bh[n]);
        }
      }
      // each warp rewrites only the columns it read; Y read S before the last barrier
#pragma unroll
      for (int m = 0; m < MT6; ++m)
#pragma unroll
        for (int n = 0; n < NPW; ++n) {
          const int col = 8 * (nst + n) + 2 * t;
          *reinterpret_cast<float2 *>(&Ss[(16 * m + g) * LDS + col]) =
              make_float2(acc[m][n][0], acc[m][n][1]);
          *reinterpret_cast<float2 *>(&Ss[(16 * m + g + 8) * LDS + col]) =
              make_float2(acc[m][n][2], acc[m][n][3]);
        }
    }
  }
  __syncthreads();
  for (int idx = tid; idx < D * D / 4; idx += kPrefillThreads) {
    const int r = idx / (D / 4), c4 = (idx % (D / 4)) * 4;
    st_stream4(Sg + (size_t)r * D + c4, *reinterpret_cast<const float4 *>(&Ss[r * LDS + c4]));
  }
}

template <typename KT, int VARIANT, int D>
cudaError_t run_prefill(const PoolView &P, const RowBatch &rows, const TokenIO &io,
                        cudaStream_t stream) {
  using Sh = PrefillShape<KT, D>;
  cudaError_t e = ensure_smem((const void *)prefill_kernel<KT, VARIANT, D>, Sh::BYTES);
  if (e != cudaSuccess) return e;
  dim3 grid(P.Hv, rows.count);
  prefill_kernel<KT, VARIANT, D><<<grid, kPrefillThreads, Sh::BYTES, stream>>>(P, rows, io);
  return cudaGetLastError();
}

template <typename KT, int VARIANT>
cudaError_t prefill_d(const PoolView &P, const RowBatch &rows, const TokenIO &io, int d,
                      cudaStream_t s) {
  if (d == 128) return run_prefill<KT, VARIANT, 128>(P, rows, io, s);
  if (d == 64) return run_prefill<KT, VARIANT, 64>(P, rows, io, s);
  return kUnsupported;
}

template <typename KT>
cudaError_t prefill_variant(const PoolView &P, const RowBatch &rows, const TokenIO &io,
                            int variant, int d, cudaStream_t s) {
  switch (variant) {
    case kPlain: return prefill_d<KT, kPlain>(P, rows, io, d, s);
    case kGated: return prefill_d<KT, kGated>(P, rows, io, d, s);
    case kGatedDelta: return prefill_d<KT, kGatedDelta>(P, rows, io, d, s);
  }
  return kUnsupported;
}

}  // namespace

cudaError_t launch_prefill(const PoolView &P, const RowBatch &rows, const TokenIO &io,
                           int variant, int dtype, int d, cudaStream_t stream) {
  if (rows.count <= 0) return cudaSuccess;
  if (dtype == 1 && d == 128 && (reinterpret_cast<uintptr_t>(io.o) & 15) == 0) {
    // the tensor-core kernel moves its tiles by TMA (the boundary admits only
    // 16-byte aligned token buffers); where the driver cannot encode the tensor
    // maps, the mma.sync kernel below runs instead
    PrefillMaps maps;
    if (encode_prefill_maps(&maps, io, P.Hk, P.Hv) == cudaSuccess)
      return launch_prefill_tc(P, rows, io, maps, variant, stream);
  }
  if (dtype == 0) return prefill_variant<float>(P, rows, io, variant, d, stream);
  if (dtype == 1) return prefill_variant<__nv_bfloat16>(P, rows, io, variant, d, stream);
  return kUnsupported;
}

}  // namespace kvb
