// Chunked prefill on the fifth-generation tensor cores (tcgen05, TMEM), for
// bf16 inputs at d = 128.
//
// Same chunk algebra as prefill.cu ("KVBuffer: IO-aware Serving for Linear
// Attention", abstract: chunkwise computation; the delta-rule chunk form with
// the UT transform), chunk C = 64, per (request, value head) CTA:
//   Y = [Q; K] S,  Mq = scale e^{A_i-A_j} q_i.k_j (j <= i),  Mk = beta_i e^{A_i-A_j} k_i.k_j (j < i)
//   (I + Mk) U = R,  R_i = beta_i (v_i - e^{A_i} S^T k_i)       (U = V unless the delta rule)
//   O = e^{A} scale Y_q + Mq U,   S <- e^{A_{C-1}} S + K^T diag(w) U
// Layout: four warpgroups of 128 threads; thread t of each owns TMEM lane t,
// the warpgroups splitting its column ranges.  The state lives in TMEM
// transposed (lane = value column c, columns = key rows), so that
//   Y^T = S^T X^T          (A: S^T from TMEM as bf16 hi/lo parts, B: X = [Q;K] from smem)
//   G   = X K^T            (A: X, B: the K rows of X; exact for bf16 inputs)
//   O^T = e^A Y_q^T + U^T Mq^T   (A: U^T parts from TMEM, B: Mq parts from smem)
//   S^T <- e^{A_C} S^T + (wU)^T K   (A: (wU)^T parts from TMEM, B: K^T from smem)
// leave every per-column quantity (R, the substitution, U, the output column,
// the state column) in the registers of the thread that owns that column: the
// UT transform T = (I + Mk)^{-1} is built in 16 x 16 blocks by all threads and
// applied as one more tensor-core product, U^T = R^T T^T.
// Operands that are not exact in bf16 (S, U, wU, Mq) enter as hi + lo bf16
// parts (about 16 significant bits; the lo x lo product is dropped), with fp32
// accumulation in TMEM.  Single-thread MMA issue, completion via tcgen05.commit
// on an mbarrier; every wait is bounded and a timeout sets the error word.
#include "kvb_device.cuh"

namespace kvb {
namespace {

constexpr int kC = 64, kD = 128, kThreads = 512;  // four warpgroups share every TMEM lane
// TMEM columns
constexpr uint32_t kColS = 0;     // S^T fp32            [128 lanes x 128]
constexpr uint32_t kColP = 128;   // A parts: S^T hi/lo (64 + 64), later U^T hi/lo, (wU)^T hi/lo (32 each)
constexpr uint32_t kColY = 256;   // Y^T fp32 (tokens: 0..63 q, 64..127 k); O^T in 0..63
constexpr uint32_t kColG = 384;   // G fp32 (lane = token of [Q;K], column = key token); then U^T
constexpr uint32_t kTmemCols = 512;
// shared memory (bytes)
constexpr int kXBytes = 2 * kC * kD * 2;        // [Q;K] bf16, core-matrix K-major (32 KB)
constexpr int kVBytes = kC * kD * 2;            // V bf16 [token][column] (16 KB)
constexpr int kGBytes = 2 * kC * 4;             // log-gate, beta
constexpr int kStage = (kXBytes + kVBytes + kGBytes + 1023) / 1024 * 1024;
constexpr int kKtBytes = kD * kC * 2;           // K^T bf16, core-matrix K-major (16 KB)
constexpr int kMqBytes = kC * kC * 2;           // one bf16 part of Mq (8 KB)
constexpr int kLdMk = kC + 4;                   // fp32 rows of Mk
constexpr int kMkBytes = kC * kLdMk * 4;
constexpr int kOffKt = 2 * kStage;
constexpr int kOffMq = kOffKt + kKtBytes;       // [2 parts]
constexpr int kOffMk = kOffMq + 2 * kMqBytes;
constexpr int kLdP = 20;                        // fp32 row stride of the block-product scratch
constexpr int kOffR = kOffMk + kMkBytes;        // scratch for the block products, fp32 [3][16][kLdP]
constexpr int kRBytes = 3 * 16 * kLdP * 4;
constexpr int kOffTf = kOffR + kRBytes;         // T = (I + Mk)^-1, fp32 [64][68]
constexpr int kOffTp = kOffTf + kMkBytes;       // T as bf16 hi / lo parts, core-matrix K-major
constexpr int kOffA = kOffTp + 2 * kMqBytes;    // Acum, e^A, w: [3][C]
constexpr int kSmemBytes = kOffA + 3 * kC * 4;
// core-matrix strides (bytes): 8 rows x 16 bytes per core matrix, k groups adjacent
constexpr uint32_t kLbo = 128;
constexpr uint32_t kSboX = (kD / 8) * 128;      // X: 128 dk per row group
constexpr uint32_t kSboKt = (kC / 8) * 128;     // K^T and Mq: 64 tokens per row group
static_assert(kSmemBytes <= 227 * 1024, "one CTA's shared memory");
static_assert(kStage % 1024 == 0 && kKtBytes % 1024 == 0 && kMqBytes % 1024 == 0, "alignment");

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
// shared-memory matrix descriptor: K-major, no swizzle (core matrices of 8 rows x
// 16 bytes; lbo = distance between k groups, sbo = distance between row groups)
__device__ __forceinline__ uint64_t sdesc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
  return (uint64_t)((addr >> 4) & 0x3FFF) | ((uint64_t)((lbo >> 4) & 0x3FFF) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3FFF) << 32) | ((uint64_t)1 << 46);
}
// instruction descriptor: bf16 x bf16 -> fp32, both K-major, M x N
__host__ __device__ constexpr uint32_t idesc_bf16(int m, int n) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(m >> 4) << 24);
}
__device__ __forceinline__ void mma_ss(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
               "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}"
               ::"r"(d), "l"(a), "l"(b), "r"(idesc), "r"(acc));
}
__device__ __forceinline__ void mma_ts(uint32_t d, uint32_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
               "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}"
               ::"r"(d), "r"(a), "l"(b), "r"(idesc), "r"(acc));
}
__device__ __forceinline__ void mma_commit(uint32_t mbar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(mbar));
}
// Bounded wait on an mbarrier phase: at most `polls` polls (the default is about
// 50 ms); false on timeout.
constexpr int kWaitPolls = 1 << 20;
__device__ __forceinline__ bool mbar_wait(uint32_t mbar, uint32_t parity, int polls = kWaitPolls) {
  for (int it = 0; it < polls; ++it) {
    uint32_t done;
    asm volatile("{\n\t.reg .pred p;\n\tmbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
                 "selp.u32 %0, 1, 0, p;\n\t}"
                 : "=r"(done) : "r"(mbar), "r"(parity));
    if (done) return true;
    __nanosleep(32);
  }
  return false;
}
__device__ __forceinline__ void fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// 32 consecutive TMEM columns of this thread's lane
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// x = hi + lo, both bf16 (hi = round(x), lo = round(x - hi), to nearest even), two
// values at once: {x0, x1} (x0 in the low half) as hi and lo pairs
__device__ __forceinline__ void split_pair(float x0, float x1, uint32_t &hi, uint32_t &lo) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(x0, x1);
  const float2 hf = __bfloat1622float2(h);
  const __nv_bfloat162 l = __floats2bfloat162_rn(x0 - hf.x, x1 - hf.y);
  hi = *reinterpret_cast<const uint32_t *>(&h);
  lo = *reinterpret_cast<const uint32_t *>(&l);
}
__device__ __forceinline__ void split16(const float (&x)[16], uint32_t (&hi)[8], uint32_t (&lo)[8]) {
#pragma unroll
  for (int j = 0; j < 8; ++j) split_pair(x[2 * j], x[2 * j + 1], hi[j], lo[j]);
}
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_st8(uint32_t taddr, const uint32_t (&r)[8]) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};"
               ::"r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]),
                 "r"(r[7])
               : "memory");
}

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};"
      ::"r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
        "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}

// Block products for the UT inverse on the tensor cores.  A fp32 value x enters
// as bf16 hi + lo parts (x ~ hi + lo to about 16 significant bits); a product is
// hi*hi + hi*lo + lo*hi with fp32 accumulation, the lo*lo term dropped, as the
// chunk's other tensor-core products take their non-bf16 operands.
__device__ __forceinline__ void mma_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
// d += A B for the 16 x 16 block of A at (ar, ac) (row stride lda) and the 16 x 8
// block of B at (br, bc) (row stride ldb), both fp32 in shared memory; lane
// (g, t) = (lane / 4, lane % 4) holds rows g, g + 8 and columns 2t, 2t + 1 of d
__device__ __forceinline__ void mma3_f32(float (&d)[4], const float *A, int lda, int ar, int ac,
                                         const float *B, int ldb, int br, int bc, int lane) {
  const int g = lane >> 2, t = lane & 3;
  uint32_t ah[4], al[4], bh[2], bl[2];
  const float *a0 = A + (ar + g) * lda + ac + 2 * t, *a1 = a0 + 8 * lda;
  split_pair(a0[0], a0[1], ah[0], al[0]);
  split_pair(a1[0], a1[1], ah[1], al[1]);
  split_pair(a0[8], a0[9], ah[2], al[2]);
  split_pair(a1[8], a1[9], ah[3], al[3]);
  const float *b0 = B + (br + 2 * t) * ldb + bc + g;
  split_pair(b0[0], b0[ldb], bh[0], bl[0]);
  split_pair(b0[8 * ldb], b0[9 * ldb], bh[1], bl[1]);
  mma_16816(d, ah, bh[0], bh[1]);
  mma_16816(d, ah, bl[0], bl[1]);
  mma_16816(d, al, bh[0], bh[1]);
}
// the 16 x 8 tile d (times s) into C at columns c0 .. c0 + 7 (row stride ldc)
__device__ __forceinline__ void store_tile(float *C, int ldc, int c0, const float (&d)[4], float s, int lane) {
  const int g = lane >> 2, t = lane & 3;
  *reinterpret_cast<float2 *>(C + g * ldc + c0 + 2 * t) = make_float2(s * d[0], s * d[1]);
  *reinterpret_cast<float2 *>(C + (g + 8) * ldc + c0 + 2 * t) = make_float2(s * d[2], s * d[3]);
}

// T = (I + Mk)^{-1} for the strictly lower 64 x 64 Mk (fp32, row stride kLdMk),
// in 16 x 16 blocks: T_aa = (I + Mk_aa)^{-1} by forward substitution (one
// column per thread), then T_ab = -T_aa sum_{b<=c<a} Mk_ac T_cb level by level
// (a - b = 1, 2, 3) as tensor-core block products.  Writes T (zero above
// the diagonal) to Tf; P is scratch for three 16 x 16 blocks.  All threads.
__device__ __forceinline__ void ut_inverse(const float *Mk, float *Tf, float *Pb, int tid) {
  if (tid < 64) {  // diagonal blocks: block a, column j
    const int a = tid >> 4, j = tid & 15, o = a * 16;
    float t[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      float acc = i == j ? 1.f : 0.f;
#pragma unroll
      for (int l = 0; l < i; ++l) acc = fmaf(-Mk[(o + i) * kLdMk + o + l], t[l], acc);
      t[i] = i < j ? 0.f : acc;
    }
#pragma unroll
    for (int i = 0; i < 16; ++i) Tf[(o + i) * kLdMk + o + j] = t[i];
  }
  __syncthreads();
  // level d: blocks (a, a - d), a = d .. 3; P = sum_c Mk_ac T_c,a-d, then T = -T_aa P,
  // each 16 x 16 block product as mma.sync passes: warp 2 blk + nh takes columns
  // 8 nh .. 8 nh + 7 of block blk of the level
  const int warp = tid >> 5;
  for (int dlev = 1; dlev <= 3; ++dlev) {
    const int nblk = 4 - dlev;
    const bool mine = warp < 2 * nblk;
    const int blk = warp >> 1, nh = warp & 1;
    const int a = blk + dlev, bcol = a - dlev;
    if (mine) {
      float acc[4] = {0.f, 0.f, 0.f, 0.f};
      for (int cb = bcol; cb < a; ++cb)
        mma3_f32(acc, Mk, kLdMk, a * 16, cb * 16, Tf, kLdMk, cb * 16, bcol * 16 + 8 * nh, tid & 31);
      store_tile(Pb + blk * 16 * kLdP, kLdP, 8 * nh, acc, 1.f, tid & 31);
    }
    __syncthreads();
    if (mine) {
      float acc[4] = {0.f, 0.f, 0.f, 0.f};
      mma3_f32(acc, Tf, kLdMk, a * 16, a * 16, Pb + blk * 16 * kLdP, kLdP, 0, 8 * nh, tid & 31);
      store_tile(Tf + a * 16 * kLdMk, kLdMk, bcol * 16 + 8 * nh, acc, -1.f, tid & 31);
    }
    __syncthreads();
  }
}

__device__ __forceinline__ void cp16(uint32_t dst, const void *src, bool valid) {
  const int n = valid ? 16 : 0;
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src), "r"(n) : "memory");
}
__device__ __forceinline__ void cp4(uint32_t dst, const void *src, bool valid) {
  const int n = valid ? 4 : 0;
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;\n" ::"r"(dst), "l"(src), "r"(n) : "memory");
}

template <int VARIANT>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_tc_kernel(const PoolView P, const __grid_constant__ RowBatch rows, const TokenIO io,
                      int first_polls) {
  using KT = __nv_bfloat16;
  constexpr bool DELTA = VARIANT == kGatedDelta, GATED = VARIANT != kPlain;
  extern __shared__ __align__(1024) uint8_t smem[];
  __shared__ uint64_t mbar_s;
  __shared__ uint32_t tmem_s;
  float *Acum = reinterpret_cast<float *>(smem + kOffA);
  float *eA = Acum + kC, *wL = eA + kC;
  float *Mk = reinterpret_cast<float *>(smem + kOffMk);

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int h = blockIdx.x;
  const RowDesc &d = rows.r[blockIdx.y];
  const size_t b = (size_t)rows.row0 + blockIdx.y;
  const int hq = h / (P.Hv / P.Hk);
  const int L = d.n;
  const bool from_zero = (d.flags & kFlagFromZero) != 0;
  if (L == 0 && !from_zero) return;  // nothing to do: the state stays as it is
  const int Tp = io.T;
  const int nchunks = (L + kC - 1) / kC;
  float *Sg = P.state + ((size_t)d.slot * P.Hv + h) * kD * kD;
  const uint32_t mbar = smem_u32(&mbar_s);
  const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;  // this warp's TMEM lanes

  if (tid == 0) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(mbar));
    asm volatile("fence.mbarrier_init.release.cluster;");
  }
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&tmem_s)),
                 "r"(kTmemCols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }

  const KT *qg = static_cast<const KT *>(io.q);
  const KT *kg = static_cast<const KT *>(io.k);
  const KT *vg = static_cast<const KT *>(io.v);
  // stage chunk c: q and k rows into X (core-matrix layout), v rows, gates
  auto issue = [&](int c) {
    uint8_t *st = smem + (c & 1) * kStage;
    const uint32_t xs = smem_u32(st), vs = xs + kXBytes, gs = vs + kVBytes;
    const int t0 = c * kC;
    for (int idx = tid; idx < 2 * kC * 16; idx += kThreads) {  // 128 rows x 16 pieces of 8
      const int i = idx >> 4, p = idx & 15;
      const int tok = t0 + (i & (kC - 1));
      const bool ok = tok < L;
      const size_t row = b * Tp + (ok ? tok : L - 1);
      const KT *src = (i < kC ? qg : kg) + (row * P.Hk + hq) * kD + p * 8;
      cp16(xs + (i >> 3) * kSboX + p * kLbo + (i & 7) * 16, src, ok);
    }
    for (int idx = tid; idx < kC * 16; idx += kThreads) {
      const int j = idx >> 4, p = idx & 15;
      const bool ok = t0 + j < L;
      const size_t row = b * Tp + (ok ? t0 + j : L - 1);
      cp16(vs + j * kD * 2 + p * 16, vg + (row * P.Hv + h) * kD + p * 8, ok);
    }
    if (tid < kC) {
      const bool ok = t0 + tid < L;
      const size_t row = b * Tp + (ok ? t0 + tid : L - 1);
      if (GATED) cp4(gs + tid * 4, io.log_g + row * P.Hv + h, ok);
      if (DELTA) cp4(gs + (kC + tid) * 4, io.beta + row * P.Hv + h, ok);
    }
    asm volatile("cp.async.commit_group;\n" ::: "memory");
  };
  if (nchunks > 0) issue(0);

  fence_before();
  __syncthreads();
  fence_after();
  const uint32_t tmem = tmem_s;
  const int lt = tid & 127;              // this thread's TMEM lane
  const int wg = tid >> 7;               // warpgroup: which quarter of each lane's columns
  const uint32_t my = tmem + lane_base;  // this thread's lane, column 0
  const int c = lt;                      // as a state column
  bool ok = true;
  uint32_t phase = 0;
  // poll bound of the next completion wait: the first one may be capped by the
  // failure-path test hook (first_polls > 0), every later one has the default
  int polls = first_polls > 0 ? first_polls : kWaitPolls;

  // e^A scale Y_q^T (the output accumulator), and e^{A_C} S^T (the state before
  // its update), for this thread's lane
  // (16-column rounds q0 .. q1 - 1 of each)
  auto scale_y = [&](const float *eAv, int q0, int q1) {
    uint32_t w[16];
#pragma unroll 1
    for (int q = q0; q < q1; ++q) {
      tmem_ld16(my + kColY + q * 16, w);
#pragma unroll
      for (int j = 0; j < 16; ++j) w[j] = __float_as_uint(P.scale * eAv[q * 16 + j] * __uint_as_float(w[j]));
      tmem_st16(my + kColY + q * 16, w);
    }
  };
  auto scale_s = [&](float eL, int q0, int q1) {
    uint32_t w[16];
#pragma unroll 1
    for (int q = q0; q < q1; ++q) {
      tmem_ld16(my + kColS + q * 16, w);
#pragma unroll
      for (int j = 0; j < 16; ++j) w[j] = __float_as_uint(eL * __uint_as_float(w[j]));
      tmem_st16(my + kColS + q * 16, w);
    }
  };
  // bf16 hi / lo parts of 16 state rows (16 r0 .. 16 r0 + 15) of column c into the
  // A region (the operand of Y^T = S^T X^T)
  auto put_parts16 = [&](const float (&x)[16], int r0) {
    uint32_t hi[8], lo[8];
    split16(x, hi, lo);
    tmem_st8(my + kColP + r0 * 8, hi);
    tmem_st8(my + kColP + 64 + r0 * 8, lo);
  };
  // this warpgroup's 32 state rows of column c: fp32 into S^T, and their parts
#pragma unroll 1
  for (int q = 0; q < 2; ++q) {
    const int r0 = wg * 2 + q;  // 16-row piece
    float x[16];
    uint32_t w[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      x[j] = from_zero ? 0.f : Sg[(size_t)(r0 * 16 + j) * kD + c];
      w[j] = __float_as_uint(x[j]);
    }
    tmem_st16(my + kColS + r0 * 16, w);
    put_parts16(x, r0);
  }
  tmem_wait_st();

  for (int ch = 0; ch < nchunks && ok; ++ch) {
    uint8_t *st = smem + (ch & 1) * kStage;
    const uint32_t xs = smem_u32(st);
    const KT *vs = reinterpret_cast<const KT *>(st + kXBytes);
    const float *gs = reinterpret_cast<const float *>(st + kXBytes + kVBytes);
    const float *bs = gs + kC;
    const int t0 = ch * kC;
    asm volatile("cp.async.wait_group 0;\n" ::: "memory");
    fence_async_smem();
    fence_before();
    __syncthreads();  // chunk staged; the previous chunk's MMAs are done
    fence_after();

    // K^T (B of the state update) from the K rows of X: the keys' core matrices
    // (8 tokens x 8 dims, 16-byte rows) transposed into K^T's (8 dims x 8
    // tokens) by ldmatrix.trans + stmatrix, four per warp instruction; warp w
    // takes tiles 8 w .. 8 w + 7 (token group tile & 7, dim group tile >> 3).
    // Cumulative gates (warp 3) follow.
    {
      const uint32_t xs_u = smem_u32(st), kt_u = smem_u32(smem + kOffKt);
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        const int tile = warp * 8 + q * 4 + (lane >> 3), jg = tile & 7, dg = tile >> 3, row = lane & 7;
        const uint32_t src = xs_u + ((kC >> 3) + jg) * kSboX + dg * kLbo + row * 16;
        const uint32_t dst = kt_u + dg * kSboKt + jg * kLbo + row * 16;
        uint32_t r0, r1, r2, r3;
        asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                     : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(src));
        asm volatile("stmatrix.sync.aligned.m8n8.x4.shared.b16 [%0], {%1,%2,%3,%4};"
                     ::"r"(dst), "r"(r0), "r"(r1), "r"(r2), "r"(r3) : "memory");
      }
    }
    if (warp == 3) {
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
    fence_async_smem();
    fence_before();
    __syncthreads();
    fence_after();

    // MMAs 1: G = X K^T (exact) and Y^T = S^T X^T (S^T as hi + lo parts)
    if (tid == 0) {
      const uint32_t idG = idesc_bf16(128, kC), idY = idesc_bf16(128, 2 * kC);
#pragma unroll
      for (int k0 = 0; k0 < kD; k0 += 16) {
        const uint64_t a = sdesc(xs + (k0 / 8) * kLbo, kLbo, kSboX);
        const uint64_t bk = sdesc(xs + (kC / 8) * kSboX + (k0 / 8) * kLbo, kLbo, kSboX);
        mma_ss(tmem + kColG, a, bk, idG, k0 > 0);
      }
#pragma unroll
      for (int part = 0; part < 2; ++part)
#pragma unroll
        for (int k0 = 0; k0 < kD; k0 += 16) {
          const uint64_t bx = sdesc(xs + (k0 / 8) * kLbo, kLbo, kSboX);
          mma_ts(tmem + kColY, tmem + kColP + part * 64 + k0 / 2, bx, idY, part > 0 || k0 > 0);
        }
      mma_commit(mbar);
    }
    // while the products run: the next chunk's copies (into the other stage, free
    // since the previous chunk finished)
    if (ch + 1 < nchunks) issue(ch + 1);
    ok = __syncthreads_and(mbar_wait(mbar, phase, polls)) != 0;  // CTA-uniform
    polls = kWaitPolls;
    phase ^= 1;
    fence_after();
    if (!ok) break;

    // Gram rows, key tokens split by warpgroup: thread (i, wg) builds entries
    // j = 16 wg .. 16 wg + 15 of row i of Mq (parts, smem) or Mk (fp32)
    {
      const int i = lt, j0 = wg * 16;
      float gr[16];
      {
        uint32_t w[16];
        tmem_ld16(my + kColG + j0, w);
#pragma unroll
        for (int j = 0; j < 16; ++j) gr[j] = __uint_as_float(w[j]);
      }
      if (i < kC) {  // Mq[i][j] = scale e^{A_i-A_j} q_i.k_j, j <= i
        const float Ai = Acum[i];
        float x[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) x[j] = j0 + j <= i ? P.scale * expf(Ai - Acum[j0 + j]) * gr[j] : 0.f;
        uint32_t hi[8], lo[8];
        split16(x, hi, lo);
        uint8_t *mq = smem + kOffMq;
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          const int off = (i >> 3) * kSboKt + (wg * 2 + q) * kLbo + (i & 7) * 16;
          *reinterpret_cast<uint4 *>(mq + off) = make_uint4(hi[4 * q], hi[4 * q + 1], hi[4 * q + 2], hi[4 * q + 3]);
          *reinterpret_cast<uint4 *>(mq + kMqBytes + off) =
              make_uint4(lo[4 * q], lo[4 * q + 1], lo[4 * q + 2], lo[4 * q + 3]);
        }
      } else if (DELTA) {  // Mk[i'][j] = beta_i' e^{A_i'-A_j} k_i'.k_j, j < i'
        const int ip = i - kC;
        const float Ai = Acum[ip], bi = bs[ip];
#pragma unroll
        for (int j = 0; j < 16; j += 4) {
          const int jj = j0 + j;
          float4 m4;
          m4.x = jj < ip ? bi * expf(Ai - Acum[jj]) * gr[j] : 0.f;
          m4.y = jj + 1 < ip ? bi * expf(Ai - Acum[jj + 1]) * gr[j + 1] : 0.f;
          m4.z = jj + 2 < ip ? bi * expf(Ai - Acum[jj + 2]) * gr[j + 2] : 0.f;
          m4.w = jj + 3 < ip ? bi * expf(Ai - Acum[jj + 3]) * gr[j + 3] : 0.f;
          *reinterpret_cast<float4 *>(&Mk[ip * kLdMk + jj]) = m4;
        }
      }
    }
    // column c of R (delta rule), tokens 16 wg .. 16 wg + 15, as bf16 parts into
    // TMEM: the A operand (R^T) of U^T = R^T T^T
    if (DELTA) {
      uint32_t w[16];
      tmem_ld16(my + kColY + kC + wg * 16, w);
      float r[16];
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const int jj = wg * 16 + j;
        r[j] = bs[jj] * (__bfloat162float(vs[jj * kD + c]) - eA[jj] * __uint_as_float(w[j]));
      }
      uint32_t hi[8], lo[8];
      split16(r, hi, lo);
      tmem_st8(my + kColP + wg * 8, hi);
      tmem_st8(my + kColP + 32 + wg * 8, lo);
      tmem_wait_st();
    }
    fence_async_smem();
    fence_before();
    __syncthreads();  // Mk, Mq and R complete
    fence_after();

    // the UT transform: T = (I + Mk)^{-1} in blocks, its bf16 parts (B operand,
    // rows i, k = j), then U^T = R^T T^T on the tensor cores into the G columns
    if (DELTA) {
      // meanwhile, while the first 64 threads invert the diagonal blocks:
      // warpgroup 1 scales Y_q^T, warpgroups 2 and 3 the two halves of S^T
      if (wg == 1) scale_y(eA, 0, 4);
      if (wg >= 2) scale_s(eA[kC - 1], (wg - 2) * 4, (wg - 1) * 4);
      if (wg >= 1) tmem_wait_st();
      float *Tf = reinterpret_cast<float *>(smem + kOffTf);
      ut_inverse(Mk, Tf, reinterpret_cast<float *>(smem + kOffR), tid);
      if (tid < 4 * kC) {
        const int i = tid >> 2, jq = (tid & 3) * 16;  // row i, 16 columns
        float x[16];
#pragma unroll
        for (int q = 0; q < 16; ++q) x[q] = jq + q <= i ? Tf[i * kLdMk + jq + q] : 0.f;
        uint8_t *tp = smem + kOffTp;
        uint32_t hi[8], lo[8];
        split16(x, hi, lo);
#pragma unroll
        for (int g2 = 0; g2 < 2; ++g2) {
          const int off = (i >> 3) * kSboKt + (jq / 8 + g2) * kLbo + (i & 7) * 16;
          *reinterpret_cast<uint4 *>(tp + off) = make_uint4(hi[4 * g2], hi[4 * g2 + 1], hi[4 * g2 + 2], hi[4 * g2 + 3]);
          *reinterpret_cast<uint4 *>(tp + kMqBytes + off) =
              make_uint4(lo[4 * g2], lo[4 * g2 + 1], lo[4 * g2 + 2], lo[4 * g2 + 3]);
        }
      }
      fence_async_smem();
      fence_before();
      __syncthreads();
      fence_after();
      if (tid == 0) {
        const uint32_t idU = idesc_bf16(128, kC), tpa = smem_u32(smem + kOffTp);
#pragma unroll
        for (int combo = 0; combo < 3; ++combo) {
          const int ra = combo == 2 ? 32 : 0;                   // R^T hi, hi, lo
          const uint32_t tb = tpa + (combo == 1 ? kMqBytes : 0);  // T hi, lo, hi
#pragma unroll
          for (int k0 = 0; k0 < kC; k0 += 16)
            mma_ts(tmem + kColG, tmem + kColP + ra + k0 / 2, sdesc(tb + (k0 / 8) * kLbo, kLbo, kSboKt), idU,
                   combo > 0 || k0 > 0);
        }
        mma_commit(mbar);
      }
      ok = __syncthreads_and(mbar_wait(mbar, phase, polls)) != 0;  // CTA-uniform
      polls = kWaitPolls;
      phase ^= 1;
      fence_after();
      if (!ok) break;
    }

    {
      // column c of U (from the UT product, or V), 16 tokens at a time: U^T and
      // (wU)^T parts into TMEM, the A operands of the second MMAs; without the
      // delta rule the scaling of Y_q^T and S^T (done during the inverse with it)
      // shares these warpgroups: 4 U chunks + 4 Y rounds + 8 S rounds
      auto u_parts = [&](int q) {
        float x[16];
        if (DELTA) {
          uint32_t w[16];
          tmem_ld16(my + kColG + q * 16, w);
#pragma unroll
          for (int j = 0; j < 16; ++j) x[j] = __uint_as_float(w[j]);
        } else {
#pragma unroll
          for (int j = 0; j < 16; ++j) x[j] = __bfloat162float(vs[(q * 16 + j) * kD + c]);
        }
        uint32_t hi[8], lo[8];
        split16(x, hi, lo);
        tmem_st8(my + kColP + q * 8, hi);
        tmem_st8(my + kColP + 32 + q * 8, lo);
#pragma unroll
        for (int j = 0; j < 16; ++j) x[j] *= wL[q * 16 + j];
        split16(x, hi, lo);
        tmem_st8(my + kColP + 64 + q * 8, hi);
        tmem_st8(my + kColP + 96 + q * 8, lo);
      };
      const float eL = eA[kC - 1];
      if (DELTA) {
        u_parts(wg);
      } else if (wg < 2) {
        u_parts(2 * wg);
        u_parts(2 * wg + 1);
        scale_s(eL, wg, wg + 1);
      } else if (wg == 2) {
        scale_y(eA, 0, 4);
        scale_s(eL, 2, 3);
      } else {
        scale_s(eL, 3, 8);
      }
    }
    tmem_wait_st();
    fence_before();
    __syncthreads();
    fence_after();

    // MMAs 2: O^T += U^T Mq^T (three part products), S^T += (wU)^T K
    if (tid == 0) {
      const uint32_t idO = idesc_bf16(128, kC), idS = idesc_bf16(128, kD);
      const uint32_t mq = smem_u32(smem + kOffMq), kt = smem_u32(smem + kOffKt);
#pragma unroll
      for (int combo = 0; combo < 3; ++combo) {
        const int ua = combo == 2 ? 32 : 0;                    // U^T hi, hi, lo
        const uint32_t mb = mq + (combo == 1 ? kMqBytes : 0);  // Mq hi, lo, hi
#pragma unroll
        for (int k0 = 0; k0 < kC; k0 += 16)
          mma_ts(tmem + kColY, tmem + kColP + ua + k0 / 2, sdesc(mb + (k0 / 8) * kLbo, kLbo, kSboKt),
                 idO, 1);
      }
#pragma unroll
      for (int part = 0; part < 2; ++part)
#pragma unroll
        for (int k0 = 0; k0 < kC; k0 += 16)
          mma_ts(tmem + kColS, tmem + kColP + 64 + part * 32 + k0 / 2,
                 sdesc(kt + (k0 / 8) * kLbo, kLbo, kSboKt), idS, 1);
      mma_commit(mbar);
    }
    ok = __syncthreads_and(mbar_wait(mbar, phase, polls)) != 0;  // CTA-uniform
    polls = kWaitPolls;
    phase ^= 1;
    fence_after();
    if (!ok) break;

    // outputs (tokens 16 wg .. 16 wg + 15 of column c) and the next chunk's S^T
    // parts (state rows 32 wg .. 32 wg + 31)
    {
      uint32_t w[16];
      tmem_ld16(my + kColY + wg * 16, w);
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const int i = wg * 16 + j;
        if (t0 + i < L) io.o[((b * Tp + t0 + i) * P.Hv + h) * kD + c] = __uint_as_float(w[j]);
      }
      if (ch + 1 < nchunks) {
#pragma unroll 1
        for (int q = 0; q < 2; ++q) {
          const int r0 = wg * 2 + q;
          uint32_t w16[16];
          tmem_ld16(my + kColS + r0 * 16, w16);
          float x[16];
#pragma unroll
          for (int j = 0; j < 16; ++j) x[j] = __uint_as_float(w16[j]);
          put_parts16(x, r0);
        }
        tmem_wait_st();
      }
    }
  }

  if (ok) {
    // this warpgroup's quarter of the state column back to global memory
    {
      uint32_t w[32];
      tmem_ld32(my + kColS + wg * 32, w);
#pragma unroll
      for (int j = 0; j < 32; ++j) Sg[(size_t)(wg * 32 + j) * kD + c] = __uint_as_float(w[j]);
    }
  } else {
    if (tid == 0) record_error(P.err, kErrTimeout, d.req, h);
    // the products that timed out may still be running: one more bounded wait on
    // their commit (phase already advanced) before TMEM is released; if that
    // gives up too, the more severe kind replaces the first one
    const bool drained = mbar_wait(mbar, phase ^ 1);
    if (!drained && tid == 0) {
      atomicExch(&P.err[0], (int32_t)kErrTimeoutDrain);
      P.err[1] = d.req;
      P.err[2] = h;
    }
  }
  asm volatile("cp.async.wait_group 0;\n" ::: "memory");
  fence_before();
  __syncthreads();
  fence_after();
  if (warp == 0) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols));
}

}  // namespace

cudaError_t launch_prefill_tc(const PoolView &P, const RowBatch &rows, const TokenIO &io,
                              int variant, cudaStream_t stream) {
  if (rows.count <= 0) return cudaSuccess;
  dim3 grid(P.Hv, rows.count);
  auto run = [&](auto kernel) -> cudaError_t {
    cudaError_t e = ensure_smem((const void *)kernel, kSmemBytes);
    if (e != cudaSuccess) return e;
    kernel<<<grid, kThreads, kSmemBytes, stream>>>(P, rows, io, prefill_first_wait_polls());
    return cudaGetLastError();
  };
  switch (variant) {
    case kPlain: return run(prefill_tc_kernel<kPlain>);
    case kGated: return run(prefill_tc_kernel<kGated>);
    case kGatedDelta: return run(prefill_tc_kernel<kGatedDelta>);
  }
  return kUnsupported;
}

}  // namespace kvb
