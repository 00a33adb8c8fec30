// Chunked prefill on the fifth-generation tensor cores (tcgen05, TMEM), for
// bf16 inputs at d = 128.
//
// Same chunk algebra as prefill.cu ("KVBuffer: IO-aware Serving for Linear
// Attention", abstract: chunkwise computation; the delta-rule chunk form),
// chunk C = 64, per (request, value head) CTA:
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
// leave every per-column quantity (R, U, the output column, the state column)
// with the threads that own that column: (I + Mk) U = R is solved in fp32 by a
// blocked forward substitution, warpgroup a owning tokens 16 a .. 16 a + 15.
// Operands that are not exact in bf16 (S, U, wU, Mq) enter as hi + lo bf16
// parts (about 16 significant bits; the lo x lo product is dropped), with fp32
// accumulation in TMEM.  Q, K, V arrive by TMA (Q and K in the K-major layout
// with the 128-byte swizzle), outputs leave by TMA from a staging tile.  MMAs
// are issued by single threads, completion via tcgen05.commit on mbarriers;
// every wait on the tensor cores or the copies is bounded and a timeout sets
// the error word.
#include "kvb_device.cuh"

namespace kvb {
namespace {

constexpr int kC = 64, kD = 128, kThreads = 512;  // four warpgroups share every TMEM lane
// TMEM columns
constexpr uint32_t kColS = 0;     // S^T fp32            [128 lanes x 128]
constexpr uint32_t kColP = 128;   // A parts: S^T hi/lo (64 + 64), later U^T hi/lo, (wU)^T hi/lo (32 each)
constexpr uint32_t kColY = 256;   // Y^T fp32 (tokens: 0..63 q, 64..127 k); O^T in 0..63
constexpr uint32_t kColD = 384;   // the delta rule's block products; then an output part product
constexpr uint32_t kColG = 448;   // G fp32 (lane = token of [Q;K], column = key token), a chunk ahead
constexpr uint32_t kTmemCols = 512;
// shared memory (bytes)
constexpr int kXBytes = 2 * kC * kD * 2;        // [Q;K] bf16, K-major, 128-byte swizzle (32 KB)
constexpr int kXHalf = kXBytes / 2;             // X: [d_k half][token of [Q;K]][64 elements]
constexpr int kVBytes = kC * kD * 2;            // V bf16 [token][column] (16 KB)
constexpr int kGBytes = 2 * kC * 4;             // log-gate, beta
constexpr int kStage = (kXBytes + kVBytes + kGBytes + 1023) / 1024 * 1024;
constexpr int kKtBytes = kD * kC * 2;           // K^T bf16, core-matrix K-major (16 KB), two buffers
constexpr int kMqBytes = kC * kC * 2;           // one bf16 part of Mq (8 KB)
constexpr int kLdMk = kC + 4;                   // fp32 rows of Mk
constexpr int kMkBytes = kC * kLdMk * 4;
constexpr int kOffKt = 2 * kStage;
constexpr int kOffMq = kOffKt + 2 * kKtBytes;   // [2 parts]
constexpr int kOffMk = kOffMq + 2 * kMqBytes;
constexpr int kOffMkp = kOffMk + kMkBytes;      // Mk as bf16 hi / lo parts, core-matrix K-major
constexpr int kGateF = 8 * kC;                   // floats of one chunk's gate tables (see gates())
constexpr int kOffA = kOffMkp + 2 * kMqBytes;   // gate tables per chunk parity
constexpr int kSmemBytes = kOffA + 2 * kGateF * 4;
// core-matrix strides (bytes): 8 rows x 16 bytes per core matrix, k groups adjacent
constexpr uint32_t kLbo = 128;
constexpr uint32_t kSboKt = (kC / 8) * 128;     // K^T and Mq: 64 tokens per row group
static_assert(kSmemBytes <= 227 * 1024, "one CTA's shared memory");
static_assert(kStage % 1024 == 0 && kKtBytes % 1024 == 0 && kMqBytes % 1024 == 0, "alignment");
static_assert(kMqBytes == (kC / 8) * kSboKt, "Mq's lo part continues its hi part's row groups");
static_assert(kColD == kColY + 2 * kC && kColG == kColD + kC, "the output product's 128 columns");
// completion barriers, one completion each per chunk (so phase parity = chunk &
// 1): G, Y (first products), O and S (second products), P + b (the delta rule's
// products Mk_{.,b} U_b, b = 0 .. 2); then the two stages' landing barriers
// (TMA bytes), one completion per use, each on one commit.  G is issued a chunk
// ahead (its k-th completion is chunk k's).
constexpr int kBarG = 0, kBarY = 1, kBarO = 2, kBarS = 3, kBarP = 4, kBarF = 7, kBars = 9;

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
// shared-memory matrix descriptor: K-major, no swizzle (core matrices of 8 rows x
// 16 bytes; lbo = distance between k groups, sbo = distance between row groups)
__device__ __forceinline__ uint64_t sdesc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
  return (uint64_t)((addr >> 4) & 0x3FFF) | ((uint64_t)((lbo >> 4) & 0x3FFF) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3FFF) << 32) | ((uint64_t)1 << 46);
}
// K-major operand with the 128-byte swizzle (rows of 64 bf16 = 128 bytes, 8-row
// atoms of 1024 bytes, atom-aligned): stride between row groups 1024, leading
// offset unused; a K step of 16 elements advances the start by 32 bytes
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t addr) {
  return (uint64_t)((addr >> 4) & 0x3FFF) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
         ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
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
// Bounded wait on an mbarrier phase: at most `polls` polls, false on timeout.
// try_wait lets the hardware suspend the thread until the phase completes (or a
// short time limit, about a microsecond, passes), so waiting warps wake at once
// and take no issue slots meanwhile; the default bound is some tens of ms.  A
// capped wait (fewer polls: the failure-path test hook) polls without
// suspending, so that it gives up after that many looks.
constexpr int kWaitPolls = 1 << 16;
__device__ __forceinline__ bool mbar_wait(uint32_t mbar, uint32_t parity, int polls = kWaitPolls) {
  for (int it = 0; it < polls; ++it) {
    uint32_t done;
    if (polls < kWaitPolls)
      asm volatile("{\n\t.reg .pred p;\n\tmbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
                   "selp.u32 %0, 1, 0, p;\n\t}"
                   : "=r"(done) : "r"(mbar), "r"(parity) : "memory");
    else
      asm volatile("{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
                   "selp.u32 %0, 1, 0, p;\n\t}"
                   : "=r"(done) : "r"(mbar), "r"(parity) : "memory");
    if (done) return true;
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
// 16 columns without waiting (tmem_wait_ld completes every load issued before it)
__device__ __forceinline__ void tmem_ld16_async(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
// after tmem_wait_ld: ties the loaded registers to the wait, so that no use of
// them is scheduled before it
__device__ __forceinline__ void tmem_loaded(uint32_t (&r)[16]) {
  asm volatile(""
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]),
                 "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]),
                 "+r"(r[15]));
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

// named barrier `id` over `n` threads (whole warps): arrive without waiting, or wait
__device__ __forceinline__ void named_arrive(int id, int n) {
  asm volatile("bar.arrive %0, %1;" ::"r"(id), "r"(n) : "memory");
}
__device__ __forceinline__ void named_sync(int id, int n) { asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory"); }

// TMA: a 3D box of a tensor map into shared memory, completing its bytes on mbar
__device__ __forceinline__ void tma3d(uint32_t dst, const void *map, int x, int y, int z, uint32_t mbar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], [%5];"
      ::"r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(mbar) : "memory");
}
__device__ __forceinline__ void arrive_tx(uint32_t mbar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(mbar), "r"(bytes) : "memory");
}
// bulk copy shared -> global (16-byte aligned addresses, 16-byte multiple size),
// tracked in this thread's bulk groups
__device__ __forceinline__ void bulk_store(void *dst, uint32_t src, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst), "r"(src), "r"(bytes)
               : "memory");
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// TMA: a 3D box of shared memory out to a tensor map (bulk group of this thread)
__device__ __forceinline__ void tma3d_store(const void *map, int x, int y, int z, uint32_t src) {
  asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%1, %2, %3}], [%4];"
               ::"l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(src) : "memory");
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
__device__ __forceinline__ void bulk_wait_read() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
__device__ __forceinline__ void cp4(uint32_t dst, const void *src, bool valid) {
  const int n = valid ? 4 : 0;
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;\n" ::"r"(dst), "l"(src), "r"(n) : "memory");
}

template <int VARIANT>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_tc_kernel(const PoolView P, const __grid_constant__ RowBatch rows, const TokenIO io,
                      const __grid_constant__ PrefillMaps maps, int first_polls) {
  using KT = __nv_bfloat16;
  constexpr bool DELTA = VARIANT == kGatedDelta, GATED = VARIANT != kPlain;
  extern __shared__ __align__(1024) uint8_t smem[];
  __shared__ uint64_t mbar_s[kBars];
  __shared__ uint32_t tmem_s;
  // gate tables of chunk cc: the cumulative log-gates A, e^A, w = e^{A_{C-1} - A}
  // (then a spare row) and E_{a,j} = e^{A_{16 a} - A_j} (a = 0 .. 3), so that
  // e^{A_i - A_j} = e^{A_i - A_{16 a}} E_{a,j} for any a (a factor spans at most
  // one 16-token block of growth where the other is a decay)
  auto gates = [&](int cc) { return reinterpret_cast<float *>(smem + kOffA) + (cc & 1) * kGateF; };
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
  const uint32_t mbar0 = smem_u32(&mbar_s[0]);  // barrier k at mbar0 + 8 k
  const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;  // this warp's TMEM lanes


  // stage chunk cc: q and k rows of the chunk by TMA into X (two d_k halves of
  // 64 elements, 128-byte swizzle), v rows into V, the landing barrier of the
  // stage counting the bytes (thread 64, which also sends the outputs staged in
  // X two chunks earlier: those must have left first); gates and beta as plain
  // copies, zero past the prompt (64 threads from kGateTid: under the delta rule
  // warpgroup 3, which prepares the next chunk by itself)
  constexpr int kGateTid = DELTA ? 384 : 64;
  constexpr int kYTid = 384;  // the issuer of Y (warp 12)
  auto issue = [&](int cc, int tma_tid) {
    const uint32_t st_u = smem_u32(smem + (cc & 1) * kStage);
    if (tid == tma_tid) {
      bulk_wait_read();
      const uint32_t full = mbar0 + 8 * (kBarF + (cc & 1));
      const int z = (int)(b * Tp + (size_t)cc * kC);  // first token row of the chunk
      arrive_tx(full, kXBytes + kVBytes);
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        tma3d(st_u + hf * kXHalf, &maps.q, hf * 64, hq, z, full);
        tma3d(st_u + hf * kXHalf + kC * 128, &maps.k, hf * 64, hq, z, full);
      }
      tma3d(st_u + kXBytes, &maps.v, 0, h, z, full);
    }
    if (tid >= kGateTid && tid < kGateTid + kC) {
      const int j = tid - kGateTid;
      const bool ok = cc * kC + j < L;
      const size_t row = b * Tp + (ok ? cc * kC + j : L - 1);
      const uint32_t gs = st_u + kXBytes + kVBytes;
      if (GATED) cp4(gs + j * 4, io.log_g + row * P.Hv + h, ok);
      if (DELTA) cp4(gs + (kC + j) * 4, io.beta + row * P.Hv + h, ok);
    }
    asm volatile("cp.async.commit_group;\n" ::: "memory");
  };

  // the barriers, and chunk 0's copies at once (thread 0 right after the init),
  // then the TMEM allocation
  if (tid == 0) {
#pragma unroll
    for (int k = 0; k < kBars; ++k)
      asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(mbar0 + 8 * k));
    asm volatile("fence.mbarrier_init.release.cluster;");
  }
  if (nchunks > 0) issue(0, 0);
  int pending = nchunks > 0 ? 0 : -1;  // the chunk whose copies are issued and not yet waited for
  int gpend = -1;                      // the chunk whose G is issued and not yet waited for
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&tmem_s)),
                 "r"(kTmemCols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  fence_before();
  __syncthreads();
  fence_after();
  const uint32_t tmem = tmem_s;
  const int lt = tid & 127;              // this thread's TMEM lane
  const int wg = tid >> 7;               // warpgroup: which quarter of each lane's columns
  const uint32_t my = tmem + lane_base;  // this thread's lane, column 0
  const int c = lt;                      // as a state column
  bool ok = true;
  // poll bound of the waits on the products: those of the first chunk may be
  // capped by the failure-path test hook (first_polls > 0), later ones have the
  // default
  const int cap = first_polls > 0 ? first_polls : kWaitPolls;
  auto polls_at = [&](int chn) { return chn == 0 ? cap : kWaitPolls; };

  // bf16 hi / lo parts of 16 state rows (16 r0 .. 16 r0 + 15) of column c into the
  // A region (the operand of Y^T = S^T X^T)
  auto put_parts16 = [&](const float (&x)[16], int r0) {
    uint32_t hi[8], lo[8];
    split16(x, hi, lo);
    tmem_st8(my + kColP + r0 * 8, hi);
    tmem_st8(my + kColP + 64 + r0 * 8, lo);
  };

  // K^T of chunk cc (the B operand of its state update) from the K rows of its
  // staged X, and its cumulative gates.  K^T: 8 x 8 tiles of the keys (8 tokens
  // x 8 dims, 16-byte pieces of the swizzled rows: piece p of row t sits at
  // p ^ (t & 7)) transposed into K^T's core matrices (8 dims x 8 tokens) by
  // ldmatrix.trans + stmatrix, four per warp instruction, the tiles (token group
  // tile & 7, dim group tile >> 3) split evenly over the working warps.
  auto prep = [&](int cc, int w0, int nw) {  // by warps w0 .. w0 + nw - 1 (16, or a warpgroup's 4)
    const uint8_t *stc = smem + (cc & 1) * kStage;
    const uint32_t xs_u = smem_u32(stc), kt_u = smem_u32(smem + kOffKt + (cc & 1) * kKtBytes);
    const int wr = warp - w0, per = 128 / nw;  // this warp's rank; K^T tiles per warp
#pragma unroll 2
    for (int q = 0; q < per; q += 4) {
      const int tile = wr * per + q + (lane >> 3), jg = tile & 7, dg = tile >> 3, row = lane & 7;
      const uint32_t src =
          xs_u + (dg >> 3) * kXHalf + (kC + jg * 8 + row) * 128 + (uint32_t)(((dg & 7) ^ row) << 4);
      const uint32_t dst = kt_u + dg * kSboKt + jg * kLbo + row * 16;
      uint32_t r0, r1, r2, r3;
      asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                   : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(src));
      asm volatile("stmatrix.sync.aligned.m8n8.x4.shared.b16 [%0], {%1,%2,%3,%4};"
                   ::"r"(dst), "r"(r0), "r"(r1), "r"(r2), "r"(r3) : "memory");
    }
    const int role = wr - (nw == 16 ? 4 : 0);  // gate tables: four warps scan the gates, each fills a share
    if (role >= 0 && role < 4) {
      const float *gsc = reinterpret_cast<const float *>(stc + kXBytes + kVBytes);
      float *Acum = gates(cc), *eA = Acum + kC, *wL = eA + kC, *E = wL + 2 * kC;
      float a0 = GATED ? gsc[lane] : 0.f, a1 = GATED ? gsc[lane + 32] : 0.f;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const float y0 = __shfl_up_sync(kFull, a0, off), y1 = __shfl_up_sync(kFull, a1, off);
        if (lane >= off) {
          a0 += y0;
          a1 += y1;
        }
      }
      a1 += __shfl_sync(kFull, a0, 31);
      if (role == 0) {
        Acum[lane] = a0;
        Acum[lane + 32] = a1;
        eA[lane] = expf(a0);
        eA[lane + 32] = expf(a1);
      } else if (role == 1) {
        const float AL = __shfl_sync(kFull, a1, 31);
        wL[lane] = expf(AL - a0);
        wL[lane + 32] = expf(AL - a1);
      } else {
        const int a = (role - 2) * 2;  // E rows a, a + 1 (A_{16 a}: lane 16 a of the token scan)
        const float B0 = __shfl_sync(kFull, a < 2 ? a0 : a1, 0), B1 = __shfl_sync(kFull, a < 2 ? a0 : a1, 16);
        E[a * kC + lane] = expf(B0 - a0);
        E[a * kC + lane + 32] = expf(B0 - a1);
        E[(a + 1) * kC + lane] = expf(B1 - a0);
        E[(a + 1) * kC + lane + 32] = expf(B1 - a1);
      }
    }
  };
  // CTA-uniform: chunk cc's copies landed (bounded wait on the TMA bytes, then
  // this thread's plain copies), visible to all; the rows past the prompt of a
  // last, partial chunk are zeroed (the TMA brought whatever follows it)
  auto land = [&](int cc) -> bool {
    asm volatile("cp.async.wait_group 0;\n" ::: "memory");
    ok = __syncthreads_and(mbar_wait(mbar0 + 8 * (kBarF + (cc & 1)), (cc >> 1) & 1)) != 0;
    if (!ok) return false;
    pending = -1;
    const int nv = L - cc * kC;  // valid tokens of the chunk
    if (nv < kC) {
      uint8_t *stc = smem + (cc & 1) * kStage;
      // per padded token: 4 X rows of 128 bytes (2 halves x Q, K), 1 V row of 256
      for (int idx = tid; idx < (kC - nv) * 48; idx += kThreads) {
        const int t = nv + idx / 48, pc = idx % 48;
        uint8_t *dst = pc < 32 ? stc + (pc >> 4) * kXHalf + ((pc >> 3) & 1) * (kC * 128) + t * 128 + (pc & 7) * 16
                               : stc + kXBytes + t * 256 + (pc - 32) * 16;
        *reinterpret_cast<uint4 *>(dst) = make_uint4(0u, 0u, 0u, 0u);
      }
      fence_async_smem();  // the zeros, for the tensor cores (G is issued next)
      __syncthreads();
    }
    return true;
  };
  // G = X K^T of chunk cc (exact; thread 64, after cc landed), into the G columns
  auto issue_g = [&](int cc) {
    if (tid == 64) {
      const uint32_t xg = smem_u32(smem + (cc & 1) * kStage), idG = idesc_bf16(128, kC);
#pragma unroll
      for (int ks = 0; ks < kD / 16; ++ks) {  // X rows: tokens of [Q;K]; the keys from row kC
        const uint32_t xk = xg + (ks >> 2) * kXHalf + (ks & 3) * 32;
        mma_ss(tmem + kColG, sdesc_sw128(xk), sdesc_sw128(xk + kC * 128), idG, ks > 0);
      }
      mma_commit(mbar0 + 8 * kBarG);
    }
    gpend = cc;
  };
  // this warpgroup's 32 state rows of column c, read while chunk 0 lands
  float s0[32];
#pragma unroll
  for (int j = 0; j < 32; ++j) s0[j] = from_zero ? 0.f : Sg[(size_t)(wg * 32 + j) * kD + c];
  if (nchunks > 0 && land(0)) {
    issue_g(0);
    prep(0, 0, 16);
  }
  // their parts (the operand of the first Y^T), and e^{A_{C-1}} S^T in fp32, the
  // state ready for chunk 0's update (each chunk's decay is applied when its
  // predecessor's parts are made)
  {
    __syncthreads();  // chunk 0's gates
    const float eL = nchunks > 0 ? gates(0)[kC + kC - 1] : 1.f;
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      float x[16];
      uint32_t w[16];
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        x[j] = s0[q * 16 + j];
        w[j] = __float_as_uint(eL * x[j]);
      }
      tmem_st16(my + kColS + (wg * 2 + q) * 16, w);
      put_parts16(x, wg * 2 + q);
    }
    tmem_wait_st();
  }
  // Mq's entries in rows 0 .. 31 and key columns 32 .. 63 (above the diagonal)
  // stay zero: written once here, skipped by the Gram rows
  for (int k = tid; k < 2 * 4 * 4 * 8; k += kThreads) {  // part, row group, k group, row
    const int part = k >> 7, rg = (k >> 5) & 3, kg = 4 + ((k >> 3) & 3), r = k & 7;
    *reinterpret_cast<uint4 *>(smem + kOffMq + part * kMqBytes + rg * kSboKt + kg * kLbo + r * 16) =
        make_uint4(0u, 0u, 0u, 0u);
  }
  fence_async_smem();
  fence_before();
  __syncthreads();
  fence_after();

  // the barriers committed in the current chunk (a timeout drains on each)
  uint32_t cmask = 0;
  int ch_at = 0;  // the chunk the loop is in
  // CTA-uniform bounded wait on barrier k of chunk ch (parity ch & 1)
  auto wait_bar = [&](int k, int chn) -> bool {
    ok = __syncthreads_and(mbar_wait(mbar0 + 8 * k, chn & 1, polls_at(chn))) != 0;
    fence_after();
    return ok;
  };

  for (int ch = 0; ch < nchunks && ok; ++ch) {
    ch_at = ch;
    uint8_t *st = smem + (ch & 1) * kStage;
    const uint32_t xs = smem_u32(st);
    const KT *vs = reinterpret_cast<const KT *>(st + kXBytes);
    const float *gs = reinterpret_cast<const float *>(st + kXBytes + kVBytes);
    const float *bs = gs + kC;
    const float *Acum = gates(ch), *eA = Acum + kC, *wL = eA + kC, *Eg = wL + 2 * kC;
    const int t0 = ch * kC;
    // (chunk ch staged, its K^T and gates built, S^T's parts in TMEM, S^T
    // already decayed by e^{A_{C-1}})

    // MMAs 1: Y^T = S^T X^T (S^T as hi + lo parts), by thread 384: warp 12 (like
    // warp 8) holds Gram entries that are all above the diagonal, written once
    if (tid == kYTid) {
      const uint32_t idY = idesc_bf16(128, 2 * kC);
#pragma unroll
      for (int part = 0; part < 2; ++part)
#pragma unroll
        for (int ks = 0; ks < kD / 16; ++ks) {
          const uint64_t bx = sdesc_sw128(xs + (ks >> 2) * kXHalf + (ks & 3) * 32);
          mma_ts(tmem + kColY, tmem + kColP + part * 64 + ks * 8, bx, idY, part > 0 || ks > 0);
        }
      mma_commit(mbar0 + 8 * kBarY);
    }
    // G (issued with the previous chunk): each thread waits by itself (the
    // CTA-wide check of this wait comes with the one on Y) and takes its 16 entries
    const int j0 = wg * 16;
    float gr[16];
    const bool okG = mbar_wait(mbar0 + 8 * kBarG, ch & 1, polls_at(ch));
    gpend = -1;
    fence_after();
    {
      uint32_t w[16];
      tmem_ld16(my + kColG + j0, w);
#pragma unroll
      for (int j = 0; j < 16; ++j) gr[j] = __uint_as_float(w[j]);
    }

    cmask = 1u << kBarY;
    // while the products run: the next chunk's copies (into the other stage, free
    // since the previous chunk finished)
    if (ch + 1 < nchunks) {
      issue(ch + 1, 64);
      pending = ch + 1;
    }
    // Gram rows, key tokens split by warpgroup: thread (i, wg) builds entries
    // j = 16 wg .. 16 wg + 15 of row i of Mq (parts, smem) or Mk (fp32 and parts)
    // e^{A_i - A_j} = e^{A_i - A_{j0}} E_{wg, j} (j0 = 16 wg): one exponential per
    // thread, and a table row shared by the warp
    if (warp != 8 && warp != 12) {
      const int i = lt;
      const float *Er = Eg + wg * kC + j0;
      if (i < kC) {  // Mq[i][j] = scale e^{A_i-A_j} q_i.k_j, j <= i
        const float sF = i >= j0 ? P.scale * expf(Acum[i] - Acum[j0]) : 0.f;
        float x[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) x[j] = j0 + j <= i ? sF * Er[j] * gr[j] : 0.f;
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
      } else if (DELTA && wg <= ((i - kC) >> 4)) {
        // Mk[i'][j] = beta_i' e^{A_i'-A_j} k_i'.k_j, j < i': the diagonal block in
        // fp32 (the in-register solves), the blocks below it as bf16 parts (the
        // tensor-core block products); the blocks above it are never read
        const int ip = i - kC;
        const float bF = bs[ip] * expf(Acum[ip] - Acum[j0]);
        float x[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) x[j] = j0 + j < ip ? bF * Er[j] * gr[j] : 0.f;
        if (wg == (ip >> 4)) {  // column-major: [block][column l][row i]
          float *mt = Mk + (ip >> 4) * 256 + (ip & 15);
#pragma unroll
          for (int j = 0; j < 16; ++j) mt[j * 16] = x[j];
        } else {
          uint32_t hi[8], lo[8];
          split16(x, hi, lo);
          uint8_t *mkp = smem + kOffMkp;
#pragma unroll
          for (int q = 0; q < 2; ++q) {
            const int off = (ip >> 3) * kSboKt + (wg * 2 + q) * kLbo + (ip & 7) * 16;
            *reinterpret_cast<uint4 *>(mkp + off) =
                make_uint4(hi[4 * q], hi[4 * q + 1], hi[4 * q + 2], hi[4 * q + 3]);
            *reinterpret_cast<uint4 *>(mkp + kMqBytes + off) =
                make_uint4(lo[4 * q], lo[4 * q + 1], lo[4 * q + 2], lo[4 * q + 3]);
          }
        }
      }
    }
    fence_async_smem();  // Mq, for the tensor cores
    ok = __syncthreads_and(okG && mbar_wait(mbar0 + 8 * kBarY, ch & 1, polls_at(ch))) != 0;  // Mk, Mq complete
    fence_after();
    if (!ok) break;

    bool okP = true, okL = true;
    {
      // U^T and (wU)^T parts (tokens 16 q .. 16 q + 15 of column c) into TMEM,
      // the A operands of the second MMAs
      auto u_parts = [&](float (&x)[16], int q, bool weighted) {
        uint32_t hi[8], lo[8];
        if (weighted) {
          float y[16];
#pragma unroll
          for (int j = 0; j < 16; ++j) y[j] = x[j] * wL[q * 16 + j];
          split16(y, hi, lo);
          tmem_st8(my + kColP + 64 + q * 8, hi);
          tmem_st8(my + kColP + 96 + q * 8, lo);
        } else {
          split16(x, hi, lo);
          tmem_st8(my + kColP + q * 8, hi);
          tmem_st8(my + kColP + 32 + q * 8, lo);
        }
      };
      if (DELTA) {
        // (I + Mk) U = R by blocked forward substitution: warpgroup a holds R and
        // then U for tokens 16 a .. 16 a + 15 of column c.  Its diagonal block is
        // solved in fp32 in registers, each solved value updating the rows below
        // it at once (a chain of 15 FMAs); the blocks below the diagonal enter as
        // tensor-core products, D^T += U_b^T Mk_{.,b}^T (U_b^T parts from TMEM,
        // Mk parts from smem; three part products, rows 16 (b + 1) .. 63 into the
        // G columns), issued by thread 0 as soon as warpgroup b has written U_b's
        // parts (named barrier 1 + b), each completing on barrier P + b.
        float u[16];
        {
          uint32_t w[16];
          tmem_ld16(my + kColY + kC + wg * 16, w);
#pragma unroll
          for (int j = 0; j < 16; ++j) {  // R_i = beta_i (v_i - e^{A_i} S^T k_i)
            const int jj = wg * 16 + j;
            u[j] = bs[jj] * (__bfloat162float(vs[jj * kD + c]) - eA[jj] * __uint_as_float(w[j]));
          }
        }
        auto solve = [&]() {  // the diagonal block, column-major: column l in 16 floats
          const float4 *md = reinterpret_cast<const float4 *>(Mk + wg * 256);
#pragma unroll
          for (int l = 0; l < 15; ++l)
#pragma unroll
            for (int i4 = (l + 1) >> 2; i4 < 4; ++i4) {
              const float4 m = md[l * 4 + i4];
              if (4 * i4 > l) u[4 * i4] = fmaf(-m.x, u[l], u[4 * i4]);
              if (4 * i4 + 1 > l) u[4 * i4 + 1] = fmaf(-m.y, u[l], u[4 * i4 + 1]);
              if (4 * i4 + 2 > l) u[4 * i4 + 2] = fmaf(-m.z, u[l], u[4 * i4 + 2]);
              u[4 * i4 + 3] = fmaf(-m.w, u[l], u[4 * i4 + 3]);
            }
        };
        // thread 0: the products of block b (after fence_after)
        auto issue_sub = [&](int bb) {
          const int n0 = 16 * (bb + 1);
          const uint32_t idP = idesc_bf16(128, kC - n0), mkp = smem_u32(smem + kOffMkp);
#pragma unroll
          for (int combo = 0; combo < 3; ++combo) {
            const int ua = combo == 2 ? 32 : 0;                      // U_b^T hi, hi, lo
            const uint32_t mb = mkp + (combo == 1 ? kMqBytes : 0);   // Mk hi, lo, hi
            mma_ts(tmem + kColD + n0, tmem + kColP + ua + bb * 8,
                   sdesc(mb + (n0 >> 3) * kSboKt + 2 * bb * kLbo, kLbo, kSboKt), idP, bb > 0 || combo > 0);
          }
          mma_commit(mbar0 + 8 * (kBarP + bb));
        };
        if (wg == 3 && ch + 1 < nchunks) {
          // meanwhile: chunk ch + 1 landed (the TMA bytes, this warpgroup's own
          // gate copies; a partial last chunk's rows past the prompt zeroed), its
          // K^T and gate tables (named barrier 5 over the warpgroup)
          asm volatile("cp.async.wait_group 0;\n" ::: "memory");
          okL = mbar_wait(mbar0 + 8 * (kBarF + ((ch + 1) & 1)), ((ch + 1) >> 1) & 1);
          const int nv = L - (ch + 1) * kC;
          if (nv < kC) {
            uint8_t *stc = smem + ((ch + 1) & 1) * kStage;
            for (int idx = tid - 384; idx < (kC - nv) * 48; idx += 128) {
              const int t = nv + idx / 48, pc = idx % 48;
              uint8_t *dst = pc < 32 ? stc + (pc >> 4) * kXHalf + ((pc >> 3) & 1) * (kC * 128) + t * 128 + (pc & 7) * 16
                                     : stc + kXBytes + t * 256 + (pc - 32) * 16;
              *reinterpret_cast<uint4 *>(dst) = make_uint4(0u, 0u, 0u, 0u);
            }
            fence_async_smem();
          }
          named_sync(5, 128);
          prep(ch + 1, 12, 4);
          fence_async_smem();  // K^T, for the tensor cores
        }
        if (wg > 0) {  // the products of the blocks above
          okP = mbar_wait(mbar0 + 8 * (kBarP + wg - 1), ch & 1, polls_at(ch));
          fence_after();
          uint32_t w[16];
          tmem_ld16(my + kColD + wg * 16, w);
#pragma unroll
          for (int j = 0; j < 16; ++j) u[j] -= __uint_as_float(w[j]);
        }
        solve();
        u_parts(u, wg, false);
        if (wg < 3) {
          tmem_wait_st();
          fence_before();
        }
        if (wg == 0) {
          named_sync(1, 128);  // U_0's parts in TMEM
          if (warp == 0) {
            if (lane == 0) {
              fence_after();
              issue_sub(0);
            }
            named_sync(2, 160);  // U_1's parts
            if (lane == 0) {
              fence_after();
              issue_sub(1);
            }
            named_sync(3, 160);  // U_2's parts
            if (lane == 0) {
              fence_after();
              issue_sub(2);
            }
          }
        } else if (wg < 3) {
          named_arrive(1 + wg, 160);
        }
        u_parts(u, wg, true);  // (wU)^T, for the state update only
      } else {  // U = V, tokens 16 wg .. 16 wg + 15
        float x[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) x[j] = __bfloat162float(vs[(wg * 16 + j) * kD + c]);
        u_parts(x, wg, false);
        u_parts(x, wg, true);
      }
    }
    if (DELTA) cmask |= 7u << kBarP;
    tmem_wait_st();
    fence_before();
    ok = __syncthreads_and(okP && okL) != 0;  // the waits on the block products (and landing), CTA-wide
    fence_after();
    if (!ok) break;

    // MMAs 2, from two issuing threads: U^T Mq^T (thread 0) and S^T += (wU)^T K
    // (thread 96).  Mq's hi and lo parts lie back to back (8 row groups each), so
    // U^T hi [Mq hi; Mq lo]^T is one product of 128 columns (the K half of Y, read
    // by now, and the D columns), and U^T lo Mq hi^T adds onto its first half:
    // O^T = e^A scale Y_q^T + both halves
    if (tid == 0) {
      const uint32_t idO2 = idesc_bf16(128, 2 * kC), idO = idesc_bf16(128, kC), mq = smem_u32(smem + kOffMq);
#pragma unroll
      for (int k0 = 0; k0 < kC; k0 += 16)
        mma_ts(tmem + kColY + kC, tmem + kColP + k0 / 2, sdesc(mq + (k0 / 8) * kLbo, kLbo, kSboKt), idO2, k0 > 0);
#pragma unroll
      for (int k0 = 0; k0 < kC; k0 += 16)
        mma_ts(tmem + kColY + kC, tmem + kColP + 32 + k0 / 2, sdesc(mq + (k0 / 8) * kLbo, kLbo, kSboKt), idO, 1);
      mma_commit(mbar0 + 8 * kBarO);
    } else if (tid == 96) {
      const uint32_t idS = idesc_bf16(128, kD), kt = smem_u32(smem + kOffKt + (ch & 1) * kKtBytes);
#pragma unroll
      for (int part = 0; part < 2; ++part)
#pragma unroll
        for (int k0 = 0; k0 < kC; k0 += 16)
          mma_ts(tmem + kColS, tmem + kColP + 64 + part * 32 + k0 / 2,
                 sdesc(kt + (k0 / 8) * kLbo, kLbo, kSboKt), idS, 1);
      mma_commit(mbar0 + 8 * kBarS);
    }
    cmask |= (1u << kBarO) | (1u << kBarS);
    // while they run: the next chunk's K^T (the other buffer) and gates (this
    // chunk's are no longer read)
    if (ch + 1 < nchunks) {
      if (DELTA) {  // landed and prepared by warpgroup 3 during the substitution
        pending = -1;
      } else {
        if (!land(ch + 1)) break;
        prep(ch + 1, 0, 16);
      }
      issue_g(ch + 1);  // the G columns were read by this chunk's Gram rows
    }
    if (!wait_bar(kBarO, ch)) break;

    // outputs (tokens 16 wg .. 16 wg + 15 of column c, the sum of the three
    // part products) into a staging tile [token][column] over this chunk's X
    // (read by now), leaving by one TMA store (thread 64), or one bulk copy of
    // 512 bytes per prompt token for a last, partial chunk; then the next
    // chunk's S^T parts (state rows 32 wg .. 32 wg + 31)
    {
      uint32_t w[16], w1[16], w2[16];
      tmem_ld16_async(my + kColY + wg * 16, w);
      tmem_ld16_async(my + kColY + kC + wg * 16, w1);
      tmem_ld16_async(my + kColD + wg * 16, w2);
      tmem_wait_ld();
      tmem_loaded(w);
      tmem_loaded(w1);
      tmem_loaded(w2);
      float *ost = reinterpret_cast<float *>(st);
#pragma unroll
      for (int j = 0; j < 16; ++j)
        ost[(wg * 16 + j) * kD + c] =
            fmaf(P.scale * eA[wg * 16 + j], __uint_as_float(w[j]), __uint_as_float(w1[j])) + __uint_as_float(w2[j]);
      fence_async_smem();
    }
    if (!wait_bar(kBarS, ch)) break;
    if (t0 + kC <= L) {
      if (tid == 64) tma3d_store(&maps.o, 0, h, (int)(b * Tp + t0), xs);
    } else if (tid < L - t0) {
      bulk_store(io.o + ((b * Tp + t0 + tid) * P.Hv + h) * kD, xs + tid * kD * 4, kD * 4);
    }
    if (ch + 1 < nchunks) {
      // the next chunk's S^T parts, and its decay e^{A_{C-1}} applied to S^T
      const float eLn = gates(ch + 1)[kC + kC - 1];
      uint32_t wa[16], wb[16];
      tmem_ld16_async(my + kColS + wg * 32, wa);
      tmem_ld16_async(my + kColS + wg * 32 + 16, wb);
      tmem_wait_ld();
      tmem_loaded(wa);
      tmem_loaded(wb);
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        uint32_t (&w16)[16] = q ? wb : wa;
        float x[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          x[j] = __uint_as_float(w16[j]);
          w16[j] = __float_as_uint(eLn * x[j]);
        }
        put_parts16(x, wg * 2 + q);
        tmem_st16(my + kColS + wg * 32 + q * 16, w16);
      }
      tmem_wait_st();
    }
    fence_async_smem();  // the next stage's copies and K^T, for the tensor cores
    fence_before();
    __syncthreads();
    fence_after();
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
    // the products and copies that timed out may still be running: one more
    // bounded wait on the last commit and on the copies in flight before TMEM
    // and shared memory are released; if that gives up too, the more severe
    // kind replaces the first one
    bool drained = true;
    for (int k = 0; k < kBarF; ++k)
      if (cmask & (1u << k)) drained = mbar_wait(mbar0 + 8 * k, ch_at & 1) && drained;
    if (gpend >= 0) drained = mbar_wait(mbar0 + 8 * kBarG, gpend & 1) && drained;
    if (pending >= 0) drained = mbar_wait(mbar0 + 8 * (kBarF + (pending & 1)), (pending >> 1) & 1) && drained;
    if (!drained && tid == 0) {
      atomicExch(&P.err[0], (int32_t)kErrTimeoutDrain);
      P.err[1] = d.req;
      P.err[2] = h;
    }
  }
  asm volatile("cp.async.wait_group 0;\n" ::: "memory");
  bulk_wait_all();  // this thread's output copies
  fence_before();
  __syncthreads();
  fence_after();
  if (warp == 0) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols));
}

}  // namespace

cudaError_t launch_prefill_tc(const PoolView &P, const RowBatch &rows, const TokenIO &io,
                              const PrefillMaps &maps, int variant, cudaStream_t stream) {
  if (rows.count <= 0) return cudaSuccess;
  dim3 grid(P.Hv, rows.count);
  auto run = [&](auto kernel) -> cudaError_t {
    cudaError_t e = ensure_smem((const void *)kernel, kSmemBytes);
    if (e != cudaSuccess) return e;
    kernel<<<grid, kThreads, kSmemBytes, stream>>>(P, rows, io, maps, prefill_first_wait_polls());
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
