// Parallel verification of T draft tokens on the fifth-generation tensor cores
// (tcgen05 + TMA), bf16 pools at d = 128.
//
// KVBuffer ("KVBuffer: IO-aware Serving for Linear Attention", Figure 2): the
// drafts' KVs go into the buffer and every draft's output comes from the same
// state S0 plus the buffer, with no temporary state.  With n tokens buffered
// since the last fold and the drafts at chunk positions n .. n+T-1
// (A = cumulative log-gate over the chunk):
//   y_j = S0^T q_j,  z_j = S0^T k_j                    2T mat-vecs over S0
//   u_j = beta_j (v_j - e^{A_j} z_j - sum_{l<j} e^{A_j-A_l} (k_j.k_l) u_l)   (delta rule)
//   o_j = scale (e^{A_j} y_j + sum_{l<=j} e^{A_j-A_l} (q_j.k_l) u_l)
//
// The mat-vecs are one tensor-core product per (row, value head) unit:
//   Y^T = S0^T X,   X = [q_0 .. q_{T-1}, k_0 .. k_{T-1}]  (d_k x V, V <= 16)
// M = 128 state columns (TMEM lanes), N = 16 vectors, K = d_k, kind::tf32 with
// fp32 accumulation in TMEM.  S0 is the A operand read straight from shared
// memory in its stored orientation (value columns contiguous, i.e. MN-major);
// the tensor cores accept an MN-major tf32 operand only in the 128-byte swizzle
// with 32-byte atoms, which is exactly what a TMA tensor copy with the
// 128B_ATOM_32B swizzle writes: each (slot, head) tile arrives as four
// {32 columns x 128 rows} boxes, and no thread ever touches the state.  The
// hardware truncates S0 to tf32 (relative error < 2^-10 per element); q and k
// are bf16 and exact.
//
// Each CTA is persistent (one per SM) and walks units u, u + grid, ...; unit k
// of a CTA belongs to consumer group g = k mod G (G = 2 when shared memory
// allows).  The roles form a pipeline, every hand-off an mbarrier:
//  * the TMA warp streams the state tiles through a ring of 64 KB stages,
//    refilling a stage as soon as the tensor cores have read it;
//  * one staging warp per group copies each unit's small operands (draft q, k,
//    v; buffered keys, u / v and gates; draft gates and betas) into one of the
//    group's small stages: rows by bulk copies (one per lane), gates by 4-byte
//    cp.async, so no register round trip;
//  * one builder group (4 warps) per group turns a unit's staged q and k into
//    X (fp32, canonical K-major layout) in one of two X buffers, then forms the
//    drafts' cumulative gates and, with one mma.sync pass, the score dots
//    q_j.k_l, k_j.k_l and their decay weights in one of two weight buffers;
//  * one MMA warp per group issues the unit's product into one of the group's
//    two TMEM accumulators once its tile has landed and its X is built;
//  * the consumer group (4 warps; thread c owns state column c and TMEM lane
//    c) reads its column of Y^T, runs the forward substitution over the drafts
//    and writes the outputs and the drafts' buffer entries.
// With two buffers of X, weights and accumulator per group, the builder and the
// tensor cores work on unit k + 2G while the consumers finish unit k.  A
// single warp issuing every product, with the consumers building X between
// their own phases, kept the tensor cores and the consumers waiting on each
// other: the product of one tile (16 MMAs) took about as long to issue as the
// HBM share of a tile.
//
// Every wait is bounded: a timeout records the error word (kErrTimeout), stops
// every role, waits (bounded) for the copies and products still in flight,
// releases TMEM and returns.
#include <cuda.h>

#include <type_traits>

#include "kvb_device.cuh"

namespace kvb {
namespace {

constexpr int kVtCons = 128;               // threads of one consumer (or builder) group
constexpr int kVtMaxGroups = 2;            // unit pipelines per CTA
// per group: consumers, builders, its MMA warp and staging warp; + the TMA warp
constexpr int kVtGroupThreads = 2 * kVtCons + 64;
constexpr int kVtMaxThreads = kVtMaxGroups * kVtGroupThreads + 32;
constexpr int kVtXS = 128 + 8;             // bf16 row stride of staged vectors and keys (272 B)
constexpr int kVtMaxL = 16;                // chunk tokens (buffered + drafts)
constexpr int kVtMaxV = 16;                // vectors of the product (its N)
constexpr int kVtMaxStages = 3;            // state tiles in flight
constexpr int kVtPolls = 1 << 16;          // try_wait bound of every wait (each up to ~a microsecond)
constexpr uint32_t kTileBytes = 128 * 128 * 4;
constexpr uint32_t kTmemCols = 128;  // per group two accumulators of up to 16 columns
constexpr uint32_t kVtSmemMax = 227 * 1024 - 10 * 1024;  // dynamic bytes (1 KB static aside, and margin)

// Byte offsets of one small stage (16-byte aligned parts).
struct VtStage {
  uint32_t xr, kr, us, vs, acum, lg, bt, koff, voff, meta, bytes;
};
__host__ __device__ inline VtStage vt_stage(int variant, int T, int LM) {
  const bool delta = variant == kGatedDelta;
  auto up = [](uint32_t x) { return (x + 15u) & ~15u; };
  const uint32_t LP = (uint32_t)(LM + 7) / 8 * 8;
  VtStage s;
  s.xr = 0;                                                  // [T][XS] bf16 draft q
  s.kr = s.xr + up((uint32_t)T * kVtXS * 2);                 // [LP][XS] bf16 chunk keys
  s.us = s.kr + up(LP * kVtXS * 2);                          // u (fp32) or v (bf16) rows
  // u rows of the buffered tokens (delta rule: at most LM - T of them; the
  // drafts' u stay in registers), or v rows of the whole chunk
  s.vs = s.us + up((uint32_t)(delta ? LM - T : LM) * 128 * (delta ? 4 : 2));  // [T][128] bf16 draft v
  s.acum = s.vs + (delta ? up((uint32_t)T * 128 * 2) : 0);   // [LM] cumulative log-gates
  s.lg = s.acum + up((uint32_t)LM * 4);                      // [T] draft log-gates
  s.bt = s.lg + up((uint32_t)T * 4);                         // [T] draft betas
  s.koff = s.bt + up((uint32_t)T * 4);                       // [LM] key row offsets (elements)
  s.voff = s.koff + up((uint32_t)LM * 8);                    // [LM] value row indices
  s.meta = s.voff + up((uint32_t)LM * 8);                    // {row, head, n, bad, slot, req}
  s.bytes = s.meta + 32;
  return s;
}
// Whole dynamic shared memory: `ns` state tiles (1024-aligned); per group two
// X buffers (fp32, K-major core matrices, VP = V rounded up to 8 vectors) and
// two weight buffers (weighted q.k, weighted k.k, e^{A_j}); `nst` small stages
// per group.
struct VtLayout {
  uint32_t tile, grp, xf, xbuf, sw, cw, ea, wbuf, grp_bytes, stage, stage_bytes, total;
};
__host__ __device__ inline VtLayout vt_layout(int variant, int T, int LM, int ns, int groups, int nst) {
  VtLayout l;
  const uint32_t V = (uint32_t)(variant == kGatedDelta ? 2 * T : T);
  const uint32_t VP = (V + 7) & ~7u;
  const uint32_t TP = (uint32_t)(T + 3) & ~3u;   // weight row stride (float4 reads)
  l.tile = 0;
  l.grp = (uint32_t)ns * kTileBytes;              // group parts, group g at grp + g * grp_bytes
  l.xf = 0;                                       // X buffer b at xf + b * xbuf
  l.xbuf = VP * 128 * 4;
  l.sw = 2 * l.xbuf;                              // weight buffer b at + b * wbuf:
  l.cw = l.sw + (uint32_t)LM * TP * 4;            //   [LM][TP] weighted q.k, token-major,
  l.ea = l.cw + (uint32_t)LM * TP * 4;            //   [LM][TP] weighted k.k, [TP] e^{A_j}
  l.wbuf = (2 * (uint32_t)LM + 1) * TP * 4;
  l.grp_bytes = (l.sw + 2 * l.wbuf + 127) / 128 * 128;
  l.stage = l.grp + (uint32_t)groups * l.grp_bytes;  // small stage s at stage + s * stage_bytes
  l.stage_bytes = (vt_stage(variant, T, LM).bytes + 127) / 128 * 128;
  l.total = l.stage + (uint32_t)(nst * groups) * l.stage_bytes;
  return l;
}
// The launch shape: groups, state stages and small stages per group.  Two
// groups first (one leaves the SM idle between its phases); then the most
// small stages (with three the staging warp and the builders run a unit ahead
// of the consumers), then the most state stages that fit (false: none fits).
__host__ __device__ inline bool vt_shape(int variant, int T, int LM, int &groups, int &ns, int &nst) {
  for (groups = kVtMaxGroups; groups >= 1; --groups)
    for (nst = 3; nst >= 2; --nst)
      for (ns = kVtMaxStages; ns >= 2; --ns)
        if (vt_layout(variant, T, LM, ns, groups, nst).total <= kVtSmemMax) return true;
  return false;
}

__device__ __forceinline__ uint32_t su32(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
// shared-memory matrix descriptor (sm_100 form): start, leading / stride byte
// offsets, fixed version bits, layout type (0 none, 1 128B with 32B atoms)
__device__ __forceinline__ uint64_t vt_desc(uint32_t addr, uint32_t lbo, uint32_t sbo, uint32_t layout) {
  return (uint64_t)((addr >> 4) & 0x3FFF) | ((uint64_t)((lbo >> 4) & 0x3FFF) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3FFF) << 32) | ((uint64_t)1 << 46) | ((uint64_t)(layout & 7) << 61);
}
// instruction descriptor: tf32 x tf32 -> fp32, A MN-major, B K-major, M x N
__host__ __device__ constexpr uint32_t vt_idesc(int m, int n) {
  return (1u << 4) | (2u << 7) | (2u << 10) | (1u << 15) | ((uint32_t)(n >> 3) << 17) |
         ((uint32_t)(m >> 4) << 24);
}
// Bounded wait on an mbarrier phase.  try_wait lets the hardware suspend the
// thread until the phase completes (or a short time limit passes), so waiting
// warps do not take issue slots from the working ones; kVtPolls of them bound
// the wait.
__device__ __forceinline__ bool vt_wait(uint32_t mbar, uint32_t parity) {
  for (int it = 0; it < kVtPolls; ++it) {
    uint32_t done;
    asm volatile("{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
                 "selp.u32 %0, 1, 0, p;\n\t}"
                 : "=r"(done) : "r"(mbar), "r"(parity) : "memory");
    if (done) return true;
  }
  return false;
}
// The same wait, given up early once another role has stopped the CTA (*abort
// set): 1 = the phase completed, 0 = timed out, -1 = stopped.
__device__ __forceinline__ int vt_wait_ab(uint32_t mbar, uint32_t parity, const int *abort) {
  for (int it = 0; it < kVtPolls; ++it) {
    uint32_t done;
    asm volatile("{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
                 "selp.u32 %0, 1, 0, p;\n\t}"
                 : "=r"(done) : "r"(mbar), "r"(parity) : "memory");
    if (done) return 1;
    if ((it & 15) == 15 && *(const volatile int *)abort) return -1;
  }
  return 0;
}
__device__ __forceinline__ void vt_arrive(uint32_t mbar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(mbar) : "memory");
}
__device__ __forceinline__ void vt_arrive_tx(uint32_t mbar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(mbar), "r"(bytes) : "memory");
}
// 1D bulk copy global -> shared, completing `bytes` on mbar (16-byte multiples, aligned)
__device__ __forceinline__ void vt_bulk(uint32_t dst, const void *src, uint32_t bytes, uint32_t mbar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
               ::"r"(dst), "l"(src), "r"(bytes), "r"(mbar) : "memory");
}
// 4-byte cp.async global -> shared; vt_cp_arrive makes `mbar` wait for this
// thread's earlier cp.async copies (its pending count rises by one until they land)
__device__ __forceinline__ void vt_cp4(uint32_t dst, const void *src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void vt_cp_arrive(uint32_t mbar) {
  asm volatile("cp.async.mbarrier.arrive.shared.b64 [%0];" ::"r"(mbar) : "memory");
}
__device__ __forceinline__ void vt_tma2d(uint32_t dst, const void *map, int x, int y, uint32_t mbar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];"
      ::"r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(mbar) : "memory");
}
// the 128 threads of one consumer group only (named barrier `id`, 1 + group)
__device__ __forceinline__ void cons_sync(int id) { asm volatile("bar.sync %0, 128;" ::"r"(id) : "memory"); }
__device__ __forceinline__ bool cons_and(int id, bool p) {
  uint32_t r;
  asm volatile("{\n\t.reg .pred a, b;\n\tsetp.ne.u32 a, %2, 0;\n\t"
               "barrier.cta.red.and.pred b, %1, 128, a;\n\tselp.u32 %0, 1, 0, b;\n\t}"
               : "=r"(r) : "r"(id), "r"((uint32_t)p) : "memory");
  return r != 0;
}
__device__ __forceinline__ void mma_bf16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
template <int N>
__device__ __forceinline__ void tmem_ldn(uint32_t taddr, float (&v)[N]) {
  uint32_t r[N];
  if constexpr (N == 8) {
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
                   "=r"(r[7])
                 : "r"(taddr));
  } else {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
  }
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < N; ++i) v[i] = __uint_as_float(r[i]);
}

template <int VARIANT, bool TREE>
__global__ void __launch_bounds__(kVtMaxThreads, 1)
    verify_tc_kernel(const PoolView P, const __grid_constant__ RowBatch rows, const TokenIO io,
                     const __grid_constant__ TreeArg<TREE> tree, const __grid_constant__ StateMap smap,
                     int units, FastDiv hv_div, int NS, int G, int NST) {
  using KT = __nv_bfloat16;
  constexpr int D = 128, XS = kVtXS;
  constexpr bool DELTA = VARIANT == kGatedDelta, GATED = VARIANT != kPlain;
  using UT = typename std::conditional<DELTA, float, KT>::type;  // staged u (or v)
  constexpr int UROW = D * (int)sizeof(UT);                       // bytes of one u / v row
  constexpr int JMAX = DELTA ? 8 : 16;                            // most drafts per unit
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int T = io.T, LM = io.lmax;
  const int V = DELTA ? 2 * T : T, VP = (V + 7) & ~7;
  const int TP = (T + 3) & ~3;
  const int group = P.Hv / P.Hk;
  const int NSM = NST * G;  // small stages; unit k uses stage k % NSM
  const VtLayout lay = vt_layout(VARIANT, T, LM, NS, G, NST);
  const VtStage sl = vt_stage(VARIANT, T, LM);
  // warps: 4 G consumers, 4 G builders, the TMA warp, G MMA warps, G staging warps
  const int w_bld = 4 * G, w_tma = 8 * G, w_mma = w_tma + 1, w_stage = w_mma + G;

  extern __shared__ __align__(1024) uint8_t smem[];
  // per group g and buffer b (index 2 g + b): X built, weights built, product
  // done, accumulator and X buffer free again, weight buffer free again
  __shared__ uint64_t bar_full[kVtMaxStages], bar_empty[kVtMaxStages], bar_sfull[3 * kVtMaxGroups],
      bar_sempty[3 * kVtMaxGroups], bar_xready[2 * kVtMaxGroups], bar_wready[2 * kVtMaxGroups],
      bar_mmad[2 * kVtMaxGroups], bar_afree[2 * kVtMaxGroups], bar_wfree[2 * kVtMaxGroups];
  __shared__ uint32_t tmem_s;
  __shared__ int s_abort;
  __shared__ unsigned long long anc[kVtMaxGroups][kVtMaxL];  // draft trees: ancestor sets

  // barriers (8 bytes apart within each array) and stage memory
  auto bar = [](uint64_t *b, int i) { return su32(b) + 8u * (uint32_t)i; };
  auto stage_base = [&](int s) { return smem + lay.stage + (uint32_t)s * lay.stage_bytes; };
  auto group_base = [&](int g) { return smem + lay.grp + (uint32_t)g * lay.grp_bytes; };

  if (tid == 0) {
    // one arrival completes a phase, except where each consumer warp arrives
    auto init = [&](uint64_t *b, int n, uint32_t count) {
      for (int i = 0; i < n; ++i)
        asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar(b, i)), "r"(count));
    };
    init(bar_full, kVtMaxStages, 1);
    init(bar_empty, kVtMaxStages, 1);
    init(bar_sfull, 3 * kVtMaxGroups, 1);
    init(bar_sempty, 3 * kVtMaxGroups, kVtCons / 32);
    init(bar_xready, 2 * kVtMaxGroups, 1);
    init(bar_wready, 2 * kVtMaxGroups, 1);
    init(bar_mmad, 2 * kVtMaxGroups, 1);
    init(bar_afree, 2 * kVtMaxGroups, kVtCons / 32);
    init(bar_wfree, 2 * kVtMaxGroups, kVtCons / 32);
    s_abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;");
  }
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(su32(&tmem_s)),
                 "r"(kTmemCols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  const uint32_t tmem = tmem_s;
  auto stop = [&](int kind, int req, int value) {
    record_error(P.err, kind, req, value);
    s_abort = 1;
  };

  if (warp == w_tma) {
    // ------------------------------------------------------------- state tiles
    if (lane == 0) {
      uint32_t armed = 0u, phases = 0u;  // bit ks: stage armed; its phase parity
      for (int k = 0;; ++k) {
        const int u = blockIdx.x + k * gridDim.x;
        if (u >= units || *(volatile int *)&s_abort) break;
        const int ks = k % NS;
        if (k >= NS) {  // the tile of unit k - NS has been read
          const int w = vt_wait_ab(bar(bar_empty, ks), ((k / NS) - 1) & 1, &s_abort);
          if (w <= 0) {
            if (w == 0) stop(kErrTimeout, -1, 10);
            break;
          }
        }
        const int y = fast_div(u, hv_div), h = u - y * P.Hv;
        const int slot = rows.r[y].slot;  // the parameter block, read in place
        if (slot >= 0) {
          vt_arrive_tx(bar(bar_full, ks), kTileBytes);
          const uint32_t dst = su32(smem + lay.tile) + (uint32_t)ks * kTileBytes;
          const int y0 = (slot * P.Hv + h) * D;
#pragma unroll
          for (int g4 = 0; g4 < 4; ++g4) vt_tma2d(dst + g4 * 16384, &smap, 32 * g4, y0, bar(bar_full, ks));
        } else {
          vt_arrive(bar(bar_full, ks));  // no state: the consumers take S = 0
        }
        armed |= 1u << ks;
        phases = (phases & ~(1u << ks)) | ((uint32_t)((k / NS) & 1) << ks);
      }
      // tiles still in flight (only after a stop) land before the CTA exits
      if (*(volatile int *)&s_abort)
        for (int ks = 0; ks < NS; ++ks)
          if (armed & (1u << ks)) vt_wait(bar(bar_full, ks), (phases >> ks) & 1u);
    }
  } else if (warp >= w_stage) {
    // ------------------------------------------------------------- small operands
    // staging warp g stages the units k = g + G i of group g
    const int gs = warp - w_stage;
    uint32_t armed = 0u, phases = 0u;  // lane 0: bit s: stage armed; its phase parity
    for (int k = gs;; k += G) {
      const int u = blockIdx.x + k * gridDim.x;
      if (u >= units || __shfl_sync(kFull, *(volatile int *)&s_abort, 0)) break;
      const int s = k % NSM;
      uint8_t *st = stage_base(s);
      if (k >= NSM) {  // unit k - NSM has released this stage
        int w = lane == 0 ? vt_wait_ab(bar(bar_sempty, s), ((k / NSM) - 1) & 1, &s_abort) : 0;
        w = __shfl_sync(kFull, w, 0);
        if (w <= 0) {
          if (lane == 0 && w == 0) stop(kErrTimeout, -1, 11);
          break;
        }
      }
      const int y = fast_div(u, hv_div), h = u - y * P.Hv;
      const RowDesc &d = rows.r[y];
      const size_t b = (size_t)rows.row0 + y;
      const int hq = h / group, n = d.n, L = n + T;
      size_t *koff = reinterpret_cast<size_t *>(st + sl.koff);
      size_t *voff = reinterpret_cast<size_t *>(st + sl.voff);
      int anybad = 0;
      for (int i = lane; i < L; i += 32) {
        const int gr = buffer_row(P, d, i);
        anybad |= gr < 0;
        koff[i] = gr >= 0 ? kv_row(P, gr, hq, P.Hk) * D : 0;
        voff[i] = gr >= 0 ? kv_row(P, gr, h, P.Hv) : 0;
      }
      anybad = __any_sync(kFull, anybad);
      __syncwarp();  // every lane's offsets are visible to the others
      if (lane == 0) {
        int *meta = reinterpret_cast<int *>(st + sl.meta);
        meta[0] = y;
        meta[1] = h;
        meta[2] = n;
        meta[3] = anybad;
        meta[4] = d.slot;
        meta[5] = d.req;
      }
      const uint32_t sb = su32(st);
      if (!anybad) {
        // gates by 4-byte copies: buffered cumulative gates, draft log-gates, betas
        float *lg = reinterpret_cast<float *>(st + sl.lg);
        float *bt = reinterpret_cast<float *>(st + sl.bt);
        if (GATED)
          for (int i = lane; i < n; i += 32) vt_cp4(sb + sl.acum + 4 * i, P.gbuf + voff[i]);
        for (int j = lane; j < T; j += 32) {
          if (GATED && io.log_g)
            vt_cp4(sb + sl.lg + 4 * j, io.log_g + (b * T + j) * P.Hv + h);
          else
            lg[j] = 0.f;
          if (DELTA)
            vt_cp4(sb + sl.bt + 4 * j, io.beta + (b * T + j) * P.Hv + h);
          else
            bt[j] = 0.f;
        }
        vt_cp_arrive(bar(bar_sfull, s));  // the stage also waits for these lanes' copies
        // one bulk copy per row, issued by the row's lane: T draft q, T draft k, n
        // buffered keys, u / v rows, (delta rule) T draft v; the stage's barrier
        // expects their bytes
        const KT *qg = static_cast<const KT *>(io.q) + b * T * P.Hk * D;
        const KT *kg = static_cast<const KT *>(io.k) + b * T * P.Hk * D;
        const KT *vg = static_cast<const KT *>(io.v) + b * T * P.Hv * D;
        const int urows = DELTA ? n : L;
        const int r_q = T, r_k = r_q + T, r_b = r_k + n, r_u = r_b + urows;
        const int nrows = r_u + (DELTA ? T : 0);
        const uint32_t bytes = (uint32_t)(r_b + (DELTA ? T : 0)) * D * 2 + (uint32_t)urows * UROW;
        __syncwarp();
        if (lane == 0) vt_arrive_tx(bar(bar_sfull, s), bytes);
        __syncwarp();
        for (int r = lane; r < nrows; r += 32) {
          uint32_t dst, nb = D * 2;
          const void *src;
          if (r < r_q) {
            dst = sb + sl.xr + r * XS * 2;
            src = qg + ((size_t)r * P.Hk + hq) * D;
          } else if (r < r_k) {
            dst = sb + sl.kr + (n + r - r_q) * XS * 2;
            src = kg + ((size_t)(r - r_q) * P.Hk + hq) * D;
          } else if (r < r_b) {
            dst = sb + sl.kr + (r - r_k) * XS * 2;
            src = static_cast<const KT *>(P.kbuf) + koff[r - r_k];
          } else if (r < r_u) {
            const int i = r - r_b;
            dst = sb + sl.us + i * UROW;
            nb = UROW;
            if (DELTA)
              src = P.ubuf + voff[i] * D;
            else if (i < n)
              src = static_cast<const KT *>(P.vbuf) + voff[i] * D;
            else
              src = vg + ((size_t)(i - n) * P.Hv + h) * D;
          } else {
            dst = sb + sl.vs + (r - r_u) * D * 2;
            src = vg + ((size_t)(r - r_u) * P.Hv + h) * D;
          }
          vt_bulk(dst, src, nb, bar(bar_sfull, s));
        }
      } else {
        __syncwarp();
        if (lane == 0) vt_arrive(bar(bar_sfull, s));  // with a bad block id the unit is skipped
      }
      if (lane == 0) {
        armed |= 1u << s;
        phases = (phases & ~(1u << s)) | ((uint32_t)((k / NSM) & 1) << s);
      }
    }
    // after a stop, copies still in flight land before the CTA exits (without
    // one, the consumers have waited for every stage)
    if (lane == 0 && *(volatile int *)&s_abort)
      for (int s = gs; s < NSM; s += G)
        if (armed & (1u << s)) vt_wait(bar(bar_sfull, s), (phases >> s) & 1u);
  } else if (warp >= w_mma) {
    // ------------------------------------------------------------- products
    // MMA warp g: Y^T = S0^T X for the units k = g + G i of its group, each once
    // its tile has landed and its X is built, into accumulator i & 1 (TMEM
    // columns 32 g + 16 (i & 1) ...); the commits free the tile's stage and tell
    // the consumers
    const int g = warp - w_mma;
    if (lane == 0) {
      uint32_t pending = 0u, phases = 0u;  // bit b: a product in flight into accumulator b; its parity
      const uint32_t id = vt_idesc(128, VP);
      for (int i = 0;; ++i) {
        const int k = g + i * G;
        const int u = blockIdx.x + k * gridDim.x;
        if (u >= units || *(volatile int *)&s_abort) break;
        const int ks = k % NS, bb = i & 1;
        const int *meta = reinterpret_cast<const int *>(stage_base(k % NSM) + sl.meta);
        int w = vt_wait_ab(bar(bar_xready, 2 * g + bb), (i >> 1) & 1, &s_abort);
        if (w > 0) w = vt_wait_ab(bar(bar_full, ks), (k / NS) & 1, &s_abort);
        if (w <= 0) {
          if (w == 0) stop(kErrTimeout, -1, 30);
          break;
        }
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        if (meta[4] >= 0 && !meta[3]) {  // a state, and the unit's tokens located
          const uint32_t ta = su32(smem + lay.tile) + (uint32_t)ks * kTileBytes;
          const uint32_t xa = su32(group_base(g) + lay.xf) + (uint32_t)bb * lay.xbuf;
          const uint32_t dt = tmem + 32u * (uint32_t)g + 16u * (uint32_t)bb;
          // K steps of 8 rows: A advances 1024 bytes (8 rows of 128), B 256 (two
          // core matrices); the start-address field counts 16-byte units.  A
          // rolled loop keeps this warp's code small: unrolled, its instruction
          // fetches competed with the other roles' and issue took twice as long.
          uint64_t adesc = vt_desc(ta, 16384, 512, 1), bdesc = vt_desc(xa, 128, 4096, 0);
#pragma unroll 1
          for (int kk = 0; kk < 16; ++kk) {
            asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
                         "tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n\t}"
                         ::"r"(dt), "l"(adesc), "l"(bdesc), "r"(id), "r"((uint32_t)(kk > 0)));
            adesc += 1024 >> 4;
            bdesc += 256 >> 4;
          }
        }
        asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
                     ::"r"(bar(bar_empty, ks)) : "memory");
        asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
                     ::"r"(bar(bar_mmad, 2 * g + bb)) : "memory");
        pending |= 1u << bb;
        phases = (phases & ~(1u << bb)) | ((uint32_t)((i >> 1) & 1) << bb);
      }
      // products still in flight (only after a stop) finish before TMEM is released
      if (*(volatile int *)&s_abort)
        for (int bb = 0; bb < 2; ++bb)
          if (pending & (1u << bb)) vt_wait(bar(bar_mmad, 2 * g + bb), (phases >> bb) & 1u);
    }
  } else if (warp >= w_bld) {
    // ------------------------------------------------------------- builders
    // Builder group g, for the units k = g + G i of its group: X into X buffer
    // i & 1 once unit i - 2 has read its product (the MMA warp may then issue
    // the product); then, once unit i - 2 is finished, the drafts' cumulative
    // gates, e^{A_j} and the decay-weighted scores into weight buffer i & 1.
    const int g = (warp - w_bld) >> 2;
    const int bid = 1 + G + g;     // the group's named barrier
    const int c = tid & 127;
    const int qw = warp & 3;       // warp within the group
    const int gq = lane >> 2, t = lane & 3;
    uint8_t *gp = group_base(g);
    unsigned long long *ancg = anc[g];
    for (int i = 0;; ++i) {
      const int k = g + i * G;
      if (blockIdx.x + k * gridDim.x >= units) break;
      const int bb = i & 1, s = k % NSM;
      int w = 1;
      if (i >= 2) w = vt_wait_ab(bar(bar_afree, 2 * g + bb), ((i >> 1) - 1) & 1, &s_abort);
      if (w > 0) w = vt_wait_ab(bar(bar_sfull, s), (k / NSM) & 1, &s_abort);
      if (!cons_and(bid, w > 0)) {
        if (c == 0 && w == 0) stop(kErrTimeout, -1, 40);
        break;
      }
      uint8_t *st = stage_base(s);
      const int *meta = reinterpret_cast<const int *>(st + sl.meta);
      const int y = meta[0], n = meta[2], bad = meta[3], L = n + T;
      const KT *Xr = reinterpret_cast<const KT *>(st + sl.xr);
      const KT *Kr = reinterpret_cast<const KT *>(st + sl.kr);
      // K-major core matrices (8 vectors x 16 bytes), vector v at
      // (v / 8) * 4096 + (r / 4) * 128 + (v % 8) * 16; consecutive threads take
      // consecutive vectors of a core matrix, so a warp's stores cover 512
      // contiguous bytes
      if (!bad) {
        uint8_t *Xf = gp + lay.xf + (uint32_t)bb * lay.xbuf;
        for (int idx = c; idx < VP * 32; idx += kVtCons) {
          const int v = (idx & 7) | ((idx >> 8) << 3), c4 = (idx >> 3) & 31;
          if (v >= V) continue;
          const KT *src = v < T ? Xr + v * XS : Kr + (n + v - T) * XS;
          *reinterpret_cast<float4 *>(Xf + (v >> 3) * 4096 + c4 * 128 + (v & 7) * 16) = ld4(src + c4 * 4);
        }
      }
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // X for the tensor cores
      cons_sync(bid);
      if (c == 0) vt_arrive(bar(bar_xready, 2 * g + bb));

      // weight buffer bb: free once unit i - 2 is finished
      w = 1;
      if (i >= 2) w = vt_wait_ab(bar(bar_wfree, 2 * g + bb), ((i >> 1) - 1) & 1, &s_abort);
      if (!cons_and(bid, w > 0)) {
        if (c == 0 && w == 0) stop(kErrTimeout, -1, 41);
        break;
      }
      float *Acum = reinterpret_cast<float *>(st + sl.acum);
      const float *lgs = reinterpret_cast<const float *>(st + sl.lg);
      uint8_t *wb = gp + (uint32_t)bb * lay.wbuf;
      float *sw = reinterpret_cast<float *>(wb + lay.sw);
      float *cw = reinterpret_cast<float *>(wb + lay.cw);
      float *eA = reinterpret_cast<float *>(wb + lay.ea);
      // cumulative gates of the drafts (the group's first warp): along each
      // draft's path for trees, else a prefix over the chain
      if (qw == 0 && !bad) {
        const float A_prev = GATED && n > 0 ? Acum[n - 1] : 0.f;
        if constexpr (TREE) {
          for (int j = lane; j < T; j += 32) Acum[n + j] = GATED ? lgs[j] : 0.f;
          __syncwarp();
          if (lane == 0) tree_walk(tree.p[y], T, GATED ? A_prev : 0.f, GATED ? Acum + n : nullptr, ancg);
          __syncwarp();
          for (int j = lane; j < T; j += 32) eA[j] = GATED ? expf(Acum[n + j]) : 1.f;
        } else {
          for (int j = lane; j < T; j += 32) {
            float a = 0.f;
            for (int i2 = 0; i2 <= j; ++i2) a += lgs[i2];
            a += A_prev;
            if (GATED) Acum[n + j] = a;
            eA[j] = GATED ? expf(a) : 1.f;
          }
        }
        if (!GATED)
          for (int j = lane; j < L; j += 32) Acum[j] = 0.f;
      }
      cons_sync(bid);  // the gates (and tree paths) for the score warps

      // score dots q_j.k_l, k_j.k_l as one mma.sync pass (warps 0, 1: key tiles
      // 0, 1); the lanes holding them write the decay-weighted scores,
      // token-major: sw[l][j] = scale e^{A_{n+j}-A_l} q_j.k_l (l <= n+j),
      // cw[l][j] = e^{A_{n+j}-A_l} k_{n+j}.k_l (l < n+j); a tree draft sees the
      // buffer and its own path only
      const int LP = (L + 7) >> 3;
      if (!bad && qw < LP) {
        auto arow = [&](int v) -> const KT * {
          return v < T ? Xr + v * XS : (v < V ? Kr + (n + v - T) * XS : nullptr);
        };
        const KT *a0 = arow(gq), *a1 = arow(gq + 8);
        const KT *kr = Kr + (qw * 8 + gq) * XS;
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int ks2 = 0; ks2 < 8; ++ks2) {
          const int o = ks2 * 16 + 2 * t;
          const uint32_t a[4] = {a0 ? *reinterpret_cast<const uint32_t *>(a0 + o) : 0u,
                                 a1 ? *reinterpret_cast<const uint32_t *>(a1 + o) : 0u,
                                 a0 ? *reinterpret_cast<const uint32_t *>(a0 + o + 8) : 0u,
                                 a1 ? *reinterpret_cast<const uint32_t *>(a1 + o + 8) : 0u};
          mma_bf16(acc, a, *reinterpret_cast<const uint32_t *>(kr + o),
                   *reinterpret_cast<const uint32_t *>(kr + o + 8));
        }
        // acc[2 hi + x]: vector gq + 8 hi against key l = tile * 8 + 2t + x
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int v = gq + 8 * (e >> 1), l = qw * 8 + 2 * t + (e & 1);
          if (v >= V || l >= LM) continue;
          const bool isq = v < T;
          const int j = isq ? v : v - T;
          float wgt = 0.f;
          const bool inside = isq ? l <= n + j : l < n + j;
          const bool on_path = !TREE || l < n || ((ancg[j] >> (l - n)) & 1ull);
          if (l < L && inside && on_path) wgt = (GATED ? expf(Acum[n + j] - Acum[l]) : 1.f) * acc[e];
          if (isq)
            sw[l * TP + j] = P.scale * wgt;
          else
            cw[l * TP + j] = wgt;
        }
      }
      cons_sync(bid);
      if (c == 0) vt_arrive(bar(bar_wready, 2 * g + bb));
    }
  } else {
    // ------------------------------------------------------------- consumers
    // Consumer group g, for the units k = g + G i of its group: once the weights
    // and the product are ready, this column of Y^T from accumulator i & 1 (the
    // accumulator is then released), the forward substitution over the drafts,
    // the outputs and the drafts' buffer entries; then the stage and the weight
    // buffer are released.
    const int g = warp >> 2;
    const int bid = 1 + g;     // the group's named barrier
    const int c = tid & 127;   // state column, TMEM lane
    const int qw = warp & 3;   // warp within the group
    const uint32_t my_tmem = tmem + 32u * (uint32_t)g + ((uint32_t)(qw * 32) << 16);
    uint8_t *gp = group_base(g);
    for (int i = 0;; ++i) {
      const int k = g + i * G;
      if (blockIdx.x + k * gridDim.x >= units) break;
      const int bb = i & 1, s = k % NSM;
      int w = vt_wait_ab(bar(bar_wready, 2 * g + bb), (i >> 1) & 1, &s_abort);
      if (w > 0) w = vt_wait_ab(bar(bar_sfull, s), (k / NSM) & 1, &s_abort);
      if (w > 0) w = vt_wait_ab(bar(bar_mmad, 2 * g + bb), (i >> 1) & 1, &s_abort);
      const bool go = cons_and(bid, w > 0);  // uniform over the group
      asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
      if (!go) {
        if (c == 0 && w == 0) stop(kErrTimeout, -1, 50);
        break;
      }
      const uint8_t *st = stage_base(s);
      const int *meta = reinterpret_cast<const int *>(st + sl.meta);
      const int y = meta[0], h = meta[1], n = meta[2], bad = meta[3], slot = meta[4];
      const size_t b = (size_t)rows.row0 + y;
      const bool has_state = slot >= 0 && !bad;
      const KT *Kr = reinterpret_cast<const KT *>(st + sl.kr);
      const UT *us = reinterpret_cast<const UT *>(st + sl.us);
      const float *Acum = reinterpret_cast<const float *>(st + sl.acum);
      const float *bts = reinterpret_cast<const float *>(st + sl.bt);
      const size_t *koff = reinterpret_cast<const size_t *>(st + sl.koff);
      const size_t *voff = reinterpret_cast<const size_t *>(st + sl.voff);
      const uint8_t *wb = gp + (uint32_t)bb * lay.wbuf;
      const float *sw = reinterpret_cast<const float *>(wb + lay.sw);
      const float *cw = reinterpret_cast<const float *>(wb + lay.cw);
      const float *eA = reinterpret_cast<const float *>(wb + lay.ea);

      float po[JMAX], pc[DELTA ? JMAX : 1];
      if (has_state) {
        tmem_ldn<JMAX>(my_tmem + 16u * (uint32_t)bb, po);
        if constexpr (DELTA) tmem_ldn<JMAX>(my_tmem + 16u * (uint32_t)bb + (uint32_t)T, pc);
      } else {
#pragma unroll
        for (int j = 0; j < JMAX; ++j) {
          po[j] = 0.f;
          if constexpr (DELTA) pc[j] = 0.f;
        }
      }
      // this warp is done with accumulator bb (and so with X buffer bb): the
      // builders and the tensor cores may take unit i + 2
      asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
      __syncwarp();
      if (lane == 0) vt_arrive(bar(bar_afree, 2 * g + bb));

      // per draft in order: u (the delta rule's forward substitution) and o,
      // and the drafts' buffer entries for this column
      if (!bad) {
#pragma unroll
        for (int j = 0; j < JMAX; ++j) {
          if (j < T) {
            po[j] *= eA[j] * P.scale;
            if constexpr (DELTA) pc[j] *= eA[j];
          }
        }
        // the buffered tokens, for all drafts at once
        for (int l = 0; l < n; ++l) {
          const float ul = to_float(us[l * D + c]);
#pragma unroll
          for (int j4 = 0; j4 < JMAX; j4 += 4) {
            if (j4 >= T) break;
            const float4 wq = *reinterpret_cast<const float4 *>(sw + l * TP + j4);
            po[j4] = fmaf(wq.x, ul, po[j4]);
            po[j4 + 1] = fmaf(wq.y, ul, po[j4 + 1]);
            po[j4 + 2] = fmaf(wq.z, ul, po[j4 + 2]);
            po[j4 + 3] = fmaf(wq.w, ul, po[j4 + 3]);
            if constexpr (DELTA) {
              const float4 wk = *reinterpret_cast<const float4 *>(cw + l * TP + j4);
              pc[j4] = fmaf(wk.x, ul, pc[j4]);
              pc[j4 + 1] = fmaf(wk.y, ul, pc[j4 + 1]);
              pc[j4 + 2] = fmaf(wk.z, ul, pc[j4 + 2]);
              pc[j4 + 3] = fmaf(wk.w, ul, pc[j4 + 3]);
            }
          }
        }
        // the drafts in order; each one's u goes into the later drafts' sums
        const KT *vdr = DELTA ? reinterpret_cast<const KT *>(st + sl.vs)
                              : reinterpret_cast<const KT *>(us) + (size_t)n * D;
        const bool keys = h % group == 0;
#pragma unroll
        for (int j = 0; j < JMAX; ++j) {
          if (j >= T) break;
          const int tp = n + j;
          const KT vraw = vdr[j * D + c];
          float ut = to_float(vraw);
          if constexpr (DELTA) ut = bts[j] * (ut - pc[j]);
          const float *swr = sw + tp * TP;
          const float *cwr = cw + tp * TP;
          __stcs(io.o + ((b * T + j) * P.Hv + h) * D + c, fmaf(swr[j], ut, po[j]));
#pragma unroll
          for (int j2 = j + 1; j2 < JMAX; ++j2) {
            if (j2 < T) {
              po[j2] = fmaf(swr[j2], ut, po[j2]);
              if constexpr (DELTA) pc[j2] = fmaf(cwr[j2], ut, pc[j2]);
            }
          }
          const size_t vo = voff[tp];
          static_cast<KT *>(P.vbuf)[vo * D + c] = vraw;
          if constexpr (DELTA) P.ubuf[vo * D + c] = ut;
          if (keys) static_cast<KT *>(P.kbuf)[koff[tp] + c] = Kr[tp * XS + c];
          if (c == j) {
            P.gbuf[vo] = Acum[tp];  // cumulative since the last fold
            P.bbuf[vo] = DELTA ? bts[j] : 0.f;
          }
        }
      }
      // this warp is done with the stage and weight buffer bb (the stage is
      // refilled by copies that need no proxy fence after generic reads)
      __syncwarp();
      if (lane == 0) {
        vt_arrive(bar(bar_sempty, s));
        vt_arrive(bar(bar_wfree, 2 * g + bb));
      }
    }
  }

  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  if (warp == 0) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols));
}

template <int VARIANT, bool TREE>
cudaError_t run_verify_tc(const PoolView &P, const RowBatch &rows, const TokenIO &io,
                          const TreeArg<TREE> &tree, const StateMap &smap, cudaStream_t stream) {
  int groups = 0, ns = 0, nst = 0;
  if (!vt_shape(VARIANT, io.T, io.lmax, groups, ns, nst)) return kUnsupported;
  const size_t smem = vt_layout(VARIANT, io.T, io.lmax, ns, groups, nst).total;
  const int threads = groups * kVtGroupThreads + 32;
  const void *fn = (const void *)verify_tc_kernel<VARIANT, TREE>;
  int cap = 0;
  cudaError_t e = resident_ctas(fn, threads, smem, &cap);
  if (e != cudaSuccess) return e;
  if (cap <= 0) return kUnsupported;
  const int units = rows.count * P.Hv;
  const int grid = units < cap ? units : cap;
  verify_tc_kernel<VARIANT, TREE><<<grid, threads, smem, stream>>>(
      P, rows, io, tree, smap, units, make_fastdiv((uint32_t)P.Hv), ns, groups, nst);
  return cudaGetLastError();
}

}  // namespace

bool verify_tc_fits(int variant, int T, int lmax) {
  const int V = variant == kGatedDelta ? 2 * T : T;
  if (T < 1 || V > kVtMaxV || lmax > kVtMaxL) return false;
  int groups = 0, ns = 0, nst = 0;
  return vt_shape(variant, T, lmax, groups, ns, nst);
}

template <bool TREE>
cudaError_t launch_verify_tc(const PoolView &P, const RowBatch &rows, const TokenIO &io, int variant,
                             const TreeArg<TREE> &tree, const StateMap &smap, cudaStream_t stream) {
  switch (variant) {
    case kPlain: return run_verify_tc<kPlain, TREE>(P, rows, io, tree, smap, stream);
    case kGated: return run_verify_tc<kGated, TREE>(P, rows, io, tree, smap, stream);
    case kGatedDelta: return run_verify_tc<kGatedDelta, TREE>(P, rows, io, tree, smap, stream);
  }
  return kUnsupported;
}
template cudaError_t launch_verify_tc<false>(const PoolView &, const RowBatch &, const TokenIO &, int,
                                             const TreeArg<false> &, const StateMap &, cudaStream_t);
template cudaError_t launch_verify_tc<true>(const PoolView &, const RowBatch &, const TokenIO &, int,
                                            const TreeArg<true> &, const StateMap &, cudaStream_t);

}  // namespace kvb
