// Internal types shared by the host library (kvb_host.cpp) and the kernels.
// Plain structs only: this header is included by both g++ and nvcc sources.
#pragma once

#include <cstddef>
#include <cstdint>

#include <cuda_runtime_api.h>

#include "kvb.h"

namespace kvb {

// Most batch rows one launch carries in its parameter block; longer batches
// are split into several launches by the host library.
constexpr int kMaxRows = 256;
// Leading block ids of each request carried in its row descriptor, so the
// kernels find the first kRowBlocks * block_size buffer slots without a
// dependent load of the block table.
constexpr int kRowBlocks = 8;

// Device view of a pool: raw pointers into the caller's regions plus shapes.
struct PoolView {
  float *state;       // [slots][Hv][dk][dv]
  void *kbuf;         // [rows][Hk][dk]  kv dtype
  void *vbuf;         // [rows][Hv][dv]  kv dtype
  float *ubuf;        // [rows][Hv][dv]  (gated delta) pseudo-values
  float *gbuf;        // [rows][Hv]      log-gates
  float *bbuf;        // [rows][Hv]      beta
  const int32_t *table;  // [max_requests][max_blocks]
  int32_t *dlen;      // [max_requests] device-side lengths
  int32_t *err;       // [4] error word: kind, request, value, count
  int Hk, Hv, bs, max_blocks, num_blocks;
  float scale;
  int bs_shift;  // log2(bs) when bs is a power of two, else -1
};

// Division by a fixed divisor d >= 1 for 0 <= n < 2^31 as a multiply and a
// shift: n / d = (umulhi(n, m) + n) >> s with s = ceil(log2 d) and
// m = floor(2^32 (2^s - d) / d) + 1 (the round-up method of Granlund and
// Montgomery, "Division by invariant integers using multiplication").
struct FastDiv {
  uint32_t m;
  int s;
};
inline FastDiv make_fastdiv(uint32_t d) {
  int s = 0;
  while ((1ull << s) < d) ++s;
  const uint64_t m = ((((uint64_t)1 << s) - d) << 32) / d + 1;
  return FastDiv{(uint32_t)m, s};
}

// One batch row: which request, its buffer length before this call, its
// state slot (-1 = none), flags, and its first block ids (-1 past its table).
struct RowDesc {
  int32_t req, n, slot, flags;
  int32_t blk[kRowBlocks];
};
constexpr int32_t kFlagFlush = 1;  // decode: fold the buffer (incl. this token) into S
constexpr int32_t kFlagFromZero = 2;  // flush: start from S = 0 instead of the slot's state

// Rows of one launch, passed by value in the kernel parameter block.
struct RowBatch {
  int32_t count;  // rows in this launch (== gridDim.y)
  int32_t row0;   // index of rows[0] in the caller's input arrays
  RowDesc r[kMaxRows];
};

// Buffered tokens the persistent decode (decode_stream.cu) stages per item;
// launches whose rows hold more take decode_kernel.
constexpr int kStageTok = 8;

// Draft trees of one launch, carried in the kernel parameter block: for row i
// of the launch and draft j, p[i][j] is the parent draft (-1: the last
// accepted token), always < j.  Accept reuses it for the accepted path (the
// draft index at each path position).  Chain launches pass the empty form.
constexpr int kTreeRows = kMaxRows;  // rows per tree launch (16 KB of parents: within the 32 KB parameter block)
template <bool TREE>
struct TreeArg {};
template <>
struct TreeArg<true> {
  int8_t p[kTreeRows][KVB_MAX_DRAFTS];
};

// A TMA tensor map (the driver's CUtensorMap: 128 bytes, 64-byte aligned) of a
// pool's state region viewed as a 2D fp32 array {d_v columns, slots * Hv * d_k
// rows}, copied in {32 x 128} boxes with the 128-byte swizzle of 32-byte atoms:
// the layout the tensor cores read as an MN-major tf32 operand.
struct alignas(64) StateMap {
  uint64_t opaque[16];
};
// Encode the map of `rows` state rows of 128 fp32 at `state` (d = 128 pools).
cudaError_t encode_state_map(StateMap *out, float *state, uint64_t rows);

// Input / output pointers of a decode or verify launch (device).
struct TokenIO {
  const void *q, *k, *v;  // kv dtype
  const float *log_g, *beta;
  float *o;
  int T;     // tokens per row (1 for decode)
  int lmax;  // most tokens any row of the launch stages in shared memory
  int nrows = 0;  // rows of the token buffers (prefill: the whole batch), for tensor maps
};

// TMA tensor maps of a prefill's token buffers at d = 128, each viewed as {128
// elements, heads, nrows * T tokens}: q and k (bf16) copied in {64, 1, 64}
// boxes with the 128-byte swizzle (the K-major layout the tensor cores read), v
// (bf16) in {128, 1, 64} boxes as plain rows, o (fp32, Hv heads) written in
// {128, 1, 64} boxes.  Encoding fails (cudaErrorNotSupported) for buffers that
// are not 16-byte aligned or too many tokens for the coordinates.
struct alignas(64) TmaMap {
  uint64_t opaque[16];
};
struct PrefillMaps {
  TmaMap q, k, v, o;
};
cudaError_t encode_prefill_maps(PrefillMaps *out, const TokenIO &io, int Hk, int Hv);

// kErrTimeout: a bounded wait on the tensor cores gave up (the launch's outputs
// and states are invalid); kErrTimeoutDrain: the wait that follows, for the
// products still in flight before TMEM is released, gave up as well.
enum ErrKind : int32_t { kErrNone = 0, kErrBlockRange = 1, kErrTimeout = 2, kErrTimeoutDrain = 3 };

// Per-device launch set-up (device_setup.cpp).  A kernel's dynamic
// shared-memory limit and its occupancy belong to one device, so both helpers
// act on the current device and cache per (device, kernel); they are safe to
// call from several host threads.
// Raise `kernel`'s dynamic shared-memory limit on the current device to >= bytes.
cudaError_t ensure_smem(const void *kernel, size_t bytes);
// CTAs of `kernel` (threads, dynamic smem) resident on the whole current device
// (SM count x CTAs per SM), the grid of a persistent launch; 0 if none fit.
cudaError_t resident_ctas(const void *kernel, int threads, size_t smem, int *out);
// SM count of the current device.
cudaError_t sm_count(int *out);
// Poll bound of the first completion wait of every tensor-core prefill CTA
// (0 = the default bound); set by kvb_set_prefill_wait_limit.
int prefill_first_wait_polls();
void set_prefill_first_wait_polls(int polls);

// Launchers (kernels.cu).  `dtype` is KVB_F32 / KVB_BF16; `d` is d_k == d_v.
// Return cudaSuccess or the launch error; kUnsupported for a missing instance.
constexpr cudaError_t kUnsupported = cudaErrorNotSupported;

// nmax: the largest buffer length of any row; flush_len: the most tokens any
// row folds (0 if none).
cudaError_t launch_decode(const PoolView &P, const RowBatch &rows, const TokenIO &io, int variant,
                          int dtype, int d, bool recurrent, int flush_len, int nmax,
                          cudaStream_t stream);
cudaError_t launch_short(const PoolView &P, const RowBatch &rows, const TokenIO &io, int variant,
                         int dtype, int d, cudaStream_t stream);
// smap: the pool's state map, or nullptr when it has none (the tensor-core
// verify then falls back to the mma.sync kernel).
cudaError_t launch_verify(const PoolView &P, const RowBatch &rows, const TokenIO &io, int variant,
                          int dtype, int d, int max_len, cudaStream_t stream,
                          const TreeArg<true> *tree = nullptr, const StateMap *smap = nullptr);
// The tcgen05 / TMA verify (bf16, d = 128): whether a launch of T drafts and
// chunks of at most lmax tokens fits it, and the launch itself.
bool verify_tc_fits(int variant, int T, int lmax);
template <bool TREE>
cudaError_t launch_verify_tc(const PoolView &P, const RowBatch &rows, const TokenIO &io, int variant,
                             const TreeArg<TREE> &tree, const StateMap &smap, cudaStream_t stream);
// Move each row's accepted draft path to the front of its draft slots: row i
// (RowDesc.n = length before the drafts, RowDesc.flags = path length) copies
// the entry of draft path.p[i][l] into slot n + l, l in path order.
cudaError_t launch_tree_compact(const PoolView &P, const RowBatch &rows,
                                const TreeArg<true> &path, int variant, int dtype, int d,
                                cudaStream_t stream);
cudaError_t launch_flush(const PoolView &P, const RowBatch &rows, int variant, int dtype, int d,
                         int max_len, cudaStream_t stream);
cudaError_t launch_verify_tempstate(const PoolView &P, const RowBatch &rows, const TokenIO &io,
                                    int variant, int dtype, int d, float *temp,
                                    cudaStream_t stream);
cudaError_t launch_accept_tempstate(const PoolView &P, const RowBatch &rows, const float *temp,
                                    int T, int d, cudaStream_t stream);
// The same two launches with the temporary states in the library's fixed
// device array (kvb_verify_tempstate_static).
cudaError_t launch_verify_tempstate_static(const PoolView &P, const RowBatch &rows,
                                           const TokenIO &io, int variant, int dtype, int d,
                                           cudaStream_t stream);
cudaError_t launch_accept_tempstate_static(const PoolView &P, const RowBatch &rows, int T, int d,
                                           cudaStream_t stream);
// Buffered decode (d = 128, at most kStageTok buffered tokens per row) as a
// persistent pipelined kernel.
cudaError_t launch_decode_stream(const PoolView &P, const RowBatch &rows, const TokenIO &io,
                                 int variant, int dtype, cudaStream_t stream);
// Whether a launch of `units` (row, value head) pairs is large enough for it.
bool decode_stream_pays(int units, int variant, int dtype);
// The fold (kvb_flush and accepts that fill the buffer) with the same streaming,
// for rows of at most kStageTok tokens at d = 128, and its size rule.
bool flush_stream_pays(int units, int variant, int dtype);
cudaError_t launch_flush_stream(const PoolView &P, const RowBatch &rows, int variant, int dtype,
                                cudaStream_t stream);
// Chunked prefill on tcgen05 / TMEM (bf16 inputs, d = 128).
cudaError_t launch_prefill_tc(const PoolView &P, const RowBatch &rows, const TokenIO &io,
                              const PrefillMaps &maps, int variant, cudaStream_t stream);
// Chunked prefill of rows.r[i].n prompt tokens per row (io.T = padded length).
cudaError_t launch_prefill(const PoolView &P, const RowBatch &rows, const TokenIO &io,
                           int variant, int dtype, int d, cudaStream_t stream);
cudaError_t launch_set_lengths(const PoolView &P, const RowBatch &rows, cudaStream_t stream);
cudaError_t launch_copy_probe(const void *src, void *dst, size_t bytes, cudaStream_t stream);

}  // namespace kvb
