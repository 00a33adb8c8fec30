/*
 * kvb.h - C ABI of libkvb, KV-buffered linear-attention decoding on GB300 (sm_103a).
 *
 * The method is KVBuffer ("KVBuffer: IO-aware Serving for Linear Attention",
 * Zou and Zhong).  A linear-attention request keeps a fixed-size state S in a
 * state slot; recent keys and values are kept in a KV buffer made of
 * fixed-size blocks; decoding reads S together with the buffered KVs and
 * does not write S; when the buffer is full, all buffered KVs are folded
 * into S in one update and S is written back to its slot (Figure 1 and its
 * caption).  The same buffer verifies speculative draft tokens without
 * temporary states (Figure 2), and short-context requests are served from
 * buffered KVs alone, with no state (abstract).
 *
 * Recurrence (the pages print none; standard forms of the cited works):
 *   plain        S_t = S_{t-1} + k_t v_t^T
 *   gated        S_t = g_t S_{t-1} + k_t v_t^T,                 g_t = exp(log_g_t)
 *   gated delta  S_t = g_t (I - beta_t k_t k_t^T) S_{t-1} + beta_t k_t v_t^T
 *   output       o_t = scale * S_t^T q_t   (after the current token's update)
 * Every entry point computes exactly these outputs (up to fp32 rounding);
 * only the time at which S is updated, and how often it crosses HBM, differ.
 *
 * Conventions for every call:
 *  - All device memory (state, buffer, metadata, inputs, outputs) is allocated
 *    by the caller and borrowed; no call allocates device memory.  The one
 *    piece of device memory the library holds itself is the fixed
 *    KVB_STATIC_TEMP_BYTES array of kvb_verify_tempstate_static, a file-scope
 *    device array that every GPU loading the library keeps until the process
 *    exits.  The library owns the small host-side pool handle.
 *  - A process may drive several GPUs (one pool per GPU): every call works on
 *    the current device, and per-device launch set-up is done once per device.
 *  - Pointers named q, k, v, log_g, beta, o are DEVICE pointers, contiguous,
 *    16-byte aligned.  Pointers named req_ids, block_ids, n_accepted and
 *    host_out are HOST pointers.
 *  - Calls are asynchronous on `stream` (a cudaStream_t; NULL = legacy default
 *    stream) unless stated otherwise.  Argument errors are detected on the
 *    host before anything is launched and leave the pool unchanged.
 *  - Return value: KVB_OK (0) or a negative KVB_E_* code; kvb_strerror()
 *    names it.  Nothing traps: a check that fails on the device records an
 *    error word, which kvb_get_error() reports.
 *  - One pool must not be used from two host threads at once.
 *  - Layer shapes: d_k, d_v in {64, 128} with d_k == d_v; n_v_heads a multiple
 *    of n_qk_heads (value head h uses q/k head h / (n_v_heads / n_qk_heads)).
 */
#ifndef KVB_H
#define KVB_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *kvb_stream_t; /* same type as cudaStream_t */
typedef struct kvb_pool kvb_pool;         /* opaque host-side handle */

/* status codes */
#define KVB_OK 0
#define KVB_E_ARG (-1)         /* bad argument: null/misaligned pointer, bad size, duplicate request */
#define KVB_E_CAPACITY (-2)    /* the request's buffer cannot hold the new tokens */
#define KVB_E_RANGE (-3)       /* request, block or state-slot id out of range */
#define KVB_E_STATE (-4)       /* call does not fit the request's kind or phase */
#define KVB_E_CUDA (-5)        /* a CUDA runtime call failed (launch, memset, copy) */
#define KVB_E_DEVICE (-6)      /* a device-side check recorded an error (kvb_get_error) */
#define KVB_E_UNSUPPORTED (-7) /* shape or dtype not built into this library */

/* variants */
#define KVB_PLAIN 0
#define KVB_GATED 1
#define KVB_GATED_DELTA 2

/* dtypes of q, k, v and of the buffered K/V (the state and outputs are always fp32) */
#define KVB_F32 0
#define KVB_BF16 1

#define KVB_MAX_CAPACITY 64 /* largest buffer (slots) one request may own */
#define KVB_MAX_DRAFTS 64   /* largest T of one kvb_verify call */

typedef struct kvb_config {
  int32_t variant;            /* KVB_PLAIN | KVB_GATED | KVB_GATED_DELTA */
  int32_t kv_dtype;           /* KVB_F32 | KVB_BF16 */
  int32_t n_qk_heads;         /* H_k */
  int32_t n_v_heads;          /* H_v, a multiple of H_k */
  int32_t d_k;                /* key dim, 64 or 128 */
  int32_t d_v;                /* value dim, == d_k */
  int32_t m;                  /* buffer size: flush when a request holds m tokens;
                                 0 = recurrent decoding (S read and written every token) */
  int32_t block_size;         /* slots per buffer block (Figure 1 uses 6) */
  int32_t num_blocks;         /* blocks in the shared buffer pool */
  int32_t num_state_slots;    /* slots in the state pool */
  int32_t max_requests;       /* request ids are 0 .. max_requests-1 */
  int32_t max_blocks_per_req; /* width of the block table */
  float scale;                /* multiplies q (1.0 for pre-scaled inputs) */
} kvb_config;

/*
 * Pool memory, three caller-allocated device regions (each 256-byte aligned):
 *  state: fp32 [num_state_slots][n_v_heads][d_k][d_v], row-major (d_v fastest).
 *         The caller may read or write a slot's state directly between calls
 *         (e.g. to load a prefilled state); byte offset of (slot, head) is
 *         ((slot * n_v_heads + head) * d_k * d_v) * 4.
 *  kv:    the block-partitioned buffer; offsets of its parts in kvb_layout.
 *         Token slot p of a request lives in block table[p / block_size] at
 *         position p % block_size.  Within a block, each head's positions are
 *         contiguous (so a request's buffered tokens for one head form one
 *         contiguous run per block):
 *           K    [block][n_qk_heads][block_size][d_k]  kv dtype
 *           V    [block][n_v_heads][block_size][d_v]   kv dtype
 *           U    [block][n_v_heads][block_size][d_v]   fp32, gated delta only:
 *                the token's pseudo-value (the delta-rule value correction,
 *                computed once when the token enters the buffer)
 *           LOGG [block][n_v_heads][block_size]        fp32 cumulative log-gate
 *                A_i = a_1 + ... + a_i of the buffer's tokens since the last
 *                fold (0 for plain)
 *           BETA [block][n_v_heads][block_size]        fp32 (gated delta only)
 *  meta:  block tables, device lengths and the error word (layout private).
 */
typedef struct kvb_layout {
  size_t state_bytes, kv_bytes, meta_bytes;
  size_t k_off, v_off, u_off, logg_off, beta_off; /* byte offsets inside kv */
  size_t state_slot_stride;                       /* bytes per state slot */
} kvb_layout;

/* Sizes and offsets of the three regions for `cfg`.  Host only.
   KVB_E_ARG / KVB_E_UNSUPPORTED for an invalid or unbuilt configuration. */
int kvb_pool_layout(const kvb_config *cfg, kvb_layout *out);

/* Create a pool handle over caller memory (sizes from kvb_pool_layout).
   Zeroes the meta region (synchronously); leaves state and kv untouched.
   All requests start inactive.  *out is set only on success. */
int kvb_alloc_pool(const kvb_config *cfg, void *state_mem, void *kv_mem, void *meta_mem,
                   kvb_pool **out);

/* Destroy the host handle.  Does not free the caller's device memory.
   The caller synchronizes any stream still using the pool first. */
int kvb_free_pool(kvb_pool *pool);

/* Admit request `req` (Figure 1: a state slot per request, a list of buffer
   blocks per request).  state_slot = -1 admits a short-context request with
   no state (abstract: outputs computed directly from buffered KVs).
   block_ids: host array of n_blocks ids; its capacity is n_blocks *
   block_size slots (at most KVB_MAX_CAPACITY).  The buffer starts empty.
   Errors: KVB_E_RANGE for ids out of range or a state slot / block already
   owned by another active request; KVB_E_STATE if `req` is active.
   Writes the block table row with an async copy on `stream`. */
int kvb_set_request(kvb_pool *pool, int32_t req, int32_t state_slot, int32_t n_blocks,
                    const int32_t *block_ids, kvb_stream_t stream);

/* Retire request `req`: its state slot and blocks become free.  Host only. */
int kvb_release_request(kvb_pool *pool, int32_t req);

/* One decode step for B long-context requests (Figure 1: load the state along
   with the buffered KVs, compute the output; when the buffer is full, update
   the state with all buffered KVs and write it back to the slot).
   Row b of the inputs belongs to request req_ids[b] (host array, no
   duplicates; every request must own a state slot, else KVB_E_STATE).
     q, k:  [B][n_qk_heads][d_k]  kv dtype
     v:     [B][n_v_heads][d_v]   kv dtype
     log_g: [B][n_v_heads] fp32   required for gated, optional (NULL = 0) for
                                  gated delta, ignored for plain
     beta:  [B][n_v_heads] fp32   required for gated delta, else ignored
     o:     [B][n_v_heads][d_v] fp32 (written)
   The token is appended to the buffer at slot n (n = the request's length).
   With auto_flush != 0 and m > 0, a request whose buffer reaches m tokens
   folds all of them into its state in the same launch and its length becomes
   0.  With m == 0 this is recurrent decoding: no buffer, S updated in place.
   KVB_E_CAPACITY if a buffer is already full. */
int kvb_decode(kvb_pool *pool, int32_t B, const int32_t *req_ids, const void *q, const void *k,
               const void *v, const float *log_g, const float *beta, float *o, int32_t auto_flush,
               kvb_stream_t stream);

/* Short-context decode (abstract: compute outputs directly from buffered
   keys and values, without creating or updating the state).  Same arguments
   as kvb_decode without auto_flush; every request must be stateless
   (state_slot = -1, else KVB_E_STATE).  The output is the recurrence from
   S = 0 over the request's whole history, which must fit its buffer
   (KVB_E_CAPACITY otherwise). */
int kvb_short_ctx(kvb_pool *pool, int32_t B, const int32_t *req_ids, const void *q, const void *k,
                  const void *v, const float *log_g, const float *beta, float *o,
                  kvb_stream_t stream);

/* Fold all buffered tokens of each listed request into its state, write the
   state back and empty the buffer (Figure 1, deferred state update).
   Requests with an empty buffer are skipped; stateless requests give
   KVB_E_STATE. */
int kvb_flush(kvb_pool *pool, int32_t n_req, const int32_t *req_ids, kvb_stream_t stream);

/* Chunked prefill: run each listed request's prompt through its state, 64
   tokens per chunk, on the tensor cores (the chunkwise form of linear
   attention that KVBuffer's buffer also uses; abstract).  Request req_ids[b]
   processes lengths[b] tokens (host array; NULL means L each, 0 <= lengths[b]
   <= L) taken from inputs laid out [B][L][heads][dim] (log_g, beta:
   [B][L][n_v_heads]); o: [B][L][n_v_heads][d_v] fp32 receives every prompt
   token's output (rows past lengths[b] are not written).  The state starts
   from the request's slot, or from S = 0 when from_zero is nonzero (a new
   request; then the slot's contents are never read), and holds the state
   after the prompt when the call completes.  Requires a state slot, an empty
   buffer and no pending verify (KVB_E_STATE otherwise: flush first), and
   d_k = d_v in {64, 128} (KVB_E_UNSUPPORTED otherwise).  The buffer is not
   touched. */
int kvb_prefill(kvb_pool *pool, int32_t B, int32_t L, const int32_t *req_ids,
                const int32_t *lengths, const void *q, const void *k, const void *v,
                const float *log_g, const float *beta, float *o, int32_t from_zero,
                kvb_stream_t stream);

/* Short-to-long promotion: a short-context request (no state slot) that is
   to continue past what its buffer holds is given its own state.  Short
   requests are served from buffered keys and values alone, with no state
   (abstract); this call creates the state at the point where that stops:
   request req_ids[b] takes the free state slot state_slots[b] (host array),
   its buffered tokens are folded into that slot starting from S = 0 (the
   Figure 1 state update with an all-zero state), and its buffer is emptied.
   A request with an empty buffer gets an all-zero state.  Afterwards the
   request is a state-backed request like any other (kvb_decode, kvb_verify,
   kvb_flush) and keeps its blocks as its buffer.
   Errors: KVB_E_STATE if a request already has a state or has a pending
   verify; KVB_E_RANGE if a slot is out of range, owned, or listed twice. */
int kvb_promote(kvb_pool *pool, int32_t B, const int32_t *req_ids, const int32_t *state_slots,
                kvb_stream_t stream);

/* Verify T draft tokens per request in parallel (Figure 2: the drafts' KVs go
   into the buffer and no temporary state is stored).  Inputs are laid out
   [B][T][heads][dim] (log_g, beta: [B][T][n_v_heads]); o: [B][T][n_v_heads][d_v].
   Draft j's output is the recurrent output after the request's history and
   drafts 0..j.  The drafts occupy buffer slots n .. n+T-1; the state is
   only read.  Stateless requests verify against S = 0.
   Requires m > 0, 1 <= T <= KVB_MAX_DRAFTS and n + T <= capacity
   (KVB_E_CAPACITY); a verify must be followed by kvb_accept before the
   request is used again (KVB_E_STATE otherwise). */
int kvb_verify(kvb_pool *pool, int32_t B, int32_t T, const int32_t *req_ids, const void *q,
               const void *k, const void *v, const float *log_g, const float *beta, float *o,
               kvb_stream_t stream);

/* Accept a prefix of the verified drafts: request req_ids[b] keeps its first
   n_accepted[b] drafts (0 <= n_accepted[b] <= T, host array); the rest are
   dropped by setting its length to n + n_accepted[b].  A request with a
   state whose buffer then holds >= m tokens folds all of them into its state
   (launched on `stream`).  Every listed request must have a pending
   kvb_verify (KVB_E_STATE otherwise); requests not listed stay pending. */
int kvb_accept(kvb_pool *pool, int32_t B, const int32_t *req_ids, const int32_t *n_accepted,
               kvb_stream_t stream);

/* Verify a tree of T draft tokens per request (tree-shaped speculation, as
   in the draft trees the page cites for speculative decoding; Figure 2's
   buffered verification with each draft seeing only its own path).
   parents (host, [B][T]): parents[b*T + j] is the draft that draft j
   continues, -1 for a child of the last accepted token; it must be < j
   (KVB_E_ARG otherwise), so drafts come in topological order.  Draft j's
   output is the recurrent output after the request's history and the drafts
   on the path from the root to j.  As in kvb_verify, the drafts occupy buffer
   slots n .. n+T-1 and the state is only read; inputs and o are laid out as
   there.  A verify_tree must be followed by kvb_accept_tree (kvb_accept gives
   KVB_E_STATE).  Launches carry at most 256 rows each. */
int kvb_verify_tree(kvb_pool *pool, int32_t B, int32_t T, const int32_t *req_ids,
                    const int32_t *parents, const void *q, const void *k, const void *v,
                    const float *log_g, const float *beta, float *o, kvb_stream_t stream);

/* Accept one path of a verified draft tree: request req_ids[b] keeps the
   drafts on the path from the root to draft accepted[b] (host array; -1
   keeps none), in path order, and drops the rest; its length grows by the
   path length.  Entries of the kept drafts are moved to the front of the
   draft slots on `stream` when the path is not already the leading drafts;
   a buffer that then holds >= m tokens is folded into the state as in
   kvb_accept.  Also accepts after a chain kvb_verify (the path to draft j is
   drafts 0..j).  Every listed request must have a pending verify
   (KVB_E_STATE otherwise). */
int kvb_accept_tree(kvb_pool *pool, int32_t B, const int32_t *req_ids, const int32_t *accepted,
                    kvb_stream_t stream);

/* The comparison baseline of Figure 2: a serving system with only a state pool
   verifies T drafts with the recurrent form and stores a temporary state after
   every draft.  For pools with m == 0 (KVB_E_STATE otherwise); every request
   must own a state slot.  Inputs and o as in kvb_verify.  temp_states: device
   fp32 [B][T][n_v_heads][d_k][d_v], caller-allocated, 16-byte aligned; row b
   belongs to req_ids[b] and entry j receives the state after drafts 0..j.  The
   requests' own states are only read. */
int kvb_verify_tempstate(kvb_pool *pool, int32_t B, int32_t T, const int32_t *req_ids,
                         const void *q, const void *k, const void *v, const float *log_g,
                         const float *beta, float *o, float *temp_states, kvb_stream_t stream);

/* Accept for the baseline: request req_ids[b] takes temporary state
   n_accepted[b] - 1 from the same temp_states layout as its state (Figure 2:
   the state is replaced by the temporary state of the last accepted draft);
   n_accepted[b] = 0 keeps the state.  0 <= n_accepted[b] <= T (KVB_E_ARG). */
int kvb_accept_tempstate(kvb_pool *pool, int32_t B, int32_t T, const int32_t *req_ids,
                         const int32_t *n_accepted, const float *temp_states,
                         kvb_stream_t stream);

/* Allocation-free kvb_verify_tempstate, for callers that cannot allocate device
   memory: an engine whose memory planner has already handed all device memory
   out, or code that must not call cudaMalloc because it synchronizes the device
   inside a latency-critical loop.  The paper has no counterpart; this is a
   library convenience.  The temporary states live in a fixed array inside the
   library (KVB_STATIC_TEMP_BYTES of device memory, held by every GPU that loads
   the library until the process exits), so B * T * n_v_heads * d_k * d_v * 4
   bytes must fit in it (KVB_E_CAPACITY otherwise, before anything runs).
   Inputs, o and the rules are those of kvb_verify_tempstate.  n_accepted (host,
   may be NULL) applies kvb_accept_tempstate in the same call: request
   req_ids[b] takes the state after its first n_accepted[b] drafts.
   The first call on a device looks up the array's device address; make it
   before any stream capture.  The address is kept for the process, so a
   cudaDeviceReset() after that first call is not supported (the array would
   then be reached through a stale address).  All calls share the array and it keeps the last
   call's contents (every temporary state is written before it is read, so
   nothing needs clearing); calls whose GPU work overlaps, from other streams or
   threads, race on it.  Calls no allocator. */
#define KVB_STATIC_TEMP_BYTES ((size_t)64 << 20)
int kvb_verify_tempstate_static(kvb_pool *pool, int32_t B, int32_t T, const int32_t *req_ids,
                                const void *q, const void *k, const void *v, const float *log_g,
                                const float *beta, float *o, const int32_t *n_accepted,
                                kvb_stream_t stream);

/* Host copy of every request's buffer length (max_requests int32). Host only,
   no synchronization: the host keeps an exact mirror of the device lengths. */
int kvb_get_lengths(const kvb_pool *pool, int32_t *host_out);

/* Copy the device-side lengths (max_requests int32) to host_out; synchronizes
   `stream`.  Equal to kvb_get_lengths whenever the pool is used correctly. */
int kvb_get_device_lengths(kvb_pool *pool, int32_t *host_out, kvb_stream_t stream);

/* Synchronize `stream` and read the device error word.  Returns KVB_OK, or
   KVB_E_DEVICE with detail[0..2] = {kind, request, value} when detail is not
   NULL, and clears the word.  Kinds:
     1  block id out of range (value = the id); the row was skipped;
     2  a bounded wait of the tensor-core prefill gave up (value = head); the
        CTA released its tensor memory and returned: every output and state of
        that kvb_prefill launch is invalid;
     3  as 2, and the wait for the products still in flight gave up too, so the
        tensor memory was released while they may still have been running:
        treat the device as unreliable for that stream. */
int kvb_get_error(kvb_pool *pool, kvb_stream_t stream, int32_t *detail);

/* Testing hook for the device-side failure path (host only, process-wide).
   The tensor-core prefill (bf16, d = 128) waits for its tensor-core products
   and copies with bounded polls.  This caps the first wait on its products in
   every CTA of later kvb_prefill launches at `polls` non-blocking polls (0
   restores the default bound of 2^16 blocking polls, each up to about a
   microsecond), so a test can make that wait run out without any fault: the CTA
   records kind 2 in the error word, waits with the full bound for the products
   still in flight, releases its tensor memory and returns, and the context
   stays usable.  KVB_E_ARG for polls < 0. */
int kvb_set_prefill_wait_limit(int32_t polls);

/* Name of a status code (static string). */
const char *kvb_strerror(int status);

/* HBM copy probe: dst[i] = src[i] for `bytes` bytes (multiple of 16, both
   pointers 16-byte aligned) with 128-bit loads and stores; used to measure
   the achievable HBM bandwidth in the same run as the decode benchmark. */
int kvb_copy_probe(const void *src, void *dst, size_t bytes, kvb_stream_t stream);

/* Library version, e.g. "libkvb 0.2 sm_103a". */
const char *kvb_version(void);

#ifdef __cplusplus
}
#endif
#endif /* KVB_H */
