// libkvb host side: the C ABI of include/kvb.h.
//
// The host keeps an exact mirror of every request's buffer length, its state
// slot and its block list (the state pool, block-partitioned KV buffer and
// per-request buffer length of "KVBuffer: IO-aware Serving for Linear
// Attention", Figures 1 and 2).  From the mirror it validates every call
// before launching anything, decides which requests fold their buffer into
// the state in this step, and packs the per-row descriptors (request, length,
// slot, flags) into the kernels' parameter block, so a step needs no device
// synchronization and no host-to-device copy.
#include <cmath>
#include <cstdint>
#include <cstring>
#include <new>
#include <vector>

#include <cuda_runtime_api.h>

#include "kvb.h"
#include "kvb_internal.h"

namespace {

constexpr size_t kAlign = 256;
size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }
bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

struct MetaLayout {
  size_t table_off, len_off, err_off, bytes;
};

bool mul_ok(size_t a, size_t b, size_t *out) {
  if (a != 0 && b > SIZE_MAX / a) return false;
  *out = a * b;
  return true;
}

int check_config(const kvb_config *c) {
  if (!c) return KVB_E_ARG;
  if (c->variant < KVB_PLAIN || c->variant > KVB_GATED_DELTA) return KVB_E_ARG;
  if (c->kv_dtype != KVB_F32 && c->kv_dtype != KVB_BF16) return KVB_E_ARG;
  if (c->n_qk_heads <= 0 || c->n_v_heads <= 0 || c->n_v_heads % c->n_qk_heads) return KVB_E_ARG;
  if (c->d_k != c->d_v) return KVB_E_UNSUPPORTED;
  if (c->d_k != 64 && c->d_k != 128) return KVB_E_UNSUPPORTED;
  if (c->m < 0 || c->m > KVB_MAX_CAPACITY) return KVB_E_ARG;
  if (c->block_size <= 0 || c->num_blocks < 0 || c->num_state_slots < 0) return KVB_E_ARG;
  if (c->max_requests <= 0 || c->max_blocks_per_req < 0) return KVB_E_ARG;
  if (!std::isfinite(c->scale)) return KVB_E_ARG;
  return KVB_OK;
}

int compute_layout(const kvb_config *c, kvb_layout *L, MetaLayout *M) {
  int st = check_config(c);
  if (st) return st;
  const size_t esz = c->kv_dtype == KVB_BF16 ? 2 : 4;
  size_t per_slot, state, rows, kb, vb, ub, gb;
  if (!mul_ok((size_t)c->n_v_heads * c->d_k * c->d_v, 4, &per_slot)) return KVB_E_ARG;
  if (!mul_ok(per_slot, (size_t)c->num_state_slots, &state)) return KVB_E_ARG;
  if (!mul_ok((size_t)c->num_blocks, (size_t)c->block_size, &rows)) return KVB_E_ARG;
  if (!mul_ok(rows, (size_t)c->n_qk_heads * c->d_k * esz, &kb)) return KVB_E_ARG;
  if (!mul_ok(rows, (size_t)c->n_v_heads * c->d_v * esz, &vb)) return KVB_E_ARG;
  if (c->variant == KVB_GATED_DELTA) {
    if (!mul_ok(rows, (size_t)c->n_v_heads * c->d_v * 4, &ub)) return KVB_E_ARG;
  } else {
    ub = 0;
  }
  if (!mul_ok(rows, (size_t)c->n_v_heads * 4, &gb)) return KVB_E_ARG;
  L->state_slot_stride = per_slot;
  L->state_bytes = align_up(state);
  L->k_off = 0;
  L->v_off = align_up(L->k_off + kb);
  L->u_off = align_up(L->v_off + vb);
  L->logg_off = align_up(L->u_off + ub);
  L->beta_off = align_up(L->logg_off + gb);
  L->kv_bytes = align_up(L->beta_off + gb);
  M->table_off = 0;
  M->len_off = align_up((size_t)c->max_requests * c->max_blocks_per_req * 4);
  M->err_off = align_up(M->len_off + (size_t)c->max_requests * 4);
  M->bytes = align_up(M->err_off + 4 * sizeof(int32_t));
  L->meta_bytes = M->bytes;
  return KVB_OK;
}

}  // namespace

struct kvb_pool {
  kvb_config cfg;
  kvb_layout layout;
  MetaLayout meta;
  kvb::PoolView view;
  int32_t *d_len = nullptr;
  int32_t *d_err = nullptr;
  int32_t *d_table = nullptr;
  // host mirror
  std::vector<int32_t> len, slot, nblk, pending_T, table;
  std::vector<uint8_t> active;
  std::vector<int32_t> slot_owner, block_owner;
  std::vector<uint32_t> stamp;
  uint32_t stamp_gen = 0;
  kvb::RowBatch rows;  // parameter block under construction (8 KB, kept off the stack)
  // draft trees: parents of each request's pending tree verify, and the tree
  // parameter block under construction (8 KB)
  std::vector<int8_t> tree_host;
  std::vector<uint8_t> pending_tree;
  kvb::TreeArg<true> tree_arg;
  // TMA map of the state region (d = 128 pools with a state pool), for the
  // tensor-core verify; has_map is false when it could not be encoded
  kvb::StateMap state_map;
  bool has_map = false;

  int capacity(int r) const { return nblk[r] * cfg.block_size; }
};

namespace {

// Checks shared by the batch calls: ids in range, active, not repeated.
int check_reqs(kvb_pool *p, int32_t B, const int32_t *req_ids) {
  if (B < 0) return KVB_E_ARG;
  if (B == 0) return KVB_OK;
  if (!req_ids) return KVB_E_ARG;
  if (++p->stamp_gen == 0) {
    std::fill(p->stamp.begin(), p->stamp.end(), 0u);
    p->stamp_gen = 1;
  }
  for (int32_t b = 0; b < B; ++b) {
    const int32_t r = req_ids[b];
    if (r < 0 || r >= p->cfg.max_requests) return KVB_E_RANGE;
    if (!p->active[r]) return KVB_E_STATE;
    if (p->stamp[r] == p->stamp_gen) return KVB_E_ARG;  // duplicate: rows would race
    p->stamp[r] = p->stamp_gen;
  }
  return KVB_OK;
}

int check_io(const kvb_pool *p, const void *q, const void *k, const void *v, const float *log_g,
             const float *beta, const float *o) {
  if (!q || !k || !v || !o) return KVB_E_ARG;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16)) return KVB_E_ARG;
  if (p->cfg.variant == KVB_GATED && !log_g) return KVB_E_ARG;
  if (p->cfg.variant == KVB_GATED_DELTA && !beta) return KVB_E_ARG;
  if ((log_g && !aligned(log_g, 4)) || (beta && !aligned(beta, 4))) return KVB_E_ARG;
  return KVB_OK;
}

int cuda_status(cudaError_t e) {
  if (e == cudaSuccess) return KVB_OK;
  if (e == kvb::kUnsupported) return KVB_E_UNSUPPORTED;
  return KVB_E_CUDA;
}

// A row descriptor from the host mirror: request, length, slot, flags and the
// request's first block ids.
kvb::RowDesc make_row(const kvb_pool *p, int32_t r, int32_t n, int32_t flags) {
  kvb::RowDesc d;
  d.req = r;
  d.n = n;
  d.slot = p->slot[r];
  d.flags = flags;
  const int32_t *row = p->table.data() + (size_t)r * p->cfg.max_blocks_per_req;
  for (int i = 0; i < kvb::kRowBlocks; ++i) d.blk[i] = i < p->nblk[r] ? row[i] : -1;
  return d;
}

enum Mode { kDecode, kShort };

int decode_like(kvb_pool *p, int32_t B, const int32_t *req_ids, const void *q, const void *k,
                const void *v, const float *log_g, const float *beta, float *o, bool auto_flush,
                Mode mode, cudaStream_t stream) {
  if (!p) return KVB_E_ARG;
  int st = check_reqs(p, B, req_ids);
  if (st || B == 0) return st;
  if ((st = check_io(p, q, k, v, log_g, beta, o))) return st;
  const kvb_config &c = p->cfg;
  const bool recurrent = (mode == kDecode && c.m == 0);
  for (int32_t b = 0; b < B; ++b) {
    const int32_t r = req_ids[b];
    if (p->pending_T[r]) return KVB_E_STATE;
    if (mode == kDecode && p->slot[r] < 0) return KVB_E_STATE;
    if (mode == kShort && p->slot[r] >= 0) return KVB_E_STATE;
    if (!recurrent && p->len[r] + 1 > p->capacity(r)) return KVB_E_CAPACITY;
  }
  const kvb::TokenIO io{q, k, v, log_g, beta, o, 1, 0};
  for (int32_t base = 0; base < B; base += kvb::kMaxRows) {
    const int32_t cnt = B - base < kvb::kMaxRows ? B - base : kvb::kMaxRows;
    p->rows.count = cnt;
    p->rows.row0 = base;
    int lmax = recurrent ? 1 : 0, nmax = 0;
    for (int32_t i = 0; i < cnt; ++i) {
      const int32_t r = req_ids[base + i];
      kvb::RowDesc &d = p->rows.r[i];
      d = make_row(p, r, recurrent ? 0 : p->len[r], 0);
      if (d.n > nmax) nmax = d.n;
      if (mode == kDecode && !recurrent && auto_flush && c.m > 0 && d.n + 1 >= c.m) {
        d.flags = kvb::kFlagFlush;
        if (d.n + 1 > lmax) lmax = d.n + 1;
      }
    }
    kvb::TokenIO io_short = io;
    io_short.lmax = nmax;  // most buffered tokens any row stages
    cudaError_t e = mode == kShort
                        ? kvb::launch_short(p->view, p->rows, io_short, c.variant, c.kv_dtype, c.d_k, stream)
                        : kvb::launch_decode(p->view, p->rows, io, c.variant, c.kv_dtype, c.d_k,
                                             recurrent, lmax, nmax, stream);
    if (e != cudaSuccess) return cuda_status(e);
    if (!recurrent) {
      for (int32_t i = 0; i < cnt; ++i) {
        const kvb::RowDesc &d = p->rows.r[i];
        p->len[d.req] = (d.flags & kvb::kFlagFlush) ? 0 : d.n + 1;
      }
    }
  }
  return KVB_OK;
}

int launch_fold(kvb_pool *p, const std::vector<int32_t> &reqs, cudaStream_t stream,
                int32_t flags = 0) {
  const kvb_config &c = p->cfg;
  for (size_t base = 0; base < reqs.size(); base += kvb::kMaxRows) {
    const size_t cnt = reqs.size() - base < (size_t)kvb::kMaxRows ? reqs.size() - base : kvb::kMaxRows;
    p->rows.count = (int32_t)cnt;
    p->rows.row0 = 0;
    int lmax = 0;
    for (size_t i = 0; i < cnt; ++i) {
      const int32_t r = reqs[base + i];
      p->rows.r[i] = make_row(p, r, p->len[r], flags);
      if (p->len[r] > lmax) lmax = p->len[r];
    }
    cudaError_t e = kvb::launch_flush(p->view, p->rows, c.variant, c.kv_dtype, c.d_k, lmax, stream);
    if (e != cudaSuccess) return cuda_status(e);
    for (size_t i = 0; i < cnt; ++i) p->len[reqs[base + i]] = 0;
  }
  return KVB_OK;
}

}  // namespace

extern "C" {

int kvb_pool_layout(const kvb_config *cfg, kvb_layout *out) {
  if (!out) return KVB_E_ARG;
  MetaLayout m;
  kvb_layout l;
  int st = compute_layout(cfg, &l, &m);
  if (st) return st;
  *out = l;
  return KVB_OK;
}

int kvb_alloc_pool(const kvb_config *cfg, void *state_mem, void *kv_mem, void *meta_mem,
                   kvb_pool **out) {
  if (!out) return KVB_E_ARG;
  kvb_layout l;
  MetaLayout m;
  int st = compute_layout(cfg, &l, &m);
  if (st) return st;
  if (!meta_mem || !aligned(meta_mem, kAlign)) return KVB_E_ARG;
  if (cfg->num_state_slots > 0 && (!state_mem || !aligned(state_mem, kAlign))) return KVB_E_ARG;
  if (l.kv_bytes > 0 && cfg->num_blocks > 0 && (!kv_mem || !aligned(kv_mem, kAlign)))
    return KVB_E_ARG;
  kvb_pool *p = new (std::nothrow) kvb_pool();
  if (!p) return KVB_E_ARG;
  p->cfg = *cfg;
  p->layout = l;
  p->meta = m;
  char *kv = static_cast<char *>(kv_mem);
  char *meta = static_cast<char *>(meta_mem);
  p->d_table = reinterpret_cast<int32_t *>(meta + m.table_off);
  p->d_len = reinterpret_cast<int32_t *>(meta + m.len_off);
  p->d_err = reinterpret_cast<int32_t *>(meta + m.err_off);
  kvb::PoolView &v = p->view;
  v.state = static_cast<float *>(state_mem);
  v.kbuf = kv ? kv + l.k_off : nullptr;
  v.vbuf = kv ? kv + l.v_off : nullptr;
  v.ubuf = kv ? reinterpret_cast<float *>(kv + l.u_off) : nullptr;
  v.gbuf = kv ? reinterpret_cast<float *>(kv + l.logg_off) : nullptr;
  v.bbuf = kv ? reinterpret_cast<float *>(kv + l.beta_off) : nullptr;
  v.table = p->d_table;
  v.dlen = p->d_len;
  v.err = p->d_err;
  v.Hk = cfg->n_qk_heads;
  v.Hv = cfg->n_v_heads;
  v.bs = cfg->block_size;
  v.bs_shift = -1;
  for (int sh = 0; sh < 31; ++sh)
    if (cfg->block_size == (1 << sh)) v.bs_shift = sh;
  v.max_blocks = cfg->max_blocks_per_req;
  v.num_blocks = cfg->num_blocks;
  v.scale = cfg->scale;
  const size_t R = (size_t)cfg->max_requests;
  p->len.assign(R, 0);
  p->slot.assign(R, -1);
  p->nblk.assign(R, 0);
  p->pending_T.assign(R, 0);
  p->pending_tree.assign(R, 0);
  p->tree_host.assign(R * (size_t)KVB_MAX_DRAFTS, -1);
  p->active.assign(R, 0);
  p->stamp.assign(R, 0u);
  p->table.assign(R * (size_t)cfg->max_blocks_per_req, -1);
  p->slot_owner.assign((size_t)cfg->num_state_slots, -1);
  p->block_owner.assign((size_t)cfg->num_blocks, -1);
  if (cudaMemset(meta_mem, 0, m.bytes) != cudaSuccess) {
    delete p;
    return KVB_E_CUDA;
  }
  if (cfg->d_k == 128 && cfg->kv_dtype == KVB_BF16 && cfg->num_state_slots > 0)
    p->has_map = kvb::encode_state_map(&p->state_map, v.state,
                                       (uint64_t)cfg->num_state_slots * cfg->n_v_heads * cfg->d_k) ==
                 cudaSuccess;
  *out = p;
  return KVB_OK;
}

int kvb_free_pool(kvb_pool *pool) {
  if (!pool) return KVB_E_ARG;
  delete pool;
  return KVB_OK;
}

int kvb_set_request(kvb_pool *p, int32_t req, int32_t state_slot, int32_t n_blocks,
                    const int32_t *block_ids, kvb_stream_t stream) {
  if (!p) return KVB_E_ARG;
  const kvb_config &c = p->cfg;
  if (req < 0 || req >= c.max_requests) return KVB_E_RANGE;
  if (p->active[req]) return KVB_E_STATE;
  if (state_slot < -1 || state_slot >= c.num_state_slots) return KVB_E_RANGE;
  if (state_slot >= 0 && p->slot_owner[state_slot] >= 0) return KVB_E_RANGE;
  if (n_blocks < 0 || n_blocks > c.max_blocks_per_req) return KVB_E_RANGE;
  if ((int64_t)n_blocks * c.block_size > KVB_MAX_CAPACITY) return KVB_E_CAPACITY;
  if (n_blocks > 0 && !block_ids) return KVB_E_ARG;
  if (state_slot < 0 && n_blocks == 0) return KVB_E_ARG;  // a stateless request needs a buffer
  for (int32_t i = 0; i < n_blocks; ++i) {
    const int32_t bid = block_ids[i];
    if (bid < 0 || bid >= c.num_blocks || p->block_owner[bid] >= 0) return KVB_E_RANGE;
    for (int32_t j = 0; j < i; ++j)
      if (block_ids[j] == bid) return KVB_E_RANGE;
  }
  int32_t *row = p->table.data() + (size_t)req * c.max_blocks_per_req;
  for (int32_t i = 0; i < c.max_blocks_per_req; ++i) row[i] = i < n_blocks ? block_ids[i] : -1;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (c.max_blocks_per_req > 0) {
    if (cudaMemcpyAsync(p->d_table + (size_t)req * c.max_blocks_per_req, row,
                        (size_t)c.max_blocks_per_req * 4, cudaMemcpyHostToDevice, s) != cudaSuccess)
      return KVB_E_CUDA;
  }
  if (cudaMemsetAsync(p->d_len + req, 0, 4, s) != cudaSuccess) return KVB_E_CUDA;
  for (int32_t i = 0; i < n_blocks; ++i) p->block_owner[block_ids[i]] = req;
  if (state_slot >= 0) p->slot_owner[state_slot] = req;
  p->active[req] = 1;
  p->slot[req] = state_slot;
  p->nblk[req] = n_blocks;
  p->len[req] = 0;
  p->pending_T[req] = 0;
  p->pending_tree[req] = 0;
  return KVB_OK;
}

int kvb_release_request(kvb_pool *p, int32_t req) {
  if (!p) return KVB_E_ARG;
  if (req < 0 || req >= p->cfg.max_requests) return KVB_E_RANGE;
  if (!p->active[req]) return KVB_E_STATE;
  const int32_t *row = p->table.data() + (size_t)req * p->cfg.max_blocks_per_req;
  for (int32_t i = 0; i < p->nblk[req]; ++i) p->block_owner[row[i]] = -1;
  if (p->slot[req] >= 0) p->slot_owner[p->slot[req]] = -1;
  p->active[req] = 0;
  p->slot[req] = -1;
  p->nblk[req] = 0;
  p->len[req] = 0;
  p->pending_T[req] = 0;
  p->pending_tree[req] = 0;
  return KVB_OK;
}

int kvb_decode(kvb_pool *pool, int32_t B, const int32_t *req_ids, const void *q, const void *k,
               const void *v, const float *log_g, const float *beta, float *o, int32_t auto_flush,
               kvb_stream_t stream) {
  return decode_like(pool, B, req_ids, q, k, v, log_g, beta, o, auto_flush != 0, kDecode,
                     reinterpret_cast<cudaStream_t>(stream));
}

int kvb_short_ctx(kvb_pool *pool, int32_t B, const int32_t *req_ids, const void *q, const void *k,
                  const void *v, const float *log_g, const float *beta, float *o,
                  kvb_stream_t stream) {
  return decode_like(pool, B, req_ids, q, k, v, log_g, beta, o, false, kShort,
                     reinterpret_cast<cudaStream_t>(stream));
}

int kvb_flush(kvb_pool *p, int32_t n_req, const int32_t *req_ids, kvb_stream_t stream) {
  if (!p) return KVB_E_ARG;
  int st = check_reqs(p, n_req, req_ids);
  if (st || n_req == 0) return st;
  std::vector<int32_t> todo;
  for (int32_t i = 0; i < n_req; ++i) {
    const int32_t r = req_ids[i];
    if (p->slot[r] < 0 || p->pending_T[r]) return KVB_E_STATE;
    if (p->len[r] > 0) todo.push_back(r);
  }
  return launch_fold(p, todo, reinterpret_cast<cudaStream_t>(stream));
}

int kvb_prefill(kvb_pool *p, int32_t B, int32_t L, const int32_t *req_ids,
                const int32_t *lengths, const void *q, const void *k, const void *v,
                const float *log_g, const float *beta, float *o, int32_t from_zero,
                kvb_stream_t stream) {
  if (!p) return KVB_E_ARG;
  if (L < 0) return KVB_E_ARG;
  int st = check_reqs(p, B, req_ids);
  if (st || B == 0) return st;
  if ((st = check_io(p, q, k, v, log_g, beta, o))) return st;
  const kvb_config &c = p->cfg;
  if (c.d_k != c.d_v || (c.d_k != 64 && c.d_k != 128)) return KVB_E_UNSUPPORTED;
  for (int32_t b = 0; b < B; ++b) {
    const int32_t r = req_ids[b];
    if (p->slot[r] < 0 || p->len[r] != 0 || p->pending_T[r]) return KVB_E_STATE;
    if (lengths && (lengths[b] < 0 || lengths[b] > L)) return KVB_E_ARG;
  }
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const kvb::TokenIO io{q, k, v, log_g, beta, o, L, 0, B};
  const int32_t flags = from_zero ? kvb::kFlagFromZero : 0;
  for (int32_t base = 0; base < B; base += kvb::kMaxRows) {
    const int32_t cnt = B - base < kvb::kMaxRows ? B - base : kvb::kMaxRows;
    p->rows.count = cnt;
    p->rows.row0 = base;
    for (int32_t i = 0; i < cnt; ++i)
      p->rows.r[i] = make_row(p, req_ids[base + i], lengths ? lengths[base + i] : L, flags);
    cudaError_t e = kvb::launch_prefill(p->view, p->rows, io, c.variant, c.kv_dtype, c.d_k, s);
    if (e != cudaSuccess) return cuda_status(e);
  }
  return KVB_OK;
}

int kvb_promote(kvb_pool *p, int32_t B, const int32_t *req_ids, const int32_t *state_slots,
                kvb_stream_t stream) {
  if (!p) return KVB_E_ARG;
  int st = check_reqs(p, B, req_ids);
  if (st || B == 0) return st;
  if (!state_slots) return KVB_E_ARG;
  const kvb_config &c = p->cfg;
  for (int32_t b = 0; b < B; ++b) {
    const int32_t r = req_ids[b], sl = state_slots[b];
    if (p->slot[r] >= 0 || p->pending_T[r]) return KVB_E_STATE;
    if (sl < 0 || sl >= c.num_state_slots || p->slot_owner[sl] >= 0) return KVB_E_RANGE;
    for (int32_t j = 0; j < b; ++j)
      if (state_slots[j] == sl) return KVB_E_RANGE;
  }
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const size_t state_bytes = (size_t)c.n_v_heads * c.d_k * c.d_v * sizeof(float);
  std::vector<int32_t> fold;
  for (int32_t b = 0; b < B; ++b) {
    const int32_t r = req_ids[b], sl = state_slots[b];
    p->slot[r] = sl;
    p->slot_owner[sl] = r;
    if (p->len[r] > 0) {
      fold.push_back(r);
    } else if (cudaMemsetAsync(p->view.state + (size_t)sl * state_bytes / sizeof(float), 0,
                               state_bytes, s) != cudaSuccess) {
      return KVB_E_CUDA;
    }
  }
  return launch_fold(p, fold, s, kvb::kFlagFromZero);
}

}  // extern "C"

namespace {

// Verify of a chain (parents == nullptr) or of a draft tree (host parents [B][T]).
int verify_impl(kvb_pool *p, int32_t B, int32_t T, const int32_t *req_ids,
                const int32_t *parents, const void *q, const void *k, const void *v,
                const float *log_g, const float *beta, float *o, cudaStream_t stream) {
  if (!p) return KVB_E_ARG;
  if (p->cfg.m == 0) return KVB_E_STATE;
  if (T < 1 || T > KVB_MAX_DRAFTS) return KVB_E_ARG;
  int st = check_reqs(p, B, req_ids);
  if (st || B == 0) return st;
  if ((st = check_io(p, q, k, v, log_g, beta, o))) return st;
  for (int32_t b = 0; b < B; ++b) {
    const int32_t r = req_ids[b];
    if (p->pending_T[r]) return KVB_E_STATE;
    if (p->len[r] + T > p->capacity(r)) return KVB_E_CAPACITY;
    if (parents)
      for (int32_t j = 0; j < T; ++j) {
        const int32_t par = parents[(size_t)b * T + j];
        if (par < -1 || par >= j) return KVB_E_ARG;
      }
  }
  const kvb_config &c = p->cfg;
  const kvb::TokenIO io{q, k, v, log_g, beta, o, T, 0};
  const int32_t per_launch = parents ? kvb::kTreeRows : kvb::kMaxRows;
  for (int32_t base = 0; base < B; base += per_launch) {
    const int32_t cnt = B - base < per_launch ? B - base : per_launch;
    p->rows.count = cnt;
    p->rows.row0 = base;
    int lmax = 0;
    for (int32_t i = 0; i < cnt; ++i) {
      const int32_t r = req_ids[base + i];
      p->rows.r[i] = make_row(p, r, p->len[r], 0);
      if (p->len[r] + T > lmax) lmax = p->len[r] + T;
      if (parents)
        for (int32_t j = 0; j < T; ++j)
          p->tree_arg.p[i][j] = static_cast<int8_t>(parents[(size_t)(base + i) * T + j]);
    }
    cudaError_t e = kvb::launch_verify(p->view, p->rows, io, c.variant, c.kv_dtype, c.d_k, lmax,
                                       stream, parents ? &p->tree_arg : nullptr,
                                       p->has_map ? &p->state_map : nullptr);
    if (e != cudaSuccess) return cuda_status(e);
    for (int32_t i = 0; i < cnt; ++i) {
      const int32_t r = req_ids[base + i];
      p->pending_T[r] = T;
      p->pending_tree[r] = parents != nullptr;
      if (parents)
        for (int32_t j = 0; j < T; ++j)
          p->tree_host[(size_t)r * KVB_MAX_DRAFTS + j] = p->tree_arg.p[i][j];
    }
  }
  return KVB_OK;
}

// Lengths after an accept: fold the rows whose buffer reached m, set the
// device length of the others.
int finish_accept(kvb_pool *p, const std::vector<int32_t> &reqs, cudaStream_t s) {
  std::vector<int32_t> fold, keep;
  for (int32_t r : reqs) {
    if (p->slot[r] >= 0 && p->cfg.m > 0 && p->len[r] >= p->cfg.m)
      fold.push_back(r);
    else
      keep.push_back(r);
  }
  for (size_t base = 0; base < keep.size(); base += kvb::kMaxRows) {
    const size_t cnt = keep.size() - base < (size_t)kvb::kMaxRows ? keep.size() - base : kvb::kMaxRows;
    p->rows.count = (int32_t)cnt;
    p->rows.row0 = 0;
    for (size_t i = 0; i < cnt; ++i) {
      const int32_t r = keep[base + i];
      p->rows.r[i] = make_row(p, r, p->len[r], 0);
    }
    cudaError_t e = kvb::launch_set_lengths(p->view, p->rows, s);
    if (e != cudaSuccess) return cuda_status(e);
  }
  return launch_fold(p, fold, s);
}

}  // namespace

extern "C" {

int kvb_verify(kvb_pool *p, int32_t B, int32_t T, const int32_t *req_ids, const void *q,
               const void *k, const void *v, const float *log_g, const float *beta, float *o,
               kvb_stream_t stream) {
  return verify_impl(p, B, T, req_ids, nullptr, q, k, v, log_g, beta, o,
                     reinterpret_cast<cudaStream_t>(stream));
}

int kvb_verify_tree(kvb_pool *p, int32_t B, int32_t T, const int32_t *req_ids,
                    const int32_t *parents, const void *q, const void *k, const void *v,
                    const float *log_g, const float *beta, float *o, kvb_stream_t stream) {
  if (!parents) return KVB_E_ARG;
  return verify_impl(p, B, T, req_ids, parents, q, k, v, log_g, beta, o,
                     reinterpret_cast<cudaStream_t>(stream));
}

int kvb_accept_tree(kvb_pool *p, int32_t B, const int32_t *req_ids, const int32_t *accepted,
                    kvb_stream_t stream) {
  if (!p) return KVB_E_ARG;
  int st = check_reqs(p, B, req_ids);
  if (st || B == 0) return st;
  if (!accepted) return KVB_E_ARG;
  for (int32_t b = 0; b < B; ++b) {
    const int32_t r = req_ids[b];
    if (!p->pending_T[r]) return KVB_E_STATE;
    if (accepted[b] < -1 || accepted[b] >= p->pending_T[r]) return KVB_E_ARG;
  }
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const kvb_config &c = p->cfg;
  // accepted paths, root first; rows whose path is not already the leading drafts
  // are compacted on the device before the lengths change
  std::vector<int32_t> reqs(B);
  int32_t cnt = 0;
  auto flush_compact = [&]() -> int {
    if (cnt == 0) return KVB_OK;
    p->rows.count = cnt;
    p->rows.row0 = 0;
    cudaError_t e = kvb::launch_tree_compact(p->view, p->rows, p->tree_arg, c.variant,
                                             c.kv_dtype, c.d_k, s);
    cnt = 0;
    return e == cudaSuccess ? KVB_OK : cuda_status(e);
  };
  for (int32_t b = 0; b < B; ++b) {
    const int32_t r = req_ids[b];
    reqs[b] = r;
    int8_t path[KVB_MAX_DRAFTS];
    int32_t len = 0;
    if (p->pending_tree[r]) {
      int8_t rev[KVB_MAX_DRAFTS];
      for (int32_t j = accepted[b]; j >= 0; j = p->tree_host[(size_t)r * KVB_MAX_DRAFTS + j])
        rev[len++] = static_cast<int8_t>(j);
      for (int32_t l = 0; l < len; ++l) path[l] = rev[len - 1 - l];
    } else {
      for (int32_t l = 0; l <= accepted[b]; ++l) path[len++] = static_cast<int8_t>(l);
    }
    bool moved = false;
    for (int32_t l = 0; l < len; ++l) moved |= path[l] != l;
    if (moved) {
      p->rows.r[cnt] = make_row(p, r, p->len[r], len);
      for (int32_t l = 0; l < len; ++l) p->tree_arg.p[cnt][l] = path[l];
      if (++cnt == kvb::kTreeRows && (st = flush_compact())) return st;
    }
    p->len[r] += len;
    p->pending_T[r] = 0;
    p->pending_tree[r] = 0;
  }
  if ((st = flush_compact())) return st;
  return finish_accept(p, reqs, s);
}


int kvb_accept(kvb_pool *p, int32_t B, const int32_t *req_ids, const int32_t *n_accepted,
               kvb_stream_t stream) {
  if (!p) return KVB_E_ARG;
  int st = check_reqs(p, B, req_ids);
  if (st || B == 0) return st;
  if (!n_accepted) return KVB_E_ARG;
  for (int32_t b = 0; b < B; ++b) {
    const int32_t r = req_ids[b];
    if (!p->pending_T[r] || p->pending_tree[r]) return KVB_E_STATE;
    if (n_accepted[b] < 0 || n_accepted[b] > p->pending_T[r]) return KVB_E_ARG;
  }
  std::vector<int32_t> reqs(B);
  for (int32_t b = 0; b < B; ++b) {
    const int32_t r = req_ids[b];
    reqs[b] = r;
    p->len[r] += n_accepted[b];
    p->pending_T[r] = 0;
  }
  return finish_accept(p, reqs, reinterpret_cast<cudaStream_t>(stream));
}

int kvb_verify_tempstate(kvb_pool *p, int32_t B, int32_t T, const int32_t *req_ids,
                         const void *q, const void *k, const void *v, const float *log_g,
                         const float *beta, float *o, float *temp_states, kvb_stream_t stream) {
  if (!p) return KVB_E_ARG;
  if (p->cfg.m != 0) return KVB_E_STATE;
  if (T < 1 || T > KVB_MAX_DRAFTS) return KVB_E_ARG;
  int st = check_reqs(p, B, req_ids);
  if (st || B == 0) return st;
  if ((st = check_io(p, q, k, v, log_g, beta, o))) return st;
  if (!temp_states || !aligned(temp_states, 16)) return KVB_E_ARG;
  for (int32_t b = 0; b < B; ++b)
    if (p->slot[req_ids[b]] < 0) return KVB_E_STATE;
  const kvb_config &c = p->cfg;
  const kvb::TokenIO io{q, k, v, log_g, beta, o, T, 0};
  for (int32_t base = 0; base < B; base += kvb::kMaxRows) {
    const int32_t cnt = B - base < kvb::kMaxRows ? B - base : kvb::kMaxRows;
    p->rows.count = cnt;
    p->rows.row0 = base;
    for (int32_t i = 0; i < cnt; ++i) p->rows.r[i] = make_row(p, req_ids[base + i], 0, 0);
    cudaError_t e = kvb::launch_verify_tempstate(p->view, p->rows, io, c.variant, c.kv_dtype, c.d_k,
                                                 temp_states, reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_status(e);
  }
  return KVB_OK;
}

int kvb_accept_tempstate(kvb_pool *p, int32_t B, int32_t T, const int32_t *req_ids,
                         const int32_t *n_accepted, const float *temp_states,
                         kvb_stream_t stream) {
  if (!p) return KVB_E_ARG;
  if (p->cfg.m != 0) return KVB_E_STATE;
  if (T < 1 || T > KVB_MAX_DRAFTS) return KVB_E_ARG;
  int st = check_reqs(p, B, req_ids);
  if (st || B == 0) return st;
  if (!n_accepted || !temp_states || !aligned(temp_states, 16)) return KVB_E_ARG;
  for (int32_t b = 0; b < B; ++b) {
    if (n_accepted[b] < 0 || n_accepted[b] > T) return KVB_E_ARG;
    if (p->slot[req_ids[b]] < 0) return KVB_E_STATE;
  }
  // only rows that accepted something copy a state; row0 keeps the temp_states row
  int32_t i = 0;
  for (int32_t b = 0; b < B; ++b) {
    if (n_accepted[b] == 0) continue;
    if (i == kvb::kMaxRows || (i > 0 && b != p->rows.row0 + i)) {
      cudaError_t e = kvb::launch_accept_tempstate(p->view, p->rows, temp_states, T, p->cfg.d_k,
                                                   reinterpret_cast<cudaStream_t>(stream));
      if (e != cudaSuccess) return cuda_status(e);
      i = 0;
    }
    if (i == 0) p->rows.row0 = b;
    p->rows.r[i++] = make_row(p, req_ids[b], n_accepted[b], 0);
    p->rows.count = i;
  }
  if (i > 0) {
    cudaError_t e = kvb::launch_accept_tempstate(p->view, p->rows, temp_states, T, p->cfg.d_k,
                                                 reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_status(e);
  }
  return KVB_OK;
}

int kvb_verify_tempstate_static(kvb_pool *p, int32_t B, int32_t T, const int32_t *req_ids,
                                const void *q, const void *k, const void *v, const float *log_g,
                                const float *beta, float *o, const int32_t *n_accepted,
                                kvb_stream_t stream) {
  if (!p) return KVB_E_ARG;
  if (p->cfg.m != 0) return KVB_E_STATE;
  if (T < 1 || T > KVB_MAX_DRAFTS) return KVB_E_ARG;
  int st = check_reqs(p, B, req_ids);
  if (st || B == 0) return st;
  if ((st = check_io(p, q, k, v, log_g, beta, o))) return st;
  const kvb_config &c = p->cfg;
  const size_t need = (size_t)B * T * c.n_v_heads * c.d_k * c.d_v * sizeof(float);
  if (need > KVB_STATIC_TEMP_BYTES) return KVB_E_CAPACITY;
  for (int32_t b = 0; b < B; ++b) {
    if (p->slot[req_ids[b]] < 0) return KVB_E_STATE;
    if (n_accepted && (n_accepted[b] < 0 || n_accepted[b] > T)) return KVB_E_ARG;
  }
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const kvb::TokenIO io{q, k, v, log_g, beta, o, T, 0};
  for (int32_t base = 0; base < B; base += kvb::kMaxRows) {
    const int32_t cnt = B - base < kvb::kMaxRows ? B - base : kvb::kMaxRows;
    p->rows.count = cnt;
    p->rows.row0 = base;
    for (int32_t i = 0; i < cnt; ++i) p->rows.r[i] = make_row(p, req_ids[base + i], 0, 0);
    cudaError_t e = kvb::launch_verify_tempstate_static(p->view, p->rows, io, c.variant,
                                                        c.kv_dtype, c.d_k, s);
    if (e != cudaSuccess) return cuda_status(e);
  }
  if (!n_accepted) return KVB_OK;
  // rows that accepted something take their temporary state; consecutive rows per launch
  int32_t i = 0;
  for (int32_t b = 0; b < B; ++b) {
    if (n_accepted[b] == 0) continue;
    if (i == kvb::kMaxRows || (i > 0 && b != p->rows.row0 + i)) {
      cudaError_t e = kvb::launch_accept_tempstate_static(p->view, p->rows, T, c.d_k, s);
      if (e != cudaSuccess) return cuda_status(e);
      i = 0;
    }
    if (i == 0) p->rows.row0 = b;
    p->rows.r[i++] = make_row(p, req_ids[b], n_accepted[b], 0);
    p->rows.count = i;
  }
  if (i > 0) {
    cudaError_t e = kvb::launch_accept_tempstate_static(p->view, p->rows, T, c.d_k, s);
    if (e != cudaSuccess) return cuda_status(e);
  }
  return KVB_OK;
}

int kvb_get_lengths(const kvb_pool *p, int32_t *host_out) {
  if (!p || !host_out) return KVB_E_ARG;
  std::memcpy(host_out, p->len.data(), p->len.size() * sizeof(int32_t));
  return KVB_OK;
}

int kvb_get_device_lengths(kvb_pool *p, int32_t *host_out, kvb_stream_t stream) {
  if (!p || !host_out) return KVB_E_ARG;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (cudaMemcpyAsync(host_out, p->d_len, (size_t)p->cfg.max_requests * 4, cudaMemcpyDeviceToHost,
                      s) != cudaSuccess)
    return KVB_E_CUDA;
  return cudaStreamSynchronize(s) == cudaSuccess ? KVB_OK : KVB_E_CUDA;
}

int kvb_get_error(kvb_pool *p, kvb_stream_t stream, int32_t *detail) {
  if (!p) return KVB_E_ARG;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  int32_t w[4] = {0, 0, 0, 0};
  if (cudaMemcpyAsync(w, p->d_err, sizeof(w), cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return KVB_E_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return KVB_E_CUDA;
  if (w[0] == 0) return KVB_OK;
  if (detail) {
    detail[0] = w[0];
    detail[1] = w[1];
    detail[2] = w[2];
  }
  if (cudaMemsetAsync(p->d_err, 0, sizeof(w), s) != cudaSuccess) return KVB_E_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return KVB_E_CUDA;
  return KVB_E_DEVICE;
}

const char *kvb_strerror(int status) {
  switch (status) {
    case KVB_OK: return "ok";
    case KVB_E_ARG: return "invalid argument";
    case KVB_E_CAPACITY: return "buffer capacity exceeded";
    case KVB_E_RANGE: return "id out of range or already owned";
    case KVB_E_STATE: return "call does not fit the request's kind or phase";
    case KVB_E_CUDA: return "CUDA runtime error";
    case KVB_E_DEVICE: return "device-side check failed";
    case KVB_E_UNSUPPORTED: return "shape or dtype not supported";
  }
  return "unknown status";
}

int kvb_copy_probe(const void *src, void *dst, size_t bytes, kvb_stream_t stream) {
  if (!src || !dst || bytes % 16 || !aligned(src, 16) || !aligned(dst, 16)) return KVB_E_ARG;
  if (bytes == 0) return KVB_OK;
  return cuda_status(kvb::launch_copy_probe(src, dst, bytes, reinterpret_cast<cudaStream_t>(stream)));
}

int kvb_set_prefill_wait_limit(int32_t polls) {
  if (polls < 0) return KVB_E_ARG;
  kvb::set_prefill_first_wait_polls(polls);
  return KVB_OK;
}

const char *kvb_version(void) { return "libkvb 0.2 sm_103a"; }

}  // extern "C"
