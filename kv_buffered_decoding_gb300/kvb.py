"""Python binding of libkvb (include/kvb.h): argument marshalling only.

Every step of the path runs in libkvb's CUDA kernels.  This module loads the
in-tree ``_lib/libkvb.so`` and fails loudly if it is missing; there is no
fallback.  PyTorch supplies device memory and the current CUDA stream.

Two layers:
* ``kvb_*`` functions with the C names, taking raw pointers / integers;
* ``Pool``, which allocates the three pool regions as torch tensors and turns
  torch tensors into the pointers, shapes and stream the C calls take.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_lib", "libkvb.so")

KVB_OK = 0
KVB_E_ARG, KVB_E_CAPACITY, KVB_E_RANGE, KVB_E_STATE = -1, -2, -3, -4
KVB_E_CUDA, KVB_E_DEVICE, KVB_E_UNSUPPORTED = -5, -6, -7
KVB_PLAIN, KVB_GATED, KVB_GATED_DELTA = 0, 1, 2
KVB_F32, KVB_BF16 = 0, 1
KVB_MAX_CAPACITY = 64
KVB_MAX_DRAFTS = 64
KVB_STATIC_TEMP_BYTES = 64 << 20

# every symbol include/kvb.h declares
EXPORTS = ("kvb_pool_layout", "kvb_alloc_pool", "kvb_free_pool", "kvb_set_request",
           "kvb_release_request", "kvb_decode", "kvb_short_ctx", "kvb_flush", "kvb_prefill",
           "kvb_promote",
           "kvb_verify",
           "kvb_accept", "kvb_verify_tree", "kvb_accept_tree", "kvb_verify_tempstate",
           "kvb_accept_tempstate",
           "kvb_verify_tempstate_static", "kvb_get_lengths", "kvb_get_device_lengths", "kvb_get_error",
           "kvb_strerror", "kvb_set_prefill_wait_limit", "kvb_copy_probe", "kvb_version")


class KvbConfig(ctypes.Structure):
    _fields_ = [("variant", ctypes.c_int32), ("kv_dtype", ctypes.c_int32),
                ("n_qk_heads", ctypes.c_int32), ("n_v_heads", ctypes.c_int32),
                ("d_k", ctypes.c_int32), ("d_v", ctypes.c_int32), ("m", ctypes.c_int32),
                ("block_size", ctypes.c_int32), ("num_blocks", ctypes.c_int32),
                ("num_state_slots", ctypes.c_int32), ("max_requests", ctypes.c_int32),
                ("max_blocks_per_req", ctypes.c_int32), ("scale", ctypes.c_float)]


class KvbLayout(ctypes.Structure):
    _fields_ = [(name, ctypes.c_size_t) for name in
                ("state_bytes", "kv_bytes", "meta_bytes", "k_off", "v_off", "u_off", "logg_off",
                 "beta_off", "state_slot_stride")]


class KvbError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {kvb_strerror(status)} ({status})")


_lib = None
_P = ctypes.c_void_p
_I32 = ctypes.c_int32
_I32P = ctypes.POINTER(ctypes.c_int32)


def load_library(path: str = LIB_PATH):
    """Load libkvb.so (built by ``__graft_entry__.build()``); raise if it is absent."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"libkvb.so not found at {path}: build it first "
                           "(python -m kv_buffered_decoding_gb300.build)")
    lib = ctypes.CDLL(path)
    sig = {
        "kvb_pool_layout": (ctypes.c_int, [ctypes.POINTER(KvbConfig), ctypes.POINTER(KvbLayout)]),
        "kvb_alloc_pool": (ctypes.c_int, [ctypes.POINTER(KvbConfig), _P, _P, _P,
                                          ctypes.POINTER(_P)]),
        "kvb_free_pool": (ctypes.c_int, [_P]),
        "kvb_set_request": (ctypes.c_int, [_P, _I32, _I32, _I32, _I32P, _P]),
        "kvb_release_request": (ctypes.c_int, [_P, _I32]),
        "kvb_decode": (ctypes.c_int, [_P, _I32, _I32P, _P, _P, _P, _P, _P, _P, _I32, _P]),
        "kvb_short_ctx": (ctypes.c_int, [_P, _I32, _I32P, _P, _P, _P, _P, _P, _P, _P]),
        "kvb_flush": (ctypes.c_int, [_P, _I32, _I32P, _P]),
        "kvb_verify": (ctypes.c_int, [_P, _I32, _I32, _I32P, _P, _P, _P, _P, _P, _P, _P]),
        "kvb_accept": (ctypes.c_int, [_P, _I32, _I32P, _I32P, _P]),
        "kvb_verify_tempstate": (ctypes.c_int, [_P, _I32, _I32, _I32P, _P, _P, _P, _P, _P, _P, _P,
                                                _P]),
        "kvb_accept_tempstate": (ctypes.c_int, [_P, _I32, _I32, _I32P, _I32P, _P, _P]),
        "kvb_promote": (ctypes.c_int, [_P, _I32, _I32P, _I32P, _P]),
        "kvb_verify_tree": (ctypes.c_int, [_P, _I32, _I32, _I32P, _I32P, _P, _P, _P, _P, _P, _P,
                                           _P]),
        "kvb_accept_tree": (ctypes.c_int, [_P, _I32, _I32P, _I32P, _P]),
        "kvb_prefill": (ctypes.c_int, [_P, _I32, _I32, _I32P, _I32P, _P, _P, _P, _P, _P, _P,
                                       _I32, _P]),
        "kvb_verify_tempstate_static": (ctypes.c_int, [_P, _I32, _I32, _I32P, _P, _P, _P, _P, _P,
                                                       _P, _I32P, _P]),
        "kvb_get_lengths": (ctypes.c_int, [_P, _I32P]),
        "kvb_get_device_lengths": (ctypes.c_int, [_P, _I32P, _P]),
        "kvb_get_error": (ctypes.c_int, [_P, _P, _I32P]),
        "kvb_strerror": (ctypes.c_char_p, [ctypes.c_int]),
        "kvb_set_prefill_wait_limit": (ctypes.c_int, [_I32]),
        "kvb_copy_probe": (ctypes.c_int, [_P, _P, ctypes.c_size_t, _P]),
        "kvb_version": (ctypes.c_char_p, []),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def kvb_strerror(status: int) -> str:
    return load_library().kvb_strerror(status).decode()


def kvb_version() -> str:
    return load_library().kvb_version().decode()


def set_prefill_wait_limit(polls: int):
    """Cap the first bounded wait of every tensor-core prefill CTA (0 = default)."""
    _check(load_library().kvb_set_prefill_wait_limit(int(polls)), "kvb_set_prefill_wait_limit")


def _check(status: int, where: str):
    if status != KVB_OK:
        raise KvbError(status, where)


def _i32(arr):
    a = np.ascontiguousarray(np.asarray(arr, dtype=np.int32))
    return a, a.ctypes.data_as(_I32P)


def make_config(variant, kv_dtype, n_qk_heads, n_v_heads, d_k, d_v, m, block_size, num_blocks,
                num_state_slots, max_requests, max_blocks_per_req, scale=1.0) -> KvbConfig:
    return KvbConfig(variant, kv_dtype, n_qk_heads, n_v_heads, d_k, d_v, m, block_size,
                     num_blocks, num_state_slots, max_requests, max_blocks_per_req, scale)


def kvb_pool_layout(cfg: KvbConfig) -> KvbLayout:
    out = KvbLayout()
    _check(load_library().kvb_pool_layout(ctypes.byref(cfg), ctypes.byref(out)), "kvb_pool_layout")
    return out


# ----------------------------------------------------------------------------- Pool
class Pool:
    """A pool over torch-allocated device memory (state, KV buffer, metadata).

    Tensor views of the regions:
      state  [num_state_slots, Hv, d_k, d_v] fp32
      kbuf   [num_blocks, Hk, block_size, d_k]  kv dtype
      vbuf   [num_blocks, Hv, block_size, d_v]  kv dtype
      ubuf   [num_blocks, Hv, block_size, d_v]  fp32 (gated delta only, else None)
      gbuf, bbuf [num_blocks, Hv, block_size]   fp32
    """

    def __init__(self, cfg: KvbConfig, device=None):
        import torch
        self.torch = torch
        self.cfg = cfg
        self.lib = load_library()
        self.device = torch.device(device or "cuda")
        lay = kvb_pool_layout(cfg)
        self.layout = lay

        def region(nbytes):
            # 256-byte aligned: the caching allocator returns 512-byte aligned blocks
            return torch.empty(max(int(nbytes), 256), dtype=torch.uint8, device=self.device)

        self._state_mem = region(lay.state_bytes)
        self._kv_mem = region(lay.kv_bytes)
        self._meta_mem = region(lay.meta_bytes)
        self.kv_torch_dtype = torch.bfloat16 if cfg.kv_dtype == KVB_BF16 else torch.float32
        S, Hk, Hv, dk, dv = (cfg.num_state_slots, cfg.n_qk_heads, cfg.n_v_heads, cfg.d_k, cfg.d_v)
        nb, bs = cfg.num_blocks, cfg.block_size
        self.state = self._state_mem[: S * Hv * dk * dv * 4].view(torch.float32).view(S, Hv, dk, dv)

        def sub(off, count, dtype, shape):
            nbytes = count * (2 if dtype == torch.bfloat16 else 4)
            return self._kv_mem[off: off + nbytes].view(dtype).view(*shape)

        rows = nb * bs
        self.kbuf = sub(lay.k_off, rows * Hk * dk, self.kv_torch_dtype, (nb, Hk, bs, dk))
        self.vbuf = sub(lay.v_off, rows * Hv * dv, self.kv_torch_dtype, (nb, Hv, bs, dv))
        self.ubuf = (sub(lay.u_off, rows * Hv * dv, torch.float32, (nb, Hv, bs, dv))
                     if cfg.variant == KVB_GATED_DELTA else None)
        self.gbuf = sub(lay.logg_off, rows * Hv, torch.float32, (nb, Hv, bs))
        self.bbuf = sub(lay.beta_off, rows * Hv, torch.float32, (nb, Hv, bs))
        h = _P()
        _check(self.lib.kvb_alloc_pool(ctypes.byref(cfg), self._state_mem.data_ptr(),
                                       self._kv_mem.data_ptr(), self._meta_mem.data_ptr(),
                                       ctypes.byref(h)), "kvb_alloc_pool")
        self.handle = h

    # -- lifetime -----------------------------------------------------------
    def close(self):
        if getattr(self, "handle", None):
            self.torch.cuda.synchronize(self.device)
            self.lib.kvb_free_pool(self.handle)
            self.handle = None

    def __del__(self):
        try:
            if getattr(self, "handle", None):
                self.lib.kvb_free_pool(self.handle)
                self.handle = None
        except Exception:
            pass

    # -- helpers ------------------------------------------------------------
    def _stream(self):
        return self.torch.cuda.current_stream(self.device).cuda_stream

    def _ptr(self, t, dtype, shape, name):
        if t is None:
            return None
        if t.device != self.device and not (t.is_cuda and self.device.index is None):
            raise ValueError(f"{name} must be on {self.device}")
        if t.dtype != dtype:
            raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
        if tuple(t.shape) != tuple(shape):
            raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
        return t.data_ptr()

    def _token_ptrs(self, lead, q, k, v, log_g, beta, o):
        c, tdt, f32 = self.cfg, self.kv_torch_dtype, self.torch.float32
        return (self._ptr(q, tdt, lead + (c.n_qk_heads, c.d_k), "q"),
                self._ptr(k, tdt, lead + (c.n_qk_heads, c.d_k), "k"),
                self._ptr(v, tdt, lead + (c.n_v_heads, c.d_v), "v"),
                self._ptr(log_g, f32, lead + (c.n_v_heads,), "log_g"),
                self._ptr(beta, f32, lead + (c.n_v_heads,), "beta"),
                self._ptr(o, f32, lead + (c.n_v_heads, c.d_v), "o"))

    # -- the C calls ----------------------------------------------------------
    def set_request(self, req: int, state_slot: int, block_ids):
        ids, p = _i32(block_ids)
        _check(self.lib.kvb_set_request(self.handle, req, state_slot, len(ids), p, self._stream()),
               "kvb_set_request")

    def release_request(self, req: int):
        _check(self.lib.kvb_release_request(self.handle, req), "kvb_release_request")

    def decode(self, req_ids, q, k, v, log_g=None, beta=None, o=None, auto_flush=True):
        ids, p = _i32(req_ids)
        B = len(ids)
        if o is None:
            o = self.torch.empty(B, self.cfg.n_v_heads, self.cfg.d_v, dtype=self.torch.float32,
                                 device=self.device)
        ptrs = self._token_ptrs((B,), q, k, v, log_g, beta, o)
        _check(self.lib.kvb_decode(self.handle, B, p, *ptrs, int(bool(auto_flush)), self._stream()),
               "kvb_decode")
        return o

    def short_ctx(self, req_ids, q, k, v, log_g=None, beta=None, o=None):
        ids, p = _i32(req_ids)
        B = len(ids)
        if o is None:
            o = self.torch.empty(B, self.cfg.n_v_heads, self.cfg.d_v, dtype=self.torch.float32,
                                 device=self.device)
        ptrs = self._token_ptrs((B,), q, k, v, log_g, beta, o)
        _check(self.lib.kvb_short_ctx(self.handle, B, p, *ptrs, self._stream()), "kvb_short_ctx")
        return o

    def flush(self, req_ids):
        ids, p = _i32(req_ids)
        _check(self.lib.kvb_flush(self.handle, len(ids), p, self._stream()), "kvb_flush")

    def verify(self, req_ids, q, k, v, log_g=None, beta=None, o=None):
        ids, p = _i32(req_ids)
        B = len(ids)
        T = q.shape[1]
        if o is None:
            o = self.torch.empty(B, T, self.cfg.n_v_heads, self.cfg.d_v, dtype=self.torch.float32,
                                 device=self.device)
        ptrs = self._token_ptrs((B, T), q, k, v, log_g, beta, o)
        _check(self.lib.kvb_verify(self.handle, B, T, p, *ptrs, self._stream()), "kvb_verify")
        return o

    def accept(self, req_ids, n_accepted):
        ids, p = _i32(req_ids)
        acc, pa = _i32(n_accepted)
        if len(acc) != len(ids):
            raise ValueError("n_accepted must have one entry per request")
        _check(self.lib.kvb_accept(self.handle, len(ids), p, pa, self._stream()), "kvb_accept")

    def prefill(self, req_ids, q, k, v, log_g=None, beta=None, o=None, lengths=None,
                from_zero=True):
        """kvb_prefill: run prompts [B, L, heads, dim] through the requests' states in
        64-token chunks; returns o [B, L, Hv, d_v] (rows past lengths[b] untouched)."""
        ids, p = _i32(req_ids)
        B, L = len(ids), q.shape[1]
        c = self.cfg
        if o is None:
            o = self.torch.empty(B, L, c.n_v_heads, c.d_v, dtype=self.torch.float32,
                                 device=self.device)
        ptrs = self._token_ptrs((B, L), q, k, v, log_g, beta, o)
        lp = None
        if lengths is not None:
            lens, lp = _i32(lengths)
            if len(lens) != B:
                raise ValueError("prefill: one length per request")
        _check(self.lib.kvb_prefill(self.handle, B, L, p, lp, *ptrs, int(bool(from_zero)),
                                    self._stream()), "kvb_prefill")
        return o

    def promote(self, req_ids, state_slots):
        """kvb_promote: give short-context requests a state slot, folding their buffered
        tokens into it from S = 0."""
        ids, p = _i32(req_ids)
        sl, ps = _i32(state_slots)
        if len(sl) != len(ids):
            raise ValueError("promote: one state slot per request")
        _check(self.lib.kvb_promote(self.handle, len(ids), p, ps, self._stream()), "kvb_promote")

    def verify_tree(self, req_ids, parents, q, k, v, log_g=None, beta=None, o=None):
        """kvb_verify_tree: drafts [B, T, ...] with parents [B, T] (host ints, -1 = root)."""
        ids, p = _i32(req_ids)
        B, T = len(ids), q.shape[1]
        par, pp = _i32(np.asarray(parents).reshape(B, T))
        c = self.cfg
        if o is None:
            o = self.torch.empty(B, T, c.n_v_heads, c.d_v, dtype=self.torch.float32,
                                 device=self.device)
        ptrs = self._token_ptrs((B, T), q, k, v, log_g, beta, o)
        _check(self.lib.kvb_verify_tree(self.handle, B, T, p, pp, *ptrs, self._stream()),
               "kvb_verify_tree")
        return o

    def accept_tree(self, req_ids, accepted):
        """kvb_accept_tree: keep the root path of draft accepted[b] (-1: none)."""
        ids, p = _i32(req_ids)
        acc, pa = _i32(accepted)
        _check(self.lib.kvb_accept_tree(self.handle, len(ids), p, pa, self._stream()),
               "kvb_accept_tree")

    def verify_tempstate(self, req_ids, q, k, v, log_g=None, beta=None, temp=None, o=None):
        """The recurrent verify of the comparison baseline: returns (o, temp) where temp
        [B, T, Hv, d_k, d_v] holds the state after each draft."""
        ids, p = _i32(req_ids)
        B, T = len(ids), q.shape[1]
        c = self.cfg
        if o is None:
            o = self.torch.empty(B, T, c.n_v_heads, c.d_v, dtype=self.torch.float32,
                                 device=self.device)
        if temp is None:
            temp = self.torch.empty(B, T, c.n_v_heads, c.d_k, c.d_v, dtype=self.torch.float32,
                                    device=self.device)
        ptrs = self._token_ptrs((B, T), q, k, v, log_g, beta, o)
        tp = self._ptr(temp, self.torch.float32, (B, T, c.n_v_heads, c.d_k, c.d_v), "temp")
        _check(self.lib.kvb_verify_tempstate(self.handle, B, T, p, *ptrs, tp, self._stream()),
               "kvb_verify_tempstate")
        return o, temp

    def accept_tempstate(self, req_ids, n_accepted, temp):
        ids, p = _i32(req_ids)
        acc, pa = _i32(n_accepted)
        B, T = len(ids), temp.shape[1]
        c = self.cfg
        tp = self._ptr(temp, self.torch.float32, (B, T, c.n_v_heads, c.d_k, c.d_v), "temp")
        _check(self.lib.kvb_accept_tempstate(self.handle, B, T, p, pa, tp, self._stream()),
               "kvb_accept_tempstate")

    def verify_tempstate_static(self, req_ids, q, k, v, log_g=None, beta=None, o=None,
                                n_accepted=None):
        """kvb_verify_tempstate_static: the baseline verify with the temporary states in
        the library's fixed device array (no allocation); optional accept in the same call."""
        ids, p = _i32(req_ids)
        B, T = len(ids), q.shape[1]
        c = self.cfg
        if o is None:
            o = self.torch.empty(B, T, c.n_v_heads, c.d_v, dtype=self.torch.float32,
                                 device=self.device)
        ptrs = self._token_ptrs((B, T), q, k, v, log_g, beta, o)
        acc_p = None
        if n_accepted is not None:
            acc, acc_p = _i32(n_accepted)
        _check(self.lib.kvb_verify_tempstate_static(self.handle, B, T, p, *ptrs, acc_p,
                                                    self._stream()),
               "kvb_verify_tempstate_static")
        return o

    def get_lengths(self) -> np.ndarray:
        out = np.zeros(self.cfg.max_requests, dtype=np.int32)
        _check(self.lib.kvb_get_lengths(self.handle, out.ctypes.data_as(_I32P)), "kvb_get_lengths")
        return out

    def get_device_lengths(self) -> np.ndarray:
        out = np.zeros(self.cfg.max_requests, dtype=np.int32)
        _check(self.lib.kvb_get_device_lengths(self.handle, out.ctypes.data_as(_I32P),
                                               self._stream()), "kvb_get_device_lengths")
        return out

    def get_error(self):
        """Return None, or (kind, request, value) of the first device-side error (cleared)."""
        detail = np.zeros(3, dtype=np.int32)
        st = self.lib.kvb_get_error(self.handle, self._stream(), detail.ctypes.data_as(_I32P))
        if st == KVB_OK:
            return None
        if st == KVB_E_DEVICE:
            return tuple(int(x) for x in detail)
        raise KvbError(st, "kvb_get_error")


def copy_probe(src, dst):
    """128-bit device copy of src into dst (same byte size) on the current stream."""
    import torch
    nbytes = src.numel() * src.element_size()
    if dst.numel() * dst.element_size() != nbytes:
        raise ValueError("src and dst must have the same byte size")
    _check(load_library().kvb_copy_probe(src.data_ptr(), dst.data_ptr(), nbytes,
                                         torch.cuda.current_stream(src.device).cuda_stream),
           "kvb_copy_probe")
