"""Python binding of libkvr: retrieval-based sparse decode attention on GB300.

The functions below carry the C ABI's names (include/kvr.h) and only marshal
arguments: torch CUDA tensors become device pointers, shapes become the
``kvr_shape`` / ``kvr_select_params`` structs, and the caller's current CUDA
stream is passed through. Every step of the computation runs in the CUDA
kernels of ``libkvr.so``; there is no CPU or PyTorch fallback, and a missing
library raises.
"""
from __future__ import annotations

import ctypes
import os

import torch

from . import _build

__all__ = [
    "KvrError", "Shape", "SelectParams", "load", "kvr_status_string", "kvr_version",
    "kvr_encode_keys", "kvr_select_workspace_size", "kvr_select_workspace_views",
    "kvr_select", "kvr_select_static_scratch", "kvr_attend_workspace_size",
    "kvr_sparse_attend", "kvr_read_error",
    "DEFAULT_LUT", "DEVERR", "SELECT_STORE_COARSE", "SELECT_EARLY_INPUTS",
    "SELECT_MAGNITUDE_VOTES", "kvr_codes_bytes",
    "codes_buffer",
    "WINDOW", "TIER_BF16", "TIER_INT2", "TIER_EVICTED", "TierState", "kvr_ledger_bytes",
    "kvr_tier_init", "kvr_tiered_attend_workspace_size", "kvr_sparse_attend_tiered",
    "kvr_tier_update_workspace_size", "kvr_tier_update",
    "kvr_rsq_record_bytes", "kvr_rsq_tables", "kvr_encode_rsq", "rsq_buffer",
    "kvr_sparse_attend_regions", "kvr_regions_update", "kvr_decode_step", "DecodeStep",
    "kvr_select_attend", "SelectAttend",
]

KVR_F32, KVR_BF16 = 0, 1
DEFAULT_LUT = (3, 2, 1, 0, 0, 0, 0, 0, 0)
DEVERR = {"seq_len": 0x1, "position": 0x2, "index": 0x4, "nonfinite": 0x8, "timeout": 0x10,
          "tier": 0x20, "range": 0x40}
WINDOW = 64
TIER_BF16, TIER_INT2, TIER_EVICTED = 0, 1, 2


class KvrError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__("%s: %s (status %d)" % (where, kvr_status_string(status), status))


class _Shape(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int), ("Hq", ctypes.c_int), ("Hkv", ctypes.c_int),
                ("d", ctypes.c_int), ("cap", ctypes.c_int64), ("dtype", ctypes.c_int)]


class _Params(ctypes.Structure):
    _fields_ = [("C", ctypes.c_int), ("k", ctypes.c_int), ("W", ctypes.c_int),
                ("lut", ctypes.c_int * 9), ("flags", ctypes.c_int),
                ("V_prefetch", ctypes.c_void_p), ("rsq_records", ctypes.c_void_p),
                ("sink", ctypes.c_int), ("region_end", ctypes.c_void_p)]


SELECT_STORE_COARSE = 0x1
SELECT_EARLY_INPUTS = 0x2
SELECT_MAGNITUDE_VOTES = 0x4


class _Views(ctypes.Structure):
    _fields_ = [("coarse", ctypes.c_size_t), ("cand_idx", ctypes.c_size_t),
                ("cand_score", ctypes.c_size_t), ("cand_count", ctypes.c_size_t),
                ("qbar", ctypes.c_size_t)]


class _TierState(ctypes.Structure):
    _fields_ = [("n_win", ctypes.c_int64), ("tier", ctypes.c_void_p), ("score", ctypes.c_void_p),
                ("has_ledger", ctypes.c_void_p), ("ledger", ctypes.c_void_p),
                ("quota", ctypes.c_void_p), ("budget", ctypes.c_void_p)]


class Shape:
    """Cache / query shape: K, V [B, Hkv, cap, d]; q [B, Hq, d]."""

    def __init__(self, B, Hq, Hkv, d, cap, dtype):
        self.B, self.Hq, self.Hkv, self.d, self.cap = int(B), int(Hq), int(Hkv), int(d), int(cap)
        if dtype in (torch.bfloat16, "bf16"):
            self.dtype = torch.bfloat16
        elif dtype in (torch.float32, "f32"):
            self.dtype = torch.float32
        else:
            raise ValueError("dtype must be bf16 or f32")

    @classmethod
    def of(cls, K: torch.Tensor, q: torch.Tensor) -> "Shape":
        B, Hkv, cap, d = K.shape
        return cls(B, q.shape[1], Hkv, d, cap, K.dtype)

    def c(self) -> _Shape:
        return _Shape(self.B, self.Hq, self.Hkv, self.d, self.cap,
                      KVR_BF16 if self.dtype == torch.bfloat16 else KVR_F32)


class SelectParams:
    """kvr_select_params. ``V_prefetch``: optional V cache tensor of a
    kvr_sparse_attend that follows (an L2 prefetch hint; results unchanged).
    ``rsq_records``: optional uint8 records of the pool keys (kvr_encode_rsq);
    when given, candidates are ranked by the calibrated estimate.
    ``sink`` / ``region_end``: cache regions (the first ``sink`` tokens are
    never candidates; ``region_end`` int32 [B] ends the Retrieval pool,
    kvr_regions_update)."""

    def __init__(self, C, k, W, lut=DEFAULT_LUT, flags=0, V_prefetch=None, rsq_records=None,
                 sink=0, region_end=None):
        self.C, self.k, self.W = int(C), int(k), int(W)
        self.lut = tuple(int(v) for v in lut)
        self.flags = int(flags)
        if len(self.lut) != 9:
            raise ValueError("lut needs 9 entries (Hamming distance 0..8)")
        if V_prefetch is not None and (not isinstance(V_prefetch, torch.Tensor)
                                       or not V_prefetch.is_cuda):
            raise TypeError("V_prefetch must be a CUDA tensor or None")
        self.V_prefetch = V_prefetch
        if rsq_records is not None:
            _cuda(rsq_records, "rsq_records", torch.uint8)
        self.rsq_records = rsq_records
        if region_end is not None:
            _cuda(region_end, "region_end", torch.int32)
        self.sink = int(sink)
        self.region_end = region_end

    def c(self) -> _Params:
        vp = None if self.V_prefetch is None else self.V_prefetch.data_ptr()
        rp = None if self.rsq_records is None else self.rsq_records.data_ptr()
        re = None if self.region_end is None else self.region_end.data_ptr()
        return _Params(self.C, self.k, self.W, (ctypes.c_int * 9)(*self.lut), self.flags, vp, rp,
                       self.sink, re)


_lib = None
_P = ctypes.c_void_p


def load(build_if_missing: bool = True):
    """Load libkvr.so (built in-tree by ``_build.build``). Raises if unavailable."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(_build.LIB) or not _build.up_to_date():
        if not build_if_missing:
            raise RuntimeError("libkvr.so is not built; run sparse_decode_attention_gb300._build")
        _build.build()
    L = ctypes.CDLL(_build.LIB)
    S, Pp, V = ctypes.POINTER(_Shape), ctypes.POINTER(_Params), ctypes.POINTER(_Views)
    L.kvr_status_string.argtypes = [ctypes.c_int]
    L.kvr_status_string.restype = ctypes.c_char_p
    L.kvr_version.restype = ctypes.c_int
    L.kvr_codes_bytes.argtypes = [S]
    L.kvr_codes_bytes.restype = ctypes.c_size_t
    L.kvr_encode_keys.argtypes = [S, _P, _P, ctypes.c_int, _P, _P, _P, _P]
    L.kvr_select_workspace_size.argtypes = [S, Pp]
    L.kvr_select_workspace_size.restype = ctypes.c_size_t
    L.kvr_select_workspace_views.argtypes = [S, Pp, V]
    L.kvr_select.argtypes = [S, Pp, _P, _P, _P, _P, _P, _P, _P, _P, ctypes.c_size_t, _P, _P]
    L.kvr_select_static_scratch.argtypes = [S, Pp, _P, _P, _P, _P, _P, _P, _P, _P, _P]
    L.kvr_attend_workspace_size.argtypes = [S, ctypes.c_int, ctypes.c_int]
    L.kvr_attend_workspace_size.restype = ctypes.c_size_t
    L.kvr_sparse_attend.argtypes = [S, _P, _P, _P, _P, ctypes.c_int, _P, _P, ctypes.c_int,
                                    ctypes.c_float, _P, _P, ctypes.c_size_t, _P, _P]
    L.kvr_read_error.argtypes = [_P, _P, _P]
    T = ctypes.POINTER(_TierState)
    L.kvr_ledger_bytes.argtypes = [ctypes.c_int]
    L.kvr_ledger_bytes.restype = ctypes.c_size_t
    L.kvr_tier_init.argtypes = [S, T, _P, _P, _P, _P, _P, _P]
    L.kvr_tiered_attend_workspace_size.argtypes = [S, ctypes.c_int64]
    L.kvr_tiered_attend_workspace_size.restype = ctypes.c_size_t
    L.kvr_sparse_attend_tiered.argtypes = [S, T, _P, _P, _P, _P, ctypes.c_float, _P, _P, _P,
                                           ctypes.c_size_t, _P, _P]
    L.kvr_tier_update_workspace_size.argtypes = [S, ctypes.c_int64]
    L.kvr_tier_update_workspace_size.restype = ctypes.c_size_t
    L.kvr_tier_update.argtypes = [S, T, _P, _P, _P, _P, _P, _P, ctypes.c_size_t, _P, _P]
    L.kvr_rsq_record_bytes.argtypes = [ctypes.c_int]
    L.kvr_rsq_record_bytes.restype = ctypes.c_size_t
    L.kvr_rsq_tables.argtypes = [_P, _P]
    L.kvr_encode_rsq.argtypes = [S, _P, _P, ctypes.c_int, _P, _P, _P, _P]
    L.kvr_sparse_attend_regions.argtypes = [S, _P, _P, _P, _P, ctypes.c_int, _P, _P, ctypes.c_int,
                                            _P, ctypes.c_float, _P, _P, ctypes.c_size_t, _P, _P]
    L.kvr_regions_update.argtypes = [ctypes.c_int, _P, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                     ctypes.c_int, _P, _P, _P]
    L.kvr_decode_step.argtypes = [S, Pp, _P, _P, _P, _P, _P, _P, _P, _P, _P, ctypes.c_float, _P,
                                  _P, ctypes.c_size_t, _P, _P]
    L.kvr_select_attend.argtypes = [S, Pp, _P, _P, _P, _P, _P, _P, ctypes.c_float, _P, _P, _P, _P,
                                    ctypes.c_size_t, _P, _P]
    L.kvr_testing_tiered_withheld_copy.argtypes = [S, T, _P, _P, _P, _P, ctypes.c_float, _P, _P,
                                                   _P, ctypes.c_size_t, _P, _P, ctypes.c_int64]
    for fn in ("kvr_encode_keys", "kvr_select_workspace_views", "kvr_select",
               "kvr_select_static_scratch", "kvr_tier_init", "kvr_sparse_attend_tiered",
               "kvr_tier_update", "kvr_rsq_tables", "kvr_encode_rsq",
               "kvr_sparse_attend_regions", "kvr_regions_update", "kvr_decode_step",
               "kvr_select_attend", "kvr_sparse_attend", "kvr_read_error",
               "kvr_testing_tiered_withheld_copy"):
        getattr(L, fn).restype = ctypes.c_int
    _lib = L
    return L


def kvr_status_string(status: int) -> str:
    return load().kvr_status_string(int(status)).decode()


def kvr_codes_bytes(shape: Shape) -> int:
    """Bytes of the bit-plane code buffer for a cache of this shape."""
    return int(load().kvr_codes_bytes(ctypes.byref(shape.c())))


def codes_buffer(shape: Shape, device="cuda") -> torch.Tensor:
    """A zeroed device buffer for the codes of a cache of this shape."""
    return torch.zeros(max(kvr_codes_bytes(shape), 16), dtype=torch.uint8, device=device)


def kvr_version() -> int:
    return load().kvr_version()


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _check(status, where):
    if status != 0:
        raise KvrError(status, where)


def _cuda(t, name, dtype=None):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError("%s must be a CUDA tensor" % name)
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    if dtype is not None and t.dtype != dtype:
        raise TypeError("%s must be %s, got %s" % (name, dtype, t.dtype))
    return t


def _kv(t, name):
    """A K or V cache: a CUDA tensor, or a page-locked host tensor that the
    kernels read through the device's mapping of it (host-resident cache)."""
    if not isinstance(t, torch.Tensor) or not (t.is_cuda or t.is_pinned()):
        raise TypeError("%s must be a CUDA tensor or a page-locked (pinned) host tensor" % name)
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    return t


def _device(*tensors):
    """The one CUDA device of the CUDA tensors among `tensors` (host-resident
    caches are skipped); raises when they are spread over devices."""
    devs = {t.device for t in tensors if isinstance(t, torch.Tensor) and t.is_cuda}
    if len(devs) != 1:
        raise ValueError("the tensors of one call must all be on one CUDA device, got %s"
                         % sorted(str(d) for d in devs))
    return devs.pop()


def _records(params, shape):
    """The reranker records, when given, must hold every key of the cache."""
    if params.rsq_records is not None and (
            params.rsq_records.numel() < shape.B * shape.Hkv * shape.cap * kvr_rsq_record_bytes(shape.d)):
        raise ValueError("rsq_records buffer too small")


def _codes(codes, shape):
    _cuda(codes, "codes", torch.uint8)
    if codes.numel() < kvr_codes_bytes(shape):
        raise ValueError("codes holds %d bytes, the cache needs %d (kvr_codes_bytes)"
                         % (codes.numel(), kvr_codes_bytes(shape)))


def kvr_encode_keys(K, pos0, n_new, srht_sign, codes, err=None, stream=None, shape=None):
    """Encode rows [pos0[b], pos0[b] + n_new) of every unit of K into codes."""
    _kv(K, "K")
    shape = shape or Shape(K.shape[0], K.shape[1], K.shape[1], K.shape[3], K.shape[2], K.dtype)
    _cuda(pos0, "pos0", torch.int32)
    _cuda(srht_sign, "srht_sign", torch.int8)
    _codes(codes, shape)
    with torch.cuda.device(_device(K, pos0, srht_sign, codes, err)):
        st = load().kvr_encode_keys(ctypes.byref(shape.c()), _ptr(K), _ptr(pos0), int(n_new),
                                    _ptr(srht_sign), _ptr(codes), _ptr(err), _stream(stream))
    _check(st, "kvr_encode_keys")


def kvr_select_workspace_size(shape: Shape, params: SelectParams) -> int:
    return int(load().kvr_select_workspace_size(ctypes.byref(shape.c()),
                                                ctypes.byref(params.c())))


def kvr_select_workspace_views(shape: Shape, params: SelectParams) -> dict:
    v = _Views()
    st = load().kvr_select_workspace_views(ctypes.byref(shape.c()), ctypes.byref(params.c()),
                                           ctypes.byref(v))
    _check(st, "kvr_select_workspace_views")
    return {f: int(getattr(v, f)) for f, _ in _Views._fields_}


def kvr_select(q, K, codes, seq_len, srht_sign, params: SelectParams, out_idx, out_count,
               workspace, err=None, stream=None):
    """Coarse score, candidate set, exact rescoring and top-k for every unit."""
    shape = Shape.of(_kv(K, "K"), _cuda(q, "q", K.dtype))
    _codes(codes, shape)
    _cuda(seq_len, "seq_len", torch.int32)
    _cuda(srht_sign, "srht_sign", torch.int8)
    _cuda(out_idx, "out_idx", torch.int32)
    _cuda(out_count, "out_count", torch.int32)
    _cuda(workspace, "workspace")
    _records(params, shape)
    dev = _device(q, K, codes, seq_len, srht_sign, out_idx, out_count, workspace, err,
                  params.V_prefetch, params.rsq_records, params.region_end)
    with torch.cuda.device(dev):
        st = load().kvr_select(ctypes.byref(shape.c()), ctypes.byref(params.c()), _ptr(q), _ptr(K),
                               _ptr(codes), _ptr(seq_len), _ptr(srht_sign), _ptr(out_idx),
                               _ptr(out_count), _ptr(workspace),
                               workspace.numel() * workspace.element_size(), _ptr(err),
                               _stream(stream))
    _check(st, "kvr_select")


def kvr_select_static_scratch(q, K, codes, seq_len, srht_sign, params: SelectParams, out_idx,
                              out_count, err=None, stream=None):
    """kvr_select for callers that cannot allocate: scratch is a fixed device
    array inside the library (16 MiB per GPU), shared by every call on a device."""
    shape = Shape.of(_kv(K, "K"), _cuda(q, "q", K.dtype))
    _codes(codes, shape)
    _cuda(seq_len, "seq_len", torch.int32)
    _cuda(srht_sign, "srht_sign", torch.int8)
    _cuda(out_idx, "out_idx", torch.int32)
    _cuda(out_count, "out_count", torch.int32)
    _records(params, shape)
    # the scratch array used is the current device's: make it the tensors' device
    dev = _device(q, K, codes, seq_len, srht_sign, out_idx, out_count, err, params.V_prefetch,
                  params.rsq_records, params.region_end)
    with torch.cuda.device(dev):
        st = load().kvr_select_static_scratch(ctypes.byref(shape.c()), ctypes.byref(params.c()),
                                              _ptr(q), _ptr(K), _ptr(codes), _ptr(seq_len),
                                              _ptr(srht_sign), _ptr(out_idx), _ptr(out_count),
                                              _ptr(err), _stream(stream))
    _check(st, "kvr_select_static_scratch")


def kvr_attend_workspace_size(shape: Shape, kmax: int, W: int) -> int:
    return int(load().kvr_attend_workspace_size(ctypes.byref(shape.c()), int(kmax), int(W)))


def kvr_sparse_attend(q, K, V, idx, count, seq_len, W, scale, out, workspace, err=None,
                      stream=None):
    """Gather + online-softmax attention over idx[b, h, :count] plus the window."""
    shape = Shape.of(_kv(K, "K"), _cuda(q, "q", K.dtype))
    _kv(V, "V")
    if V.dtype != K.dtype or V.shape != K.shape:
        raise TypeError("V must have K's dtype and shape")
    _cuda(idx, "idx", torch.int32)
    _cuda(count, "count", torch.int32)
    _cuda(seq_len, "seq_len", torch.int32)
    _cuda(out, "out", torch.float32)
    _cuda(workspace, "workspace")
    kmax = idx.shape[-1]
    dev = _device(q, K, V, idx, count, seq_len, out, workspace, err)
    with torch.cuda.device(dev):
        st = load().kvr_sparse_attend(ctypes.byref(shape.c()), _ptr(q), _ptr(K), _ptr(V),
                                      _ptr(idx), int(kmax), _ptr(count), _ptr(seq_len), int(W),
                                      float(scale), _ptr(out), _ptr(workspace),
                                      workspace.numel() * workspace.element_size(), _ptr(err),
                                      _stream(stream))
    _check(st, "kvr_sparse_attend")


def kvr_read_error(err, stream=None) -> int:
    """Synchronise, return and clear the device error bits."""
    bits = ctypes.c_int32(0)
    st = load().kvr_read_error(_ptr(err), ctypes.byref(bits), _stream(stream))
    if st not in (0, 5):
        _check(st, "kvr_read_error")
    return int(bits.value)


# --------------------------------------------------------------------------
# tiered window cache
# --------------------------------------------------------------------------

def kvr_ledger_bytes(d: int) -> int:
    return int(load().kvr_ledger_bytes(int(d)))


class TierState:
    """Device arrays of the tiered cache (kvr_tier_state): for U = B * Hkv
    units and n_win windows each, tier int8, score int64, has_ledger uint8,
    ledger uint8 [U, n_win, 48 d], quota int32 [U], budget int64 [U]."""

    def __init__(self, U: int, n_win: int, d: int, device="cuda"):
        self.U, self.n_win, self.d = int(U), int(n_win), int(d)
        self.tier = torch.zeros((U, n_win), dtype=torch.int8, device=device)
        self.score = torch.zeros((U, n_win), dtype=torch.int64, device=device)
        self.has_ledger = torch.zeros((U, n_win), dtype=torch.uint8, device=device)
        self.ledger = torch.zeros((U, n_win, kvr_ledger_bytes(d)), dtype=torch.uint8,
                                  device=device)
        self.quota = torch.zeros(U, dtype=torch.int32, device=device)
        self.budget = torch.zeros(U, dtype=torch.int64, device=device)

    def c(self) -> _TierState:
        return _TierState(self.n_win, self.tier.data_ptr(), self.score.data_ptr(),
                          self.has_ledger.data_ptr(), self.ledger.data_ptr(),
                          self.quota.data_ptr(), self.budget.data_ptr())


def kvr_tier_init(state: TierState, initial_tier, K, V, seq_len, q_heads: int, err=None,
                  stream=None):
    """Tiers, scores, ledgers of the initially INT2 windows, quota, budget."""
    _cuda(K, "K", torch.bfloat16)
    _cuda(V, "V", torch.bfloat16)
    _cuda(initial_tier, "initial_tier", torch.int8)
    _cuda(seq_len, "seq_len", torch.int32)
    if initial_tier.numel() < state.U * state.n_win:
        raise ValueError("initial_tier must hold [U, n_win] entries")
    B, Hkv, cap, d = K.shape
    shape = Shape(B, q_heads, Hkv, d, cap, torch.bfloat16)
    with torch.cuda.device(_device(initial_tier, K, V, seq_len, err, state.tier)):
        st = load().kvr_tier_init(ctypes.byref(shape.c()), ctypes.byref(state.c()),
                                  _ptr(initial_tier), _ptr(K), _ptr(V), _ptr(seq_len), _ptr(err),
                                  _stream(stream))
    _check(st, "kvr_tier_init")


def kvr_tiered_attend_workspace_size(shape: Shape, n_win: int) -> int:
    return int(load().kvr_tiered_attend_workspace_size(ctypes.byref(shape.c()), int(n_win)))


def kvr_sparse_attend_tiered(state: TierState, q, K, V, seq_len, scale, out, window_mass,
                             workspace, err=None, stream=None):
    """Attention over bf16 + INT2 windows + the open window; window masses."""
    shape = Shape.of(_cuda(K, "K", torch.bfloat16), _cuda(q, "q", torch.bfloat16))
    _cuda(V, "V", torch.bfloat16)
    _cuda(seq_len, "seq_len", torch.int32)
    _cuda(out, "out", torch.float32)
    _cuda(window_mass, "window_mass", torch.float32)
    _cuda(workspace, "workspace")
    if window_mass.numel() < state.U * state.n_win:
        raise ValueError("window_mass must hold [U, n_win] entries")
    with torch.cuda.device(_device(q, K, V, seq_len, out, window_mass, workspace, err,
                                   state.tier)):
        st = load().kvr_sparse_attend_tiered(ctypes.byref(shape.c()), ctypes.byref(state.c()),
                                             _ptr(q), _ptr(K), _ptr(V), _ptr(seq_len),
                                             float(scale), _ptr(out), _ptr(window_mass),
                                             _ptr(workspace),
                                             workspace.numel() * workspace.element_size(),
                                             _ptr(err), _stream(stream))
    _check(st, "kvr_sparse_attend_tiered")


def kvr_tier_update_workspace_size(shape: Shape, n_win: int) -> int:
    return int(load().kvr_tier_update_workspace_size(ctypes.byref(shape.c()), int(n_win)))


def kvr_tier_update(state: TierState, window_mass, seq_len, K, V, q_heads: int, stats,
                    workspace, err=None, stream=None):
    """One routing step: scores, ranks, tiers, ledger writes and promotions."""
    _cuda(K, "K", torch.bfloat16)
    _cuda(V, "V", torch.bfloat16)
    _cuda(window_mass, "window_mass", torch.float32)
    _cuda(seq_len, "seq_len", torch.int32)
    _cuda(workspace, "workspace")
    if stats is not None:
        _cuda(stats, "stats", torch.int32)
    B, Hkv, cap, d = K.shape
    shape = Shape(B, q_heads, Hkv, d, cap, torch.bfloat16)
    with torch.cuda.device(_device(window_mass, seq_len, K, V, stats, workspace, err,
                                   state.tier)):
        st = load().kvr_tier_update(ctypes.byref(shape.c()), ctypes.byref(state.c()),
                                    _ptr(window_mass), _ptr(seq_len), _ptr(K), _ptr(V),
                                    _ptr(stats), _ptr(workspace),
                                    workspace.numel() * workspace.element_size(), _ptr(err),
                                    _stream(stream))
    _check(st, "kvr_tier_update")


def workspace(nbytes: int, device="cuda") -> torch.Tensor:
    """A 256-byte aligned device buffer of at least nbytes (torch allocation)."""
    return torch.empty(max(int(nbytes), 256), dtype=torch.uint8, device=device)


def kvr_rsq_record_bytes(d: int) -> int:
    """Bytes of one key's reranker record (0 for an unsupported d)."""
    return int(load().kvr_rsq_record_bytes(int(d)))


def kvr_rsq_tables():
    """(bsq, lev): the float32 squared bin edges and levels of the 3-bit
    magnitude quantiser, as the library computed them."""
    bsq = (ctypes.c_float * 8)()
    lev = (ctypes.c_float * 8)()
    _check(load().kvr_rsq_tables(ctypes.cast(bsq, ctypes.c_void_p),
                                 ctypes.cast(lev, ctypes.c_void_p)), "kvr_rsq_tables")
    return list(bsq), list(lev)


def rsq_buffer(K, device=None):
    """Zeroed uint8 device records [B, Hkv, cap, record bytes] for a K cache
    [B, Hkv, cap, d] (on K's device, or the current CUDA device for a
    host-resident K)."""
    B, Hkv, cap, d = K.shape
    rb = kvr_rsq_record_bytes(d)
    if rb == 0:
        raise ValueError("the reranker supports d = 64 or 128")
    if device is None:
        device = K.device if K.is_cuda else torch.device("cuda", torch.cuda.current_device())
    return torch.zeros((B, Hkv, cap, rb), dtype=torch.uint8, device=device)


def kvr_encode_rsq(K, pos0, n_new, srht_sign, records, err=None, stream=None):
    """Reranker records of rows [pos0[b], pos0[b] + n_new) of every unit of K."""
    _kv(K, "K")
    shape = Shape(K.shape[0], K.shape[1], K.shape[1], K.shape[3], K.shape[2], K.dtype)
    _cuda(pos0, "pos0", torch.int32)
    _cuda(srht_sign, "srht_sign", torch.int8)
    _cuda(records, "records", torch.uint8)
    if records.numel() < K.shape[0] * K.shape[1] * K.shape[2] * kvr_rsq_record_bytes(K.shape[3]):
        raise ValueError("records buffer too small")
    with torch.cuda.device(_device(K, pos0, srht_sign, records, err)):
        st = load().kvr_encode_rsq(ctypes.byref(shape.c()), _ptr(K), _ptr(pos0), int(n_new),
                                   _ptr(srht_sign), _ptr(records), _ptr(err), _stream(stream))
    _check(st, "kvr_encode_rsq")


def kvr_sparse_attend_regions(q, K, V, idx, count, seq_len, sink, region_end, scale, out,
                              workspace, err=None, stream=None):
    """Attention over the Sink, idx[b, h, :count] and [region_end[b], N)."""
    shape = Shape.of(_kv(K, "K"), _cuda(q, "q", K.dtype))
    _kv(V, "V")
    if V.dtype != K.dtype or V.shape != K.shape:
        raise TypeError("V must have K's dtype and shape")
    _cuda(idx, "idx", torch.int32)
    _cuda(count, "count", torch.int32)
    _cuda(seq_len, "seq_len", torch.int32)
    _cuda(region_end, "region_end", torch.int32)
    _cuda(out, "out", torch.float32)
    _cuda(workspace, "workspace")
    with torch.cuda.device(_device(q, K, V, idx, count, seq_len, region_end, out, workspace,
                                   err)):
        st = load().kvr_sparse_attend_regions(ctypes.byref(shape.c()), _ptr(q), _ptr(K),
                                              _ptr(V), _ptr(idx), int(idx.shape[-1]),
                                              _ptr(count), _ptr(seq_len), int(sink),
                                              _ptr(region_end), float(scale), _ptr(out),
                                              _ptr(workspace),
                                              workspace.numel() * workspace.element_size(),
                                              _ptr(err), _stream(stream))
    _check(st, "kvr_sparse_attend_regions")


def kvr_regions_update(seq_len, sink, local, buffer, region_end, init=False, err=None,
                       stream=None):
    """Retrieval end of every batch entry after appends (or at set-up)."""
    _cuda(seq_len, "seq_len", torch.int32)
    _cuda(region_end, "region_end", torch.int32)
    if region_end.numel() < seq_len.numel():
        raise ValueError("region_end needs one entry per batch entry")
    with torch.cuda.device(_device(seq_len, region_end, err)):
        st = load().kvr_regions_update(int(seq_len.numel()), _ptr(seq_len), int(sink),
                                       int(local), int(buffer), 1 if init else 0,
                                       _ptr(region_end), _ptr(err), _stream(stream))
    _check(st, "kvr_regions_update")


def _decode_args(q, K, V, codes, seq_len, pos_new, srht_sign, params, out_idx, out_count, scale,
                 out, workspace, err, stream):
    shape = Shape.of(_kv(K, "K"), _cuda(q, "q", K.dtype))
    _kv(V, "V")
    if V.dtype != K.dtype or V.shape != K.shape:
        raise TypeError("V must have K's dtype and shape")
    _codes(codes, shape)
    for t, n, dt in ((seq_len, "seq_len", torch.int32), (pos_new, "pos_new", torch.int32),
                     (srht_sign, "srht_sign", torch.int8), (out_idx, "out_idx", torch.int32),
                     (out_count, "out_count", torch.int32), (out, "out", torch.float32)):
        _cuda(t, n, dt)
    _cuda(workspace, "workspace")
    if out_idx.shape[-1] != params.k:
        raise ValueError("out_idx rows must hold params.k entries")
    _records(params, shape)
    dev = _device(q, K, V, codes, seq_len, pos_new, srht_sign, out_idx, out_count, out,
                  workspace, err, params.rsq_records, params.region_end)
    with torch.cuda.device(dev):
        strm = _stream(stream)
    return (ctypes.byref(shape.c()), ctypes.byref(params.c()), _ptr(q), _ptr(K), _ptr(V),
            _ptr(codes), _ptr(seq_len), _ptr(pos_new), _ptr(srht_sign), _ptr(out_idx),
            _ptr(out_count), float(scale), _ptr(out), _ptr(workspace),
            workspace.numel() * workspace.element_size(), _ptr(err), strm), dev


def kvr_decode_step(q, K, V, codes, seq_len, pos_new, srht_sign, params: SelectParams, out_idx,
                    out_count, scale, out, workspace, err=None, stream=None):
    """Code (and record) of the appended key at pos_new, selection and
    attention, in one library call."""
    args, dev = _decode_args(q, K, V, codes, seq_len, pos_new, srht_sign, params, out_idx,
                             out_count, scale, out, workspace, err, stream)
    with torch.cuda.device(dev):
        _check(load().kvr_decode_step(*args), "kvr_decode_step")


class DecodeStep:
    """kvr_decode_step with its arguments marshalled once: calling it enqueues
    the step on the stream given at construction with no per-call argument
    conversion (the tensors must stay alive and in place)."""

    def __init__(self, q, K, V, codes, seq_len, pos_new, srht_sign, params: SelectParams, out_idx,
                 out_count, scale, out, workspace, err=None, stream=None):
        self._keep = (q, K, V, codes, seq_len, pos_new, srht_sign, params, out_idx, out_count,
                      out, workspace, err, stream)
        self._args, self._dev = _decode_args(q, K, V, codes, seq_len, pos_new, srht_sign, params,
                                             out_idx, out_count, scale, out, workspace, err,
                                             stream)
        self._fn = load().kvr_decode_step

    def __call__(self):
        with torch.cuda.device(self._dev):
            st = self._fn(*self._args)
        if st != 0:
            raise KvrError(st, "kvr_decode_step")


def _select_attend_args(q, K, V, codes, seq_len, srht_sign, params, scale, out_idx, out_count, out,
                        workspace, err, stream):
    shape = Shape.of(_kv(K, "K"), _cuda(q, "q", K.dtype))
    _kv(V, "V")
    if V.dtype != K.dtype or V.shape != K.shape:
        raise TypeError("V must have K's dtype and shape")
    _codes(codes, shape)
    for t, n, dt in ((seq_len, "seq_len", torch.int32), (srht_sign, "srht_sign", torch.int8),
                     (out_idx, "out_idx", torch.int32), (out_count, "out_count", torch.int32),
                     (out, "out", torch.float32)):
        _cuda(t, n, dt)
    _cuda(workspace, "workspace")
    if out_idx.shape[-1] != params.k:
        raise ValueError("out_idx rows must hold params.k entries")
    _records(params, shape)
    dev = _device(q, K, V, codes, seq_len, srht_sign, out_idx, out_count, out, workspace, err,
                  params.rsq_records, params.region_end)
    with torch.cuda.device(dev):
        strm = _stream(stream)
    return (ctypes.byref(shape.c()), ctypes.byref(params.c()), _ptr(q), _ptr(K), _ptr(V),
            _ptr(codes), _ptr(seq_len), _ptr(srht_sign), float(scale), _ptr(out_idx),
            _ptr(out_count), _ptr(out), _ptr(workspace),
            workspace.numel() * workspace.element_size(), _ptr(err), strm), dev


def kvr_select_attend(q, K, V, codes, seq_len, srht_sign, params: SelectParams, scale, out_idx,
                      out_count, out, workspace, err=None, stream=None):
    """kvr_select, then the attention over its top-k and the window (one
    kernel launch for groups of up to 4 heads with exact rescoring)."""
    args, dev = _select_attend_args(q, K, V, codes, seq_len, srht_sign, params, scale, out_idx,
                                    out_count, out, workspace, err, stream)
    with torch.cuda.device(dev):
        _check(load().kvr_select_attend(*args), "kvr_select_attend")


class SelectAttend:
    """kvr_select_attend with its arguments marshalled once (the tensors must
    stay alive and in place); calling it enqueues the call."""

    def __init__(self, q, K, V, codes, seq_len, srht_sign, params: SelectParams, scale, out_idx,
                 out_count, out, workspace, err=None, stream=None):
        self._keep = (q, K, V, codes, seq_len, srht_sign, params, out_idx, out_count, out,
                      workspace, err, stream)
        self._args, self._dev = _select_attend_args(q, K, V, codes, seq_len, srht_sign, params,
                                                    scale, out_idx, out_count, out, workspace,
                                                    err, stream)
        self._fn = load().kvr_select_attend

    def __call__(self):
        with torch.cuda.device(self._dev):
            st = self._fn(*self._args)
        if st != 0:
            raise KvrError(st, "kvr_select_attend")


def _testing_tiered_withheld_copy(state: TierState, q, K, V, seq_len, scale, out, window_mass,
                                  workspace, wait_ns, err=None, stream=None):
    """Test hook (kvr_testing.h): the tiered attention with each CTA's last
    bulk copy withheld and every copy wait limited to wait_ns; its wait runs
    out and sets the timeout bit. Outputs are invalid afterwards."""
    shape = Shape.of(_cuda(K, "K", torch.bfloat16), _cuda(q, "q", torch.bfloat16))
    _cuda(V, "V", torch.bfloat16)
    _cuda(seq_len, "seq_len", torch.int32)
    _cuda(out, "out", torch.float32)
    _cuda(window_mass, "window_mass", torch.float32)
    _cuda(workspace, "workspace")
    st = load().kvr_testing_tiered_withheld_copy(
        ctypes.byref(shape.c()), ctypes.byref(state.c()), _ptr(q), _ptr(K), _ptr(V),
        _ptr(seq_len), float(scale), _ptr(out), _ptr(window_mass), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _ptr(err), _stream(stream), int(wait_ns))
    _check(st, "kvr_testing_tiered_withheld_copy")
