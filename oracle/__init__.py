"""CPU oracle for retrieval-based sparse decode attention.

TEST INFRASTRUCTURE. Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference leg of ``bench.py`` may import this package. The
CUDA library and its Python binding never import it, and it imports nothing
from them.

The arithmetic lives in ``kvr_oracle.c`` (plain single-threaded C, built with
``-O2 -ffp-contract=off``); this module only builds it, loads it with ctypes
and loops over the independent (batch, kv-head) units. Inputs are numpy
arrays or CPU torch tensors; bf16 tensors are widened to fp32 exactly.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = [os.path.join(_HERE, "kvr_oracle.c"), os.path.join(_HERE, "kvr_tiers_oracle.c"),
        os.path.join(_HERE, "kvr_rsq_oracle.c"), os.path.join(_HERE, "kvr_regions_oracle.c"),
        os.path.join(_HERE, "kvr_votes_oracle.c")]
_LIB = os.path.join(_HERE, "libkvr_oracle.so")
_lib = None

_P = ctypes.c_void_p
_I64 = ctypes.c_int64
_I32 = ctypes.c_int


def build(force: bool = False) -> str:
    """Compile the oracle into ``oracle/libkvr_oracle.so`` (gcc, no fast-math)."""
    srcs = [s for s in _SRC if os.path.exists(s)]
    newest = max(os.path.getmtime(s) for s in srcs)
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= newest:
        return _LIB
    tmp = _LIB + ".tmp%d" % os.getpid()
    cmd = ["gcc", "-O2", "-ffp-contract=off", "-fno-fast-math", "-std=c11", "-fPIC",
           "-shared", "-o", tmp] + srcs + ["-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def lib():
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(_LIB)
        L.orc_fwht_f32.argtypes = [_P, _I32]
        L.orc_srht_unit_f64.argtypes = [_P, _I32, _P, _P]
        L.orc_encode.argtypes = [_P, _I64, _I32, _P, _P]
        L.orc_group_mean.argtypes = [_P, _I32, _I32, _P]
        L.orc_coarse_scores.argtypes = [_P, _I64, _I32, _P, _P, _P]
        L.orc_top_by_int.argtypes = [_P, _I64, _I64, _P]
        L.orc_top_by_int.restype = _I64
        L.orc_top_by_float.argtypes = [_P, _P, _I64, _I64, _P]
        L.orc_top_by_float.restype = _I64
        L.orc_exact_score.argtypes = [_P, _P, _I32]
        L.orc_exact_score.restype = ctypes.c_float
        L.orc_select_unit.argtypes = [_P, _I32, _P, _P, _I64, _I32, _P, _I64, _I64, _I64,
                                      _P, _P, _P, _P, _P, _P, _P]
        L.orc_attend_unit.argtypes = [_P, _I32, _P, _P, _I64, _I32, _P, _I64, _I64,
                                      ctypes.c_float, _P]
        _tier_signatures(L)
        _rsq_signatures(L)
        _region_signatures(L)
        L.orc_flip_cost.argtypes = [_P, ctypes.c_uint]
        L.orc_flip_cost.restype = ctypes.c_float
        L.orc_mag_vote_table.argtypes = [_P, _I32, _P, _P]
        L.orc_mag_vote_table.restype = _I32
        L.orc_select_unit_mag.argtypes = [_P, _I32, _P, _P, _I64, _I32, _P, _I64, _I64, _I64, _P,
                                          _P, _P, _P, _P, _P, _P]
        L.orc_select_unit_mag.restype = _I32
        _lib = L
    return _lib


def _region_signatures(L):
    L.orc_region_init.argtypes = [_I64, _I64, _I64]
    L.orc_region_init.restype = _I64
    L.orc_region_advance.argtypes = [_I64, _I64, _I64, _I64, _I64]
    L.orc_region_advance.restype = _I64
    L.orc_select_unit_regions.argtypes = [_P, _I32, _P, _P, _P, _I64, _I32, _P, _I64, _I64, _I64,
                                          _I64, _P, _P, _P, _P, _P, _P]
    L.orc_select_unit_regions.restype = _I32
    L.orc_attend_unit_regions.argtypes = [_P, _I32, _P, _P, _I64, _I32, _I64, _I64, _P, _I64,
                                          ctypes.c_float, _P]
    L.orc_attend_unit_regions.restype = _I32


def _rsq_signatures(L):
    L.orc_rsq_table.argtypes = [_I32, _P, _P]
    L.orc_rsq_table.restype = _I32
    L.orc_rsq_float_tables.argtypes = [_I32, _P, _P]
    L.orc_rsq_float_tables.restype = _I32
    L.orc_rsq_record_bytes.argtypes = [_I32]
    L.orc_rsq_record_bytes.restype = _I64
    L.orc_rsq_encode.argtypes = [_P, _I64, _I32, _P, _P]
    L.orc_rsq_encode.restype = _I32
    L.orc_rsq_score.argtypes = [_P, _P, _I32]
    L.orc_rsq_score.restype = ctypes.c_float
    L.orc_select_unit_rsq.argtypes = [_P, _I32, _P, _P, _I64, _I32, _P, _I64, _I64, _I64, _P,
                                      _P, _P, _P, _P]
    L.orc_select_unit_rsq.restype = _I32


def _tier_signatures(L):
    u16 = ctypes.c_uint16
    L.orc_f32_to_f16_rd.argtypes = [ctypes.c_float]
    L.orc_f32_to_f16_rd.restype = u16
    L.orc_f32_to_f16_ru.argtypes = [ctypes.c_float]
    L.orc_f32_to_f16_ru.restype = u16
    L.orc_f16_to_f32.argtypes = [u16]
    L.orc_f16_to_f32.restype = ctypes.c_float
    L.orc_f16_next_up.argtypes = [u16]
    L.orc_f16_next_up.restype = u16
    L.orc_bf16_round.argtypes = [ctypes.c_float]
    L.orc_bf16_round.restype = ctypes.c_float
    L.orc_f32_to_f16_array.argtypes = [_P, _I64, _I32, _P]
    L.orc_bf16_round_array.argtypes = [_P, _I64, _P]
    L.orc_int2_quantize_group.argtypes = [_P, _P, _P, _P]
    L.orc_int2_quantize_group.restype = _I32
    L.orc_int2_dequantize_group.argtypes = [_P, u16, u16, _P]
    L.orc_ledger_bytes.argtypes = [_I32]
    L.orc_ledger_bytes.restype = _I64
    L.orc_ledger_write_window.argtypes = [_P, _P, _I32, _P]
    L.orc_ledger_write_window.restype = _I32
    L.orc_ledger_read_window.argtypes = [_P, _I32, _P, _P]
    L.orc_tiered_attend_unit.argtypes = [_P, _I32, _P, _P, _P, _P, _I64, _I32,
                                         ctypes.c_float, _P, _P]
    L.orc_tiered_attend_unit.restype = _I32
    L.orc_tier_init_unit.argtypes = [_P, _P, _P, _I64, _I32, _I64, _P, _P, _P, _P, _P, _P]
    L.orc_tier_init_unit.restype = _I32
    L.orc_tier_update_unit.argtypes = [_P, _P, _P, _P, _P, _P, _P, _I64, _I32, _I32, _I64, _P]
    L.orc_tier_update_unit.restype = _I32


# --------------------------------------------------------------------------
# array helpers
# --------------------------------------------------------------------------

def f32(x) -> np.ndarray:
    """fp32 C-contiguous numpy copy; bf16 / fp16 torch tensors widen exactly."""
    try:
        import torch
        if isinstance(x, torch.Tensor):
            return np.ascontiguousarray(x.detach().to("cpu", torch.float32).numpy())
    except ImportError:  # pragma: no cover
        pass
    return np.ascontiguousarray(np.asarray(x, dtype=np.float32))


def _c(a, dtype):
    return np.ascontiguousarray(np.asarray(a, dtype=dtype))


def _p(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


# --------------------------------------------------------------------------
# the steps, exposed one by one
# --------------------------------------------------------------------------

def fwht(x) -> np.ndarray:
    """Natural-order FWHT of each row of x (fp32, canonical stage order)."""
    a = f32(x).copy()
    d = a.shape[-1]
    flat = a.reshape(-1, d)
    for r in range(flat.shape[0]):
        row = np.ascontiguousarray(flat[r])
        lib().orc_fwht_f32(_p(row), d)
        flat[r] = row
    return flat.reshape(a.shape)


def srht_unit(x, sgn) -> np.ndarray:
    """fp64 rotated unit vector (1/sqrt(d)) H D x / ||x|| of one vector."""
    a = f32(x)
    s = _c(sgn, np.int8)
    y = np.zeros(a.shape[-1], dtype=np.float64)
    lib().orc_srht_unit_f64(_p(a), a.shape[-1], _p(s), _p(y))
    return y


def encode(x, sgn) -> np.ndarray:
    """Sign codes [..., d/8] uint8 of the rows of x [..., d]."""
    a = f32(x)
    d = a.shape[-1]
    n = a.size // d
    s = _c(sgn, np.int8)
    out = np.zeros(a.shape[:-1] + (d // 8,), dtype=np.uint8)
    rc = lib().orc_encode(_p(a), n, d, _p(s), _p(out))
    if rc != 0:
        raise ValueError("unsupported head_dim %d" % d)
    return out


def group_mean(q) -> np.ndarray:
    """Mean query q_bar [d] of the group's heads q [G, d]."""
    a = f32(q)
    G, d = a.shape
    out = np.zeros(d, dtype=np.float32)
    lib().orc_group_mean(_p(a), G, d, _p(out))
    return out


def coarse_scores(codes, qcode, lut) -> np.ndarray:
    c = _c(codes, np.uint8)
    nb = c.shape[-1]
    n = c.size // nb
    qc = _c(qcode, np.uint8)
    lt = _c(lut, np.int32)
    out = np.zeros(n, dtype=np.int32)
    lib().orc_coarse_scores(_p(c), n, nb, _p(qc), _p(lt), _p(out))
    return out


def top_by_int(score, c) -> np.ndarray:
    s = _c(score, np.int32)
    out = np.zeros(max(1, min(c, s.size)), dtype=np.int64)
    n = lib().orc_top_by_int(_p(s), s.size, c, _p(out))
    return out[:n]


def top_by_float(score, index, c) -> np.ndarray:
    s = _c(score, np.float32)
    ix = _c(index, np.int64)
    out = np.zeros(max(1, min(c, s.size)), dtype=np.int64)
    n = lib().orc_top_by_float(_p(s), _p(ix), s.size, c, _p(out))
    if n < 0:
        raise ValueError("NaN exact score")
    return out[:n]


def exact_score(qbar, k) -> np.float32:
    a = f32(qbar)
    b = f32(k)
    return np.float32(lib().orc_exact_score(_p(a), _p(b), a.shape[-1]))


# --------------------------------------------------------------------------
# whole calls over [B, H, ...] tensors
# --------------------------------------------------------------------------

def encode_cache(K, sgn) -> np.ndarray:
    """Codes [B, Hkv, n, d/8] of a whole cache K [B, Hkv, n, d]."""
    return encode(K, sgn)


def select_unit(q_group, K_unit, codes_unit, N, sgn, C, k, W, lut, diagnostics=False):
    """Steps 1-4 of one unit; returns (idx[k] padded -1, count[, diag dict])."""
    q = f32(q_group)
    G, d = q.shape
    Kf = f32(K_unit)
    cd = _c(codes_unit, np.uint8)
    s = _c(sgn, np.int8)
    lt = _c(lut, np.int32)
    idx = np.full(max(k, 1), -1, dtype=np.int32)
    cnt = np.zeros(1, dtype=np.int32)
    pool = max(0, N - W)
    nc = max(0, min(C, pool))
    cand = np.full(max(nc, 1), -1, dtype=np.int32)
    candS = np.zeros(max(nc, 1), dtype=np.float32)
    coarse = np.zeros(max(pool, 1), dtype=np.int32)
    qcode = np.zeros(d // 8, dtype=np.uint8)
    if diagnostics:
        extra = (_p(cand), _p(candS), _p(coarse), _p(qcode))
    else:
        extra = (None, None, None, None)
    rc = lib().orc_select_unit(_p(q), G, _p(Kf), _p(cd), N, d, _p(s), C, k, W, _p(lt),
                               _p(idx), _p(cnt), *extra)
    if rc != 0:
        raise ValueError("oracle selection failed (NaN score or bad shape)")
    if not diagnostics:
        return idx[:k], int(cnt[0])
    return idx[:k], int(cnt[0]), dict(cand=cand[:nc], cand_S=candS[:nc],
                                      coarse=coarse[:pool], qcode=qcode)


def select(q, K, codes, seq_len, sgn, C, k, W, lut, units=None):
    """kvr_select over all units. q [B,Hq,d]; K [B,Hkv,cap,d]; codes [B,Hkv,cap,nb].

    Returns idx [B, Hkv, k] int32 (ascending, -1 padded) and count [B, Hkv].
    ``units`` optionally restricts the work to a list of (b, h) pairs (the
    other rows are left at -1 / 0).
    """
    B, Hq, d = q.shape
    Hkv = K.shape[1]
    G = Hq // Hkv
    out = np.full((B, Hkv, k), -1, dtype=np.int32)
    cnt = np.zeros((B, Hkv), dtype=np.int32)
    todo = units if units is not None else [(b, h) for b in range(B) for h in range(Hkv)]
    for b, h in todo:
        N = int(seq_len[b])
        i, c = select_unit(q[b, h * G:(h + 1) * G], K[b, h, :N], codes[b, h, :N], N, sgn,
                           C, k, W, lut)
        out[b, h] = i
        cnt[b, h] = c
    return out, cnt


def attend_unit(q_group, K_unit, V_unit, N, idx, count, W, scale) -> np.ndarray:
    q = f32(q_group)
    G, d = q.shape
    Kf = f32(K_unit)
    Vf = f32(V_unit)
    ix = _c(idx, np.int32)
    out = np.zeros((G, d), dtype=np.float64)
    rc = lib().orc_attend_unit(_p(q), G, _p(Kf), _p(Vf), N, d, _p(ix), count, W,
                               float(scale), _p(out))
    if rc != 0:
        raise ValueError("selected index outside the pool")
    return out


def attend(q, K, V, idx, count, seq_len, W, scale, units=None):
    """kvr_sparse_attend over all units; returns out [B, Hq, d] fp64."""
    B, Hq, d = q.shape
    Hkv = K.shape[1]
    G = Hq // Hkv
    out = np.zeros((B, Hq, d), dtype=np.float64)
    todo = units if units is not None else [(b, h) for b in range(B) for h in range(Hkv)]
    for b, h in todo:
        N = int(seq_len[b])
        c = int(count[b, h])
        out[b, h * G:(h + 1) * G] = attend_unit(q[b, h * G:(h + 1) * G], K[b, h, :N],
                                                V[b, h, :N], N, idx[b, h, :c], c, W, scale)
    return out


# --------------------------------------------------------------------------
# tiered window cache (kvr_tiers_oracle.c)
# --------------------------------------------------------------------------

WINDOW = 64
BF16, INT2, EVICTED = 0, 1, 2


def f16_round(x, direction: str) -> np.ndarray:
    """fp16 bit patterns (uint16) of x rounded 'down' (toward -inf) or 'up'."""
    a = f32(x).ravel()
    out = np.zeros(a.size, dtype=np.uint16)
    lib().orc_f32_to_f16_array(_p(a), a.size, -1 if direction == "down" else 1, _p(out))
    return out.reshape(np.shape(x))


def f16_value(h) -> np.ndarray:
    """fp32 values of fp16 bit patterns."""
    a = _c(h, np.uint16).ravel()
    return np.array([lib().orc_f16_to_f32(int(v)) for v in a], dtype=np.float32).reshape(
        np.shape(h))


def bf16_round(x) -> np.ndarray:
    """Nearest bfloat16 (ties to even) of each fp32 value, as fp32."""
    a = f32(x).ravel()
    out = np.zeros(a.size, dtype=np.float32)
    lib().orc_bf16_round_array(_p(a), a.size, _p(out))
    return out.reshape(np.shape(x))


def int2_quantize_group(x):
    """(codes uint8[8], scale fp16 bits, zero fp16 bits, ok) of 32 values."""
    a = f32(x)
    assert a.size == 32
    codes = np.zeros(8, dtype=np.uint8)
    s = np.zeros(1, dtype=np.uint16)
    z = np.zeros(1, dtype=np.uint16)
    rc = lib().orc_int2_quantize_group(_p(a), _p(codes), _p(s), _p(z))
    return codes, int(s[0]), int(z[0]), rc == 0


def int2_dequantize_group(codes, scale: int, zero: int) -> np.ndarray:
    c = _c(codes, np.uint8)
    out = np.zeros(32, dtype=np.float32)
    lib().orc_int2_dequantize_group(_p(c), scale, zero, _p(out))
    return out


def ledger_bytes(d: int) -> int:
    return int(lib().orc_ledger_bytes(d))


def ledger_write_window(Kw, Vw) -> np.ndarray:
    """Ledger bytes of one window from its [64, d] K and V rows."""
    K = f32(Kw)
    V = f32(Vw)
    d = K.shape[-1]
    out = np.zeros(ledger_bytes(d), dtype=np.uint8)
    lib().orc_ledger_write_window(_p(K), _p(V), d, _p(out))
    return out


def ledger_read_window(ledger, d: int):
    """Dequantised fp32 (K [64, d], V [64, d]) of one window's ledger."""
    lg = _c(ledger, np.uint8)
    K = np.zeros((WINDOW, d), dtype=np.float32)
    V = np.zeros((WINDOW, d), dtype=np.float32)
    lib().orc_ledger_read_window(_p(lg), d, _p(K), _p(V))
    return K, V


class TierUnit:
    """Tier state of one (batch, kv-head) unit, with its own fp32 copy of the
    unit's K and V rows (bf16 values), which promotions overwrite."""

    def __init__(self, init_tiers, K_unit, V_unit, N: int, n_win: int):
        self.K = f32(K_unit).copy()
        self.V = f32(V_unit).copy()
        self.d = self.K.shape[-1]
        assert self.K.shape[0] >= n_win * WINDOW or self.K.shape[0] >= N
        self.n_win = n_win
        self.tier = np.zeros(n_win, dtype=np.int8)
        self.score = np.zeros(n_win, dtype=np.int64)
        self.has_ledger = np.zeros(n_win, dtype=np.uint8)
        self.ledger = np.zeros((n_win, ledger_bytes(self.d)), dtype=np.uint8)
        init = np.zeros(n_win, dtype=np.int8)
        it = _c(init_tiers, np.int8)
        init[:min(n_win, it.size)] = it[:n_win]
        q = np.zeros(1, dtype=np.int32)
        b = np.zeros(1, dtype=np.int64)
        self._pad()
        rc = lib().orc_tier_init_unit(_p(init), _p(self.K), _p(self.V), N, self.d, n_win,
                                      _p(self.tier), _p(self.score), _p(self.has_ledger),
                                      _p(self.ledger), _p(q), _p(b))
        if rc < 0:
            raise ValueError("bad initial tier value")
        self.quota = int(q[0])
        self.budget = int(b[0])

    def _pad(self):
        rows = self.n_win * WINDOW
        if self.K.shape[0] < rows:
            pad = np.zeros((rows - self.K.shape[0], self.d), dtype=np.float32)
            self.K = np.ascontiguousarray(np.concatenate([self.K, pad]))
            self.V = np.ascontiguousarray(np.concatenate([self.V, pad]))

    def attend(self, q_group, N: int, scale: float):
        """(out [G, d] fp64, mass [ceil(N/64)] fp64) of the tiered attention."""
        q = f32(q_group)
        G, d = q.shape
        nw = -(-N // WINDOW)
        out = np.zeros((G, d), dtype=np.float64)
        mass = np.zeros(max(nw, 1), dtype=np.float64)
        rc = lib().orc_tiered_attend_unit(_p(q), G, _p(self.K), _p(self.V), _p(self.ledger),
                                          _p(self.tier), N, d, float(scale), _p(out), _p(mass))
        if rc != 0:
            raise ValueError("bad tier value")
        return out, mass[:nw]

    def update(self, mass, N: int):
        """One routing step from fp32 window masses; returns [promotions,
        demotions, evictions]."""
        nw = -(-N // WINDOW)
        m = np.zeros(self.n_win, dtype=np.float32)
        mm = f32(mass).ravel()
        m[:min(nw, mm.size)] = mm[:nw]
        stats = np.zeros(3, dtype=np.int32)
        rc = lib().orc_tier_update_unit(_p(self.tier), _p(self.score), _p(self.has_ledger),
                                        _p(self.ledger), _p(self.K), _p(self.V), _p(m), N,
                                        self.d, self.quota, self.budget, _p(stats))
        if rc < 0:
            raise ValueError("bad tier value")
        return stats

    def tier_bytes(self, N: int) -> int:
        closed = N // WINDOW
        t = self.tier[:closed]
        return int((t == BF16).sum()) * WINDOW * 4 * self.d + int((t == INT2).sum()) * \
            ledger_bytes(self.d)


# --------------------------------------------------------------------------
# calibrated inner-product reranker (kvr_rsq_oracle.c)
# --------------------------------------------------------------------------

def rsq_table(m: int = 8):
    """(bin edges [9], levels [8]) of the 3-bit magnitude quantiser, fp64."""
    bound = np.zeros(9, dtype=np.float64)
    level = np.zeros(8, dtype=np.float64)
    if lib().orc_rsq_table(m, _p(bound), _p(level)):
        raise ValueError("m must be >= 3")
    return bound, level


def rsq_float_tables(m: int = 8):
    """(fl(edge^2) [8] with entry 0 = 0, fl(level) [8]): the fp32 tables."""
    bsq = np.zeros(8, dtype=np.float32)
    lev = np.zeros(8, dtype=np.float32)
    lib().orc_rsq_float_tables(m, _p(bsq), _p(lev))
    return bsq, lev


def rsq_record_bytes(d: int) -> int:
    return int(lib().orc_rsq_record_bytes(d))


def rsq_encode(x, sgn) -> np.ndarray:
    """Records [..., 6 d/8] uint8 of the rows x [..., d]."""
    a = f32(x)
    d = a.shape[-1]
    n = a.size // d
    s = _c(sgn, np.int8)
    out = np.zeros(a.shape[:-1] + (rsq_record_bytes(d),), dtype=np.uint8)
    if lib().orc_rsq_encode(_p(a), n, d, _p(s), _p(out)):
        raise ValueError("unsupported head_dim %d" % d)
    return out


def rsq_score(record, zq) -> np.float32:
    r = _c(record, np.uint8)
    z = f32(zq)
    return np.float32(lib().orc_rsq_score(_p(r), _p(z), z.shape[-1]))


def select_unit_rsq(q_group, codes_unit, rec_unit, N, sgn, C, k, W, lut, diagnostics=False):
    """Selection of one unit with the reranker; (idx[k] padded -1, count[, diag])."""
    q = f32(q_group)
    G, d = q.shape
    cd = _c(codes_unit, np.uint8)
    rc_ = _c(rec_unit, np.uint8)
    s = _c(sgn, np.int8)
    lt = _c(lut, np.int32)
    idx = np.full(max(k, 1), -1, dtype=np.int32)
    cnt = np.zeros(1, dtype=np.int32)
    pool = max(0, N - W)
    nc = max(0, min(C, pool))
    cand = np.full(max(nc, 1), -1, dtype=np.int32)
    candS = np.zeros(max(nc, 1), dtype=np.float32)
    rc = lib().orc_select_unit_rsq(_p(q), G, _p(cd), _p(rc_), N, d, _p(s), C, k, W, _p(lt),
                                   _p(idx), _p(cnt), _p(cand), _p(candS))
    if rc != 0:
        raise ValueError("oracle selection failed")
    if not diagnostics:
        return idx[:k], int(cnt[0])
    return idx[:k], int(cnt[0]), dict(cand=cand[:nc], cand_S=candS[:nc])


# --------------------------------------------------------------------------
# cache regions: sink, retrieval, local + update buffer (kvr_regions_oracle.c)
# --------------------------------------------------------------------------

def region_init(N, S, L) -> int:
    """Retrieval end at set-up: Local holds the L newest tokens, buffer empty."""
    return int(lib().orc_region_init(int(N), int(S), int(L)))


def region_advance(N, R, S, L, U) -> int:
    """Retrieval end after appends up to length N (buffer of U tokens)."""
    return int(lib().orc_region_advance(int(N), int(R), int(S), int(L), int(U)))


def select_unit_regions(q_group, K_unit, codes_unit, N, S, R, sgn, C, k, lut, rec_unit=None,
                        diagnostics=False):
    """Selection of one unit over the retrieval region [S', R'); exact scores,
    or the reranker's estimates when rec_unit is given."""
    q = f32(q_group)
    G, d = q.shape
    Kf = f32(K_unit) if K_unit is not None else np.zeros((1, d), dtype=np.float32)
    cd = _c(codes_unit, np.uint8)
    rc_ = None if rec_unit is None else _c(rec_unit, np.uint8)
    s = _c(sgn, np.int8)
    lt = _c(lut, np.int32)
    lo = min(S, N)
    hi = min(max(R, lo), N)
    pool = hi - lo
    nc = max(0, min(C, pool))
    idx = np.full(max(k, 1), -1, dtype=np.int32)
    cnt = np.zeros(1, dtype=np.int32)
    cand = np.full(max(nc, 1), -1, dtype=np.int32)
    candS = np.zeros(max(nc, 1), dtype=np.float32)
    coarse = np.zeros(max(pool, 1), dtype=np.int32)
    rc = lib().orc_select_unit_regions(_p(q), G, _p(Kf), _p(cd), None if rc_ is None else _p(rc_),
                                       N, d, _p(s), C, k, S, R, _p(lt), _p(idx), _p(cnt),
                                       _p(cand), _p(candS), _p(coarse))
    if rc != 0:
        raise ValueError("oracle selection failed")
    if not diagnostics:
        return idx[:k], int(cnt[0])
    return idx[:k], int(cnt[0]), dict(cand=cand[:nc], cand_S=candS[:nc], coarse=coarse[:pool])


def attend_unit_regions(q_group, K_unit, V_unit, N, S, R, idx, count, scale) -> np.ndarray:
    """Attention over [0, S') + idx + [R', N) of one unit, fp64."""
    q = f32(q_group)
    G, d = q.shape
    Kf = f32(K_unit)
    Vf = f32(V_unit)
    ix = _c(idx, np.int32)
    out = np.zeros((G, d), dtype=np.float64)
    rc = lib().orc_attend_unit_regions(_p(q), G, _p(Kf), _p(Vf), N, d, S, R, _p(ix), count,
                                       float(scale), _p(out))
    if rc != 0:
        raise ValueError("selected index outside the retrieval region")
    return out


# --------------------------------------------------------------------------
# magnitude-aware coarse votes (kvr_votes_oracle.c)
# --------------------------------------------------------------------------

def flip_cost(a8, x) -> np.float32:
    """fp32 sum of a8[j] over the set bits j of x, ascending from +0."""
    a = f32(a8)
    return np.float32(lib().orc_flip_cost(_p(a), int(x)))


def mag_vote_table(zq, lut) -> np.ndarray:
    """Vote tables [d/8, 256] int32 of the rotated query zq [d]."""
    z = f32(zq)
    d = z.shape[-1]
    T = np.zeros((d // 8, 256), dtype=np.int32)
    if lib().orc_mag_vote_table(_p(z), d, _p(_c(lut, np.int32)), _p(T)):
        raise ValueError("unsupported head_dim %d" % d)
    return T


def select_unit_mag(q_group, K_unit, codes_unit, N, sgn, C, k, W, lut, diagnostics=False):
    """Selection of one unit with magnitude-aware votes; (idx[k] padded -1,
    count[, diag with cand, cand_S, coarse, table])."""
    q = f32(q_group)
    G, d = q.shape
    Kf = f32(K_unit)
    cd = _c(codes_unit, np.uint8)
    s = _c(sgn, np.int8)
    lt = _c(lut, np.int32)
    pool = max(0, N - W)
    nc = max(0, min(C, pool))
    idx = np.full(max(k, 1), -1, dtype=np.int32)
    cnt = np.zeros(1, dtype=np.int32)
    cand = np.full(max(nc, 1), -1, dtype=np.int32)
    candS = np.zeros(max(nc, 1), dtype=np.float32)
    coarse = np.zeros(max(pool, 1), dtype=np.int32)
    table = np.zeros((d // 8, 256), dtype=np.int32)
    rc = lib().orc_select_unit_mag(_p(q), G, _p(Kf), _p(cd), N, d, _p(s), C, k, W, _p(lt),
                                   _p(idx), _p(cnt), _p(cand), _p(candS), _p(coarse), _p(table))
    if rc != 0:
        raise ValueError("oracle selection failed")
    if not diagnostics:
        return idx[:k], int(cnt[0])
    return idx[:k], int(cnt[0]), dict(cand=cand[:nc], cand_S=candS[:nc], coarse=coarse[:pool],
                                      table=table)
