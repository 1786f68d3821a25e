"""Pins of the cache-region oracle (ParisKV, "Meccanismo di Aggiornamento a
Finestra Scorrevole": Sink, Local, Retrieval and Update Buffer regions).

Checked against: an explicit simulation of the four regions as lists of
token positions (the buffer filling up and moving the oldest local tokens to
retrieval), a Python restatement of the selection over the retrieval region
from the pinned step functions, textbook numpy attention over the explicit
token set, and the reduction to the plain window path (S = 0, R = N - W).
"""
import math

import numpy as np
import pytest

import oracle
import workloads as wl

RNG = np.random.default_rng(91)


class Regions:
    """The four regions as explicit lists of positions."""

    def __init__(self, N, S, L):
        self.S, self.L = S, L
        self.sink = list(range(min(S, N)))
        rest = list(range(len(self.sink), N))
        self.local = rest[max(0, len(rest) - L):]
        self.retrieval = rest[:max(0, len(rest) - L)]
        self.buffer = []

    def append(self, t, U):
        if t < self.S:               # the first S positions are the sink
            self.sink.append(t)
            return
        if len(self.local) < self.L:  # Local fills up first
            self.local.append(t)
            return
        self.buffer.append(t)
        if len(self.buffer) == U:     # full: the U oldest local tokens retire
            moved, self.local = self.local[:U], self.local[U:] + self.buffer
            self.retrieval += moved
            self.buffer = []

    def retrieval_end(self):
        return len(self.sink) + len(self.retrieval)


@pytest.mark.parametrize("N0,S,L,U", [(1000, 4, 128, 64), (300, 16, 64, 1), (50, 64, 16, 8),
                                      (130, 4, 128, 32), (0, 4, 8, 4)])
def test_region_rule_matches_the_explicit_simulation(N0, S, L, U):
    reg = Regions(N0, S, L)
    R = oracle.region_init(N0, S, L)
    assert R == reg.retrieval_end()
    for N in range(N0 + 1, N0 + 700):
        reg.append(N - 1, U)
        R_new = oracle.region_advance(N, R, S, L, U)
        assert R_new == reg.retrieval_end(), (N, R_new)
        # retrieval grows in blocks of U (past the sink, which fills one by one)
        assert R_new >= R and ((R_new - R) % U == 0 or R_new <= S)
        # Local + buffer hold the newest L .. L + U - 1 tokens past the sink
        if N >= S + L:
            assert L <= N - R_new < L + U
        assert sorted(reg.sink + reg.retrieval + reg.local + reg.buffer) == list(range(N))
        R = R_new


def brute_select(q, K, codes, N, S, R, sgn, C, k, lut):
    lo = min(S, N)
    hi = min(max(R, lo), N)
    qbar = oracle.group_mean(q)
    qcode = oracle.encode(qbar[None, :], sgn)[0]
    coarse = oracle.coarse_scores(codes[:N], qcode, lut)
    pool = list(range(lo, hi))
    cand = sorted(pool, key=lambda t: (-int(coarse[t]), t))[:C]
    cand = sorted(cand)
    score = {t: float(oracle.exact_score(qbar, K[t])) for t in cand}
    top = sorted(cand, key=lambda t: (-score[t], t))[:k]
    return sorted(top), cand


@pytest.mark.parametrize("N,S,R", [(3000, 4, 2872), (3000, 64, 2900), (3000, 0, 2500),
                                   (200, 300, 250), (500, 100, 50), (500, 4, 900)])
def test_selection_over_the_retrieval_region(N, S, R):
    d, G = 64, 4
    w = wl.Workload("r", B=1, Hq=G, Hkv=1, d=d, N=N, dtype="f32", rank=16, planted=8, seed=N + S)
    K, V, q = wl.make_cache(w, device="cpu", cap=N)
    sgn = wl.srht_signs(d).numpy()
    Ku = oracle.f32(K[0, 0])
    codes = oracle.encode(Ku, sgn)
    qg = oracle.f32(q[0])
    C, k = 300, 80
    idx, cnt, dg = oracle.select_unit_regions(qg, Ku, codes, N, S, R, sgn, C, k, wl.DEFAULT_LUT,
                                              diagnostics=True)
    ref, cand = brute_select(qg, Ku, codes, N, S, R, sgn, C, k, wl.DEFAULT_LUT)
    assert list(dg["cand"]) == cand
    assert cnt == len(ref) and list(idx[:cnt]) == ref
    assert np.all(idx[cnt:] == -1)


def test_plain_window_is_the_special_case():
    w = wl.TINY
    K, V, qb = wl.make_cache(w)
    sgn = wl.srht_signs(w.d).numpy()
    Ku = oracle.f32(K[0, 1])
    codes = oracle.encode(Ku, sgn)
    rec = oracle.rsq_encode(Ku, sgn)
    q = oracle.f32(qb[0, 1:2])
    N = w.N
    a = oracle.select_unit_regions(q, Ku, codes, N, 0, N - w.W, sgn, w.C, w.k, w.lut)
    b = oracle.select_unit(q, Ku, codes, N, sgn, w.C, w.k, w.W, w.lut)
    assert a[1] == b[1] and np.array_equal(a[0], b[0])
    a = oracle.select_unit_regions(q, None, codes, N, 0, N - w.W, sgn, w.C, w.k, w.lut, rec_unit=rec)
    b = oracle.select_unit_rsq(q, codes, rec, N, sgn, w.C, w.k, w.W, w.lut)
    assert a[1] == b[1] and np.array_equal(a[0], b[0])
    Vu = oracle.f32(V[0, 1])
    o1 = oracle.attend_unit_regions(q, Ku, Vu, N, 0, N - w.W, b[0][:b[1]], b[1], 0.125)
    o2 = oracle.attend_unit(q, Ku, Vu, N, b[0][:b[1]], b[1], w.W, 0.125)
    assert np.array_equal(o1, o2)


@pytest.mark.parametrize("N,S,R", [(400, 4, 300), (400, 0, 400), (10, 16, 12), (400, 50, 20)])
def test_attention_over_the_regions_is_textbook_attention(N, S, R):
    d, G = 32, 2
    K = RNG.normal(0, 1, (N, d)).astype(np.float32)
    V = RNG.normal(0, 1, (N, d)).astype(np.float32)
    q = RNG.normal(0, 1, (G, d)).astype(np.float32)
    lo = min(S, N)
    hi = min(max(R, lo), N)
    idx = np.sort(RNG.choice(np.arange(lo, hi), size=min(20, hi - lo), replace=False)).astype(np.int32)
    out = oracle.attend_unit_regions(q, K, V, N, S, R, idx, len(idx), 0.3)
    T = list(range(lo)) + list(idx) + list(range(hi, N))
    s = (q.astype(np.float64) @ K[T].astype(np.float64).T) * np.float64(np.float32(0.3))
    p = np.exp(s - s.max(1, keepdims=True))
    p /= p.sum(1, keepdims=True)
    ref = p @ V[T].astype(np.float64)
    assert np.abs(out - ref).max() < 1e-12


def test_attention_rejects_indices_outside_the_retrieval_region():
    N, d = 100, 16
    K = np.zeros((N, d), np.float32)
    q = np.zeros((1, d), np.float32)
    with pytest.raises(ValueError):
        oracle.attend_unit_regions(q, K, K, N, 8, 60, np.array([3], np.int32), 1, 1.0)   # in the sink
    with pytest.raises(ValueError):
        oracle.attend_unit_regions(q, K, K, N, 8, 60, np.array([60], np.int32), 1, 1.0)  # local
