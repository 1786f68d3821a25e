"""Pins of the magnitude-aware vote oracle (ParisKV, "Pipeline di Recupero
Nativa su GPU in Due Stadi": top-rho most similar centroids per sub-space,
tiered votes).

Checked against: the ranking of all 256 sign-pattern centroids by their
float64 inner product with the rotated query sub-vector, the Hamming-ring
votes when a sub-block's magnitudes are equal (table and whole selection),
and a Python restatement of the coarse score and the selection.
"""
import numpy as np
import pytest

import oracle
import workloads as wl

RNG = np.random.default_rng(23)
LUT = (3, 2, 1, 0, 0, 0, 0, 0, 0)
RING_END = [1, 9, 37, 93, 163, 219, 247, 255, 256]


def tier(r):
    return next(t for t, e in enumerate(RING_END) if r < e)


def test_ranking_is_by_inner_product_with_the_centroids():
    d = 128
    zq = RNG.normal(0, 1, d).astype(np.float32)
    lut = (8, 7, 6, 5, 4, 3, 2, 1, 0)          # every tier distinct: the table shows the rank's tier
    T = oracle.mag_vote_table(zq, lut)
    signs = np.array([[-1.0 if (x >> j) & 1 else 1.0 for j in range(8)] for x in range(256)])
    for b in range(d // 8):
        z = zq[8 * b:8 * b + 8].astype(np.float64)
        qcode = sum(1 << j for j in range(8) if z[j] < 0)
        # centroid of flip set x: the query's signs with the bits of x flipped
        c = np.sign(np.where(z == 0, 1.0, z))[None, :] * signs
        sim = c @ z
        order = sorted(range(256), key=lambda x: (-sim[x], x))
        for r, x in enumerate(order):
            assert T[b, x] == lut[tier(r)], (b, x, r)
        assert T[b, 0] == lut[0] and qcode >= 0


def test_equal_magnitudes_give_the_hamming_ring_votes():
    zq = np.where(RNG.random(64) < 0.5, -0.37, 0.37).astype(np.float32)
    T = oracle.mag_vote_table(zq, LUT)
    pc = np.array([bin(x).count("1") for x in range(256)])
    for b in range(8):
        assert np.array_equal(T[b], np.array(LUT)[pc])


def test_flip_cost_is_the_left_to_right_fp32_sum():
    a = RNG.random(8).astype(np.float32)
    for x in (0, 1, 0x81, 0xff, 0x5a):
        f = np.float32(0)
        for j in range(8):
            if (x >> j) & 1:
                f = np.float32(f + a[j])
        assert oracle.flip_cost(a, x) == f


def brute(q, K, codes, N, sgn, C, k, W, T):
    qbar = oracle.group_mean(q)
    qcode = oracle.encode(qbar[None, :], sgn)[0]
    pool = max(0, N - W)
    nb = codes.shape[1]
    coarse = np.array([sum(int(T[b, codes[i, b] ^ qcode[b]]) for b in range(nb))
                       for i in range(pool)], dtype=np.int64)
    cand = sorted(sorted(range(pool), key=lambda i: (-coarse[i], i))[:C])
    S = {i: float(oracle.exact_score(qbar, K[i])) for i in cand}
    top = sorted(sorted(cand, key=lambda i: (-S[i], i))[:k])
    return coarse, cand, top


def test_selection_restated():
    d, G, N = 64, 4, 1500
    w = wl.Workload("v", B=1, Hq=G, Hkv=1, d=d, N=N, dtype="f32", rank=16, planted=8, seed=3)
    K, V, q = wl.make_cache(w, device="cpu", cap=N)
    sgn = wl.srht_signs(d).numpy()
    Ku = oracle.f32(K[0, 0])
    codes = oracle.encode(Ku, sgn)
    qg = oracle.f32(q[0])
    idx, cnt, dg = oracle.select_unit_mag(qg, Ku, codes, N, sgn, 200, 50, 64, LUT,
                                          diagnostics=True)
    coarse, cand, top = brute(qg, Ku, codes, N, sgn, 200, 50, 64, dg["table"])
    assert np.array_equal(dg["coarse"], coarse)
    assert list(dg["cand"]) == cand
    assert cnt == len(top) and list(idx[:cnt]) == top
    # the table is the one of the query's own rotation
    qbar = oracle.group_mean(qg)
    zq = oracle.fwht((qbar * sgn).astype(np.float32))
    assert np.array_equal(dg["table"], oracle.mag_vote_table(zq, LUT))


def test_equal_magnitude_query_selects_like_the_hamming_reading():
    d, N = 128, 3000
    sgn = wl.srht_signs(d).numpy()
    z = np.where(RNG.random(d) < 0.5, -1.0, 1.0)
    H = np.where(np.bitwise_count(np.arange(d)[:, None] & np.arange(d)[None, :]) % 2, -1.0, 1.0)
    q = ((H @ z) / d * sgn).astype(np.float32)[None, :]          # FWHT(D q) = z exactly
    assert np.array_equal(np.abs(oracle.fwht((q[0] * sgn).astype(np.float32))), np.ones(d))
    K = RNG.normal(0, 1, (N, d)).astype(np.float32)
    codes = oracle.encode(K, sgn)
    a = oracle.select_unit_mag(q, K, codes, N, sgn, 300, 60, 128, LUT)
    b = oracle.select_unit(q, K, codes, N, sgn, 300, 60, 128, LUT)
    assert a[1] == b[1] and np.array_equal(a[0], b[0])


def test_ties_across_a_ring_boundary_go_by_pattern():
    """Magnitudes 1,1,2,2,2,2,2,2: the cost-2 patterns 3 (bits 0 and 1), 4,
    8, 16, 32, 64, 128 tie and take ranks 3..9 in pattern order, so the ring
    boundary at rank 9 puts 128 alone in the next tier (hand-derived)."""
    zq = np.array([1, 1, 2, 2, 2, 2, 2, 2], dtype=np.float32)
    lut = (8, 7, 6, 5, 4, 3, 2, 1, 0)
    T = oracle.mag_vote_table(zq, lut)[0]
    assert T[0] == 8
    assert all(T[x] == 7 for x in (1, 2, 3, 4, 8, 16, 32, 64))
    assert T[128] == 6
    assert T[5] == 6 and T[6] == 6                   # cost 3 (bits 0 or 1 with bit 2)
