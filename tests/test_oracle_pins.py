"""Pins of the CPU oracle against what the pages and the mathematics fix.

Every check here compares the oracle with something other than itself: a
Hadamard matrix built independently from its closed form, exact rational
arithmetic, brute force over all 2^8 centroids of a sub-block, explicit
enumeration of Hamming rings, Python's own sort, fsum-exact dot products with
a rounding-error bound, and textbook dense softmax attention. Sizes are tiny
so the whole file runs in seconds on the CPU.
"""
import itertools
import math
import os
from fractions import Fraction

import numpy as np
import pytest

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
U32 = 2.0 ** -24  # unit roundoff of fp32


def hadamard(d):
    """Sylvester Hadamard matrix from its closed form (-1)^popcount(i & j)."""
    return np.array([[(-1) ** bin(i & j).count("1") for j in range(d)] for i in range(d)],
                    dtype=np.int64)


def rng(seed):
    return np.random.default_rng(seed)


# ---------------------------------------------------------------- rotation

@pytest.mark.parametrize("d", [64, 128])
def test_hadamard_closed_form_is_orthogonal(d):
    H = hadamard(d)
    assert np.array_equal(H @ H.T, d * np.eye(d, dtype=np.int64))


@pytest.mark.parametrize("d", [64, 128])
def test_fwht_columns_equal_hadamard(orc, d):
    H = hadamard(d)
    eye = np.eye(d, dtype=np.float32)
    out = orc.fwht(eye)  # row j = FWHT(e_j) = column j of H
    assert np.array_equal(out.T.astype(np.int64), H)


@pytest.mark.parametrize("d", [64, 128])
def test_fwht_matches_dense_product_within_bound(orc, d):
    H = hadamard(d).astype(np.float64)
    x = rng(d).standard_normal((50, d)).astype(np.float32)
    got = orc.fwht(x).astype(np.float64)
    ref = x.astype(np.float64) @ H.T
    bound = math.log2(d) * U32 * np.abs(x.astype(np.float64)).sum(axis=1, keepdims=True)
    assert np.all(np.abs(got - ref) <= 1.01 * bound)


@pytest.mark.parametrize("d", [64, 128])
def test_srht_preserves_norms_and_angles(orc, d):
    r = rng(3 + d)
    sgn = (r.integers(0, 2, d) * 2 - 1).astype(np.int8)
    x = r.standard_normal(d).astype(np.float32)
    y = r.standard_normal(d).astype(np.float32)
    rx, ry = orc.srht_unit(x, sgn), orc.srht_unit(y, sgn)
    assert abs(np.linalg.norm(rx) - 1.0) < 1e-12
    cos = float(x.astype(np.float64) @ y) / (np.linalg.norm(x.astype(np.float64)) *
                                             np.linalg.norm(y.astype(np.float64)))
    assert abs(float(rx @ ry) - cos) < 1e-12


# ---------------------------------------------------------------- sign codes

def brute_force_code(z_exact, d):
    """argmax over all 2^8 centroids of each sub-block (ties -> lowest byte).

    Centroid byte c has component t equal to -1/sqrt(8) if bit t is set, else
    +1/sqrt(8); the common 1/sqrt(8) factor does not change the argmax.
    """
    out = []
    for b in range(d // 8):
        sub = z_exact[8 * b:8 * b + 8]
        best, best_c = None, None
        for c in range(256):
            v = sum((-s if (c >> t) & 1 else s) for t, s in enumerate(sub))
            if best is None or v > best:
                best, best_c = v, c
        out.append(best_c)
    return np.array(out, dtype=np.uint8)


def exact_rotation(x, sgn, H):
    """H D x in exact rational arithmetic (positive scale dropped)."""
    xs = [Fraction(float(v)) * int(s) for v, s in zip(x, sgn)]
    return [sum(int(H[i, j]) * xs[j] for j in range(len(xs))) for i in range(len(xs))]


@pytest.mark.parametrize("d", [64, 128])
def test_code_is_nearest_centroid_integer_inputs(orc, d):
    """Small-integer inputs: every fp32 partial sum is exact, so codes must agree
    with the brute-force nearest centroid of the exact rotated vector, including
    the exact zeros (ties) these inputs produce."""
    r = rng(11 + d)
    H = hadamard(d)
    sgn = (r.integers(0, 2, d) * 2 - 1).astype(np.int8)
    rows = [r.integers(-3, 4, d).astype(np.float32) for _ in range(12)]
    rows.append(np.zeros(d, np.float32))
    rows.append(np.full(d, -0.0, np.float32))
    e = np.zeros(d, np.float32)
    e[0], e[1] = 1, 1  # H(e0+e1) has exact zeros at every odd coordinate
    rows.append(e)
    x = np.stack(rows)
    codes = orc.encode(x, sgn)
    n_zero = 0
    for i, row in enumerate(x):
        z = exact_rotation(row, sgn, H)
        n_zero += sum(1 for v in z if v == 0)
        assert np.array_equal(codes[i], brute_force_code(z, d)), i
    assert n_zero > 0  # the tie rule was exercised


@pytest.mark.parametrize("d", [64, 128])
def test_code_is_nearest_centroid_random_inputs(orc, d):
    """Random fp32 inputs: a code bit may differ from the exact nearest centroid
    only where the exact rotated coordinate lies inside the fp32 FWHT error bound."""
    r = rng(21 + d)
    H = hadamard(d)
    sgn = (r.integers(0, 2, d) * 2 - 1).astype(np.int8)
    x = r.standard_normal((6, d)).astype(np.float32)
    x[:, 3] *= 8.0  # an outlier channel, as in the tiny workload
    codes = orc.encode(x, sgn)
    for i, row in enumerate(x):
        z = exact_rotation(row, sgn, H)
        bf = brute_force_code(z, d)
        bound = math.log2(d) * U32 * float(np.abs(row.astype(np.float64)).sum()) * 1.01
        for b in range(d // 8):
            diff = int(codes[i, b]) ^ int(bf[b])
            for t in range(8):
                if (diff >> t) & 1:
                    assert abs(float(z[8 * b + t])) <= bound


def test_golden_sign_codes(orc):
    with open(os.path.join(GOLDEN, "sign_codes.txt")) as f:
        lines = [ln.split() for ln in f if ln.strip() and not ln.startswith("#")]
    assert len(lines) >= 10
    for d, j, dj, hexcode in lines:
        d, j, dj = int(d), int(j), int(dj)
        sgn = np.ones(d, np.int8)
        sgn[j] = dj
        x = np.zeros(d, np.float32)
        x[j] = 1.0
        assert orc.encode(x, sgn).tobytes().hex() == hexcode, (d, j, dj)


def test_code_of_rotated_query_matches_key_rule(orc):
    """The query code is the same map applied to q_bar (positive scale invariant)."""
    r = rng(5)
    d = 64
    sgn = (r.integers(0, 2, d) * 2 - 1).astype(np.int8)
    x = r.standard_normal(d).astype(np.float32)
    assert np.array_equal(orc.encode(x, sgn), orc.encode(x * np.float32(4.0), sgn))
    y = orc.srht_unit(x, sgn)
    bits = np.packbits((y < 0).astype(np.uint8).reshape(-1, 8)[:, ::-1], axis=1).ravel()
    assert np.array_equal(orc.encode(x, sgn), bits)


# ---------------------------------------------------------------- query mean

def test_group_mean_exact_cases(orc):
    q = np.array([[1, 2, -4, 0.5], [3, 4, 4, 0.25]] * 1, np.float32)
    q = np.pad(q, ((0, 0), (0, 60)))
    m = orc.group_mean(q)
    assert np.array_equal(m[:4], np.array([2, 3, 0, 0.375], np.float32))
    one = np.arange(64, dtype=np.float32)[None, :]
    assert np.array_equal(orc.group_mean(one), one[0])
    four = np.stack([np.full(64, v, np.float32) for v in (1, 2, 3, 6)])
    assert np.all(orc.group_mean(four) == np.float32(3.0))


# ---------------------------------------------------------------- coarse score

def ring_vote_score(key_code, qcode, lut):
    """Enumerate, per sub-block, the centroids in each Hamming ring around the
    query's centroid; the key collects the vote of the ring holding its own
    centroid."""
    s = 0
    for kb, qb in zip(key_code, qcode):
        for r in range(9):
            ring = {c for c in range(256) if bin(c ^ int(qb)).count("1") == r}
            if int(kb) in ring:
                s += lut[r]
    return s


def test_golden_coarse_scores(orc):
    with open(os.path.join(GOLDEN, "coarse_scores.txt")) as f:
        rows = [ln for ln in f if ln.strip() and not ln.startswith("#")]
    for ln in rows:
        qh, kh, lt, exp = [p.strip() for p in ln.split("|")]
        qc = np.frombuffer(bytes.fromhex(qh), np.uint8)
        kc = np.frombuffer(bytes.fromhex(kh), np.uint8)[None, :]
        lut = [int(v) for v in lt.split()]
        assert orc.coarse_scores(kc, qc, lut)[0] == int(exp)


@pytest.mark.parametrize("nb", [8, 16])
def test_coarse_scores_brute_force(orc, nb):
    r = rng(40 + nb)
    codes = r.integers(0, 256, (40, nb)).astype(np.uint8)
    qcode = r.integers(0, 256, nb).astype(np.uint8)
    codes[0] = qcode
    codes[1] = ~qcode
    for lut in ([3, 2, 1, 0, 0, 0, 0, 0, 0], list(r.integers(0, 16, 9))):
        got = orc.coarse_scores(codes, qcode, lut)
        ref = [ring_vote_score(c, qcode, lut) for c in codes]
        assert list(got) == ref


def test_linear_lut_is_pure_popcount(orc):
    r = rng(9)
    nb = 16
    codes = r.integers(0, 256, (100, nb)).astype(np.uint8)
    qcode = r.integers(0, 256, nb).astype(np.uint8)
    got = orc.coarse_scores(codes, qcode, [8, 7, 6, 5, 4, 3, 2, 1, 0])
    ham = [sum(bin(int(a) ^ int(b)).count("1") for a, b in zip(c, qcode)) for c in codes]
    assert list(got) == [8 * nb - h for h in ham]


# ---------------------------------------------------------------- orders

def test_top_by_int_matches_python_sort(orc):
    r = rng(12)
    s = r.integers(0, 6, 500).astype(np.int32)  # many ties
    for c in (0, 1, 7, 100, 499, 500, 800):
        ref = sorted(sorted(range(500), key=lambda i: (-int(s[i]), i))[:c])
        assert list(orc.top_by_int(s, c)) == ref


def test_top_by_int_special_cases(orc):
    s = np.full(300, 5, np.int32)
    assert list(orc.top_by_int(s, 40)) == list(range(40))  # all tie: lowest indices
    s = np.arange(300, dtype=np.int32)
    assert list(orc.top_by_int(s, 1000)) == list(range(300))  # c >= n: everything


def test_top_by_float_matches_python_sort(orc):
    r = rng(13)
    s = np.round(r.standard_normal(400), 1).astype(np.float32)  # ties
    s[::37] = -0.0
    s[::41] = 0.0
    index = r.permutation(10_000)[:400].astype(np.int64)
    for c in (0, 1, 10, 399, 400, 401):
        # -0.0 == +0.0 for Python floats too, so they tie and fall to the index
        ref = sorted(sorted(range(400), key=lambda j: (-float(s[j]), int(index[j])))[:c])
        assert list(orc.top_by_float(s, index, c)) == sorted(int(index[j]) for j in ref)


def test_top_by_float_rejects_nan(orc):
    s = np.array([1.0, np.nan], np.float32)
    with pytest.raises(ValueError):
        orc.top_by_float(s, np.arange(2), 1)


# ---------------------------------------------------------------- exact score

@pytest.mark.parametrize("d", [64, 128])
def test_exact_score_error_bound(orc, d):
    r = rng(50 + d)
    n_terms = d // 16 + 4  # fma chain of d/16, then four adds
    gamma = n_terms * U32 / (1 - n_terms * U32)
    for _ in range(200):
        q = r.standard_normal(d).astype(np.float32)
        k = (r.standard_normal(d) * r.uniform(0.1, 10)).astype(np.float32)
        prods = [float(a) * float(b) for a, b in zip(q, k)]  # exact in fp64
        exact = math.fsum(prods)
        got = float(orc.exact_score(q, k))
        assert abs(got - exact) <= gamma * math.fsum(abs(p) for p in prods)


@pytest.mark.parametrize("d", [64, 128])
def test_exact_score_single_terms(orc, d):
    """One nonzero key coordinate at a time: the score is exactly q_j k_j, so a
    dropped term, a wrong chunk bound or a transposed index fails here."""
    r = rng(60 + d)
    q = r.standard_normal(d).astype(np.float32)
    for j in range(d):
        k = np.zeros(d, np.float32)
        k[j] = np.float32(1.5)
        assert orc.exact_score(q, k) == np.float32(q[j] * np.float32(1.5))


def test_exact_score_integer_inputs_exact(orc):
    r = rng(70)
    for _ in range(50):
        q = r.integers(-50, 51, 128).astype(np.float32)
        k = r.integers(-50, 51, 128).astype(np.float32)
        assert float(orc.exact_score(q, k)) == float(np.dot(q.astype(np.int64),
                                                            k.astype(np.int64)))


# ---------------------------------------------------------------- selection

def small_unit(seed, N=300, d=64, G=2, dtype=np.float32):
    r = rng(seed)
    K = r.standard_normal((N, d)).astype(dtype)
    q = r.standard_normal((G, d)).astype(dtype)
    sgn = (r.integers(0, 2, d) * 2 - 1).astype(np.int8)
    return K, q, sgn


def test_select_unit_composition(orc):
    """The per-unit selection equals its pinned parts composed by hand."""
    K, q, sgn = small_unit(80)
    N, W, C, k = 300, 20, 64, 16
    lut = [3, 2, 1, 0, 0, 0, 0, 0, 0]
    codes = orc.encode(K, sgn)
    idx, cnt, dg = orc.select_unit(q, K, codes, N, sgn, C, k, W, lut, diagnostics=True)
    qbar = orc.group_mean(q)
    qcode = orc.encode(qbar, sgn)
    s = orc.coarse_scores(codes[:N - W], qcode, lut)
    assert np.array_equal(dg["coarse"], s)
    cand = sorted(sorted(range(N - W), key=lambda i: (-int(s[i]), i))[:C])
    assert list(dg["cand"]) == cand
    S = np.array([orc.exact_score(qbar, K[i]) for i in cand], np.float32)
    assert np.array_equal(dg["cand_S"], S)
    top = sorted(sorted(range(C), key=lambda j: (-float(S[j]), cand[j]))[:k])
    assert cnt == k and list(idx) == sorted(cand[j] for j in top)


def test_select_unit_clamps(orc):
    K, q, sgn = small_unit(81, N=50)
    codes = orc.encode(K, sgn)
    lut = [3, 2, 1, 0, 0, 0, 0, 0, 0]
    idx, cnt = orc.select_unit(q, K, codes, 50, sgn, 100, 60, 10, lut)  # C, k > pool
    assert cnt == 40 and list(idx[:40]) == list(range(40)) and np.all(idx[40:] == -1)
    idx, cnt = orc.select_unit(q, K, codes, 50, sgn, 8, 4, 50, lut)  # window covers all
    assert cnt == 0 and np.all(idx == -1)
    idx, cnt = orc.select_unit(q, K, codes, 0, sgn, 8, 4, 4, lut)  # empty cache
    assert cnt == 0


def test_select_all_tie_takes_lowest_indices(orc):
    d = 64
    K = np.tile(np.random.default_rng(1).standard_normal(d).astype(np.float32), (200, 1))
    q = np.ones((1, d), np.float32)
    sgn = np.ones(d, np.int8)
    codes = orc.encode(K, sgn)
    idx, cnt = orc.select_unit(q, K, codes, 200, sgn, 30, 10, 5, [3, 2, 1, 0, 0, 0, 0, 0, 0])
    assert cnt == 10 and list(idx) == list(range(10))


# ---------------------------------------------------------------- attention

def dense_attention(q, K, V, scale):
    """Textbook softmax attention in fp64 (separate code from the oracle)."""
    q = q.astype(np.float64)
    s = (q @ K.astype(np.float64).T) * scale
    s = s - s.max(axis=1, keepdims=True)
    p = np.exp(s)
    p /= p.sum(axis=1, keepdims=True)
    return p @ V.astype(np.float64)


def test_full_selection_is_dense_attention(orc):
    """Top-k with k = C = pool selects every token: the sparse attention is then
    dense attention over the whole context."""
    r = rng(90)
    N, d, G, W = 257, 64, 4, 16
    K = r.standard_normal((N, d)).astype(np.float32)
    V = r.standard_normal((N, d)).astype(np.float32)
    q = r.standard_normal((G, d)).astype(np.float32)
    sgn = (r.integers(0, 2, d) * 2 - 1).astype(np.int8)
    codes = orc.encode(K, sgn)
    idx, cnt = orc.select_unit(q, K, codes, N, sgn, N, N, W, [3, 2, 1, 0, 0, 0, 0, 0, 0])
    assert cnt == N - W
    scale = np.float32(1 / math.sqrt(d))
    out = orc.attend_unit(q, K, V, N, idx[:cnt], cnt, W, scale)
    assert np.max(np.abs(out - dense_attention(q, K, V, float(scale)))) < 1e-12


def test_attention_special_cases(orc):
    r = rng(91)
    N, d, G = 40, 64, 2
    K = r.standard_normal((N, d)).astype(np.float32)
    V = r.standard_normal((N, d)).astype(np.float32)
    q = r.standard_normal((G, d)).astype(np.float32)
    # |T| = 1 -> o = v
    out = orc.attend_unit(q, K, V, N, np.array([7], np.int32), 1, 0, 0.125)
    assert np.array_equal(out, np.tile(V[7].astype(np.float64), (G, 1)))
    # identical keys -> uniform weights -> mean of V over T
    Kc = np.tile(K[0], (N, 1))
    sel = np.array([1, 5, 9], np.int32)
    out = orc.attend_unit(q, Kc, V, N, sel, 3, 4, 0.125)
    T = [1, 5, 9, 36, 37, 38, 39]
    assert np.max(np.abs(out - V[T].astype(np.float64).mean(0))) < 1e-12
    # empty T -> zeros
    assert not np.any(orc.attend_unit(q, K, V, 0, np.zeros(0, np.int32), 0, 4, 0.125))
    # an index inside the window is rejected
    with pytest.raises(ValueError):
        orc.attend_unit(q, K, V, N, np.array([38], np.int32), 1, 4, 0.125)


def test_window_longer_than_context_is_dense(orc):
    """W > N: the window is the whole context (no pool, no selection), so the
    attention is dense attention over all N tokens."""
    r = rng(92)
    N, d, G = 5, 64, 3
    K = r.standard_normal((N, d)).astype(np.float32)
    V = r.standard_normal((N, d)).astype(np.float32)
    q = r.standard_normal((G, d)).astype(np.float32)
    for W in (N, N + 1, 2 * N):
        out = orc.attend_unit(q, K, V, N, np.zeros(0, np.int32), 0, W, 0.125)
        assert np.max(np.abs(out - dense_attention(q, K, V, 0.125))) < 1e-12
