"""Pins of the reranker oracle (ParisKV, "Pipeline di Recupero Nativa su GPU in
Due Stadi": 4-bit sub-space direction codes from the rotation's Beta prior, a
calibration scale per key and sub-space, the inner-product estimate).

Independent statements checked against: scipy's Beta distribution and
quadrature for the quantiser, the dense Hadamard rotation in float64 for the
codes and scales, exactness on keys whose rotated sub-blocks are scaled sign
patterns, and a Python restatement of the candidate ranking.
"""
import math

import numpy as np
import pytest

import oracle
import workloads as wl

scipy_stats = pytest.importorskip("scipy.stats")
scipy_integrate = pytest.importorskip("scipy.integrate")

RNG = np.random.default_rng(77)
M = 8


def hadamard(d):
    i = np.arange(d)
    return np.where(np.bitwise_count(i[:, None] & i[None, :]) % 2, -1.0, 1.0)


def test_bin_edges_are_equal_probability_quantiles_of_the_beta_prior():
    bound, level = oracle.rsq_table(M)
    ref = np.sqrt(scipy_stats.beta.ppf(np.arange(1, 8) / 8, 0.5, (M - 1) / 2))
    assert bound[0] == 0 and bound[8] == 1
    assert np.abs(bound[1:8] - ref).max() < 1e-9
    # each bin holds probability 1/8 of |u_j|
    cdf = scipy_stats.beta.cdf(bound ** 2, 0.5, (M - 1) / 2)
    assert np.abs(np.diff(cdf) - 1 / 8).max() < 1e-9


def test_levels_are_conditional_means():
    bound, level = oracle.rsq_table(M)
    # density of t = |u_j|: 2 t * beta_pdf(t^2)
    f = lambda t: 2 * t * scipy_stats.beta.pdf(t * t, 0.5, (M - 1) / 2)
    for i in range(8):
        num = scipy_integrate.quad(lambda t: t * f(t), bound[i], bound[i + 1])[0]
        assert abs(level[i] - 8 * num) < 1e-8, i
        assert bound[i] < level[i] < bound[i + 1]


def test_float_tables_round_the_fp64_ones():
    bound, level = oracle.rsq_table(M)
    bsq, lev = oracle.rsq_float_tables(M)
    assert bsq[0] == 0
    assert np.array_equal(bsq[1:], (bound[1:8] ** 2).astype(np.float32))
    assert np.array_equal(lev, level.astype(np.float32))


def decode(rec, d):
    """Test-side reading of the documented record: a 32-bit word per block,
    nibble j = magnitude | sign << 3 of coordinate j, then bf16 scales."""
    nb = d // M
    words = rec[:4 * nb].view("<u4")
    nib = np.array([[(int(words[b]) >> (4 * j)) & 15 for j in range(M)] for b in range(nb)])
    sign, mag = nib >> 3, nib & 7
    scale = rec[4 * nb:].view(np.uint16).astype(np.uint32) << 16
    return sign, mag, scale.view(np.float32)


@pytest.mark.parametrize("d", [64, 128])
def test_records_against_the_float64_rotation(d):
    sgn = wl.srht_signs(d).numpy()
    K = RNG.normal(0, 1, (300, d)).astype(np.float32)
    K[5] = 0.0                                                   # a zero key
    rec = oracle.rsq_encode(K, sgn)
    assert rec.shape == (300, 6 * d // M)
    codes = oracle.encode(K, sgn)
    bound, level = oracle.rsq_table(M)
    z = (K.astype(np.float64) * sgn) @ hadamard(d).T
    near = 0
    for r in range(300):
        sign, mag, scale = decode(rec[r], d)
        # sign bits are the analytic centroid code
        assert np.array_equal(np.packbits(sign, axis=1, bitorder="little")[:, 0], codes[r])
        for b in range(d // M):
            zb = z[r, 8 * b:8 * b + 8]
            n2 = (zb ** 2).sum()
            if n2 == 0:
                # 0 >= edge * 0 for every edge: the top bin, and no weight
                assert scale[b] == 0 and np.all(mag[b] == 7)
                continue
            u2 = zb ** 2 / n2
            ref = (u2[:, None] >= bound[None, 1:8] ** 2).sum(1)
            gap = np.abs(u2[:, None] - bound[None, 1:8] ** 2).min(1)
            bad = ref != mag[b]
            assert np.all(gap[bad] < 1e-5)                    # only on a bin edge
            near += int(bad.sum())
            # w = ||z_b|| / <u_b, v_b>, stored as bf16
            v = level[mag[b]]
            w_ref = n2 / (np.abs(zb) * v).sum()
            assert abs(scale[b] - w_ref) <= 2 ** -8 * w_ref + 1e-12
    assert near <= 3


def sign_pattern_keys(n, d, sgn):
    """Keys whose rotated sub-blocks are sign patterns with random positive
    scales: then the dequantised direction is parallel to the true one."""
    nb = d // M
    signs = RNG.choice([-1.0, 1.0], (n, nb, M))
    alpha = RNG.uniform(0.5, 3.0, (n, nb, 1))
    z = (signs * alpha).reshape(n, d)
    # z = H D k  =>  k = D H z / d
    k = (z @ hadamard(d).T) / d * sgn
    return k.astype(np.float32), z


@pytest.mark.parametrize("d", [64, 128])
def test_estimate_is_exact_for_sign_pattern_keys(d):
    sgn = wl.srht_signs(d).numpy()
    K, z_exact = sign_pattern_keys(50, d, sgn)
    rec = oracle.rsq_encode(K, sgn)
    q = RNG.normal(0, 1, d).astype(np.float32)
    zq = oracle.fwht((q * sgn).astype(np.float32))
    zk = (K.astype(np.float64) * sgn) @ hadamard(d).T
    for r in range(50):
        est = float(oracle.rsq_score(rec[r], zq))
        exact = float(zk[r] @ zq.astype(np.float64))
        scale = np.abs(zk[r]).max() * np.abs(zq).sum()
        assert abs(est - exact) <= 2 ** -7 * scale, (r, est, exact)


def test_estimate_ranks_like_the_exact_score():
    d = 128
    sgn = wl.srht_signs(d).numpy()
    K = RNG.normal(0, 1, (3000, d)).astype(np.float32)
    rec = oracle.rsq_encode(K, sgn)
    q = RNG.normal(0, 1, d).astype(np.float32)
    zq = oracle.fwht((q * sgn).astype(np.float32))
    est = np.array([oracle.rsq_score(rec[i], zq) for i in range(3000)], dtype=np.float64)
    exact = K.astype(np.float64) @ q.astype(np.float64)
    assert np.corrcoef(est, exact)[0, 1] > 0.99
    assert abs(np.median(est / exact) - d) < 0.1 * d          # ~ <z_k, z_q> = d <k, q>


def test_selection_ranks_the_candidates_by_the_estimate():
    w = wl.TINY
    K, V, qb = wl.make_cache(w)
    sgn = wl.srht_signs(w.d).numpy()
    Ku = oracle.f32(K[0, 1])
    codes = oracle.encode(Ku, sgn)
    rec = oracle.rsq_encode(Ku, sgn)
    q = oracle.f32(qb[0, 1:2])
    N = w.N
    idx, cnt, dg = oracle.select_unit_rsq(q, codes, rec, N, sgn, w.C, w.k, w.W, w.lut,
                                          diagnostics=True)
    # the candidate set is the exact-rescoring path's
    _, _, dg_exact = oracle.select_unit(q, Ku, codes, N, sgn, w.C, w.k, w.W, w.lut,
                                        diagnostics=True)
    assert np.array_equal(dg["cand"], dg_exact["cand"])
    qbar = oracle.group_mean(q)
    zq = oracle.fwht((qbar * sgn).astype(np.float32))
    S = np.array([oracle.rsq_score(rec[i], zq) for i in dg["cand"]], dtype=np.float32)
    assert np.array_equal(S, dg["cand_S"])
    order = sorted(range(len(S)), key=lambda j: (-float(S[j]), int(dg["cand"][j])))
    ref = np.sort(dg["cand"][order[:w.k]])
    assert cnt == min(w.k, len(S)) and np.array_equal(idx[:cnt], ref)


def test_library_tables_equal_the_oracle_tables(kvr_lib):
    """The CUDA library builds its quantiser tables on the host from its own
    incomplete-beta code; they must round to the same fp32 values (host call,
    no GPU)."""
    bsq, lev = kvr_lib.kvr_rsq_tables()
    obsq, olev = oracle.rsq_float_tables(M)
    assert np.array_equal(np.array(bsq, dtype=np.float32), obsq)
    assert np.array_equal(np.array(lev, dtype=np.float32), olev)
