"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle.

Codes, coarse scores, candidate sets, exact scores and top-k index sets must
match bit for bit; attention outputs within max-abs 2e-3 of the oracle's fp64
result over the same token set.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import workloads as wl
import sparse_decode_attention_gb300 as kvr
from gpu_cases import (attend_gpu, codes_bytes_gpu, compare_select_unit, encode_gpu, select_gpu,
                       shape_of_cache)

pytestmark = pytest.mark.gpu
ATOL = 2e-3


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    kvr.load()
    oracle.build()


def lowrank_case(B, Hq, Hkv, d, cap, seq, seed, planted=16, W=128):
    w = wl.Workload("case", B=B, Hq=Hq, Hkv=Hkv, d=d, N=max(seq), dtype="bf16", W=W, rank=32,
                    planted=planted, seed=seed)
    K, V, q = wl.make_cache(w, device="cpu", cap=cap, seq_len=seq)
    return K, V, q


# ------------------------------------------------------------------ encode

@pytest.mark.parametrize("d,dtype", [(64, torch.float32), (128, torch.bfloat16),
                                     (64, torch.bfloat16), (128, torch.float32)])
def test_encode_bit_exact(d, dtype):
    g = torch.Generator().manual_seed(d)
    B, Hkv, cap = 2, 3, 1000
    K = torch.randn((B, Hkv, cap, d), generator=g)
    K[0, 0, 0] = 0.0
    K[0, 0, 1] = -0.0
    K[0, 1, 2] = torch.randint(-3, 4, (d,), generator=g).float()  # exact zeros after FWHT
    K[1, 2, 5, :2] = 1.0
    K[1, 2, 5, 2:] = 0.0
    K = K.to(dtype)
    sgn = wl.srht_signs(d)
    Kd = K.cuda()
    codes = codes_bytes_gpu(encode_gpu(Kd, sgn.cuda(), cap), Kd)
    ref = oracle.encode(K, sgn.numpy())
    assert np.array_equal(codes, ref)


def test_encode_in_pieces_matches_one_pass():
    """Appending one row at a time, or ranges that start and end inside 32-token
    blocks, leaves the same codes as encoding everything at once."""
    d = 128
    K = torch.randn((1, 2, 2100, d)).to(torch.bfloat16).cuda()
    sgn = wl.srht_signs(d).cuda()
    whole = codes_bytes_gpu(encode_gpu(K, sgn, 2100), K)
    codes = kvr.codes_buffer(shape_of_cache(K))
    for p0, n in [(0, 5), (5, 1), (6, 57), (63, 1000), (1063, 1), (1064, 1036)]:
        kvr.kvr_encode_keys(K, torch.tensor([p0], dtype=torch.int32, device="cuda"), n, sgn,
                            codes)
    assert np.array_equal(codes_bytes_gpu(codes, K), whole)


def test_encode_rows_window_and_bad_position():
    d = 128
    K = torch.randn((2, 2, 300, d)).to(torch.bfloat16).cuda()
    sgn = wl.srht_signs(d).cuda()
    codes = kvr.codes_buffer(shape_of_cache(K))
    pos0 = torch.tensor([10, 295], dtype=torch.int32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    kvr.kvr_encode_keys(K, pos0, 7, sgn, codes, err)
    assert kvr.kvr_read_error(err) == kvr.DEVERR["position"]  # rows 300, 301 of batch 1
    ref = oracle.encode(K.cpu(), sgn.cpu().numpy())
    c = codes_bytes_gpu(codes, K)
    assert np.array_equal(c[0, :, 10:17], ref[0, :, 10:17])
    assert np.array_equal(c[1, :, 295:300], ref[1, :, 295:300])
    assert not c[0, :, :10].any() and not c[0, :, 17:].any() and not c[1, :, :295].any()


# ------------------------------------------------------------------ select

def run_and_compare(K, q, seq, params, sgn, units=None, check_diag=True):
    B, Hkv, cap, d = K.shape
    G = q.shape[1] // Hkv
    Kd, qd = K.cuda(), q.cuda()
    sgn_d = sgn.cuda()
    codes = encode_gpu(Kd, sgn_d, cap)
    seq_d = torch.tensor(seq, dtype=torch.int32, device="cuda")
    res = select_gpu(qd, Kd, codes, seq_d, sgn_d, params)
    ref_codes = oracle.encode(K, sgn.numpy())
    assert np.array_equal(codes_bytes_gpu(codes, Kd), ref_codes)
    out = {}
    for u in (units if units is not None else range(B * Hkv)):
        b, h = divmod(u, Hkv)
        N = int(seq[b])
        out[u] = compare_select_unit(res, u, q[b, h * G:(h + 1) * G], K[b, h, :N],
                                     ref_codes[b, h, :N], N, sgn.numpy(), params, check_diag)
    return res, out


def test_select_tiny_decode_steps():
    """The tiny workload: fp32 d64, 4 heads, 4096 context, 16 appending steps."""
    w = wl.TINY
    K, V, qb = wl.make_cache(w, cap=w.N + w.steps)
    sgn = wl.srht_signs(w.d)
    params = kvr.SelectParams(w.C, w.k, w.W, w.lut)
    Kd, Vd, sgn_d = K.cuda(), V.cuda(), sgn.cuda()
    codes = encode_gpu(Kd, sgn_d, w.N)  # prefill
    ref_codes = oracle.encode(K, sgn.numpy())
    scale = 1.0 / math.sqrt(w.d)
    for t in range(w.steps):
        N = w.N + t + 1
        kvr.kvr_encode_keys(Kd, torch.tensor([N - 1], dtype=torch.int32, device="cuda"), 1,
                            sgn_d, codes)
        q = wl.step_query(w, qb, t)
        seq = torch.tensor([N], dtype=torch.int32, device="cuda")
        res = select_gpu(q.cuda(), Kd, codes, seq, sgn_d, params)
        assert res["err"] == 0
        for u in range(w.Hkv):
            compare_select_unit(res, u, q[0, u:u + 1], K[0, u, :N], ref_codes[0, u, :N], N,
                                sgn.numpy(), params)
        out, bits = attend_gpu(q.cuda(), Kd, Vd, torch.from_numpy(res["idx"]).cuda(),
                               torch.from_numpy(res["count"]).cuda(), seq, w.W, scale)
        assert bits == 0
        ref = oracle.attend(q, K, V, res["idx"], res["count"], [N], w.W, np.float32(scale))
        assert np.max(np.abs(out - ref)) <= ATOL


@pytest.mark.parametrize("lut", [wl.DEFAULT_LUT, wl.LINEAR_LUT, (5, 4, 4, 2, 1, 0, 0, 3, 9)])
def test_select_multi_chunk_ragged_batch(lut):
    """bf16 d128 GQA-4, two batch entries of different lengths, several 2048-key
    chunks, a ragged tail, three vote tables (one with a distance-8 weight)."""
    seq = [19000, 7001]
    K, V, q = lowrank_case(2, 8, 2, 128, 20000, seq, seed=31)
    params = kvr.SelectParams(1024, 256, 128, lut)
    res, _ = run_and_compare(K, q, seq, params, wl.srht_signs(128))
    assert res["err"] == 0


@pytest.mark.parametrize("C,k,W,seq", [
    (64, 16, 200, [150]),       # window covers the whole context: nothing selected
    (64, 16, 200, [200]),       # pool empty at exactly N == W
    (64, 16, 200, [201]),       # pool of one token
    (500, 500, 10, [300]),      # C and k larger than the pool
    (64, 64, 10, [2100]),       # k == C
    (64, 0, 10, [2100]),        # k == 0
    (0, 0, 10, [2100]),         # C == 0
    (2047, 100, 1, [4100]),     # C - 1 around a chunk boundary
    (2049, 100, 0, [2049]),     # C + 1 > pool
])
def test_select_edge_cases(C, k, W, seq):
    K, V, q = lowrank_case(1, 4, 2, 64, 4200, seq, seed=41, planted=4, W=W)
    res, _ = run_and_compare(K, q, seq, kvr.SelectParams(C, k, W), wl.srht_signs(64))
    assert res["err"] == 0


def test_select_all_ties_take_lowest_indices():
    d = 128
    row = torch.randn(d)
    K = row.expand(1, 2, 5000, d).clone().to(torch.bfloat16)
    q = torch.randn(1, 8, d).to(torch.bfloat16)
    params = kvr.SelectParams(700, 300, 32)
    res, out = run_and_compare(K, q, [5000], params, wl.srht_signs(d))
    for u in range(2):
        assert list(res["idx"][0, u]) == list(range(300))


def test_select_bad_seq_len_sets_error_and_selects_nothing():
    K, V, q = lowrank_case(2, 4, 2, 64, 1000, [900, 900], seed=5, planted=0)
    Kd = K.cuda()
    sgn = wl.srht_signs(64).cuda()
    codes = encode_gpu(Kd, sgn, 1000)
    seq = torch.tensor([900, 1001], dtype=torch.int32, device="cuda")
    res = select_gpu(q.cuda(), Kd, codes, seq, sgn, kvr.SelectParams(64, 16, 8))
    assert res["err"] & kvr.DEVERR["seq_len"]
    assert np.all(res["count"][1] == 0) and np.all(res["idx"][1] == -1)
    assert np.all(res["count"][0] == 16)


# ------------------------------------------------------------------ attend

def test_attend_parity_ragged_gqa():
    seq = [3000, 1700]
    K, V, q = lowrank_case(2, 8, 2, 128, 3000, seq, seed=51)
    params = kvr.SelectParams(512, 300, 64)
    res, _ = run_and_compare(K, q, seq, params, wl.srht_signs(128), check_diag=False)
    scale = np.float32(1 / math.sqrt(128))
    out, bits = attend_gpu(q.cuda(), K.cuda(), V.cuda(), torch.from_numpy(res["idx"]).cuda(),
                           torch.from_numpy(res["count"]).cuda(),
                           torch.tensor(seq, dtype=torch.int32, device="cuda"), 64, float(scale))
    assert bits == 0
    ref = oracle.attend(q, K, V, res["idx"], res["count"], seq, 64, scale)
    assert np.max(np.abs(out - ref)) <= ATOL


@pytest.mark.parametrize("d,dtype", [(64, torch.float32), (128, torch.bfloat16)])
def test_full_selection_equals_dense_attention(d, dtype):
    """Top-k with k = C = pool reproduces dense attention over the whole context."""
    N, W, Hq, Hkv = 700, 37, 8, 2
    g = torch.Generator().manual_seed(d + 3)
    K = torch.randn((1, Hkv, N, d), generator=g).to(dtype)
    V = torch.randn((1, Hkv, N, d), generator=g).to(dtype)
    q = torch.randn((1, Hq, d), generator=g).to(dtype)
    params = kvr.SelectParams(N - W, N - W, W)
    res, _ = run_and_compare(K, q, [N], params, wl.srht_signs(d), check_diag=False)
    assert np.all(res["count"] == N - W)
    scale = 1 / math.sqrt(d)
    out, _ = attend_gpu(q.cuda(), K.cuda(), V.cuda(), torch.from_numpy(res["idx"]).cuda(),
                        torch.from_numpy(res["count"]).cuda(),
                        torch.tensor([N], dtype=torch.int32, device="cuda"), W, scale)
    qf, Kf, Vf = q.double()[0], K.double()[0], V.double()[0]
    G = Hq // Hkv
    for hq in range(Hq):
        s = (Kf[hq // G] @ qf[hq]) * float(np.float32(scale))
        p = torch.softmax(s, 0)
        dense = (p[:, None] * Vf[hq // G]).sum(0).numpy()
        assert np.max(np.abs(out[0, hq] - dense)) <= ATOL


def test_attend_special_sets_and_bad_index():
    d, N = 128, 500
    g = torch.Generator().manual_seed(9)
    K = torch.randn((1, 1, N, d), generator=g).to(torch.bfloat16)
    V = torch.randn((1, 1, N, d), generator=g).to(torch.bfloat16)
    q = torch.randn((1, 4, d), generator=g).to(torch.bfloat16)
    seq = torch.tensor([N], dtype=torch.int32, device="cuda")
    Kd, Vd, qd = K.cuda(), V.cuda(), q.cuda()
    # |T| = 1: the output is that token's value row
    idx = torch.tensor([[[123, 0, 0]]], dtype=torch.int32, device="cuda")
    one = torch.tensor([[1]], dtype=torch.int32, device="cuda")
    out, bits = attend_gpu(qd, Kd, Vd, idx, one, seq, 0, 0.1)
    assert bits == 0
    assert np.max(np.abs(out[0] - V[0, 0, 123].float().numpy()[None, :])) <= 1e-6
    # empty T: zeros
    zero = torch.tensor([[0]], dtype=torch.int32, device="cuda")
    out, _ = attend_gpu(qd, Kd, Vd, idx, zero, seq, 0, 0.1)
    assert not np.any(out)
    # an index inside the window is reported and skipped
    idx = torch.tensor([[[5, 498, 7]]], dtype=torch.int32, device="cuda")
    three = torch.tensor([[3]], dtype=torch.int32, device="cuda")
    out, bits = attend_gpu(qd, Kd, Vd, idx, three, seq, 4, 0.1)
    assert bits & kvr.DEVERR["index"]
    ref = oracle.attend(q, K, V, np.array([[[5, 7]]], np.int32), np.array([[2]]), [N], 4,
                        np.float32(0.1))
    assert np.max(np.abs(out - ref)) <= ATOL


def test_attend_many_segments_long_list():
    """k + W spanning many 128-token segments, with a ragged last segment."""
    d, N, k, W = 128, 9000, 3000, 77
    K, V, q = lowrank_case(1, 32, 8, d, N, [N], seed=61, W=W)
    params = kvr.SelectParams(6000, k, W)
    res, _ = run_and_compare(K, q, [N], params, wl.srht_signs(d), units=[0, 5],
                             check_diag=False)
    scale = np.float32(1 / math.sqrt(d))
    out, bits = attend_gpu(q.cuda(), K.cuda(), V.cuda(), torch.from_numpy(res["idx"]).cuda(),
                           torch.from_numpy(res["count"]).cuda(),
                           torch.tensor([N], dtype=torch.int32, device="cuda"), W, float(scale))
    assert bits == 0
    ref = oracle.attend(q, K, V, res["idx"], res["count"], [N], W, scale, units=[(0, 0), (0, 5)])
    for h in (0, 5):
        sl = slice(4 * h, 4 * h + 4)
        assert np.max(np.abs(out[:, sl] - ref[:, sl])) <= ATOL


@pytest.mark.parametrize("C,k", [(4096, 1000), (6000, 5999)])
def test_select_massive_ties_take_the_all_keys_path(C, k):
    """More than 2048 candidates share the boundary score bin (identical
    keys): the selection falls back to every CTA gathering all C' scores;
    ties still go to the lowest indices, bit-exact with the oracle."""
    d = 64
    row = torch.randn(d)
    K = row.expand(1, 2, 9000, d).clone()
    q = torch.randn(1, 4, d)
    params = kvr.SelectParams(C, k, 64)
    res, out = run_and_compare(K, q, [9000], params, wl.srht_signs(d))
    for u in range(2):
        assert list(res["idx"][0, u]) == list(range(k))
    assert res["err"] == 0


def test_select_near_ties_across_the_boundary_bin():
    """Keys on a handful of distinct score levels with thousands per level:
    the boundary bin holds more than 2048 keys of several exact scores."""
    d, N = 64, 12000
    g = torch.Generator().manual_seed(5)
    base = torch.randn(4, d, generator=g)
    K = base[torch.randint(0, 4, (N,), generator=g)].reshape(1, 1, N, d).contiguous()
    q = torch.randn(1, 2, d, generator=g)
    params = kvr.SelectParams(8000, 3000, 64)
    res, out = run_and_compare(K, q, [N], params, wl.srht_signs(d))
    assert res["err"] == 0


def dense_band_case(band, seed=3):
    """Keys that are positive multiples of one unit vector u, queries equal to
    u: every code ties (the candidates are the lowest pool positions) and the
    exact score of key i is about s_i. s: one key at 1000 and one at 1 span the
    range; 546 keys in [600, 900]; the rest form a band inside one 256th of
    the range, which therefore holds the k-th largest (k = 700) and hundreds
    of keys."""
    d, N = 64, 4000
    g = np.random.default_rng(seed)
    u = g.standard_normal(d).astype(np.float32)
    u /= np.linalg.norm(u)
    nb = 2048 - 2 - 546
    if band == "spread":
        b = g.uniform(500.0, 501.5, nb)
    elif band == "identical":
        b = np.full(nb, 500.5)
    else:  # "levels<L>": L distinct scores, each repeated
        L = int(band[len("levels"):])
        b = 500.0 + 0.15 * g.integers(0, L, nb)
    s = np.concatenate([[1000.0, 1.0], g.uniform(600.0, 900.0, 546), b])
    s = np.concatenate([s[:2], g.permutation(s[2:]), g.uniform(1.0, 1000.0, N - 2048)])
    K = torch.from_numpy((s[:, None] * u[None, :]).astype(np.float32)).reshape(1, 1, N, d)
    q = torch.from_numpy(np.stack([u, u])).reshape(1, 2, d)
    return K, q, N


@pytest.mark.parametrize("band", ["spread", "identical", "levels10", "levels3"])
def test_select_dense_boundary_bin(band):
    """Hundreds of candidates in the boundary score bin: their sub-bin
    refinement, ranking by counting or by radix passes (ties inside a
    sub-bin), bit-exact with the oracle."""
    K, q, N = dense_band_case(band)
    params = kvr.SelectParams(2048, 700, 64)
    res, out = run_and_compare(K, q, [N], params, wl.srht_signs(64))
    assert res["err"] == 0
