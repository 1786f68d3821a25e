"""kvr_select_attend (selection and attention of a step, one launch when the
group has at most 4 heads and rescoring is exact) against the CPU oracle.

Index sets and counts must match the oracle's selection bit for bit (and
kvr_select's), the output the oracle's fp64 attention over the same token set
within max-abs 2e-3. The cases cover the one-exchange score histogram (the
default and narrower vote tables) and the two-level one (the linear table),
candidates rescored by the CTA that found them and, when one CTA finds more
than its share allows, by equal slices; ragged batches, GQA groups of 1, 2
and 4 (one launch) and 8 (two launches), cache regions, the edge cases of the
selection, contexts past 256K tokens on every unit, and the 128K and
million-token layers at full size on sampled units.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import workloads as wl
import sparse_decode_attention_gb300 as kvr
from gpu_cases import codes_bytes_gpu, encode_gpu

pytestmark = pytest.mark.gpu
ATOL = 2e-3
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    kvr.load()
    oracle.build()


def lowrank_case(B, Hq, Hkv, d, cap, seq, seed, planted=16, W=128, dtype="bf16"):
    w = wl.Workload("case", B=B, Hq=Hq, Hkv=Hkv, d=d, N=max(seq), dtype=dtype, W=W, rank=32,
                    planted=planted, seed=seed)
    return wl.make_cache(w, device="cpu", cap=cap, seq_len=seq)


def run_fused(q, K, V, codes, seq_d, sgn_d, params, scale):
    B, Hkv, cap, d = K.shape
    shape = kvr.Shape.of(K, q)
    ws = kvr.workspace(kvr.kvr_select_workspace_size(shape, params))
    ws.fill_(0xAB)  # stale contents must not matter
    idx = torch.full((B, Hkv, params.k), 7, dtype=torch.int32, device=DEV)
    cnt = torch.full((B, Hkv), 7, dtype=torch.int32, device=DEV)
    out = torch.full(q.shape, float("nan"), dtype=torch.float32, device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    kvr.kvr_select_attend(q, K, V, codes, seq_d, sgn_d, params, scale, idx, cnt, out, ws, err)
    bits = kvr.kvr_read_error(err)
    return idx.cpu().numpy(), cnt.cpu().numpy(), out.cpu().numpy(), bits


def check_against_oracle(K, V, q, seq, params, sgn, units=None, codes_check=True):
    """Run kvr_select_attend on the GPU and compare every (or the listed)
    unit with the oracle; returns the GPU results."""
    B, Hkv, cap, d = K.shape
    G = q.shape[1] // Hkv
    Kd, Vd, qd, sgn_d = K.to(DEV), V.to(DEV), q.to(DEV), sgn.to(DEV)
    codes = encode_gpu(Kd, sgn_d, cap)
    ref_codes = oracle.encode(K, sgn.numpy())
    if codes_check:
        assert np.array_equal(codes_bytes_gpu(codes, Kd), ref_codes)
    seq_d = torch.tensor(seq, dtype=torch.int32, device=DEV)
    scale = np.float32(1 / math.sqrt(d))
    idx, cnt, out, bits = run_fused(qd, Kd, Vd, codes, seq_d, sgn_d, params, float(scale))
    assert bits == 0
    for u in (units if units is not None else range(B * Hkv)):
        b, h = divmod(u, Hkv)
        N = int(seq[b])
        qg = q[b, h * G:(h + 1) * G]
        ref_idx, ref_cnt = oracle.select_unit(qg, K[b, h, :N], ref_codes[b, h, :N], N,
                                              sgn.numpy(), params.C, params.k, params.W,
                                              params.lut)
        ref_out = oracle.attend_unit(qg, K[b, h, :N], V[b, h, :N], N, ref_idx[:ref_cnt],
                                     ref_cnt, params.W, scale)
        assert cnt[b, h] == ref_cnt, (b, h)
        assert np.array_equal(idx[b, h], ref_idx), (b, h)
        e = np.abs(out[b, h * G:(h + 1) * G] - ref_out).max()
        assert e <= ATOL, (b, h, e)
    return idx, cnt, out


@pytest.mark.parametrize("lut", [wl.DEFAULT_LUT, wl.LINEAR_LUT, (1, 1, 0, 0, 0, 0, 0, 0, 0),
                                 (5, 4, 4, 2, 1, 0, 0, 3, 9)])
def test_select_attend_ragged_batch_vote_tables(lut):
    """bf16 d128 GQA-4, two entries of different lengths over several code
    tiles: the one-exchange histogram (6-bit and 5-bit scores) and the
    two-level one (8-bit scores)."""
    seq = [19000, 7001]
    K, V, q = lowrank_case(2, 8, 2, 128, 20000, seq, seed=31)
    check_against_oracle(K, V, q, seq, kvr.SelectParams(1024, 256, 128, lut), wl.srht_signs(128))


@pytest.mark.parametrize("d,G,dtype", [(64, 1, "f32"), (64, 2, "bf16"), (128, 2, "f32"),
                                       (128, 4, "bf16"), (64, 8, "bf16")])
def test_select_attend_group_sizes(d, G, dtype):
    """Query groups of 1, 2 and 4 heads run in one launch (heads past the
    group score a zero query and are never written); 8 heads run the two
    calls."""
    seq = [5000]
    K, V, q = lowrank_case(1, 2 * G, 2, d, 5100, seq, seed=17 + G + d, dtype=dtype)
    check_against_oracle(K, V, q, seq, kvr.SelectParams(512, 200, 64), wl.srht_signs(d))


def test_select_attend_tiny_decode_steps():
    """The tiny workload (fp32 d64, 4 heads = 4 KV heads, 4096 context): 16
    appending steps."""
    w = wl.TINY
    K, V, qb = wl.make_cache(w, cap=w.N + w.steps)
    sgn = wl.srht_signs(w.d)
    params = kvr.SelectParams(w.C, w.k, w.W, w.lut)
    Kd, Vd, sgn_d = K.to(DEV), V.to(DEV), sgn.to(DEV)
    codes = encode_gpu(Kd, sgn_d, w.N)
    ref_codes = oracle.encode(K, sgn.numpy())
    scale = np.float32(1.0 / math.sqrt(w.d))
    for t in range(w.steps):
        N = w.N + t + 1
        kvr.kvr_encode_keys(Kd, torch.tensor([N - 1], dtype=torch.int32, device=DEV), 1, sgn_d,
                            codes)
        q = wl.step_query(w, qb, t)
        seq = torch.tensor([N], dtype=torch.int32, device=DEV)
        idx, cnt, out, bits = run_fused(q.to(DEV), Kd, Vd, codes, seq, sgn_d, params, float(scale))
        assert bits == 0
        for u in range(w.Hkv):
            ri, rc = oracle.select_unit(q[0, u:u + 1], K[0, u, :N], ref_codes[0, u, :N], N,
                                        sgn.numpy(), w.C, w.k, w.W, w.lut)
            assert cnt[0, u] == rc and np.array_equal(idx[0, u], ri)
            ro = oracle.attend_unit(q[0, u:u + 1], K[0, u, :N], V[0, u, :N], N, ri[:rc], rc,
                                    w.W, scale)
            assert np.abs(out[0, u:u + 1] - ro).max() <= ATOL


@pytest.mark.parametrize("C,k,W,seq", [
    (64, 16, 200, [150]),       # the window covers the context: attention over it alone
    (64, 16, 200, [200]),       # pool empty at N == W
    (64, 16, 200, [201]),       # pool of one token
    (500, 500, 10, [300]),      # C and k larger than the pool
    (64, 64, 10, [2100]),       # k == C
    (64, 0, 10, [2100]),        # k == 0: the window only
    (0, 0, 10, [2100]),         # C == 0
    (2047, 100, 1, [4100]),     # W = 1
    (2049, 100, 0, [2049]),     # W = 0: the top-k only
])
def test_select_attend_edge_cases(C, k, W, seq):
    K, V, q = lowrank_case(1, 4, 2, 64, 4200, seq, seed=41, planted=4, W=W)
    check_against_oracle(K, V, q, seq, kvr.SelectParams(C, k, W), wl.srht_signs(64))


def test_select_attend_candidates_concentrated_in_one_cta():
    """Identical keys: the candidates are the first C' pool positions, all in
    the lowest CTAs' ranges, more than one CTA may rescore (2048), so the
    list is cut into equal slices that other CTAs rescore; ties go to the
    lowest indices."""
    d, N = 64, 40000
    g = torch.Generator().manual_seed(77)
    row = torch.randn(d, generator=g)
    K = row.expand(1, 1, N, d).clone()
    V = torch.randn((1, 1, N, d), generator=g)
    q = torch.randn((1, 4, d), generator=g)
    params = kvr.SelectParams(8192, 3000, 64)
    idx, cnt, out = check_against_oracle(K, V, q, [N], params, wl.srht_signs(d))
    assert list(idx[0, 0]) == list(range(3000))


def test_select_attend_dense_boundary_bin():
    """Hundreds of exact scores inside one bin of the top-k exchange."""
    d, N = 64, 4000
    rng = np.random.default_rng(3)
    u = rng.standard_normal(d).astype(np.float32)
    u /= np.linalg.norm(u)
    s = np.concatenate([[1000.0, 1.0], rng.uniform(600.0, 900.0, 546),
                        rng.uniform(500.0, 501.5, 1500), rng.uniform(1.0, 1000.0, N - 2048)])
    K = torch.from_numpy((s[:, None] * u[None, :]).astype(np.float32)).reshape(1, 1, N, d)
    V = torch.from_numpy(rng.standard_normal((1, 1, N, d)).astype(np.float32))
    q = torch.from_numpy(np.stack([u, u])).reshape(1, 2, d)
    check_against_oracle(K, V, q, [N], kvr.SelectParams(2048, 700, 64), wl.srht_signs(d))


def test_select_attend_regions():
    """Cache regions: selection over [S, R), attention over the Sink, the
    top-k and [R, N); a ragged batch with the Sink inside a 32-token block."""
    seq = [9000, 5000]
    K, V, q = lowrank_case(2, 8, 2, 128, 9100, seq, seed=23)
    rend = torch.tensor([8850, 4900], dtype=torch.int32)
    params = kvr.SelectParams(1024, 256, 0, wl.DEFAULT_LUT, sink=5, region_end=rend.to(DEV))
    Kd = K.to(DEV)
    B, Hkv, cap, d = K.shape
    G = 4
    sgn = wl.srht_signs(d)
    codes = encode_gpu(Kd, sgn.to(DEV), cap)
    ref_codes = oracle.encode(K, sgn.numpy())
    idx, cnt, out, bits = run_fused(q.to(DEV), Kd, V.to(DEV), codes,
                                    torch.tensor(seq, dtype=torch.int32, device=DEV),
                                    sgn.to(DEV), params, float(np.float32(1 / math.sqrt(d))))
    assert bits == 0
    scale = np.float32(1 / math.sqrt(d))
    for b in range(B):
        for h in range(Hkv):
            N = seq[b]
            qg = q[b, h * G:(h + 1) * G]
            ri, rc = oracle.select_unit_regions(qg, K[b, h, :N], ref_codes[b, h, :N], N, 5,
                                                int(rend[b]), sgn.numpy(), 1024, 256,
                                                wl.DEFAULT_LUT)
            assert cnt[b, h] == rc and np.array_equal(idx[b, h], ri), (b, h)
            ro = oracle.attend_unit_regions(qg, K[b, h, :N], V[b, h, :N], N, 5, int(rend[b]),
                                            ri[:rc], rc, scale)
            assert np.abs(out[b, h * G:(h + 1) * G] - ro).max() <= ATOL, (b, h)


@pytest.mark.parametrize("mode", ["exact", "rsq", "magnitude"])
def test_select_attend_equals_the_two_calls(mode):
    """Indices and counts equal kvr_select's bit for bit; the output equals
    kvr_sparse_attend's up to the summation order (one launch for exact
    rescoring with Hamming votes; the two calls with records or magnitude
    votes)."""
    seq = [12000, 8000]
    K, V, q = lowrank_case(2, 8, 2, 128, 12100, seq, seed=3)
    Kd, Vd, qd = K.to(DEV), V.to(DEV), q.to(DEV)
    sgn = wl.srht_signs(128, device=DEV)
    codes = encode_gpu(Kd, sgn, 12100)
    rec = None
    if mode == "rsq":
        rec = kvr.rsq_buffer(Kd)
        kvr.kvr_encode_rsq(Kd, torch.zeros(2, dtype=torch.int32, device=DEV), 12100, sgn, rec)
    flags = kvr.SELECT_MAGNITUDE_VOTES if mode == "magnitude" else 0
    params = kvr.SelectParams(2048, 512, 128, wl.DEFAULT_LUT, flags=flags, rsq_records=rec)
    seq_d = torch.tensor(seq, dtype=torch.int32, device=DEV)
    scale = 1 / math.sqrt(128)
    shape = kvr.Shape.of(Kd, qd)
    ws = kvr.workspace(kvr.kvr_select_workspace_size(shape, params))
    i1 = torch.empty((2, 2, 512), dtype=torch.int32, device=DEV)
    c1 = torch.empty((2, 2), dtype=torch.int32, device=DEV)
    o1 = torch.empty((2, 8, 128), dtype=torch.float32, device=DEV)
    kvr.kvr_select(qd, Kd, codes, seq_d, sgn, params, i1, c1, ws)
    kvr.kvr_sparse_attend(qd, Kd, Vd, i1, c1, seq_d, 128, scale, o1, kvr.workspace(0))
    i2, c2, o2, bits = run_fused(qd, Kd, Vd, codes, seq_d, sgn, params, scale)
    assert bits == 0
    assert np.array_equal(i1.cpu().numpy(), i2) and np.array_equal(c1.cpu().numpy(), c2)
    assert np.abs(o1.cpu().numpy() - o2).max() <= 1e-5


def test_select_attend_long_ranges_every_unit():
    """Contexts past 256K tokens: every CTA scans 32 or more half-tiles and
    keeps most of its score planes in global memory (past the 512 blocks it
    holds on chip); a capacity past 512K tokens also puts the 8 units'
    clusters on SMs of their own (12 CTAs each on a GB300). Every unit of a
    ragged batch of 8 against the oracle, and kvr_select's index sets equal
    to the one-launch call's."""
    seq = [300000, 280000]
    K, V, q = lowrank_case(2, 16, 4, 128, 560000, seq, seed=77)
    params = kvr.SelectParams(4096, 1024, 128)
    sgn = wl.srht_signs(128)
    idx, cnt, _ = check_against_oracle(K, V, q, seq, params, sgn, codes_check=False)
    Kd, qd, sgn_d = K.to(DEV), q.to(DEV), sgn.to(DEV)
    codes = encode_gpu(Kd, sgn_d, 560000)
    seq_d = torch.tensor(seq, dtype=torch.int32, device=DEV)
    ws = kvr.workspace(kvr.kvr_select_workspace_size(kvr.Shape.of(Kd, qd), params))
    idx2 = torch.full((2, 4, 1024), 7, dtype=torch.int32, device=DEV)
    cnt2 = torch.zeros((2, 4), dtype=torch.int32, device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    kvr.kvr_select(qd, Kd, codes, seq_d, sgn_d, params, idx2, cnt2, ws, err)
    assert kvr.kvr_read_error(err) == 0
    assert np.array_equal(idx2.cpu().numpy(), idx) and np.array_equal(cnt2.cpu().numpy(), cnt)


def test_select_attend_128k_full_size_chain():
    """The 128K Llama-shaped layer at full size in the benchmark's launch
    form: kvr_select_attend with early inputs, chained over appending steps
    with no host synchronisation; every unit checked against the oracle after
    the last step."""
    w = wl.LLAMA_128K
    steps = 3
    K, V, qb = wl.make_cache(w, device=DEV, cap=w.N + steps)
    sgn = wl.srht_signs(w.d, device=DEV)
    shape = kvr.Shape.of(K, qb)
    codes = kvr.codes_buffer(shape, DEV)
    kvr.kvr_encode_keys(K, torch.zeros(1, dtype=torch.int32, device=DEV), w.N, sgn, codes)
    params = kvr.SelectParams(w.C, w.k, w.W, w.lut, flags=kvr.SELECT_EARLY_INPUTS)
    ws = kvr.workspace(kvr.kvr_select_workspace_size(shape, params))
    idx = torch.empty((1, w.Hkv, w.k), dtype=torch.int32, device=DEV)
    cnt = torch.empty((1, w.Hkv), dtype=torch.int32, device=DEV)
    out = torch.empty((1, w.Hq, w.d), dtype=torch.float32, device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    seq = torch.full((1,), w.N, dtype=torch.int32, device=DEV)
    pos = torch.full((1,), w.N - 1, dtype=torch.int32, device=DEV)
    scale = 1.0 / math.sqrt(w.d)
    qs = [wl.step_query(w, qb, t).contiguous() for t in range(steps)]
    torch.cuda.synchronize()
    for t in range(steps):
        seq.add_(1)
        pos.add_(1)
        kvr.kvr_decode_step(qs[t], K, V, codes, seq, pos, sgn, params, idx, cnt, scale, out, ws,
                            err)
    torch.cuda.synchronize()
    assert kvr.kvr_read_error(err) == 0
    N = w.N + steps
    q = qs[-1].float().cpu().numpy()
    sg = sgn.cpu().numpy()
    idx_h, cnt_h, out_h = idx.cpu().numpy(), cnt.cpu().numpy(), out.cpu().numpy()
    for h in range(w.Hkv):
        Ku = oracle.f32(K[0, h, :N].cpu())
        Vu = oracle.f32(V[0, h, :N].cpu())
        cu = oracle.encode(Ku, sg)
        qg = q[0, h * w.G:(h + 1) * w.G]
        ri, rc = oracle.select_unit(qg, Ku, cu, N, sg, w.C, w.k, w.W, w.lut)
        assert cnt_h[0, h] == rc and np.array_equal(idx_h[0, h], ri), h
        ro = oracle.attend_unit(qg, Ku, Vu, N, ri[:rc], rc, w.W, np.float32(scale))
        assert np.abs(out_h[0, h * w.G:(h + 1) * w.G] - ro).max() <= ATOL, h


def test_select_attend_million_token_sampled_units():
    """The million-token layer (2^20 tokens, C 16384, k 4096, W 256) at full
    size, device-resident: two sampled units against the oracle."""
    w = wl.MILLION
    K, V, qb = wl.make_cache(w, device=DEV, cap=w.N)
    sgn = wl.srht_signs(w.d, device=DEV)
    shape = kvr.Shape.of(K, qb)
    codes = kvr.codes_buffer(shape, DEV)
    kvr.kvr_encode_keys(K, torch.zeros(1, dtype=torch.int32, device=DEV), w.N, sgn, codes)
    params = kvr.SelectParams(w.C, w.k, w.W, w.lut)
    ws = kvr.workspace(kvr.kvr_select_workspace_size(shape, params))
    seq = torch.full((1,), w.N, dtype=torch.int32, device=DEV)
    q = wl.step_query(w, qb, 0).contiguous()
    idx, cnt, out, bits = run_fused(q, K, V, codes, seq, sgn, params, 1.0 / math.sqrt(w.d))
    assert bits == 0
    qn = q.float().cpu().numpy()
    sg = sgn.cpu().numpy()
    scale = np.float32(1.0 / math.sqrt(w.d))
    for h in (0, 5):
        Ku = oracle.f32(K[0, h].cpu())
        Vu = oracle.f32(V[0, h].cpu())
        cu = oracle.encode(Ku, sg)
        qg = qn[0, h * w.G:(h + 1) * w.G]
        ri, rc = oracle.select_unit(qg, Ku, cu, w.N, sg, w.C, w.k, w.W, w.lut)
        assert cnt[0, h] == rc and np.array_equal(idx[0, h], ri), h
        ro = oracle.attend_unit(qg, Ku, Vu, w.N, ri[:rc], rc, w.W, scale)
        assert np.abs(out[0, h * w.G:(h + 1) * w.G] - ro).max() <= ATOL, h
