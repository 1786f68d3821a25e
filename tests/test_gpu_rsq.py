"""GPU parity of the calibrated inner-product reranker (ParisKV, "Pipeline di
Recupero Nativa su GPU in Due Stadi", candidate reranking) against the oracle.

Records (a sign and 3-bit magnitude nibble per coordinate, bf16 calibration
scales) must match byte for byte; the selection with records ranks the same
candidate set as the exact path by estimates that must match bit for bit, and
the top-k index sets must be equal; attention over those sets within 2e-3.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import workloads as wl
import sparse_decode_attention_gb300 as kvr
from gpu_cases import attend_gpu, codes_bytes_gpu, encode_gpu, select_gpu

pytestmark = pytest.mark.gpu
ATOL = 2e-3


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    kvr.load()
    oracle.build()


def records_gpu(Kd, sgn_d, rows, pos0=0):
    rec = kvr.rsq_buffer(Kd)
    rec.fill_(0x5A)                                   # rows not written keep this
    p0 = torch.full((Kd.shape[0],), pos0, dtype=torch.int32, device=Kd.device)
    err = torch.zeros(1, dtype=torch.int32, device=Kd.device)
    kvr.kvr_encode_rsq(Kd, p0, rows, sgn_d, rec, err)
    return rec, kvr.kvr_read_error(err)


@pytest.mark.parametrize("d,dtype", [(64, torch.float32), (128, torch.bfloat16),
                                     (64, torch.bfloat16), (128, torch.float32)])
def test_records_bit_exact(d, dtype):
    g = torch.Generator().manual_seed(100 + d)
    B, Hkv, cap = 2, 3, 700
    K = torch.randn((B, Hkv, cap, d), generator=g) * torch.rand((B, Hkv, cap, 1), generator=g) * 4
    K[0, 0, 0] = 0.0                                          # zero key: top bin, no weight
    K[0, 0, 1] = -0.0
    K[0, 1, 2] = torch.randint(-3, 4, (d,), generator=g).float()  # exact zeros after FWHT
    K[1, 2, 5, :2] = 1.0
    K[1, 2, 5, 2:] = 0.0
    K[1, 0, 9] = 1e-20                                         # sub-normal squares
    K[1, 1, 11] = 1e15                                         # large squares, still finite
    K = K.to(dtype)
    sgn = wl.srht_signs(d)
    Kd = K.cuda()
    rec, bits = records_gpu(Kd, sgn.cuda(), cap)
    assert bits == 0
    ref = oracle.rsq_encode(K, sgn.numpy())
    assert np.array_equal(rec.cpu().numpy(), ref)


def test_records_appended_rows_and_bad_position():
    """Rows [pos0, pos0 + n) only; a range past the capacity sets the position
    bit and writes nothing outside the cache."""
    d, cap = 128, 300
    g = torch.Generator().manual_seed(3)
    K = torch.randn((2, 2, cap, d), generator=g).to(torch.bfloat16)
    sgn = wl.srht_signs(d)
    Kd, sgn_d = K.cuda(), sgn.cuda()
    rec, bits = records_gpu(Kd, sgn_d, 7, pos0=290)
    assert bits == 0
    got = rec.cpu().numpy()
    ref = oracle.rsq_encode(K, sgn.numpy())
    assert np.array_equal(got[:, :, 290:297], ref[:, :, 290:297])
    assert np.all(got[:, :, :290] == 0x5A) and np.all(got[:, :, 297:] == 0x5A)
    rec, bits = records_gpu(Kd, sgn_d, 20, pos0=290)
    assert bits & kvr.DEVERR["position"]
    got = rec.cpu().numpy()
    assert np.array_equal(got[:, :, 290:300], ref[:, :, 290:300])


def lowrank_case(B, Hq, Hkv, d, cap, seq, seed, planted=16, W=128, dtype="bf16"):
    w = wl.Workload("case", B=B, Hq=Hq, Hkv=Hkv, d=d, N=max(seq), dtype=dtype, W=W, rank=32,
                    planted=planted, seed=seed)
    return wl.make_cache(w, device="cpu", cap=cap, seq_len=seq)


def run_rsq(K, q, seq, C, k, W, lut, sgn, units=None):
    """GPU codes, records and reranked selection; each unit against the oracle."""
    B, Hkv, cap, d = K.shape
    G = q.shape[1] // Hkv
    Kd, qd, sgn_d = K.cuda(), q.cuda(), sgn.cuda()
    codes = encode_gpu(Kd, sgn_d, cap)
    rec, bits = records_gpu(Kd, sgn_d, cap)
    assert bits == 0
    params = kvr.SelectParams(C, k, W, lut, rsq_records=rec)
    seq_d = torch.tensor(seq, dtype=torch.int32, device="cuda")
    res = select_gpu(qd, Kd, codes, seq_d, sgn_d, params)
    ref_codes = oracle.encode(K, sgn.numpy())
    assert np.array_equal(codes_bytes_gpu(codes, Kd), ref_codes)
    ref_rec = oracle.rsq_encode(K, sgn.numpy())
    assert np.array_equal(rec.cpu().numpy(), ref_rec)
    for u in (units if units is not None else range(B * Hkv)):
        b, h = divmod(u, Hkv)
        N = int(seq[b])
        idx, cnt, dg = oracle.select_unit_rsq(q[b, h * G:(h + 1) * G], ref_codes[b, h, :N],
                                              ref_rec[b, h, :N], N, sgn.numpy(), C, k, W, lut,
                                              diagnostics=True)
        Cp = min(C, max(0, N - W))
        assert res["cand_count"][u] == Cp
        assert np.array_equal(res["cand"][u, :Cp], dg["cand"]), "candidates differ (unit %d)" % u
        assert np.array_equal(res["cand_S"][u, :Cp].view(np.int32), dg["cand_S"].view(np.int32)), \
            "estimates differ (unit %d)" % u
        assert res["count"][b, h] == cnt, u
        assert np.array_equal(res["idx"][b, h], idx), "top-k sets differ (unit %d)" % u
    return res, Kd, qd, seq_d


@pytest.mark.parametrize("lut", [wl.DEFAULT_LUT, wl.LINEAR_LUT])
def test_rsq_select_multi_chunk_ragged_batch(lut):
    """bf16 d128 GQA-4, two batch entries of different lengths, several
    2048-key chunks and a ragged tail."""
    seq = [19000, 7001]
    K, V, q = lowrank_case(2, 8, 2, 128, 20000, seq, seed=61)
    res, *_ = run_rsq(K, q, seq, 1024, 256, 128, lut, wl.srht_signs(128))
    assert res["err"] == 0


def test_rsq_select_fp32_d64():
    seq = [5000, 4097, 3000]
    K, V, q = lowrank_case(3, 8, 4, 64, 5000, seq, seed=62, dtype="f32")
    res, *_ = run_rsq(K, q, seq, 700, 100, 64, wl.DEFAULT_LUT, wl.srht_signs(64))
    assert res["err"] == 0


def test_rsq_select_long_ranges():
    """Past 256K tokens (score planes mostly in global memory; the
    optional-mode kernel set): estimates and top-k sets of two units of a
    ragged batch against the oracle."""
    seq = [300000, 270000]
    K, V, q = lowrank_case(2, 8, 2, 128, 300000, seq, seed=63)
    res, *_ = run_rsq(K, q, seq, 2048, 512, 128, wl.DEFAULT_LUT, wl.srht_signs(128),
                      units=[0, 3])
    assert res["err"] == 0


@pytest.mark.parametrize("C,k,W,seq", [
    (64, 16, 200, [150]),       # window covers the whole context: nothing selected
    (64, 16, 200, [201]),       # pool of one token
    (500, 500, 10, [300]),      # C and k larger than the pool
    (64, 0, 10, [2100]),        # k == 0
    (2047, 100, 1, [4100]),     # C - 1 around a chunk boundary
])
def test_rsq_select_edge_cases(C, k, W, seq):
    K, V, q = lowrank_case(1, 4, 2, 64, 4200, seq, seed=63, planted=4, W=W)
    res, *_ = run_rsq(K, q, seq, C, k, W, wl.DEFAULT_LUT, wl.srht_signs(64))
    assert res["err"] == 0


def test_rsq_equal_records_take_lowest_indices():
    d = 128
    row = torch.randn(d)
    K = row.expand(1, 2, 5000, d).clone().to(torch.bfloat16)
    q = torch.randn(1, 8, d).to(torch.bfloat16)
    res, *_ = run_rsq(K, q, [5000], 700, 300, 32, wl.DEFAULT_LUT, wl.srht_signs(d))
    for u in range(2):
        assert list(res["idx"][0, u]) == list(range(300))


def test_rsq_select_then_attend():
    """Attention over the reranked sets equals the oracle's over the same sets."""
    seq = [9000, 6500]
    K, V, q = lowrank_case(2, 8, 2, 128, 9000, seq, seed=64)
    res, Kd, qd, seq_d = run_rsq(K, q, seq, 1024, 256, 128, wl.DEFAULT_LUT, wl.srht_signs(128))
    idx = torch.from_numpy(res["idx"]).cuda()
    cnt = torch.from_numpy(res["count"]).cuda()
    scale = 1.0 / math.sqrt(128)
    out, bits = attend_gpu(qd, Kd, V.cuda(), idx, cnt, seq_d, 128, scale)
    assert bits == 0
    for b in range(2):
        for h in range(2):
            N = seq[b]
            ref = oracle.attend_unit(q[b, h * 4:(h + 1) * 4], K[b, h, :N], V[b, h, :N], N,
                                     res["idx"][b, h, :res["count"][b, h]], res["count"][b, h],
                                     128, np.float32(scale))
            assert np.abs(out[b, h * 4:(h + 1) * 4] - ref).max() <= ATOL


def test_rsq_recall_of_the_exact_top_k():
    """The reranked top-k keeps most of the exact path's top-k (the estimate
    is unbiased up to the bf16 scale): a loose property, not a parity check."""
    seq = [16000]
    K, V, q = lowrank_case(1, 8, 2, 128, 16000, seq, seed=65)
    sgn = wl.srht_signs(128)
    res, Kd, qd, seq_d = run_rsq(K, q, seq, 2048, 512, 128, wl.DEFAULT_LUT, sgn, units=[])
    codes = encode_gpu(Kd, sgn.cuda(), 16000)
    exact = select_gpu(qd, Kd, codes, seq_d, sgn.cuda(), kvr.SelectParams(2048, 512, 128))
    for h in range(2):
        a = set(res["idx"][0, h].tolist())
        e = set(exact["idx"][0, h].tolist())
        assert len(a & e) >= 0.8 * 512, (h, len(a & e))
