"""GPU parity of the magnitude-aware coarse votes (ParisKV, "Pipeline di
Recupero Nativa su GPU in Due Stadi": top-rho most similar centroids per
sub-space) against the oracle: every pool key's coarse score, the candidate
set, the exact scores and the top-k sets bit for bit."""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
import sparse_decode_attention_gb300 as kvr
from gpu_cases import codes_bytes_gpu, encode_gpu, select_gpu

pytestmark = pytest.mark.gpu


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


def run_mag(K, q, seq, C, k, W, lut, sgn):
    B, Hkv, cap, d = K.shape
    G = q.shape[1] // Hkv
    Kd, qd, sgn_d = K.cuda(), q.cuda(), sgn.cuda()
    codes = encode_gpu(Kd, sgn_d, cap)
    params = kvr.SelectParams(C, k, W, lut, flags=kvr.SELECT_MAGNITUDE_VOTES)
    res = select_gpu(qd, Kd, codes, torch.tensor(seq, dtype=torch.int32, device="cuda"), sgn_d,
                     params)
    assert res["err"] == 0
    ref_codes = oracle.encode(K, sgn.numpy())
    assert np.array_equal(codes_bytes_gpu(codes, Kd), ref_codes)
    for u in range(B * Hkv):
        b, h = divmod(u, Hkv)
        N = int(seq[b])
        idx, cnt, dg = oracle.select_unit_mag(q[b, h * G:(h + 1) * G], K[b, h, :N],
                                              ref_codes[b, h, :N], N, sgn.numpy(), C, k, W, lut,
                                              diagnostics=True)
        pool = max(0, N - W)
        Cp = min(C, pool)
        assert np.array_equal(res["coarse"][u, :pool].astype(np.int32), dg["coarse"]), u
        assert res["cand_count"][u] == Cp
        assert np.array_equal(res["cand"][u, :Cp], dg["cand"]), u
        assert np.array_equal(res["cand_S"][u, :Cp].view(np.int32), dg["cand_S"].view(np.int32)), u
        assert res["count"][b, h] == cnt and np.array_equal(res["idx"][b, h], idx), u
    return res


@pytest.mark.parametrize("lut", [wl.DEFAULT_LUT, (5, 4, 4, 2, 1, 0, 0, 3, 9)])
def test_magnitude_votes_multi_chunk_ragged_batch(lut):
    seq = [19000, 7001]
    K, V, q = lowrank_case(2, 8, 2, 128, 20000, seq, seed=97)
    run_mag(K, q, seq, 1024, 256, 128, lut, wl.srht_signs(128))


def test_magnitude_votes_fp32_d64_every_tier_voted():
    seq = [5000, 3333]
    K, V, q = lowrank_case(2, 8, 4, 64, 5000, seq, seed=98, dtype="f32")
    run_mag(K, q, seq, 700, 100, 64, (8, 7, 6, 5, 4, 3, 2, 1, 1), wl.srht_signs(64))


def test_magnitude_votes_equal_magnitude_query_is_the_hamming_reading():
    """A query whose rotated sub-vectors have equal magnitudes: the magnitude
    votes equal the Hamming-ring votes, so the selection equals the plain one."""
    d, N = 128, 6000
    sgn = wl.srht_signs(d)
    rng = np.random.default_rng(5)
    z = np.where(rng.random(d) < 0.5, -1.0, 1.0)
    H = np.where(np.bitwise_count(np.arange(d)[:, None] & np.arange(d)[None, :]) % 2, -1.0, 1.0)
    qv = torch.from_numpy(((H @ z) / d * sgn.numpy()).astype(np.float32))
    q = qv.expand(1, 4, d).contiguous()                       # G = 4 equal heads: q_bar = qv
    K = torch.from_numpy(rng.normal(0, 1, (1, 1, N, d)).astype(np.float32))
    res = run_mag(K, q, [N], 600, 150, 64, wl.DEFAULT_LUT, sgn)
    plain = select_gpu(q.cuda(), K.cuda(), encode_gpu(K.cuda(), sgn.cuda(), N),
                       torch.tensor([N], dtype=torch.int32, device="cuda"), sgn.cuda(),
                       kvr.SelectParams(600, 150, 64, wl.DEFAULT_LUT))
    assert np.array_equal(res["coarse"], plain["coarse"])
    assert np.array_equal(res["idx"], plain["idx"])
