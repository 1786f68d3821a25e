"""Seeded random configurations of the main path against the oracle: head
dim, dtype, group size, batch, ragged lengths, window, candidate budget,
top-k and vote table drawn at random (including zero budgets, windows wider
than the context and arbitrary vote tables). Codes, coarse scores,
candidates, exact scores and top-k sets bit for bit; attention within 2e-3.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import workloads as wl
import sparse_decode_attention_gb300 as kvr
from gpu_cases import attend_gpu, codes_bytes_gpu, compare_select_unit, encode_gpu, select_gpu

pytestmark = pytest.mark.gpu
ATOL = 2e-3


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    kvr.load()
    oracle.build()


def draw(seed):
    r = np.random.default_rng(1000 + seed)
    d = int(r.choice([64, 128]))
    dtype = str(r.choice(["f32", "bf16"]))
    G = int(r.choice([1, 2, 4, 8, 16]))
    Hkv = int(r.integers(1, 4))
    B = int(r.integers(1, 4))
    seq = [int(x) for x in r.integers(1, 9000, size=B)]
    cap = max(seq) + int(r.integers(0, 300))
    W = int(r.choice([0, 1, 32, 128, 300, 10000]))
    C = int(r.choice([0, 1, 64, 700, 2048, 3000, 16384]))
    k = int(r.integers(0, C + 1)) if C else 0
    lut = tuple(int(x) for x in (r.integers(0, 16, size=9) if r.random() < 0.5
                                 else sorted(r.integers(0, 8, size=9), reverse=True)))
    return d, dtype, G, Hkv, B, seq, cap, W, C, k, lut


@pytest.mark.parametrize("seed", range(48))
def test_random_configuration(seed):
    d, dtype, G, Hkv, B, seq, cap, W, C, k, lut = draw(seed)
    w = wl.Workload("fuzz", B=B, Hq=Hkv * G, Hkv=Hkv, d=d, N=max(seq), dtype=dtype, W=W,
                    rank=16, planted=4, seed=seed)
    K, V, q = wl.make_cache(w, device="cpu", cap=cap, seq_len=seq)
    sgn = wl.srht_signs(d)
    Kd, Vd, qd, sgn_d = K.cuda(), V.cuda(), q.cuda(), sgn.cuda()
    codes = encode_gpu(Kd, sgn_d, cap)
    ref_codes = oracle.encode(K, sgn.numpy())
    assert np.array_equal(codes_bytes_gpu(codes, Kd), ref_codes)
    params = kvr.SelectParams(C, k, W, lut)
    seq_d = torch.tensor(seq, dtype=torch.int32, device="cuda")
    res = select_gpu(qd, Kd, codes, seq_d, sgn_d, params)
    assert res["err"] == 0
    scale = 1.0 / math.sqrt(d)
    out, bits = attend_gpu(qd, Kd, Vd, torch.from_numpy(res["idx"]).cuda(),
                           torch.from_numpy(res["count"]).cuda(), seq_d, W, scale)
    assert bits == 0
    for u in range(B * Hkv):
        b, h = divmod(u, Hkv)
        N = seq[b]
        idx, cnt = compare_select_unit(res, u, q[b, h * G:(h + 1) * G], K[b, h, :N],
                                       ref_codes[b, h, :N], N, sgn.numpy(), params)
        ref = oracle.attend_unit(q[b, h * G:(h + 1) * G], K[b, h, :N], V[b, h, :N], N,
                                 idx[:cnt], cnt, W, np.float32(scale))
        assert np.abs(out[b, h * G:(h + 1) * G] - ref).max() <= ATOL, (seed, u)
