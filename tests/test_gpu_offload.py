"""Host-resident caches (ParisKV, "Offloading tramite Indirizzamento Virtuale
Unificato"): K and V live in page-locked host memory mapped into the device's
address space; codes, records, queries and outputs live on the device. The
kernels gather rows over the host link through the same C-ABI calls.

Parity bar as for device caches: codes, records, candidates, scores and top-k
sets bit-exact against the oracle (and identical to the run with the same
cache in device memory), attention within 2e-3.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import workloads as wl
import sparse_decode_attention_gb300 as kvr
from gpu_cases import codes_bytes_gpu

pytestmark = pytest.mark.gpu
ATOL = 2e-3
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    kvr.load()
    oracle.build()


def pinned(t):
    h = torch.empty(t.shape, dtype=t.dtype, pin_memory=True)
    h.copy_(t)
    return h


def run_path(K, V, q, seq, w, sgn_d, rerank):
    """Codes (and records), selection and attention with K, V where they are."""
    B, Hkv, cap, d = K.shape
    shape = kvr.Shape.of(K, q)
    codes = kvr.codes_buffer(shape, DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    p0 = torch.zeros(B, dtype=torch.int32, device=DEV)
    kvr.kvr_encode_keys(K, p0, cap, sgn_d, codes, err)
    rec = None
    if rerank:
        rec = kvr.rsq_buffer(K)
        kvr.kvr_encode_rsq(K, p0, cap, sgn_d, rec, err)
    params = kvr.SelectParams(w.C, w.k, w.W, w.lut, rsq_records=rec)
    ws_s = kvr.workspace(kvr.kvr_select_workspace_size(shape, params))
    ws_a = kvr.workspace(kvr.kvr_attend_workspace_size(shape, w.k, w.W))
    idx = torch.empty((B, Hkv, w.k), dtype=torch.int32, device=DEV)
    cnt = torch.empty((B, Hkv), dtype=torch.int32, device=DEV)
    out = torch.empty(q.shape, dtype=torch.float32, device=DEV)
    seq_d = torch.tensor(seq, dtype=torch.int32, device=DEV)
    kvr.kvr_select(q, K, codes, seq_d, sgn_d, params, idx, cnt, ws_s, err)
    kvr.kvr_sparse_attend(q, K, V, idx, cnt, seq_d, w.W, 1.0 / math.sqrt(d), out, ws_a, err)
    torch.cuda.synchronize()
    return dict(codes=codes_bytes_gpu(codes, K), rec=None if rec is None else rec.cpu().numpy(),
                idx=idx.cpu().numpy(), cnt=cnt.cpu().numpy(), out=out.cpu().numpy(),
                err=kvr.kvr_read_error(err))


@pytest.mark.parametrize("rerank", [False, True])
def test_host_resident_cache_matches_oracle_and_device_cache(rerank):
    seq = [12000, 9000]
    w = wl.Workload("offload", B=2, Hq=8, Hkv=2, d=128, N=max(seq), dtype="bf16", C=1024, k=256,
                    W=128, rank=32, planted=16, seed=71)
    K, V, q = wl.make_cache(w, device="cpu", cap=12288, seq_len=seq)
    sgn = wl.srht_signs(w.d)
    sgn_d, qd = sgn.to(DEV), q.to(DEV)
    host = run_path(pinned(K), pinned(V), qd, seq, w, sgn_d, rerank)
    dev = run_path(K.to(DEV), V.to(DEV), qd, seq, w, sgn_d, rerank)
    assert host["err"] == 0 and dev["err"] == 0
    for key in ("codes", "rec", "idx", "cnt", "out"):
        if host[key] is not None:
            assert np.array_equal(host[key], dev[key]), key      # same kernels, same bits
    ref_codes = oracle.encode(K, sgn.numpy())
    assert np.array_equal(host["codes"], ref_codes)
    ref_rec = oracle.rsq_encode(K, sgn.numpy()) if rerank else None
    if rerank:
        assert np.array_equal(host["rec"], ref_rec)
    scale = np.float32(1.0 / math.sqrt(w.d))
    for b in range(w.B):
        N = seq[b]
        for h in range(w.Hkv):
            qg = q[b, h * w.G:(h + 1) * w.G]
            Ku = oracle.f32(K[b, h, :N])
            if rerank:
                ri, rc = oracle.select_unit_rsq(qg, ref_codes[b, h, :N], ref_rec[b, h, :N], N,
                                                sgn.numpy(), w.C, w.k, w.W, w.lut)
            else:
                ri, rc = oracle.select_unit(qg, Ku, ref_codes[b, h, :N], N, sgn.numpy(), w.C,
                                            w.k, w.W, w.lut)
            assert host["cnt"][b, h] == rc and np.array_equal(host["idx"][b, h], ri), (b, h)
            ref = oracle.attend_unit(qg, Ku, oracle.f32(V[b, h, :N]), N, ri[:rc], rc, w.W, scale)
            assert np.abs(host["out"][b, h * w.G:(h + 1) * w.G] - ref).max() <= ATOL, (b, h)


def test_host_resident_cache_with_regions_and_records():
    """The one-call step over a host-resident cache with reranker records and
    cache regions equals the same step over the device-resident cache, and the
    oracle's selection and attention over the regions."""
    seq0 = [7000, 5000]
    w = wl.Workload("offreg", B=2, Hq=8, Hkv=2, d=128, N=max(seq0) + 1, dtype="bf16", C=1024,
                    k=256, W=128, rank=32, planted=16, seed=72)
    K, V, q = wl.make_cache(w, device="cpu", cap=7200, seq_len=[n + 1 for n in seq0])
    sgn = wl.srht_signs(w.d)
    sgn_d, qd = sgn.to(DEV), q.to(DEV)
    S, L, U = 4, 128, 32
    runs = []
    for Kx, Vx in ((pinned(K), pinned(V)), (K.to(DEV), V.to(DEV))):
        shape = kvr.Shape.of(Kx, qd)
        codes = kvr.codes_buffer(shape, DEV)
        rec = kvr.rsq_buffer(Kx)
        p0 = torch.zeros(2, dtype=torch.int32, device=DEV)
        kvr.kvr_encode_keys(Kx, p0, 7000, sgn_d, codes)
        kvr.kvr_encode_rsq(Kx, p0, 7000, sgn_d, rec)
        seq = torch.tensor([n + 1 for n in seq0], dtype=torch.int32, device=DEV)
        rend = torch.zeros(2, dtype=torch.int32, device=DEV)
        kvr.kvr_regions_update(seq, S, L, U, rend, init=True)
        params = kvr.SelectParams(w.C, w.k, 0, w.lut, rsq_records=rec, sink=S, region_end=rend)
        ws = kvr.workspace(kvr.kvr_select_workspace_size(shape, params))
        idx = torch.empty((2, 2, w.k), dtype=torch.int32, device=DEV)
        cnt = torch.empty((2, 2), dtype=torch.int32, device=DEV)
        out = torch.empty(qd.shape, dtype=torch.float32, device=DEV)
        err = torch.zeros(1, dtype=torch.int32, device=DEV)
        pos = torch.tensor(seq0, dtype=torch.int32, device=DEV)
        kvr.kvr_decode_step(qd, Kx, Vx, codes, seq, pos, sgn_d, params, idx, cnt,
                            1 / math.sqrt(w.d), out, ws, err)
        torch.cuda.synchronize()
        assert kvr.kvr_read_error(err) == 0
        runs.append((idx.cpu().numpy(), cnt.cpu().numpy(), out.cpu().numpy(),
                     rend.cpu().tolist()))
    for a, b in zip(runs[0], runs[1]):
        assert np.array_equal(np.asarray(a), np.asarray(b))
    idx, cnt, out, rl = runs[0]
    sg = sgn.numpy()
    for b in range(2):
        N = seq0[b] + 1
        for h in range(2):
            Ku = oracle.f32(K[b, h, :N])
            qg = q[b, h * 4:(h + 1) * 4]
            ri, rc = oracle.select_unit_regions(qg, Ku, oracle.encode(Ku, sg), N, S, rl[b], sg,
                                                w.C, w.k, w.lut, rec_unit=oracle.rsq_encode(Ku, sg))
            assert cnt[b, h] == rc and np.array_equal(idx[b, h], ri), (b, h)
            ref = oracle.attend_unit_regions(qg, Ku, oracle.f32(V[b, h, :N]), N, S, rl[b], ri[:rc],
                                             rc, np.float32(1 / math.sqrt(w.d)))
            assert np.abs(out[b, h * 4:(h + 1) * 4] - ref).max() <= ATOL
