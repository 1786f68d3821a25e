"""GPU parity of the cache regions (ParisKV, "Meccanismo di Aggiornamento a
Finestra Scorrevole": Sink, Retrieval, Local and Update Buffer).

kvr_regions_update must reproduce the oracle's region ends bit for bit over
appending steps; kvr_select with a sink and region ends must select exactly
the oracle's candidates, scores and top-k sets over the Retrieval region; the
attention over Sink + top-k + Local/buffer within 2e-3 of the oracle.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import workloads as wl
import sparse_decode_attention_gb300 as kvr
from gpu_cases import codes_bytes_gpu, encode_gpu, select_gpu

pytestmark = pytest.mark.gpu
ATOL = 2e-3
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    kvr.load()
    oracle.build()


def test_region_update_follows_the_oracle_over_appends():
    N0 = [1000, 50, 130, 0, 4096]
    S, L, U = 64, 128, 48
    seq = torch.tensor(N0, dtype=torch.int32, device=DEV)
    rend = torch.full((len(N0),), -7, dtype=torch.int32, device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    kvr.kvr_regions_update(seq, S, L, U, rend, init=True, err=err)
    ref = [oracle.region_init(n, S, L) for n in N0]
    assert rend.cpu().tolist() == ref
    for step in range(1, 400):
        grow = [1, 1, 2, 0, 3]                      # appends per step differ per entry
        n = [a + g * step for a, g in zip(N0, grow)]
        seq.copy_(torch.tensor(n, dtype=torch.int32))
        kvr.kvr_regions_update(seq, S, L, U, rend, err=err)
        ref = [oracle.region_advance(n[b], ref[b], S, L, U) for b in range(len(n))]
        assert rend.cpu().tolist() == ref, step
    assert kvr.kvr_read_error(err) == 0
    # a negative length is reported and leaves its entry alone
    seq[1] = -5
    kvr.kvr_regions_update(seq, S, L, U, rend, err=err)
    assert kvr.kvr_read_error(err) & kvr.DEVERR["seq_len"]
    assert int(rend[1]) == ref[1]


def lowrank_case(B, Hq, Hkv, d, cap, seq, seed, planted=16, W=128, dtype="bf16"):
    w = wl.Workload("case", B=B, Hq=Hq, Hkv=Hkv, d=d, N=max(seq), dtype=dtype, W=W, rank=32,
                    planted=planted, seed=seed)
    return wl.make_cache(w, device="cpu", cap=cap, seq_len=seq)


def run_regions(K, V, q, seq, S, R, C, k, lut, sgn, rerank=False, R_none_W=None):
    """GPU selection + attention over the regions; every unit against the oracle."""
    B, Hkv, cap, d = K.shape
    G = q.shape[1] // Hkv
    Kd, Vd, qd, sgn_d = K.to(DEV), V.to(DEV), q.to(DEV), sgn.to(DEV)
    codes = encode_gpu(Kd, sgn_d, cap)
    rec = None
    if rerank:
        rec = kvr.rsq_buffer(Kd)
        kvr.kvr_encode_rsq(Kd, torch.zeros(B, dtype=torch.int32, device=DEV), cap, sgn_d, rec)
    seq_d = torch.tensor(seq, dtype=torch.int32, device=DEV)
    if R_none_W is None:
        rend = torch.tensor(R, dtype=torch.int32, device=DEV)
        params = kvr.SelectParams(C, k, 0, lut, rsq_records=rec, sink=S, region_end=rend)
    else:
        rend = torch.tensor([n - R_none_W for n in seq], dtype=torch.int32, device=DEV)
        params = kvr.SelectParams(C, k, R_none_W, lut, rsq_records=rec, sink=S)
    res = select_gpu(qd, Kd, codes, seq_d, sgn_d, params)
    assert res["err"] == 0
    idx = torch.from_numpy(res["idx"]).to(DEV)
    cnt = torch.from_numpy(res["count"]).to(DEV)
    out = torch.full(q.shape, float("nan"), dtype=torch.float32, device=DEV)
    ws = kvr.workspace(kvr.kvr_attend_workspace_size(kvr.Shape.of(Kd, qd), k, 0))
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    scale = 1.0 / math.sqrt(d)
    kvr.kvr_sparse_attend_regions(qd, Kd, Vd, idx, cnt, seq_d, S, rend, scale, out, ws, err)
    assert kvr.kvr_read_error(err) == 0
    out = out.cpu().numpy()
    ref_codes = oracle.encode(K, sgn.numpy())
    assert np.array_equal(codes_bytes_gpu(codes, Kd), ref_codes)
    ref_rec = oracle.rsq_encode(K, sgn.numpy()) if rerank else None
    rl = rend.cpu().tolist()
    for u in range(B * Hkv):
        b, h = divmod(u, Hkv)
        N = int(seq[b])
        qg = q[b, h * G:(h + 1) * G]
        Ku = oracle.f32(K[b, h, :N])
        ri, rc, dg = oracle.select_unit_regions(qg, Ku, ref_codes[b, h, :N], N, S, rl[b],
                                                sgn.numpy(), C, k, lut,
                                                rec_unit=None if ref_rec is None else ref_rec[b, h, :N],
                                                diagnostics=True)
        nc = len(dg["cand"])
        assert res["cand_count"][u] == nc, u
        assert np.array_equal(res["cand"][u, :nc], dg["cand"]), "candidates differ (unit %d)" % u
        assert np.array_equal(res["cand_S"][u, :nc].view(np.int32), dg["cand_S"].view(np.int32)), u
        assert res["count"][b, h] == rc and np.array_equal(res["idx"][b, h], ri), u
        ref = oracle.attend_unit_regions(qg, Ku, oracle.f32(V[b, h, :N]), N, S, rl[b], ri[:rc], rc,
                                         np.float32(scale))
        assert np.abs(out[b, h * G:(h + 1) * G] - ref).max() <= ATOL, u
    return res


def test_regions_ragged_batch_multi_chunk():
    """Sink ending inside a 32-token block, region ends not aligned, several
    2048-key chunks, a ragged second entry."""
    seq = [19000, 7001]
    K, V, q = lowrank_case(2, 8, 2, 128, 20000, seq, seed=81)
    run_regions(K, V, q, seq, S=37, R=[18850, 6901], C=1024, k=256, lut=wl.DEFAULT_LUT,
                sgn=wl.srht_signs(128))


def test_regions_with_the_reranker_fp32_d64():
    seq = [5000, 4097]
    K, V, q = lowrank_case(2, 8, 4, 64, 5000, seq, seed=82, dtype="f32")
    run_regions(K, V, q, seq, S=4, R=[4900, 3969], C=700, k=100, lut=wl.DEFAULT_LUT,
                sgn=wl.srht_signs(64), rerank=True)


@pytest.mark.parametrize("S,R,seq", [
    (64, [100], [60]),          # shorter than the sink: everything is sink
    (64, [20], [300]),          # region end inside the sink: clamped, empty pool
    (4, [900], [500]),          # region end past N: clamped, no Local
    (0, [250], [300]),          # no sink
    (2048, [4000], [4100]),     # sink of one chunk
])
def test_region_edge_cases(S, R, seq):
    K, V, q = lowrank_case(1, 4, 2, 64, 4200, seq, seed=83, planted=4)
    run_regions(K, V, q, seq, S=S, R=R, C=500, k=120, lut=wl.DEFAULT_LUT, sgn=wl.srht_signs(64))


def test_sink_without_region_ends_uses_the_window():
    seq = [6000]
    K, V, q = lowrank_case(1, 8, 2, 128, 6000, seq, seed=84)
    run_regions(K, V, q, seq, S=16, R=None, C=800, k=200, lut=wl.DEFAULT_LUT,
                sgn=wl.srht_signs(128), R_none_W=128)


def test_decode_loop_with_buffer_flushes():
    """Appending decode steps: codes of each new key, region ends advanced on
    the device, selection + attention over the regions; the buffer flushes
    every U steps. Sampled steps against the oracle."""
    S, L, U = 4, 128, 32
    B, Hq, Hkv, d = 2, 8, 2, 128
    N0, T = 9000, 70
    w = wl.Workload("loop", B=B, Hq=Hq, Hkv=Hkv, d=d, N=N0 + T, dtype="bf16", rank=32,
                    planted=16, seed=85)
    K, V, qb = wl.make_cache(w, device="cpu", cap=N0 + T)
    sgn = wl.srht_signs(d)
    Kd, Vd, sgn_d = K.to(DEV), V.to(DEV), sgn.to(DEV)
    codes = kvr.codes_buffer(kvr.Shape.of(Kd, qb.to(DEV)), DEV)
    kvr.kvr_encode_keys(Kd, torch.zeros(B, dtype=torch.int32, device=DEV), N0, sgn_d, codes)
    seq = torch.full((B,), N0, dtype=torch.int32, device=DEV)
    rend = torch.zeros(B, dtype=torch.int32, device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    kvr.kvr_regions_update(seq, S, L, U, rend, init=True, err=err)
    C, k = 1024, 256
    params = kvr.SelectParams(C, k, 0, wl.DEFAULT_LUT, sink=S, region_end=rend)
    shape = kvr.Shape.of(Kd, qb.to(DEV))
    ws_s = kvr.workspace(kvr.kvr_select_workspace_size(shape, params))
    ws_a = kvr.workspace(kvr.kvr_attend_workspace_size(shape, k, 0))
    idx = torch.empty((B, Hkv, k), dtype=torch.int32, device=DEV)
    cnt = torch.empty((B, Hkv), dtype=torch.int32, device=DEV)
    out = torch.empty((B, Hq, d), dtype=torch.float32, device=DEV)
    scale = 1.0 / math.sqrt(d)
    R_ref = oracle.region_init(N0, S, L)
    flushes = 0
    for t in range(T):
        N = N0 + t + 1
        seq.fill_(N)
        kvr.kvr_encode_keys(Kd, torch.full((B,), N - 1, dtype=torch.int32, device=DEV), 1, sgn_d,
                            codes, err)
        kvr.kvr_regions_update(seq, S, L, U, rend, err=err)
        q = wl.step_query(w, qb.to(DEV), t).contiguous()
        kvr.kvr_select(q, Kd, codes, seq, sgn_d, params, idx, cnt, ws_s, err)
        kvr.kvr_sparse_attend_regions(q, Kd, Vd, idx, cnt, seq, S, rend, scale, out, ws_a, err)
        R_new = oracle.region_advance(N, R_ref, S, L, U)
        flushes += R_new != R_ref
        R_ref = R_new
        assert rend.cpu().tolist() == [R_ref] * B, t
        if t % 17 == 0 or t == T - 1:
            qn, on, ix, cn = q.float().cpu().numpy(), out.cpu().numpy(), idx.cpu().numpy(), cnt.cpu().numpy()
            for b, h in ((0, 0), (1, 1)):
                Ku = oracle.f32(K[b, h, :N])
                codes_u = oracle.encode(Ku, sgn.numpy())
                qg = qn[b, h * (Hq // Hkv):(h + 1) * (Hq // Hkv)]
                ri, rc = oracle.select_unit_regions(qg, Ku, codes_u, N, S, R_ref, sgn.numpy(), C, k,
                                                    wl.DEFAULT_LUT)
                assert cn[b, h] == rc and np.array_equal(ix[b, h], ri), (t, b, h)
                ref = oracle.attend_unit_regions(qg, Ku, oracle.f32(V[b, h, :N]), N, S, R_ref,
                                                 ri[:rc], rc, np.float32(scale))
                assert np.abs(on[b, h * (Hq // Hkv):(h + 1) * (Hq // Hkv)] - ref).max() <= ATOL
    assert flushes >= 2
    assert kvr.kvr_read_error(err) == 0
