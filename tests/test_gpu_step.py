"""kvr_decode_step (encode of the appended key, selection, attention in one
library call) gives the results of the three separate calls, with the plain
window and with records + cache regions: codes, records, index sets and
counts bit for bit, the output bit for bit where the step runs the separate
attention and up to the summation order where selection and attention share
one launch; the prepared caller (DecodeStep) equals kvr_decode_step."""
import math

import numpy as np
import pytest
import torch

import oracle
import workloads as wl
import sparse_decode_attention_gb300 as kvr

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    kvr.load()
    oracle.build()


@pytest.mark.parametrize("mode", ["window", "window_rsq", "regions_rsq"])
def test_decode_step_equals_the_separate_calls(mode):
    seq0 = [9000, 6000]
    w = wl.Workload("step", B=2, Hq=8, Hkv=2, d=128, N=max(seq0) + 1, dtype="bf16", rank=32,
                    planted=16, seed=93)
    K, V, qb = wl.make_cache(w, device=DEV, cap=9100)
    sgn = wl.srht_signs(128, device=DEV)
    shape = kvr.Shape.of(K, qb)
    B, Hkv = 2, 2
    runs = []
    for how in ("separate", "fused", "prepared"):
        codes = kvr.codes_buffer(shape, DEV)
        kvr.kvr_encode_keys(K, torch.zeros(B, dtype=torch.int32, device=DEV), 9000, sgn, codes)
        rec = rend = None
        S = 0
        if mode.endswith("rsq"):
            rec = kvr.rsq_buffer(K)
            kvr.kvr_encode_rsq(K, torch.zeros(B, dtype=torch.int32, device=DEV), 9000, sgn, rec)
        if mode == "regions_rsq":
            S = 4
            rend = torch.tensor([8850, 5880], dtype=torch.int32, device=DEV)
        params = kvr.SelectParams(1024, 256, 128, wl.DEFAULT_LUT, rsq_records=rec, sink=S,
                                  region_end=rend)
        seq = torch.tensor([n + 1 for n in seq0], dtype=torch.int32, device=DEV)
        pos = torch.tensor(seq0, dtype=torch.int32, device=DEV)
        ws = kvr.workspace(kvr.kvr_select_workspace_size(shape, params))
        idx = torch.full((B, Hkv, 256), 7, dtype=torch.int32, device=DEV)
        cnt = torch.zeros((B, Hkv), dtype=torch.int32, device=DEV)
        out = torch.zeros((B, 8, 128), dtype=torch.float32, device=DEV)
        err = torch.zeros(1, dtype=torch.int32, device=DEV)
        q = wl.step_query(w, qb, 3).contiguous()
        scale = 1 / math.sqrt(128)
        if how == "separate":
            kvr.kvr_encode_keys(K, pos, 1, sgn, codes, err)
            if rec is not None:
                kvr.kvr_encode_rsq(K, pos, 1, sgn, rec, err)
            kvr.kvr_select(q, K, codes, seq, sgn, params, idx, cnt, ws, err)
            if rend is not None:
                kvr.kvr_sparse_attend_regions(q, K, V, idx, cnt, seq, S, rend, scale, out,
                                              kvr.workspace(0), err)
            else:
                kvr.kvr_sparse_attend(q, K, V, idx, cnt, seq, 128, scale, out, kvr.workspace(0),
                                      err)
        elif how == "fused":
            kvr.kvr_decode_step(q, K, V, codes, seq, pos, sgn, params, idx, cnt, scale, out, ws,
                                err)
            # a copy enqueued after the call sees the finished attention
            host = torch.empty(out.shape, dtype=out.dtype).pin_memory()
            host.copy_(out, non_blocking=True)
            torch.cuda.current_stream().synchronize()
            assert torch.equal(host, out.cpu())
        else:
            kvr.DecodeStep(q, K, V, codes, seq, pos, sgn, params, idx, cnt, scale, out, ws, err)()
        torch.cuda.synchronize()
        assert kvr.kvr_read_error(err) == 0
        runs.append((codes.cpu().numpy(), None if rec is None else rec.cpu().numpy(),
                     idx.cpu().numpy(), cnt.cpu().numpy(), out.cpu().numpy()))
    for other in runs[1:]:
        for a, b in zip(runs[0][:4], other[:4]):
            if a is not None:
                assert np.array_equal(a, b)
    fused = mode == "window"   # exact rescoring, Hamming votes, 4 heads: one launch
    if fused:
        assert np.abs(runs[0][4] - runs[1][4]).max() <= 1e-5
    else:
        assert np.array_equal(runs[0][4], runs[1][4])
    assert np.array_equal(runs[1][4], runs[2][4])
    assert runs[0][3].min() > 0


def test_decode_step_flags_an_appended_key_before_the_window():
    """With a window the step writes the appended key's code after the
    attention; a key before the window (read by that selection) is flagged."""
    w = wl.Workload("step", B=1, Hq=4, Hkv=1, d=64, N=3000, dtype="f32", rank=16, planted=4,
                    seed=5)
    K, V, qb = wl.make_cache(w, device=DEV, cap=3000)
    sgn = wl.srht_signs(64, device=DEV)
    shape = kvr.Shape.of(K, qb)
    codes = kvr.codes_buffer(shape, DEV)
    kvr.kvr_encode_keys(K, torch.zeros(1, dtype=torch.int32, device=DEV), 3000, sgn, codes)
    params = kvr.SelectParams(256, 64, 32, wl.DEFAULT_LUT)
    ws = kvr.workspace(kvr.kvr_select_workspace_size(shape, params))
    idx = torch.zeros((1, 1, 64), dtype=torch.int32, device=DEV)
    cnt = torch.zeros((1, 1), dtype=torch.int32, device=DEV)
    out = torch.zeros((1, 4, 64), dtype=torch.float32, device=DEV)
    seq = torch.tensor([3000], dtype=torch.int32, device=DEV)
    for pos_new, flagged in ((2999, False), (2968, False), (2967, True)):
        err = torch.zeros(1, dtype=torch.int32, device=DEV)
        pos = torch.tensor([pos_new], dtype=torch.int32, device=DEV)
        kvr.kvr_decode_step(qb, K, V, codes, seq, pos, sgn, params, idx, cnt, 0.125, out, ws, err)
        torch.cuda.synchronize()
        assert bool(kvr.kvr_read_error(err) & kvr.DEVERR["position"]) == flagged, pos_new
