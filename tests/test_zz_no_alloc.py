"""kvr_select_static_scratch: selection for callers that may not allocate
device memory (plugin hosts that only pass inputs and outputs, runtimes that
reserve all device memory up front). Its scratch is a fixed array inside the
library; this checks, through the C ABI, that two calls in a row give exactly
what kvr_select gives with a caller-provided workspace, and that a shape too
large for the fixed array is refused. Collected last on purpose: it leaves the
shared scratch array filled, and every other test has run when it fails."""
import numpy as np
import pytest
import torch

import workloads as wl
import sparse_decode_attention_gb300 as kvr
from gpu_cases import encode_gpu

pytestmark = pytest.mark.gpu


def _case(seed, seq, cap):
    w = wl.Workload("case", B=len(seq), Hq=16, Hkv=4, d=128, N=max(seq), dtype="bf16", W=64,
                    rank=32, planted=8, seed=seed)
    K, V, q = wl.make_cache(w, device="cuda", cap=cap, seq_len=seq)
    sgn = wl.srht_signs(128, device="cuda")
    codes = encode_gpu(K, sgn, cap)
    return K, q, codes, torch.tensor(seq, dtype=torch.int32, device="cuda"), sgn


def _with_workspace(K, q, codes, seq, sgn, params):
    shape = kvr.Shape.of(K, q)
    ws = kvr.workspace(kvr.kvr_select_workspace_size(shape, params))
    idx = torch.empty((K.shape[0], K.shape[1], params.k), dtype=torch.int32, device="cuda")
    cnt = torch.empty((K.shape[0], K.shape[1]), dtype=torch.int32, device="cuda")
    kvr.kvr_select(q, K, codes, seq, sgn, params, idx, cnt, ws)
    return idx.cpu().numpy(), cnt.cpu().numpy()


def _static(K, q, codes, seq, sgn, params):
    idx = torch.full((K.shape[0], K.shape[1], params.k), 7, dtype=torch.int32, device="cuda")
    cnt = torch.full((K.shape[0], K.shape[1]), 7, dtype=torch.int32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    kvr.kvr_select_static_scratch(q, K, codes, seq, sgn, params, idx, cnt, err)
    assert kvr.kvr_read_error(err) == 0
    return idx.cpu().numpy(), cnt.cpu().numpy()


def test_static_scratch_matches_workspace_call_twice():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    # two different calls in a row: the second must not see the first's leftovers
    cases = [(_case(7, [30000, 12345], 30000), kvr.SelectParams(2048, 512, 64)),
             (_case(8, [9000], 9500), kvr.SelectParams(1000, 300, 64, wl.LINEAR_LUT))]
    for (K, q, codes, seq, sgn), params in cases:
        ref_idx, ref_cnt = _with_workspace(K, q, codes, seq, sgn, params)
        idx, cnt = _static(K, q, codes, seq, sgn, params)
        assert np.array_equal(cnt, ref_cnt)
        assert np.array_equal(idx, ref_idx)


def test_static_scratch_refuses_oversized_shapes():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    # 16 MiB cannot hold the coarse scores of 32 units x 1M tokens; nothing is read
    shape = kvr.Shape(4, 64, 8, 128, 1 << 20, "bf16")
    params = kvr.SelectParams(16384, 4096, 256)
    assert kvr.kvr_select_workspace_size(shape, params) > 16 << 20
    fake = torch.empty(16, dtype=torch.uint8, device="cuda")
    L = kvr.load()
    import ctypes
    st = L.kvr_select_static_scratch(ctypes.byref(shape.c()), ctypes.byref(params.c()),
                                     *([ctypes.c_void_p(fake.data_ptr())] * 7), None, None)
    assert st == 3  # KVR_ERR_WORKSPACE
