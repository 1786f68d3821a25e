"""kvr_select_static_scratch: selection for callers that may not allocate
device memory (plugin hosts that only pass inputs and outputs, runtimes that
reserve all device memory up front). Its scratch is a fixed array inside the
library; this checks, through the C ABI, that two calls in a row give exactly
what kvr_select gives with a caller-provided workspace (plain, with
magnitude-aware votes, whose vote lists a second kernel writes into the
scratch, and with reranker records), that the index sets equal the oracle's,
that the calls allocate no device memory, and that a shape too large for the
fixed array is refused. Collected last on purpose: it leaves the shared
scratch array filled, and every other test has run when it fails."""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
import sparse_decode_attention_gb300 as kvr
from gpu_cases import codes_bytes_gpu, encode_gpu

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


def test_static_scratch_equals_the_oracle():
    """The index sets of one call equal the oracle's selection unit by unit."""
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    oracle.build()
    seq = [20000, 7000]
    K, q, codes, seqd, sgn = _case(9, seq, 20000)
    params = kvr.SelectParams(1024, 256, 64)
    idx, cnt = _static(K, q, codes, seqd, sgn, params)
    ref_codes = codes_bytes_gpu(codes, K)
    Kc, qc, sg = K.cpu(), q.cpu(), sgn.cpu().numpy()
    G = q.shape[1] // K.shape[1]
    for b in range(K.shape[0]):
        for h in range(K.shape[1]):
            N = seq[b]
            ri, rc = oracle.select_unit(qc[b, h * G:(h + 1) * G], Kc[b, h, :N],
                                        ref_codes[b, h, :N], N, sg, params.C, params.k, params.W,
                                        params.lut)
            assert cnt[b, h] == rc, (b, h)
            assert np.array_equal(idx[b, h], ri), (b, h)


@pytest.mark.parametrize("mode", ["magnitude", "records"])
def test_static_scratch_optional_modes_twice(mode):
    """Magnitude-aware votes (vote lists written into the scratch by their own
    kernel) and reranker records, bit-exact with the workspace call, twice."""
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    for seed, seq in ((11, [15000, 6000]), (12, [8000])):
        K, q, codes, seqd, sgn = _case(seed, seq, max(seq))
        rec, flags = None, 0
        if mode == "records":
            rec = kvr.rsq_buffer(K)
            kvr.kvr_encode_rsq(K, torch.zeros(K.shape[0], dtype=torch.int32, device="cuda"),
                               max(seq), sgn, rec)
        else:
            flags = kvr.SELECT_MAGNITUDE_VOTES
        params = kvr.SelectParams(1024, 300, 64, wl.DEFAULT_LUT, flags=flags, rsq_records=rec)
        ref_idx, ref_cnt = _with_workspace(K, q, codes, seqd, sgn, params)
        idx, cnt = _static(K, q, codes, seqd, sgn, params)
        assert np.array_equal(cnt, ref_cnt) and np.array_equal(idx, ref_idx)


def test_static_scratch_allocates_nothing():
    """After the set-up call, further calls leave the device's free memory and
    the caching allocator's counters where they were."""
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    K, q, codes, seqd, sgn = _case(13, [12000], 12000)
    params = kvr.SelectParams(1024, 256, 64)
    idx = torch.empty((1, K.shape[1], params.k), dtype=torch.int32, device="cuda")
    cnt = torch.empty((1, K.shape[1]), dtype=torch.int32, device="cuda")
    kvr.kvr_select_static_scratch(q, K, codes, seqd, sgn, params, idx, cnt)  # set-up
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    alloc0, res0 = torch.cuda.memory_allocated(), torch.cuda.memory_reserved()
    for _ in range(3):
        kvr.kvr_select_static_scratch(q, K, codes, seqd, sgn, params, idx, cnt)
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0
    assert torch.cuda.memory_allocated() == alloc0 and torch.cuda.memory_reserved() == res0


def test_static_scratch_checks_the_records_size():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    K, q, codes, seqd, sgn = _case(14, [3000], 3000)
    small = torch.zeros(16, dtype=torch.uint8, device="cuda")
    params = kvr.SelectParams(256, 64, 64, rsq_records=small)
    idx = torch.empty((1, K.shape[1], 64), dtype=torch.int32, device="cuda")
    cnt = torch.empty((1, K.shape[1]), dtype=torch.int32, device="cuda")
    with pytest.raises(ValueError):
        kvr.kvr_select_static_scratch(q, K, codes, seqd, sgn, params, idx, cnt)
