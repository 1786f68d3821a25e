"""The bounded device-side wait of the tiered attention runs out and the GPU
stays usable.

The test hook (include/kvr_testing.h) withholds each attention CTA's last
bulk copy and limits every wait for a copy to 2 ms: nothing ever completes
that wait, so it gives up, sets KVR_DEVERR_TIMEOUT, and the kernel returns
with every copy it issued landed (none is abandoned in flight). No fault,
trap or hang is involved. A normal call right after it on the same context
must then match the oracle.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import sparse_decode_attention_gb300 as kvr
from test_gpu_tiers import ATOL, Run, check_mass, oracle_attend

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    kvr.load()
    oracle.build()


@pytest.mark.parametrize("d,G", [(128, 4), (64, 2)])
def test_withheld_copy_times_out_then_the_next_call_is_exact(d, G):
    B, Hkv, N = 2, 2, 3000
    run = Run(B, Hkv, G, d, cap=3100, N=N, seed=11 + d)
    g = torch.Generator(device="cuda").manual_seed(5)
    q = torch.randn((B, Hkv * G, d), generator=g, device="cuda").to(torch.bfloat16)
    scale = 1.0 / math.sqrt(d)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    kvr._testing_tiered_withheld_copy(run.st, q, run.K, run.V, run.N, scale, run.out, run.mass,
                                      run.ws_a, 2_000_000, err)
    torch.cuda.synchronize()          # the kernel returned: no hang, no fault
    bits = kvr.kvr_read_error(err)
    assert bits & kvr.DEVERR["timeout"]
    # the same context computes correctly right after
    out, mass = run.attend(q, scale)
    assert kvr.kvr_read_error(run.err) == 0
    ref, masses = oracle_attend(run, q, N, np.float32(scale))
    assert np.abs(out - ref).max() <= ATOL
    check_mass(mass, masses, N, run.n_win)


def test_hook_rejects_bad_limits():
    run = Run(1, 1, 1, 64, cap=200, N=150, seed=3)
    q = torch.zeros((1, 1, 64), dtype=torch.bfloat16, device="cuda")
    for bad in (0, -5, 10**11):
        with pytest.raises(kvr.KvrError):
            kvr._testing_tiered_withheld_copy(run.st, q, run.K, run.V, run.N, 0.125, run.out,
                                              run.mass, run.ws_a, bad)
