"""GPU run of the cache-dynamics diagnostics (QEvict, "Contributi Chiave":
Future Missed Mass, Global LIR, selection churn) against the oracle.

The full-attention window masses come from the tiered attention over an
all-bf16 state and the unmodified cache; they must match the oracle's numpy
full attention within the tiered masses' tolerance. FMM per step (from those
masses and the policy's tiers) within 1e-5 of the oracle's, LIR, leaves and
churn equal to the oracle's on the same tier history.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import workloads as wl
import sparse_decode_attention_gb300 as kvr
from oracle import diagnostics as odg
import bench_diagnostics as dg

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    kvr.load()
    oracle.build()


def test_diagnostics_over_a_routing_run():
    B, Hkv, G, d = 1, 2, 4, 64
    N0, steps = 64 * 40 + 20, 60
    cap = 64 * 42
    U, n_win = B * Hkv, -(-cap // 64)
    g = torch.Generator(device=DEV)
    g.manual_seed(11)
    K = (torch.randn((B, Hkv, cap, d), generator=g, device=DEV)).to(torch.bfloat16)
    V = (torch.randn((B, Hkv, cap, d), generator=g, device=DEV)).to(torch.bfloat16)
    K0, V0 = K.clone(), V.clone()                     # unmodified by promotions
    seq = torch.full((B,), N0, dtype=torch.int32, device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    closed = N0 // 64
    plan = np.zeros((U, n_win), np.int8)
    for u in range(U):
        plan[u, :closed] = wl.random_tier_plan(closed, seed=40 + u).numpy()
    st = kvr.TierState(U, n_win, d)
    kvr.kvr_tier_init(st, torch.from_numpy(plan).to(DEV), K, V, seq, Hkv * G, err)
    dense = dg.full_mass_state(U, n_win, d, K0, V0, seq, Hkv * G, err)
    shape = kvr.Shape(B, Hkv * G, Hkv, d, cap, torch.bfloat16)
    ws_a = kvr.workspace(kvr.kvr_tiered_attend_workspace_size(shape, n_win))
    ws_u = kvr.workspace(kvr.kvr_tier_update_workspace_size(shape, n_win))
    mass = torch.zeros((U, n_win), dtype=torch.float32, device=DEV)
    full = torch.zeros((U, n_win), dtype=torch.float32, device=DEV)
    out = torch.zeros((B, Hkv * G, d), dtype=torch.float32, device=DEV)
    stats = torch.zeros((U, 3), dtype=torch.int32, device=DEV)
    q_base = torch.randn((B, Hkv * G, d), generator=g, device=DEV)
    scale = 1 / math.sqrt(d)
    dyn = dg.CacheDynamics()
    K0n = K0.float().cpu().numpy()
    hist = [[] for _ in range(U)]
    closed_hist = []
    fmm_ref = []
    for step in range(steps):
        N = N0 + step
        seq.fill_(N)
        q = (q_base + 0.6 * torch.randn(q_base.shape, generator=g, device=DEV)).to(torch.bfloat16)
        kvr.kvr_sparse_attend_tiered(dense, q, K0, V0, seq, scale, out, full, ws_a, err)
        before = st.tier.clone()
        kvr.kvr_sparse_attend_tiered(st, q, K, V, seq, scale, out, mass, ws_a, err)
        kvr.kvr_tier_update(st, mass, seq, K, V, Hkv * G, stats, ws_u, err)
        dyn.record(full, before, st.tier, N)
        qn = q.float().cpu().numpy()
        fm = full.cpu().numpy()
        tb = before.cpu().numpy()
        nw = -(-N // 64)
        step_fmm = []
        for u in range(U):
            ref = odg.window_mass_full(qn[0, u * G:(u + 1) * G], K0n[0, u], N, scale)
            assert np.all(np.abs(fm[u, :nw] - ref) <= 1e-5 + 1e-4 * ref), (step, u)
            step_fmm.append(odg.future_missed_mass(ref, tb[u], N))
            hist[u].append(st.tier[u].cpu().numpy())
        closed_hist.append(N // 64)
        fmm_ref.append(step_fmm)
    s = dyn.summary()
    fmm_ref = np.array(fmm_ref)
    got = np.stack(dyn.fmm)
    assert np.abs(got - fmm_ref).max() <= 1e-5
    assert abs(s["fmm_mean"] - fmm_ref.mean()) <= 1e-5
    ref = odg.pooled([odg.reactivation_stats(hist[u], closed_hist) for u in range(U)])
    assert s["leaves"] == ref["leaves"] and s["reactivated"] == ref["reactivated"]
    assert s["lir"] == ref["lir"] and abs(s["churn_mean"] - ref["churn"]) < 1e-12
    assert s["leaves"] > 0 and s["fmm_mean"] > 0
    assert kvr.kvr_read_error(err) == 0
