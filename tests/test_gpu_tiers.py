"""Parity of the tiered window cache on the GPU against the oracle, through
the C ABI (QEvict, "Metodologia: QEvict" and "Meccanismi Chiave").

Bit-exact: ledger bytes (INT2 codes, fp16 scale / zero), tiers, cumulative
scores, has-ledger flags, promoted bf16 K / V rows, quota and budget; the
routing is checked at the decision level by feeding the GPU's window masses
into the oracle's routing step. Attention outputs within max-abs 2e-3 of the
oracle's fp64 softmax; window masses within 1e-5 + 1e-4 relative.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import sparse_decode_attention_gb300 as kvr
import workloads as wl

pytestmark = pytest.mark.gpu

DEV = "cuda"
ATOL = 2e-3


def bf16_cache(B, Hkv, cap, d, seed, std=1.0, outliers=True):
    g = torch.Generator(device=DEV)
    g.manual_seed(seed)
    K = torch.randn((B, Hkv, cap, d), generator=g, device=DEV) * std
    V = torch.randn((B, Hkv, cap, d), generator=g, device=DEV) * std
    if outliers:
        K[..., 3] *= 8
        V[..., 17] *= 8
    return K.to(torch.bfloat16).contiguous(), V.to(torch.bfloat16).contiguous()


def tiers_for(U, n_win, closed, seed, frac=(0.25, 0.5, 0.25)):
    t = np.zeros((U, n_win), dtype=np.int8)
    for u in range(U):
        t[u, :closed] = wl.random_tier_plan(closed, frac, seed=seed + u).numpy()
    return t


class Run:
    """GPU tier state plus one oracle TierUnit per unit on the same data."""

    def __init__(self, B, Hkv, G, d, cap, N, seed, frac=(0.25, 0.5, 0.25), init=None):
        self.B, self.Hkv, self.G, self.d, self.cap = B, Hkv, G, d, cap
        self.U = B * Hkv
        self.n_win = -(-cap // 64)
        self.K, self.V = bf16_cache(B, Hkv, cap, d, seed)
        self.N = torch.full((B,), N, dtype=torch.int32, device=DEV)
        closed = N // 64
        self.init = tiers_for(self.U, self.n_win, closed, seed) if init is None else init
        self.st = kvr.TierState(self.U, self.n_win, d)
        self.err = torch.zeros(1, dtype=torch.int32, device=DEV)
        kvr.kvr_tier_init(self.st, torch.from_numpy(self.init).to(DEV), self.K, self.V, self.N,
                          Hkv * G, self.err)
        Kc, Vc = self.K.float().cpu().numpy(), self.V.float().cpu().numpy()
        self.units = [oracle.TierUnit(self.init[u], Kc[u // Hkv, u % Hkv],
                                      Vc[u // Hkv, u % Hkv], N, self.n_win)
                      for u in range(self.U)]
        shape = kvr.Shape(B, Hkv * G, Hkv, d, cap, torch.bfloat16)
        self.ws_a = kvr.workspace(kvr.kvr_tiered_attend_workspace_size(shape, self.n_win))
        self.ws_u = kvr.workspace(kvr.kvr_tier_update_workspace_size(shape, self.n_win))
        self.mass = torch.zeros((self.U, self.n_win), dtype=torch.float32, device=DEV)
        self.out = torch.zeros((B, Hkv * G, d), dtype=torch.float32, device=DEV)
        self.stats = torch.zeros((self.U, 3), dtype=torch.int32, device=DEV)

    def attend(self, q, scale):
        self.mass.fill_(-1.0)
        kvr.kvr_sparse_attend_tiered(self.st, q, self.K, self.V, self.N, scale, self.out,
                                     self.mass, self.ws_a, self.err)
        return self.out.cpu().numpy(), self.mass.cpu().numpy()

    def update(self):
        kvr.kvr_tier_update(self.st, self.mass, self.N, self.K, self.V, self.Hkv * self.G,
                            self.stats, self.ws_u, self.err)

    def compare_state(self, what=""):
        tier = self.st.tier.cpu().numpy()
        score = self.st.score.cpu().numpy()
        hl = self.st.has_ledger.cpu().numpy()
        led = self.st.ledger.cpu().numpy()
        Kc = self.K.float().cpu().numpy()
        Vc = self.V.float().cpu().numpy()
        for u, o in enumerate(self.units):
            b, h = divmod(u, self.Hkv)
            assert np.array_equal(tier[u], o.tier), (what, u, np.flatnonzero(tier[u] != o.tier))
            assert np.array_equal(score[u], o.score), (what, u)
            assert np.array_equal(hl[u], o.has_ledger), (what, u)
            sel = o.has_ledger.astype(bool)
            assert np.array_equal(led[u][sel], o.ledger[sel]), (what, u)
            assert np.array_equal(Kc[b, h], o.K[:self.cap]), (what, u)
            assert np.array_equal(Vc[b, h], o.V[:self.cap]), (what, u)


def oracle_attend(run, q, N, scale):
    qn = q.float().cpu().numpy()
    out = np.zeros((run.B, run.Hkv * run.G, run.d))
    masses = []
    for u, o in enumerate(run.units):
        b, h = divmod(u, run.Hkv)
        ob, m = o.attend(qn[b, h * run.G:(h + 1) * run.G], N, scale)
        out[b, h * run.G:(h + 1) * run.G] = ob
        masses.append(m)
    return out, masses


def check_mass(gpu_mass, masses, N, n_win):
    nw = -(-N // 64)
    for u, m in enumerate(masses):
        g = gpu_mass[u]
        assert np.all(g[nw:] == 0)
        err = np.abs(g[:nw] - m)
        assert np.all(err <= 1e-5 + 1e-4 * m), (u, err.max())


# --------------------------------------------------------------------------
# set-up and the INT2 ledger
# --------------------------------------------------------------------------

@pytest.mark.parametrize("d,G", [(128, 4), (64, 2)])
def test_tier_init_ledgers_quota_and_budget(d, G):
    run = Run(2, 2, G, d, cap=64 * 40 + 16, N=64 * 37 + 5, seed=11)
    run.compare_state("init")
    for u, o in enumerate(run.units):
        assert int(run.st.quota[u]) == o.quota
        assert int(run.st.budget[u]) == o.budget
    assert kvr.kvr_read_error(run.err) == 0


def test_int2_groups_cover_the_directed_fp16_roundings():
    """2^20 groups whose minimum is a sample value and whose maximum lies a
    random distance above it: the zero is the fp16 rounded down from the
    sample, the scale an fp16 rounded up, both bit-exact against the oracle's
    conversions from the IEEE definition."""
    d, n_groups = 128, 1 << 20
    n_win = n_groups // (64 * 4 * 2)
    rng = np.random.default_rng(5)
    e = rng.integers(-20, 11, n_groups)          # every group stays inside the fp16 range
    v = (rng.normal(0, 1, n_groups) * np.exp2(e)).astype(np.float32)
    span = (np.abs(rng.normal(0, 1, n_groups)) * np.exp2(e + rng.integers(-4, 3, n_groups)))
    x = np.repeat(v[:, None], 32, axis=1).astype(np.float64)
    frac = rng.uniform(0, 1, (n_groups, 32))
    frac[:, 0], frac[:, 1] = 0.0, 1.0
    x = x + frac * span[:, None]
    xb = torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16)
    K = xb[: n_groups // 2].reshape(1, 1, n_win * 64, d)
    V = xb[n_groups // 2:].reshape(1, 1, n_win * 64, d)
    K, V = K.contiguous().to(DEV), V.contiguous().to(DEV)
    st = kvr.TierState(1, n_win, d)
    init = torch.ones((1, n_win), dtype=torch.int8, device=DEV)
    N = torch.tensor([n_win * 64], dtype=torch.int32, device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    kvr.kvr_tier_init(st, init, K, V, N, 1, err)
    led = st.ledger.cpu().numpy()[0]
    Kc, Vc = K.float().cpu().numpy()[0, 0], V.float().cpu().numpy()[0, 0]
    for w in range(n_win):
        ref = oracle.ledger_write_window(Kc[64 * w:64 * w + 64], Vc[64 * w:64 * w + 64])
        assert np.array_equal(led[w], ref), w
    assert kvr.kvr_read_error(err) == 0


def test_int2_special_groups():
    """Constant groups, zeros of both signs, a one-element spread, values on a
    scale / zero grid."""
    d, n_win = 128, 2
    x = np.random.default_rng(9).normal(0, 1, (2, n_win * 64, d)).astype(np.float32)
    x[0, 0, :32] = 1.5
    x[0, 1, :32] = 0.0
    x[0, 2, :32] = -0.0
    x[0, 3, :32] = 0.0
    x[0, 3, 5] = -0.0
    x[0, 4, :32] = 0.1
    x[0, 5, :32] = 2.0
    x[0, 5, 7] = 2.0078125
    x[0, 6, :32] = -1.0 + 0.5 * (np.arange(32) % 4)
    x[0, 7, 32:64] = 1e-6 * np.arange(32)
    xb = torch.from_numpy(x).to(torch.bfloat16)
    K = xb[0].reshape(1, 1, n_win * 64, d).contiguous().to(DEV)
    V = xb[1].reshape(1, 1, n_win * 64, d).contiguous().to(DEV)
    st = kvr.TierState(1, n_win, d)
    init = torch.ones((1, n_win), dtype=torch.int8, device=DEV)
    N = torch.tensor([n_win * 64], dtype=torch.int32, device=DEV)
    kvr.kvr_tier_init(st, init, K, V, N, 1)
    led = st.ledger.cpu().numpy()[0]
    Kc, Vc = K.float().cpu().numpy()[0, 0], V.float().cpu().numpy()[0, 0]
    for w in range(n_win):
        ref = oracle.ledger_write_window(Kc[64 * w:64 * w + 64], Vc[64 * w:64 * w + 64])
        assert np.array_equal(led[w], ref), w


def test_range_beyond_fp16_sets_the_error_bit():
    d = 64
    K, V = bf16_cache(1, 1, 128, d, seed=3)
    K[0, 0, 10, 4] = 1e6
    st = kvr.TierState(1, 2, d)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    kvr.kvr_tier_init(st, torch.ones((1, 2), dtype=torch.int8, device=DEV), K, V,
                      torch.tensor([128], dtype=torch.int32, device=DEV), 1, err)
    assert kvr.kvr_read_error(err) & kvr.DEVERR["range"]


# --------------------------------------------------------------------------
# tiered attention and window mass
# --------------------------------------------------------------------------

@pytest.mark.parametrize("d,G,N", [(128, 4, 64 * 50 + 37), (128, 4, 64 * 50), (64, 2, 64 * 31 + 1),
                                   (128, 1, 64 * 20 + 63), (128, 8, 64 * 12 + 9), (64, 8, 40)])
def test_tiered_attention_and_window_mass(d, G, N):
    cap = 64 * 52
    run = Run(2, 2, G, d, cap, N, seed=100 + G + d)
    g = torch.Generator(device=DEV)
    g.manual_seed(5)
    q = (torch.randn((2, 2 * G, d), generator=g, device=DEV)).to(torch.bfloat16)
    scale = 1 / math.sqrt(d)
    out, mass = run.attend(q, scale)
    ref, masses = oracle_attend(run, q, N, scale)
    assert np.abs(out - ref).max() <= ATOL
    check_mass(mass, masses, N, run.n_win)
    assert kvr.kvr_read_error(run.err) == 0


def test_tiered_attention_all_bf16_is_dense_attention():
    d, G, N, cap = 128, 4, 64 * 30 + 11, 64 * 31
    init = np.zeros((4, 31), dtype=np.int8)
    run = Run(2, 2, G, d, cap, N, seed=21, init=init)
    q = torch.randn((2, 8, d), device=DEV).to(torch.bfloat16)
    out, _ = run.attend(q, 0.1)
    Kc, Vc, qc = run.K.float().cpu().numpy(), run.V.float().cpu().numpy(), q.float().cpu().numpy()
    for u in range(4):
        b, h = divmod(u, 2)
        ref = oracle.attend_unit(qc[b, h * G:(h + 1) * G], Kc[b, h, :N], Vc[b, h, :N], N,
                                 np.zeros(0, np.int32), 0, N, np.float32(0.1))
        assert np.abs(out[b, h * G:(h + 1) * G] - ref).max() <= ATOL


def test_tiered_attention_edge_lengths():
    """N = 0 (nothing attended), every closed window evicted (open window
    only), a single token."""
    d, G, cap = 128, 4, 64 * 8
    for N, fill in [(0, 2), (64 * 5 + 3, 2), (1, 0)]:
        init = np.full((2, 8), fill, dtype=np.int8)
        run = Run(1, 2, G, d, cap, N, seed=7, init=init)
        q = torch.randn((1, 8, d), device=DEV).to(torch.bfloat16)
        out, mass = run.attend(q, 0.125)
        ref, masses = oracle_attend(run, q, N, 0.125)
        assert np.abs(out - ref).max() <= ATOL
        check_mass(mass, masses, N, run.n_win)


def test_bad_tier_value_is_flagged_and_skipped():
    d, G, N, cap = 128, 4, 64 * 6, 64 * 7
    run = Run(1, 1, G, d, cap, N, seed=8, init=np.zeros((1, 7), dtype=np.int8))
    run.st.tier[0, 2] = 5
    run.units[0].tier[2] = oracle.EVICTED
    q = torch.randn((1, 4, d), device=DEV).to(torch.bfloat16)
    out, mass = run.attend(q, 0.125)
    assert kvr.kvr_read_error(run.err) & kvr.DEVERR["tier"]
    ref, masses = oracle_attend(run, q, N, 0.125)
    assert np.abs(out - ref).max() <= ATOL
    assert mass[0, 2] == 0


# --------------------------------------------------------------------------
# routing: decision parity over appending decode steps
# --------------------------------------------------------------------------

@pytest.mark.parametrize("d,G", [(128, 4), (64, 2)])
def test_routing_steps_match_the_oracle_bit_for_bit(d, G):
    B, Hkv = 2, 2
    N0, steps = 64 * 30 + 40, 90                 # crosses two window boundaries
    cap = 64 * 34
    run = Run(B, Hkv, G, d, cap, N0, seed=31 + d)
    run.compare_state("init")
    gq = torch.Generator(device=DEV)
    gq.manual_seed(77)
    q_base = torch.randn((B, Hkv * G, d), generator=gq, device=DEV)
    scale = 1 / math.sqrt(d)
    totals = np.zeros(3, dtype=np.int64)
    for step in range(steps):
        N = N0 + step
        run.N.fill_(N)
        q = (q_base + 0.5 * torch.randn((B, Hkv * G, d), generator=gq, device=DEV)).to(
            torch.bfloat16)
        out, mass = run.attend(q, scale)
        if step % 15 == 0:
            ref, masses = oracle_attend(run, q, N, scale)
            assert np.abs(out - ref).max() <= ATOL, step
            check_mass(mass, masses, N, run.n_win)
        run.update()
        stats = run.stats.cpu().numpy()
        for u, o in enumerate(run.units):
            s = o.update(mass[u], N)
            assert list(stats[u]) == list(s), (step, u)
            totals += s
        run.compare_state("step %d" % step)
    assert totals[0] > 0 and totals[1] > 0 and totals[2] >= 2 * run.U
    assert kvr.kvr_read_error(run.err) == 0


def test_routing_with_a_frozen_evicted_score_and_no_live_windows():
    """A unit whose closed windows are all evicted routes nothing; scores of
    evicted windows stay frozen whatever mass is passed in."""
    d, G, N, cap = 64, 1, 64 * 4 + 3, 64 * 5
    run = Run(1, 1, G, d, cap, N, seed=2, init=np.full((1, 5), 2, dtype=np.int8))
    run.mass.fill_(0.25)
    run.update()
    assert run.stats.cpu().numpy().tolist() == [[0, 0, 0]]
    sc = run.st.score.cpu().numpy()[0]
    assert np.all(sc[:4] == 0) and sc[4] == int(round(0.25 * 2 ** 32))
