"""Parity at the full sizes of the workloads, on sampled units.

The GPU runs every unit of the full workload through the same C-ABI calls the
benchmark times (encode of the appended key, kvr_select, kvr_sparse_attend;
for the tiered cache kvr_sparse_attend_tiered and kvr_tier_update); the oracle
recomputes a sample of the (batch, kv head) units one by one:
  * Llama-3-8B-shaped layer, 131072 tokens, C 8192, k 2048, W 128: codes,
    candidate counts and top-k index sets bit-exact, attention within 2e-3;
  * batched drift, B 8, 32768 prefill + 4096 appending steps with a drifting
    key law, C 4096, k 1024, W 128: the same checks at three sampled steps;
  * million-token context, C 16384, k 4096, W 256;
  * tiered window cache, B 4, 131072 tokens in 2048 windows per unit:
    attention within 2e-3, window masses, and the routing state bit-exact
    after each of several appending steps (decision parity: the oracle
    routes with the GPU's masses).
"""
import math

import numpy as np
import pytest
import torch

import oracle
import sparse_decode_attention_gb300 as kvr
import workloads as wl
from gpu_cases import planes_to_bytes

pytestmark = pytest.mark.gpu

DEV = "cuda"
ATOL = 2e-3


class Path:
    """Device buffers of one retrieval workload and its three calls."""

    def __init__(self, w, cap):
        self.w = w
        self.K, self.V, self.qb = wl.make_cache(w, device=DEV, cap=cap)
        self.sgn = wl.srht_signs(w.d, device=DEV)
        self.shape = kvr.Shape.of(self.K, self.qb)
        self.params = kvr.SelectParams(w.C, w.k, w.W, w.lut, V_prefetch=self.V)
        self.ws_s = kvr.workspace(kvr.kvr_select_workspace_size(self.shape, self.params))
        self.ws_a = kvr.workspace(kvr.kvr_attend_workspace_size(self.shape, w.k, w.W))
        self.codes = kvr.codes_buffer(self.shape, DEV)
        self.idx = torch.empty((w.B, w.Hkv, w.k), dtype=torch.int32, device=DEV)
        self.cnt = torch.empty((w.B, w.Hkv), dtype=torch.int32, device=DEV)
        self.out = torch.empty((w.B, w.Hq, w.d), dtype=torch.float32, device=DEV)
        self.err = torch.zeros(1, dtype=torch.int32, device=DEV)
        self.seq = torch.full((w.B,), w.N, dtype=torch.int32, device=DEV)

    def encode(self, row0, n):
        p0 = torch.full((self.w.B,), row0, dtype=torch.int32, device=DEV)
        kvr.kvr_encode_keys(self.K, p0, n, self.sgn, self.codes, self.err)

    def step(self, q, N):
        """One decode step of length N: the appended key (row N-1) is encoded,
        then selection and attention."""
        self.seq.fill_(N)
        self.encode(N - 1, 1)
        kvr.kvr_select(q, self.K, self.codes, self.seq, self.sgn, self.params, self.idx,
                       self.cnt, self.ws_s, self.err)
        kvr.kvr_sparse_attend(q, self.K, self.V, self.idx, self.cnt, self.seq, self.w.W,
                              1.0 / math.sqrt(self.w.d), self.out, self.ws_a, self.err)

    def step_chain(self, q, N):
        """The benchmark's decode chain: selection with early inputs (the
        previous kernel on the stream is the last attention, which writes none
        of its inputs but q), then attention. The caller synchronises after any
        kernel that wrote codes, K or lengths."""
        self.seq.fill_(N)
        torch.cuda.synchronize()
        early = kvr.SelectParams(self.w.C, self.w.k, self.w.W, self.w.lut,
                                 flags=kvr.SELECT_EARLY_INPUTS, V_prefetch=self.V)
        kvr.kvr_select(q, self.K, self.codes, self.seq, self.sgn, early, self.idx, self.cnt,
                       self.ws_s, self.err)
        kvr.kvr_sparse_attend(q, self.K, self.V, self.idx, self.cnt, self.seq, self.w.W,
                              1.0 / math.sqrt(self.w.d), self.out, self.ws_a, self.err)

    def check_units(self, q, N, units, check_codes=True):
        w = self.w
        idx = self.idx.cpu().numpy()
        cnt = self.cnt.cpu().numpy()
        out = self.out.cpu().numpy()
        qn = q.float().cpu().numpy()
        sgn = self.sgn.cpu().numpy()
        cap = self.K.shape[2]
        ub = kvr.kvr_codes_bytes(self.shape) // (w.B * w.Hkv)   # code bytes of one unit
        for b, h in units:
            Ku = oracle.f32(self.K[b, h, :N].cpu())
            Vu = oracle.f32(self.V[b, h, :N].cpu())
            codes = oracle.encode(Ku, sgn)
            if check_codes:
                u = b * w.Hkv + h
                raw = self.codes[u * ub:(u + 1) * ub].cpu().numpy()
                gcodes = planes_to_bytes(raw, 1, 1, cap, w.d)[0, 0]
                assert np.array_equal(gcodes[:N], codes), (b, h)
            qg = qn[b, h * w.G:(h + 1) * w.G]
            ref_idx, ref_cnt = oracle.select_unit(qg, Ku, codes, N, sgn, w.C, w.k, w.W, w.lut)
            assert cnt[b, h] == ref_cnt, (b, h)
            assert np.array_equal(idx[b, h, :ref_cnt], ref_idx[:ref_cnt]), (b, h)
            assert np.all(idx[b, h, ref_cnt:] == -1)
            ref = oracle.attend_unit(qg, Ku, Vu, N, ref_idx[:ref_cnt], ref_cnt, w.W,
                                     np.float32(1.0 / math.sqrt(w.d)))
            err = np.abs(out[b, h * w.G:(h + 1) * w.G] - ref).max()
            assert err <= ATOL, (b, h, err)


def test_llama_128k_layer_full_size():
    w = wl.LLAMA_128K
    p = Path(w, cap=w.N)
    p.encode(0, w.N)
    q = wl.step_query(w, p.qb, 0).contiguous()
    p.step(q, w.N)
    p.check_units(q, w.N, [(0, h) for h in range(w.Hkv)])
    # the benchmark's chain: after one synchronisation, select (early inputs)
    # -> attend -> select -> attend -> ..., no host sync in between
    early = kvr.SelectParams(w.C, w.k, w.W, w.lut, flags=kvr.SELECT_EARLY_INPUTS, V_prefetch=p.V)
    torch.cuda.synchronize()
    for t in range(1, 4):
        q = wl.step_query(w, p.qb, t).contiguous()
        kvr.kvr_select(q, p.K, p.codes, p.seq, p.sgn, early, p.idx, p.cnt, p.ws_s, p.err)
        kvr.kvr_sparse_attend(q, p.K, p.V, p.idx, p.cnt, p.seq, w.W, 1.0 / math.sqrt(w.d),
                              p.out, p.ws_a, p.err)
    p.check_units(q, w.N, [(0, h) for h in range(w.Hkv)], check_codes=False)
    assert kvr.kvr_read_error(p.err) == 0


def test_batched_drift_full_size_sampled_steps():
    w = wl.DRIFT
    T = w.steps
    p = Path(w, cap=w.N + T)
    k_new, qs = wl.drift_inputs(w, p.K, w.N, T)
    p.K[:, :, w.N:w.N + T] = k_new          # the appended keys, written ahead of their steps
    p.encode(0, w.N)
    checks = {0: [(0, 0), (3, 5)], T // 2 - 1: [(5, 2), (7, 7)], T - 1: [(1, 1), (6, 4)]}
    for t in range(T):
        N = w.N + t + 1
        p.step(qs[t], N)
        if t in checks:
            p.check_units(qs[t], N, checks[t], check_codes=(t == T - 1))
    assert kvr.kvr_read_error(p.err) == 0


def test_million_token_context_full_size():
    w = wl.MILLION
    p = Path(w, cap=w.N)
    p.encode(0, w.N)
    q = wl.step_query(w, p.qb, 0).contiguous()
    p.step(q, w.N)
    p.check_units(q, w.N, [(0, 0), (0, 5)])
    q = wl.step_query(w, p.qb, 1).contiguous()
    p.step_chain(q, w.N)
    p.check_units(q, w.N, [(0, 2), (0, 7)], check_codes=False)
    assert kvr.kvr_read_error(p.err) == 0


def test_tiered_window_cache_full_size():
    w = wl.TIERED
    steps = 6
    cap = w.N + steps + 10
    n_win = -(-cap // 64)
    U = w.B * w.Hkv
    K, V, qb = wl.make_cache(w, device=DEV, cap=cap)
    closed = w.N // 64
    plan = np.zeros((U, n_win), dtype=np.int8)
    for u in range(U):
        plan[u, :closed] = wl.random_tier_plan(closed, seed=w.seed + u).numpy()
    st = kvr.TierState(U, n_win, w.d)
    seq = torch.full((w.B,), w.N, dtype=torch.int32, device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    kvr.kvr_tier_init(st, torch.from_numpy(plan).to(DEV), K, V, seq, w.Hq, err)
    shape = kvr.Shape.of(K, qb)
    ws_a = kvr.workspace(kvr.kvr_tiered_attend_workspace_size(shape, n_win))
    ws_u = kvr.workspace(kvr.kvr_tier_update_workspace_size(shape, n_win))
    mass = torch.zeros((U, n_win), dtype=torch.float32, device=DEV)
    out = torch.empty((w.B, w.Hq, w.d), dtype=torch.float32, device=DEV)
    stats = torch.zeros((U, 3), dtype=torch.int32, device=DEV)
    sample = [0, 13, 31]
    units = {}
    for u in sample:
        b, h = divmod(u, w.Hkv)
        units[u] = oracle.TierUnit(plan[u], oracle.f32(K[b, h].cpu()), oracle.f32(V[b, h].cpu()),
                                   w.N, n_win)
        assert int(st.quota[u]) == units[u].quota and int(st.budget[u]) == units[u].budget
    scale = 1.0 / math.sqrt(w.d)
    moved = 0
    for t in range(steps):
        N = w.N + t + 1
        seq.fill_(N)
        q = wl.step_query(w, qb, t).contiguous()
        kvr.kvr_sparse_attend_tiered(st, q, K, V, seq, scale, out, mass, ws_a, err)
        kvr.kvr_tier_update(st, mass, seq, K, V, w.Hq, stats, ws_u, err)
        g_out, g_mass, g_stats = out.cpu().numpy(), mass.cpu().numpy(), stats.cpu().numpy()
        g_tier, g_score = st.tier.cpu().numpy(), st.score.cpu().numpy()
        g_hl = st.has_ledger.cpu().numpy()
        qn = q.float().cpu().numpy()
        for u, o in units.items():
            b, h = divmod(u, w.Hkv)
            ref, ref_mass = o.attend(qn[b, h * w.G:(h + 1) * w.G], N, scale)
            assert np.abs(g_out[b, h * w.G:(h + 1) * w.G] - ref).max() <= ATOL, (t, u)
            nw = -(-N // 64)
            assert np.all(np.abs(g_mass[u, :nw] - ref_mass) <= 1e-5 + 1e-4 * ref_mass), (t, u)
            s = o.update(g_mass[u], N)
            assert list(g_stats[u]) == list(s), (t, u)
            moved += int(s[0] + s[1])
            assert np.array_equal(g_tier[u], o.tier), (t, u)
            assert np.array_equal(g_score[u], o.score), (t, u)
            assert np.array_equal(g_hl[u], o.has_ledger), (t, u)
        for u, o in units.items():
            b, h = divmod(u, w.Hkv)
            led = st.ledger[u].cpu().numpy()
            sel = o.has_ledger.astype(bool)
            assert np.array_equal(led[sel], o.ledger[sel]), (t, u)
            assert np.array_equal(oracle.f32(K[b, h].cpu()), o.K[:cap]), (t, u)
            assert np.array_equal(oracle.f32(V[b, h].cpu()), o.V[:cap]), (t, u)
    assert moved > 0
    assert kvr.kvr_read_error(err) == 0


def test_llama_128k_reranked_full_size():
    """The 128K layer with the calibrated reranker in the benchmark's launch
    configuration (early inputs, V hint, records): records of sampled units,
    candidate estimates and top-k sets bit-exact, attention within 2e-3."""
    w = wl.LLAMA_128K
    p = Path(w, cap=w.N)
    p.encode(0, w.N)
    rec = kvr.rsq_buffer(p.K)
    kvr.kvr_encode_rsq(p.K, torch.zeros(w.B, dtype=torch.int32, device=DEV), w.N, p.sgn, rec,
                       p.err)
    params = kvr.SelectParams(w.C, w.k, w.W, w.lut, flags=kvr.SELECT_EARLY_INPUTS,
                              V_prefetch=p.V, rsq_records=rec)
    sgn = p.sgn.cpu().numpy()
    scale = np.float32(1.0 / math.sqrt(w.d))
    for t in range(2):
        q = wl.step_query(w, p.qb, t).contiguous()
        torch.cuda.synchronize()
        kvr.kvr_select(q, p.K, p.codes, p.seq, p.sgn, params, p.idx, p.cnt, p.ws_s, p.err)
        kvr.kvr_sparse_attend(q, p.K, p.V, p.idx, p.cnt, p.seq, w.W, float(scale), p.out,
                              p.ws_a, p.err)
        idx, cnt, out = p.idx.cpu().numpy(), p.cnt.cpu().numpy(), p.out.cpu().numpy()
        qn = q.float().cpu().numpy()
        for h in ((0, 3), (5, 7))[t]:
            Ku = oracle.f32(p.K[0, h].cpu())
            codes = oracle.encode(Ku, sgn)
            ref_rec = oracle.rsq_encode(Ku, sgn)
            assert np.array_equal(rec[0, h].cpu().numpy(), ref_rec), h
            qg = qn[0, h * w.G:(h + 1) * w.G]
            ref_idx, ref_cnt = oracle.select_unit_rsq(qg, codes, ref_rec, w.N, sgn, w.C, w.k,
                                                      w.W, w.lut)
            assert cnt[0, h] == ref_cnt and np.array_equal(idx[0, h], ref_idx), h
            ref = oracle.attend_unit(qg, Ku, oracle.f32(p.V[0, h].cpu()), w.N,
                                     ref_idx[:ref_cnt], ref_cnt, w.W, scale)
            assert np.abs(out[0, h * w.G:(h + 1) * w.G] - ref).max() <= ATOL, h
    assert kvr.kvr_read_error(p.err) == 0
