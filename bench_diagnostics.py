"""Cache-dynamics diagnostics of the tiered window cache.

Source: QEvict, "Contributi Chiave": Future Missed Mass (the share of future
attention that falls on states a policy has already discarded), Global LIR
(how often windows that were inactive re-enter the active set) and selection
churn (how much the active set changes between routing steps).

This is evaluation tooling beside the benchmark, not part of the library or
its hot path (it lives next to bench.py for that reason): the
full-attention window masses come from the library's tiered attention run on
a state that keeps every window in bf16 (``full_mass_state`` +
``kvr_sparse_attend_tiered`` over the unmodified K / V), and the per-step
bookkeeping (which windows are evicted or active) runs on the host over
copies of the device tier arrays.

Definitions used:
  * FMM at a step = full-attention mass of the closed windows evicted when
    the step's attention runs / the total mass;
  * active set A_t = closed windows in bf16 after routing step t; a leave is a
    window in A_{t-1} but not in A_t; it is reactivated if the window is in
    some later A_t'; LIR = reactivated leaves / leaves over all units;
  * churn at t = |A_t xor A_{t-1}| / |A_{t-1}| over windows closed at both
    steps (0 for an empty A_{t-1}), averaged over steps and units.
"""
import numpy as np
import torch

from sparse_decode_attention_gb300 import TIER_BF16, TIER_EVICTED, WINDOW, TierState, kvr_tier_init

__all__ = ["full_mass_state", "CacheDynamics"]


def full_mass_state(U, n_win, d, K, V, seq_len, q_heads, err=None, device=None):
    """A tier state with every window in bf16 and no ledgers: the tiered
    attention over it is full attention, and its window masses are the
    full-attention masses."""
    st = TierState(U, n_win, d, device or K.device)
    plan = torch.zeros((U, n_win), dtype=torch.int8, device=device or K.device)
    kvr_tier_init(st, plan, K, V, seq_len, q_heads, err)
    return st


class CacheDynamics:
    """Accumulates FMM, LIR and churn over routing steps."""

    def __init__(self):
        self.fmm = []
        self.active = []     # bool [U, n_win] after each routing step
        self.closed = []     # closed windows at each step

    def record(self, full_mass, tiers_before, tiers_after, N):
        """One step: full-attention masses and the policy's tiers when the
        step's attention ran (tiers_before) and after its routing."""
        m = full_mass.detach().float().cpu().numpy().astype(np.float64)
        tb = tiers_before.detach().cpu().numpy()
        ta = tiers_after.detach().cpu().numpy()
        c = int(N) // WINDOW
        tot = m.sum(axis=1)
        ev = np.where(tb[:, :c] == TIER_EVICTED, m[:, :c], 0.0).sum(axis=1)
        self.fmm.append(np.where(tot > 0, ev / np.where(tot > 0, tot, 1.0), 0.0))
        act = np.zeros_like(ta, dtype=bool)
        act[:, :c] = ta[:, :c] == TIER_BF16
        self.active.append(act)
        self.closed.append(c)

    def summary(self):
        fmm = np.stack(self.fmm) if self.fmm else np.zeros((0, 0))
        A = np.stack(self.active) if self.active else np.zeros((0, 0, 0), bool)
        T = A.shape[0]
        leaves = reac = 0
        churn = []
        if T >= 2:
            # later[t] = active at some step after t
            later = np.zeros_like(A)
            for t in range(T - 2, -1, -1):
                later[t] = later[t + 1] | A[t + 1]
            for t in range(1, T):
                both = min(self.closed[t - 1], self.closed[t])
                prev, cur = A[t - 1][:, :both], A[t][:, :both]
                left = prev & ~cur
                leaves += int(left.sum())
                reac += int((left & later[t][:, :both]).sum())
                n_prev = prev.sum(axis=1)
                diff = (prev ^ cur).sum(axis=1)
                churn.append(np.where(n_prev > 0, diff / np.maximum(n_prev, 1), 0.0))
        return {
            "fmm_mean": float(fmm.mean()) if fmm.size else 0.0,
            "fmm_max": float(fmm.max()) if fmm.size else 0.0,
            "leaves": leaves, "reactivated": reac,
            "lir": reac / leaves if leaves else 0.0,
            "churn_mean": float(np.mean(churn)) if churn else 0.0,
            "steps": T,
        }
