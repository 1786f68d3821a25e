"""Cache-dynamics diagnostics of the tiered window cache, plain numpy.

TEST INFRASTRUCTURE, like the rest of ``oracle/``: only the tests and the
benchmark's evaluation passes use it; the CUDA library shares nothing with it.

Source: QEvict, "Contributi Chiave" (systematic analysis of cache dynamics):
  * Future Missed Mass (FMM): the share of future attention that falls on
    states a policy has already discarded;
  * Global LIR (latent importance reactivation): how often windows that were
    inactive re-enter the active set;
  * selection churn: how much the active set changes between consecutive
    routing steps.

Readings (the pages define the quantities in words only):
  * attention mass of a window under full attention: the softmax
    probabilities over all N tokens of its tokens, summed over the tokens and
    the group's heads (the same mass the tiered attention reports);
  * FMM at a step: the full-attention mass of the windows that are evicted
    when the step's attention runs, over the total mass (= G);
  * active set A_t: the closed windows in the bf16 tier after routing step t;
    a window leaves at t if it is in A_{t-1} and not in A_t; a leave is
    reactivated if the window is in A_t' for some later t'; LIR = reactivated
    leaves / leaves, pooled over units;
  * churn at t: |A_t symmetric-difference A_{t-1}| / |A_{t-1}| over the
    windows closed at both steps (0 when A_{t-1} is empty).
"""
import numpy as np

WINDOW = 64
BF16, INT2, EVICTED = 0, 1, 2


def window_mass_full(q_group, K_unit, N, scale):
    """Full-attention window masses [ceil(N/64)] of one unit, fp64: softmax of
    scale * q_h . k_t over t < N per head, summed per window and over heads."""
    q = np.asarray(q_group, dtype=np.float64)
    K = np.asarray(K_unit, dtype=np.float64)[:N]
    s = (q @ K.T) * float(np.float32(scale))
    s -= s.max(axis=1, keepdims=True)
    p = np.exp(s)
    p /= p.sum(axis=1, keepdims=True)
    nw = -(-N // WINDOW)
    pad = np.zeros((p.shape[0], nw * WINDOW))
    pad[:, :N] = p
    return pad.reshape(p.shape[0], nw, WINDOW).sum(axis=(0, 2))


def future_missed_mass(full_mass, tier, N):
    """Share of the full-attention mass on windows evicted at this step."""
    m = np.asarray(full_mass, dtype=np.float64)
    closed = N // WINDOW
    t = np.asarray(tier)[:closed]
    total = m.sum()
    if total <= 0:
        return 0.0
    return float(m[:closed][t == EVICTED].sum() / total)


def reactivation_stats(tier_history, closed_history):
    """Leaves, reactivated leaves, LIR and mean churn of one unit's active
    sets. tier_history[t] = tiers after routing step t; closed_history[t] =
    number of closed windows at that step."""
    active = [set(np.nonzero(np.asarray(tr)[:c] == BF16)[0].tolist())
              for tr, c in zip(tier_history, closed_history)]
    leaves, reactivated, churn = 0, 0, []
    for t in range(1, len(active)):
        both = min(closed_history[t - 1], closed_history[t])
        prev = {w for w in active[t - 1] if w < both}
        cur = {w for w in active[t] if w < both}
        churn.append(len(prev ^ cur) / len(prev) if prev else 0.0)
        for w in prev - cur:
            leaves += 1
            if any(w in active[u] for u in range(t + 1, len(active))):
                reactivated += 1
    return dict(leaves=leaves, reactivated=reactivated,
                lir=(reactivated / leaves) if leaves else 0.0,
                churn=float(np.mean(churn)) if churn else 0.0)


def pooled(stats):
    """Global LIR and mean churn over several units' reactivation_stats."""
    leaves = sum(s["leaves"] for s in stats)
    re = sum(s["reactivated"] for s in stats)
    return dict(leaves=leaves, reactivated=re, lir=(re / leaves) if leaves else 0.0,
                churn=float(np.mean([s["churn"] for s in stats])) if stats else 0.0)
