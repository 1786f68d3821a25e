"""Pins of the cache-dynamics diagnostics (QEvict, "Contributi Chiave": Future
Missed Mass, Global LIR, selection churn).

Checked against: the pinned tiered-attention oracle (all windows bf16 gives
the full-attention masses), closed forms (identical keys, one dominant key),
and hand-counted tier histories.
"""
import numpy as np
import pytest

import oracle
from oracle import diagnostics as dg

RNG = np.random.default_rng(5)


def test_full_masses_equal_the_tiered_oracle_with_every_window_bf16():
    N, d, G = 64 * 9 + 17, 64, 4
    K = RNG.normal(0, 1, (N, d)).astype(np.float32)
    V = RNG.normal(0, 1, (N, d)).astype(np.float32)
    q = RNG.normal(0, 1, (G, d)).astype(np.float32)
    n_win = -(-N // 64)
    unit = oracle.TierUnit(np.zeros(n_win, np.int8), K, V, N, n_win)
    _, mass = unit.attend(q, N, 0.125)
    full = dg.window_mass_full(q, K, N, 0.125)
    assert np.abs(full - mass).max() < 1e-12
    assert abs(full.sum() - G) < 1e-12


def test_full_masses_closed_forms():
    N, d, G = 200, 16, 2
    K = np.ones((N, d), np.float32)
    q = RNG.normal(0, 1, (G, d)).astype(np.float32)
    m = dg.window_mass_full(q, K, N, 0.5)           # identical keys: mass by token count
    assert np.allclose(m, G * np.array([64, 64, 64, 8]) / N, atol=1e-12)
    K = np.zeros((N, d), np.float32)
    K[130] = 50.0
    q = np.ones((G, d), np.float32)
    m = dg.window_mass_full(q, K, N, 1.0)           # one dominant key in window 2
    assert m[2] > G * (1 - 1e-12) and m.argmax() == 2


def test_future_missed_mass_counts_evicted_closed_windows():
    mass = np.array([1.0, 2.0, 3.0, 4.0, 0.5])      # four closed windows + the open one
    tier = np.array([dg.EVICTED, dg.BF16, dg.INT2, dg.EVICTED, dg.EVICTED], np.int8)
    N = 4 * 64 + 10
    assert abs(dg.future_missed_mass(mass, tier, N) - 5.0 / 10.5) < 1e-15
    assert dg.future_missed_mass(mass, np.zeros(5, np.int8), N) == 0.0


def test_reactivation_and_churn_hand_counted():
    B, I, E = dg.BF16, dg.INT2, dg.EVICTED
    hist = [np.array([B, B, I]), np.array([I, B, I]), np.array([B, B, I]), np.array([I, I, B])]
    s = dg.reactivation_stats(hist, [3, 3, 3, 3])
    # leaves: window 0 at step 1 (back at step 2), windows 0 and 1 at step 3 (never back)
    assert s["leaves"] == 3 and s["reactivated"] == 1
    assert abs(s["lir"] - 1 / 3) < 1e-15
    # churn: {0,1}->{1}: 1/2; {1}->{0,1}: 1/1; {0,1}->{2}: 3/2
    assert abs(s["churn"] - (0.5 + 1.0 + 1.5) / 3) < 1e-15
    # a window that closes between two steps is not a change of the active set
    s = dg.reactivation_stats([np.array([B, B, E]), np.array([B, B, B])], [2, 3])
    assert s["leaves"] == 0 and s["churn"] == 0.0
    p = dg.pooled([dict(leaves=3, reactivated=1, lir=1 / 3, churn=1.0),
                   dict(leaves=1, reactivated=1, lir=1.0, churn=0.0)])
    assert p["leaves"] == 4 and p["reactivated"] == 2 and p["lir"] == 0.5 and p["churn"] == 0.5
