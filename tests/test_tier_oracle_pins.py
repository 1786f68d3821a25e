"""Pins of the tiered-cache oracle against what the pages and mathematics fix.

QEvict, "Metodologia: QEvict" and "Meccanismi Chiave": windows routed between
a full-precision tier, a recoverable INT2 tier and an evicted tier under a
fixed byte budget, cumulative attention-mass scores, write-once ledger.

Each check compares the oracle with an independent statement of the same fact:
numpy's own float16 conversion and torch's bfloat16 conversion for the
rounding steps, enumeration of every fp16 value for the scale and zero, a
ledger decoder written here from the documented layout, textbook numpy
attention, and the routing rules restated as Python sorts and invariants.
"""
import math

import numpy as np
import pytest
import torch

import oracle

RNG = np.random.default_rng(20261202)

# every finite non-negative fp16 value, ascending, as float64
_F16_POS = np.arange(0, 0x7C00, dtype=np.uint16).view(np.float16).astype(np.float64)


def f16_val(bits):
    return np.asarray(bits, dtype=np.uint16).view(np.float16).astype(np.float64)


def fma32(a, b, c):
    """fp32 fma: the exact a*b + c (exact in float64 for fp16-sized a, b, c),
    rounded once to fp32."""
    return np.float32(np.float64(a) * np.float64(b) + np.float64(c))


def sample_floats(n):
    parts = [
        RNG.normal(0, 1, n),
        RNG.normal(0, 1e-5, n // 4),        # fp16 subnormal range
        RNG.uniform(60000, 70000, n // 8),  # around the fp16 overflow
        -RNG.uniform(60000, 70000, n // 8),
        RNG.normal(0, 300, n // 4),
    ]
    x = np.concatenate(parts).astype(np.float32)
    specials = np.array([0.0, -0.0, 1.0, -1.0, 65504.0, -65504.0, 65520.0, 2.0 ** -24,
                         -(2.0 ** -24), 2.0 ** -25, -(2.0 ** -25), 1e-30, -1e-30,
                         np.inf, -np.inf], dtype=np.float32)
    return np.concatenate([x, specials])


# --------------------------------------------------------------------------
# fp16 and bf16 rounding
# --------------------------------------------------------------------------

def test_f16_directed_rounding_brackets_numpy_nearest():
    x = sample_floats(200_000)
    rd = oracle.f16_round(x, "down")
    ru = oracle.f16_round(x, "up")
    vd, vu, xv = f16_val(rd), f16_val(ru), x.astype(np.float64)
    assert np.all(vd <= xv) and np.all(vu >= xv)
    with np.errstate(over="ignore"):
        exact = np.float16(x).astype(np.float64) == xv
    assert np.all(vd[exact] == xv[exact]) and np.all(vu[exact] == xv[exact])
    # otherwise the two are neighbours and numpy's nearest is one of them
    ne = ~exact
    with np.errstate(over="ignore"):
        nxt = np.nextafter(vd[ne].astype(np.float16), np.float16(np.inf)).astype(np.float64)
    assert np.all(nxt == vu[ne])
    with np.errstate(over="ignore"):
        near = np.float16(x[ne]).astype(np.float64)
        assert np.all((near == vd[ne]) | (near == vu[ne]))


def test_f16_directed_rounding_signs_and_overflow():
    rd = lambda v: int(oracle.f16_round(np.float32(v), "down"))
    ru = lambda v: int(oracle.f16_round(np.float32(v), "up"))
    assert rd(0.0) == 0x0000 and ru(0.0) == 0x0000
    assert rd(-0.0) == 0x8000 and ru(-0.0) == 0x8000
    assert ru(-1e-30) == 0x8000 and rd(-1e-30) == 0x8001   # -0 from a negative
    assert rd(1e-30) == 0x0000 and ru(1e-30) == 0x0001
    assert rd(1e6) == 0x7BFF and ru(1e6) == 0x7C00          # toward -inf keeps max finite
    assert rd(-1e6) == 0xFC00 and ru(-1e6) == 0xFBFF


def test_bf16_round_matches_torch():
    x = sample_floats(200_000)
    x = np.concatenate([x, np.array([3.0e38, -3.0e38, 3.4e38], dtype=np.float32)])
    ours = oracle.bf16_round(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).to(torch.float32).numpy()
    assert np.array_equal(ours.view(np.uint32), ref.view(np.uint32))


# --------------------------------------------------------------------------
# INT2 group quantiser
# --------------------------------------------------------------------------

def unpack_codes(b):
    b = np.asarray(b, dtype=np.uint8)
    return np.array([(int(b[j >> 2]) >> (2 * (j & 3))) & 3 for j in range(32)])


def random_groups(n):
    out = []
    for i in range(n):
        kind = i % 5
        if kind == 0:
            g = RNG.normal(0, 1, 32)
        elif kind == 1:
            g = RNG.normal(0, 1, 32)
            g[RNG.integers(32)] *= 40            # an outlier channel
        elif kind == 2:
            g = RNG.uniform(-3e-4, 3e-4, 32)     # subnormal-size scale
        elif kind == 3:
            g = RNG.normal(5, 0.01, 32)          # narrow range away from 0
        else:
            g = np.round(RNG.normal(0, 2, 32), 1)
        out.append(np.asarray(g, dtype=np.float32))
    return out


# (min, max) pairs where fl(3 s + z) falls short of the maximum at the first
# rounded-up scale, so the scale must step up once more (found by search)
_BUMP_CASES = [(-3.451481819152832, 6.003906726837158), (-0.006832696031779051, 0.0016899113543331623),
               (-0.2608964443206787, 0.3194580376148224), (-4.727999687194824, 0.5751953721046448),
               (-0.02407578006386757, -0.007244109641760588)]


def bump_groups():
    out = []
    for mn, mx in _BUMP_CASES:
        g = np.linspace(mn, mx, 32).astype(np.float32)
        g[0], g[-1] = np.float32(mn), np.float32(mx)
        out.append(g)
    return out


def test_int2_zero_and_scale_are_the_defined_fp16_values():
    for g in bump_groups() + random_groups(300):
        codes, s, z, ok = oracle.int2_quantize_group(g)
        assert ok
        mn, mx = np.float64(g.min()), np.float64(g.max())
        # zero: the largest fp16 at or below the group minimum
        allv = np.concatenate([-_F16_POS[::-1], _F16_POS])
        z_ref = allv[allv <= mn].max()
        assert f16_val(z) == z_ref
        # scale: the smallest fp16 at or above fl((max - z) / 3) whose
        # fl(3 s + z) reaches the maximum
        r = (np.float32(mx) - np.float32(z_ref)) / np.float32(3)
        cand = _F16_POS[_F16_POS >= np.float64(r)]
        ok_c = [c for c in cand[:64] if fma32(3.0, c, z_ref) >= np.float32(mx)]
        assert f16_val(s) == ok_c[0]


def test_int2_error_bound_and_nearest_level():
    worst = 0.0
    for g in bump_groups() + random_groups(500):
        codes, s, z, ok = oracle.int2_quantize_group(g)
        xh = oracle.int2_dequantize_group(codes, s, z)
        sv, zv = f16_val(s), f16_val(z)
        c = unpack_codes(codes)
        levels = np.array([fma32(k, sv, zv) for k in range(4)], dtype=np.float64)
        assert np.array_equal(xh.astype(np.float64), levels[c])
        err = np.abs(g.astype(np.float64) - xh)
        slack = 2 * np.spacing(np.maximum(np.abs(g), np.abs(xh)).astype(np.float32)).astype(
            np.float64) + 2 * np.spacing(np.float32(abs(zv) + 3 * sv))
        assert np.all(err <= sv / 2 + slack)
        # the chosen level is the nearest one (up to the same rounding slack)
        dist = np.abs(g.astype(np.float64)[:, None] - levels[None, :])
        assert np.all(dist[np.arange(32), c] <= dist.min(axis=1) + slack)
        worst = max(worst, float((err / np.maximum(sv, 1e-30)).max()))
    assert worst <= 0.5 + 1e-3


def test_int2_grid_values_round_trip_exactly():
    for _ in range(200):
        z = np.float16(RNG.normal(0, 2))
        s = np.float16(abs(RNG.normal(0, 0.5)) + 1e-3)
        c = RNG.integers(0, 4, 32)
        c[0], c[1] = 0, 3                                     # span the full range
        x = np.array([fma32(k, s, z) for k in c], dtype=np.float32)
        codes, s2, z2, ok = oracle.int2_quantize_group(x)
        xh = oracle.int2_dequantize_group(codes, s2, z2)
        assert np.array_equal(xh, x)


def test_int2_constant_group():
    for v in [0.0, 1.5, -2.25, 1024.0, 0.0001220703125]:        # fp16-representable
        x = np.full(32, v, dtype=np.float32)
        codes, s, z, ok = oracle.int2_quantize_group(x)
        assert s == 0 and f16_val(z) == v
        assert np.array_equal(oracle.int2_dequantize_group(codes, s, z), x)
        assert not np.any(np.asarray(codes))
    x = np.full(32, 0.1, dtype=np.float32)                       # not representable
    codes, s, z, ok = oracle.int2_quantize_group(x)
    xh = oracle.int2_dequantize_group(codes, s, z)
    assert np.all(np.abs(xh - x) <= f16_val(s) / 2 + 1e-7)


def test_int2_code_packing_layout():
    z, s = np.float16(-1.0), np.float16(0.5)
    c = np.array([j % 4 for j in range(32)])
    c = np.roll(c, 1)
    x = np.array([fma32(k, s, z) for k in c], dtype=np.float32)
    codes, _, _, _ = oracle.int2_quantize_group(x)
    expect = np.zeros(8, dtype=np.uint8)
    for j in range(32):
        expect[j // 4] |= np.uint8(c[j] << (2 * (j % 4)))
    assert np.array_equal(np.asarray(codes), expect)


def test_int2_range_beyond_fp16_is_reported():
    x = np.full(32, 1.0, dtype=np.float32)
    x[3] = -1e6
    assert not oracle.int2_quantize_group(x)[3]


# --------------------------------------------------------------------------
# ledger layout
# --------------------------------------------------------------------------

def decode_ledger(lg, d):
    """Independent reader of the documented layout: [K codes: token, group,
    8 B][K params: token, group, (fp16 scale, fp16 zero)][V codes][V params]."""
    ng = d // 32
    cb, pb = 64 * ng * 8, 64 * ng * 4
    out = []
    for kv in range(2):
        base = kv * (cb + pb)
        codes = np.asarray(lg[base:base + cb]).reshape(64, ng, 8)
        params = np.asarray(lg[base + cb:base + cb + pb]).reshape(64, ng, 2, 2)
        sz = params[..., 0].astype(np.uint16) | (params[..., 1].astype(np.uint16) << 8)
        X = np.zeros((64, d), dtype=np.float32)
        for t in range(64):
            for g in range(ng):
                sv, zv = f16_val(sz[t, g, 0]), f16_val(sz[t, g, 1])
                cc = unpack_codes(codes[t, g])
                X[t, g * 32:(g + 1) * 32] = [fma32(k, sv, zv) for k in cc]
        out.append(X)
    return out


@pytest.mark.parametrize("d", [64, 128])
def test_ledger_layout_and_round_trip(d):
    K = RNG.normal(0, 1, (64, d)).astype(np.float32)
    V = RNG.normal(0, 1, (64, d)).astype(np.float32)
    lg = oracle.ledger_write_window(K, V)
    assert lg.size == 2 * 64 * (d // 32) * 12 == 48 * d
    Kr, Vr = oracle.ledger_read_window(lg, d)
    Kd, Vd = decode_ledger(lg, d)
    assert np.array_equal(Kr, Kd) and np.array_equal(Vr, Vd)
    # each group of each token equals the group quantiser on its own
    for t in (0, 17, 63):
        for g in range(d // 32):
            codes, s, z, _ = oracle.int2_quantize_group(V[t, g * 32:(g + 1) * 32])
            assert np.array_equal(oracle.int2_dequantize_group(codes, s, z),
                                  Vr[t, g * 32:(g + 1) * 32])


# --------------------------------------------------------------------------
# tiered attention and window mass
# --------------------------------------------------------------------------

def numpy_attention(q, K, V, scale):
    s = (q.astype(np.float64) @ K.astype(np.float64).T) * scale
    s -= s.max(axis=1, keepdims=True)
    p = np.exp(s)
    p /= p.sum(axis=1, keepdims=True)
    return p @ V.astype(np.float64), p


def bf16_values(shape, std=1.0):
    x = RNG.normal(0, std, shape).astype(np.float32)
    return torch.from_numpy(x).to(torch.bfloat16).to(torch.float32).numpy()


def make_unit(n_win, N, d=128, G=4, tiers=None):
    K = bf16_values((n_win * 64, d))
    V = bf16_values((n_win * 64, d))
    if tiers is None:
        tiers = RNG.integers(0, 3, n_win).astype(np.int8)
    u = oracle.TierUnit(tiers, K, V, N, n_win)
    q = RNG.normal(0, 1, (G, d)).astype(np.float32)
    return u, q, K, V


@pytest.mark.parametrize("N", [64 * 10, 64 * 10 + 37, 64 * 9 + 1])
def test_tiered_attention_equals_dense_attention_over_the_tier_rows(N):
    n_win = 11
    u, q, K, V = make_unit(n_win, N)
    closed = N // 64
    rows_k, rows_v, win = [], [], []
    for w in range(-(-N // 64)):
        if w < closed and u.tier[w] == oracle.EVICTED:
            continue
        if w < closed and u.tier[w] == oracle.INT2:
            kd, vd = decode_ledger(u.ledger[w], 128)
        else:
            n = 64 if w < closed else N - 64 * w
            kd, vd = K[64 * w:64 * w + n], V[64 * w:64 * w + n]
        rows_k.append(kd)
        rows_v.append(vd)
        win += [w] * len(kd)
    scale = float(np.float32(1 / math.sqrt(128)))    # the oracle takes an fp32 scale
    ref, p = numpy_attention(q, np.concatenate(rows_k), np.concatenate(rows_v), scale)
    out, mass = u.attend(q, N, scale)
    assert np.abs(out - ref).max() < 1e-12
    win = np.array(win)
    ref_mass = np.array([p[:, win == w].sum() for w in range(-(-N // 64))])
    assert np.abs(mass - ref_mass).max() < 1e-12
    assert abs(mass.sum() - 4.0) < 1e-12
    assert np.all(mass[:closed][u.tier[:closed] == oracle.EVICTED] == 0)


def test_tiered_attention_all_bf16_is_dense_attention():
    n_win, N = 6, 6 * 64 - 5
    u, q, K, V = make_unit(n_win, N, tiers=np.zeros(6, dtype=np.int8))
    ref, _ = numpy_attention(q, K[:N], V[:N], 0.125)
    out, _ = u.attend(q, N, 0.125)
    assert np.abs(out - ref).max() < 1e-12


def test_tiered_attention_nothing_attended_gives_zeros():
    u, q, K, V = make_unit(4, 256, tiers=np.full(4, 2, dtype=np.int8))
    out, mass = u.attend(q, 256, 0.1)
    assert not out.any() and not mass.any()


# --------------------------------------------------------------------------
# routing
# --------------------------------------------------------------------------

def route_reference(tier, score, quota, budget, N, d):
    """The routing rule restated: rank live closed windows by (score desc,
    window asc); the first quota are bf16, the rest INT2; evict the lowest
    ranked INT2 windows while the bytes exceed the budget."""
    closed = N // 64
    live = [w for w in range(closed) if tier[w] != oracle.EVICTED]
    order = sorted(live, key=lambda w: (-int(score[w]), w))
    new = {w: (oracle.BF16 if i < quota else oracle.INT2) for i, w in enumerate(order)}
    lb = 48 * d
    nbytes = sum(256 * d if t == oracle.BF16 else lb for t in new.values())
    for w in reversed(order):
        if nbytes <= budget:
            break
        if new[w] == oracle.INT2:
            new[w] = oracle.EVICTED
            nbytes -= lb
    return new


def test_routing_steps_follow_the_rule_and_keep_the_invariants():
    d, n_win = 128, 24
    N = 20 * 64
    init = np.array([0] * 5 + [1] * 10 + [2] * 5, dtype=np.int8)
    RNG.shuffle(init)
    u, q, K, V = make_unit(n_win, N, d=d, tiers=np.concatenate([init, np.zeros(4, np.int8)]))
    assert u.quota == 5 and u.budget == 5 * 256 * d + 10 * 48 * d
    evicted = set(np.flatnonzero(init == oracle.EVICTED))
    for step in range(3 * 64 + 5):
        # a new token per step: the open window fills and joins the routing
        Ncur = N + step
        mass = RNG.dirichlet(np.ones(-(-Ncur // 64))).astype(np.float32) * 4
        before_t, before_s = u.tier.copy(), u.score.copy()
        ref_score = before_s.copy()
        for w in range(-(-Ncur // 64)):
            if before_t[w] != oracle.EVICTED:
                ref_score[w] += int(np.rint(np.float64(mass[w]) * 2.0 ** 32))
        stats = u.update(mass, Ncur)
        assert np.array_equal(u.score, ref_score)
        new = route_reference(before_t, ref_score, u.quota, u.budget, Ncur, d)
        for w, t in new.items():
            assert u.tier[w] == t, (step, w)
        closed = Ncur // 64
        now_ev = set(np.flatnonzero(u.tier[:closed] == oracle.EVICTED))
        assert evicted <= now_ev                       # evictions are permanent
        evicted = now_ev
        assert u.tier_bytes(Ncur) <= u.budget
        assert int((u.tier[:closed] == oracle.BF16).sum()) == u.quota
        joined = step > 0 and Ncur % 64 == 0           # the open window just closed
        prom = sum(1 for w in new if before_t[w] == oracle.INT2 and new[w] == oracle.BF16)
        dem = sum(1 for w in new if before_t[w] == oracle.BF16 and new[w] == oracle.INT2)
        ev = sum(1 for w in new if before_t[w] != oracle.EVICTED and new[w] == oracle.EVICTED)
        assert list(stats) == [prom, dem, ev]
        if joined:
            assert ev == 1                              # a new window forces one eviction
        was_ev = before_t == oracle.EVICTED
        assert np.array_equal(u.score[was_ev], before_s[was_ev])   # frozen scores


def test_promotion_writes_bf16_of_the_ledger_and_the_ledger_is_written_once():
    d, n_win, N = 128, 4, 4 * 64
    tiers = np.array([0, 1, 1, 0], dtype=np.int8)
    u, q, K, V = make_unit(n_win, N, d=d, tiers=tiers)
    assert u.quota == 2
    first_ledger_w0 = oracle.ledger_write_window(K[0:64], V[0:64])
    # step 1: window 1 and 2 rise above 0 and 3 -> both promoted, 0 and 3 demoted
    u.update(np.array([0.0, 2.0, 1.0, 0.0], dtype=np.float32), N)
    assert list(u.tier) == [1, 0, 0, 1]
    assert np.array_equal(u.ledger[0], first_ledger_w0)   # first demotion: from the rows
    kd, vd = decode_ledger(u.ledger[1], d)
    kb = torch.from_numpy(kd).to(torch.bfloat16).to(torch.float32).numpy()
    vb = torch.from_numpy(vd).to(torch.bfloat16).to(torch.float32).numpy()
    assert np.array_equal(u.K[64:128], kb) and np.array_equal(u.V[64:128], vb)
    led1 = u.ledger[1].copy()
    # step 2: window 1 falls back: its ledger is reused, not rewritten
    u.update(np.array([3.0, 0.0, 0.0, 3.0], dtype=np.float32), N)
    assert list(u.tier) == [0, 1, 1, 0]
    assert np.array_equal(u.ledger[1], led1)
    # step 3: promoted again: the same bf16 rows as the first promotion
    u.update(np.array([0.0, 9.0, 0.0, 0.0], dtype=np.float32), N)
    assert list(u.tier) == [0, 0, 1, 1]          # tie of windows 0 and 3: the lower wins
    assert np.array_equal(u.ledger[3], oracle.ledger_write_window(K[192:256], V[192:256]))
    assert np.array_equal(u.ledger[1], led1)
    assert np.array_equal(u.K[64:128], kb) and np.array_equal(u.V[64:128], vb)


def test_routing_ties_go_to_the_lower_window():
    d, n_win, N = 64, 6, 6 * 64
    u, q, K, V = make_unit(n_win, N, d=d, tiers=np.array([1, 1, 0, 0, 1, 1], np.int8))
    u.update(np.zeros(6, dtype=np.float32), N)
    assert list(u.tier) == [0, 0, 1, 1, 1, 1]
