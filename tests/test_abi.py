"""The C-ABI library builds, loads and exports every symbol include/kvr.h
declares; host-side validation rejects bad calls before any launch (these
calls return before touching the GPU, so they run without one)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            src = open(os.path.join(ROOT, "include", fn)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names |= set(re.findall(r"\b(kvr_[a-z0-9_]+)\s*\(", src))
    return sorted(names)


def test_header_declares_the_four_calls():
    names = declared_functions()
    for n in ("kvr_encode_keys", "kvr_select", "kvr_sparse_attend", "kvr_tier_update",
              "kvr_tier_init", "kvr_sparse_attend_tiered"):
        assert n in names, n


def test_library_exports_every_declared_symbol(kvr_lib):
    lib = kvr_lib.load()
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing


def test_status_strings(kvr_lib):
    assert kvr_lib.kvr_status_string(0) == "ok"
    assert kvr_lib.kvr_status_string(3) == "workspace too small"
    assert kvr_lib.kvr_status_string(99) == "unknown status"
    assert kvr_lib.kvr_version() >= 100


def _shape(kvr, **kw):
    base = dict(B=1, Hq=32, Hkv=8, d=128, cap=1024, dtype="bf16")
    base.update(kw)
    return kvr.Shape(**base)


def test_workspace_sizes(kvr_lib):
    kvr = kvr_lib
    s = _shape(kvr, cap=131072)
    p = kvr.SelectParams(8192, 2048, 128)
    n = kvr.kvr_select_workspace_size(s, p)
    # coarse scores (1 B per key) + candidates (8 B each) dominate
    assert n >= 8 * 131072 + 8 * 8192 * 8
    assert n < 8 * 131072 * 2 + 8 * 8192 * 8 + (1 << 22)
    v = kvr.kvr_select_workspace_views(s, p)
    assert v["coarse"] == 2 ** 64 - 1  # not stored without the flag
    assert all(x % 256 == 0 for k, x in v.items() if k != "coarse")
    pc = kvr.SelectParams(8192, 2048, 128, flags=kvr.SELECT_STORE_COARSE)
    vc = kvr.kvr_select_workspace_views(s, pc)
    assert vc["coarse"] % 256 == 0
    assert kvr.kvr_select_workspace_size(s, pc) >= n + 8 * 131072
    assert kvr.kvr_select_workspace_size(s, kvr.SelectParams(8, 4, 0, flags=8)) == 0  # unknown flag
    # magnitude-aware votes: one vote-list row per unit and sub-block on top
    pm = kvr.SelectParams(8192, 2048, 128, flags=kvr.SELECT_MAGNITUDE_VOTES)
    assert kvr.kvr_select_workspace_size(s, pm) >= n + 8 * 16 * 264 * 2
    assert kvr.kvr_codes_bytes(s) == 8 * 128 * 128 * 128  # 128 tiles of 1024 tokens per unit
    assert kvr.kvr_codes_bytes(_shape(kvr, cap=1025, d=64)) == 8 * 2 * 64 * 128
    assert kvr.kvr_select_workspace_size(_shape(kvr, d=96), p) == 0
    assert kvr.kvr_select_workspace_size(s, kvr.SelectParams(10, 20, 0)) == 0  # k > C
    assert kvr.kvr_attend_workspace_size(s, 2048, 128) == 0  # partials merge on chip


def test_validation_before_launch(kvr_lib):
    """Invalid calls return a status and enqueue nothing (no GPU involved)."""
    kvr = kvr_lib
    L = kvr.load()
    fake = ctypes.c_void_p(1 << 20)  # aligned, never dereferenced
    odd = ctypes.c_void_p((1 << 20) + 4)
    s = _shape(kvr)
    p = kvr.SelectParams(64, 16, 8)
    enc = lambda shp, K, n, codes: L.kvr_encode_keys(ctypes.byref(shp.c()), K, fake, n, fake,
                                                    codes, None, None)
    assert enc(s, None, 1, fake) == 1
    assert enc(s, odd, 1, fake) == 1
    assert enc(_shape(kvr, d=96), fake, 1, fake) == 2
    assert enc(_shape(kvr, Hq=20, Hkv=8), fake, 1, fake) == 1
    assert enc(_shape(kvr, Hq=8 * 17, Hkv=8), fake, 1, fake) == 2
    assert enc(s, fake, -1, fake) == 1
    assert enc(s, fake, 0, fake) == 0  # nothing to do

    def sel(shp, prm, ws_bytes, ws=fake):
        return L.kvr_select(ctypes.byref(shp.c()), ctypes.byref(prm.c()), fake, fake, fake, fake,
                            fake, fake, fake, ws, ws_bytes, None, None)
    need = kvr.kvr_select_workspace_size(s, p)
    assert sel(s, p, need - 1) == 3
    assert sel(s, kvr.SelectParams(64, 65, 8), need) == 1
    assert sel(s, kvr.SelectParams(40000, 16, 8), need) == 1
    assert sel(s, kvr.SelectParams(64, 16, 8, lut=(16, 0, 0, 0, 0, 0, 0, 0, 0)), need) == 1
    assert sel(s, p, need, ws=ctypes.c_void_p((1 << 20) + 16)) == 1  # ws not 256-aligned
    pv = p.c()
    pv.V_prefetch = (1 << 20) + 8                                   # misaligned V hint
    assert L.kvr_select(ctypes.byref(s.c()), ctypes.byref(pv), fake, fake, fake, fake, fake,
                        fake, fake, fake, need, None, None) == 1

    def att(shp, kmax, W, ws_bytes, scale=0.1):
        return L.kvr_sparse_attend(ctypes.byref(shp.c()), fake, fake, fake, fake, kmax, fake,
                                   fake, W, scale, fake, fake, ws_bytes, None, None)
    need = kvr.kvr_attend_workspace_size(s, 16, 8)
    assert att(s, -1, 8, need) == 1
    assert att(_shape(kvr, Hq=24, Hkv=8), 16, 8, need) == 2  # group of 3 heads
    assert att(s, 16, 8, need, scale=float("nan")) == 1


def test_tier_calls_validate_before_launch(kvr_lib):
    """The tier calls check shape, state and buffers on the host (no GPU)."""
    kvr = kvr_lib
    L = kvr.load()
    fake = 1 << 20
    s = _shape(kvr, B=4, cap=131072 + 512)
    n_win = (131072 + 512) // 64
    assert kvr.kvr_ledger_bytes(128) == 6144 and kvr.kvr_ledger_bytes(64) == 3072
    assert kvr.kvr_ledger_bytes(96) == 0
    wa = kvr.kvr_tiered_attend_workspace_size(s, n_win)
    wu = kvr.kvr_tier_update_workspace_size(s, n_win)
    assert wa >= 32 * n_win * 4 * 4 and wu >= 32 * n_win * 4
    # unsupported: fp32 cache, 16-head groups, too few windows for the capacity
    assert kvr.kvr_tiered_attend_workspace_size(_shape(kvr, dtype="f32"), 64) == 0
    assert kvr.kvr_tiered_attend_workspace_size(_shape(kvr, Hq=128, Hkv=8), 64) == 0
    assert kvr.kvr_tier_update_workspace_size(s, n_win - 1) == 0

    def state(**kw):
        f = dict(n_win=n_win, tier=fake, score=fake, has_ledger=fake, ledger=fake, quota=fake,
                 budget=fake)
        f.update(kw)
        return kvr._TierState(**f)

    def att(shp, st, ws_bytes, scale=0.1):
        return L.kvr_sparse_attend_tiered(ctypes.byref(shp.c()), ctypes.byref(st), fake, fake,
                                          fake, fake, scale, fake, fake, fake, ws_bytes, None,
                                          None)
    assert att(s, state(), wa - 1) == 3
    assert att(s, state(ledger=None), wa) == 1
    assert att(s, state(ledger=fake + 8), wa) == 1          # ledger not 16-byte aligned
    assert att(s, state(score=fake + 4), wa) == 1           # int64 array misaligned
    assert att(s, state(n_win=n_win - 1), wa) == 1          # capacity beyond the windows
    assert att(s, state(n_win=20000), wa) == 2              # above the ranking limit
    assert att(_shape(kvr, B=4, cap=131072 + 512, dtype="f32"), state(), wa) == 2
    assert att(s, state(), wa, scale=float("nan")) == 1

    def upd(shp, st, ws_bytes):
        return L.kvr_tier_update(ctypes.byref(shp.c()), ctypes.byref(st), fake, fake, fake, fake,
                                 None, fake, ws_bytes, None, None)
    assert upd(s, state(), wu - 1) == 3
    assert upd(s, state(tier=None), wu) == 1
    assert L.kvr_tier_init(ctypes.byref(s.c()), ctypes.byref(state()), None, fake, fake, fake,
                           None, None) == 1
    assert L.kvr_tier_init(ctypes.byref(s.c()), None, fake, fake, fake, fake, None, None) == 1


def test_reranker_calls_validate_before_launch(kvr_lib):
    """kvr_encode_rsq and the records field of kvr_select_params are checked
    on the host (no GPU)."""
    kvr = kvr_lib
    L = kvr.load()
    fake = ctypes.c_void_p(1 << 20)
    odd = ctypes.c_void_p((1 << 20) + 8)
    s = _shape(kvr)
    assert kvr.kvr_rsq_record_bytes(128) == 96 and kvr.kvr_rsq_record_bytes(64) == 48
    assert kvr.kvr_rsq_record_bytes(96) == 0

    def enc(shp, K, n, rec):
        return L.kvr_encode_rsq(ctypes.byref(shp.c()), K, fake, n, fake, rec, None, None)
    assert enc(s, None, 1, fake) == 1
    assert enc(s, fake, 1, None) == 1
    assert enc(s, fake, 1, odd) == 1                  # records not 16-byte aligned
    assert enc(s, fake, -1, fake) == 1
    assert enc(_shape(kvr, d=96), fake, 1, fake) == 2
    assert enc(s, fake, 0, fake) == 0                 # nothing to do
    assert L.kvr_rsq_tables(None, None) == 1
    p = kvr.SelectParams(64, 16, 8)
    need = kvr.kvr_select_workspace_size(s, p)
    pv = p.c()
    pv.rsq_records = (1 << 20) + 8                    # misaligned records
    assert L.kvr_select(ctypes.byref(s.c()), ctypes.byref(pv), fake, fake, fake, fake, fake,
                        fake, fake, fake, need, None, None) == 1


def test_pageable_host_caches_are_refused(kvr_lib):
    """K / V may be device or page-locked host memory; pageable host tensors
    are refused by the binding before any call (no GPU)."""
    import torch
    kvr = kvr_lib
    K = torch.zeros((1, 2, 64, 64), dtype=torch.bfloat16)          # pageable
    for call in (lambda: kvr.kvr_encode_keys(K, None, 1, None, None),
                 lambda: kvr.kvr_encode_rsq(K, None, 1, None, None),
                 lambda: kvr.kvr_select(None, K, None, None, None, None, None, None, None),
                 lambda: kvr.kvr_sparse_attend(None, K, K, None, None, None, 8, 0.1, None, None)):
        with pytest.raises(TypeError, match="page-locked"):
            call()


def test_region_calls_validate_before_launch(kvr_lib):
    """kvr_regions_update, kvr_sparse_attend_regions and the region fields of
    kvr_select_params are checked on the host (no GPU)."""
    kvr = kvr_lib
    L = kvr.load()
    fake = ctypes.c_void_p(1 << 20)
    odd = ctypes.c_void_p((1 << 20) + 2)
    upd = lambda B, S, Lc, U, re=fake, sl=fake: L.kvr_regions_update(B, sl, S, Lc, U, 0, re, None,
                                                                      None)
    assert upd(0, 4, 128, 64) == 0                 # nothing to do
    assert upd(2, -1, 128, 64) == 1
    assert upd(2, 4, -1, 64) == 1
    assert upd(2, 4, 128, 0) == 1                  # the buffer holds at least one token
    assert upd(2, 4, 128, 64, re=None) == 1
    assert upd(2, 4, 128, 64, re=odd) == 1
    s = _shape(kvr)
    att = lambda sink, re: L.kvr_sparse_attend_regions(ctypes.byref(s.c()), fake, fake, fake,
                                                       fake, 16, fake, fake, sink, re, 0.1, fake,
                                                       fake, 0, None, None)
    assert att(4, None) == 1                       # region_end required
    assert att(-1, fake) == 1
    assert att(4, odd) == 1
    p = kvr.SelectParams(64, 16, 8)
    need = kvr.kvr_select_workspace_size(s, p)
    pv = p.c()
    pv.sink = -3
    assert L.kvr_select(ctypes.byref(s.c()), ctypes.byref(pv), fake, fake, fake, fake, fake,
                        fake, fake, fake, need, None, None) == 1
    pv = p.c()
    pv.region_end = (1 << 20) + 2                  # int32 array misaligned
    assert L.kvr_select(ctypes.byref(s.c()), ctypes.byref(pv), fake, fake, fake, fake, fake,
                        fake, fake, fake, need, None, None) == 1


def test_decode_step_validates_before_launch(kvr_lib):
    kvr = kvr_lib
    L = kvr.load()
    fake = ctypes.c_void_p(1 << 20)
    s = _shape(kvr)
    p = kvr.SelectParams(64, 16, 8)
    need = kvr.kvr_select_workspace_size(s, p)

    def step(prm, pos=fake, V=fake, out=fake, scale=0.1, ws=need):
        return L.kvr_decode_step(ctypes.byref(s.c()), ctypes.byref(prm.c()), fake, fake, V, fake,
                                 fake, pos, fake, fake, fake, scale, out, fake, ws, None, None)
    assert step(p, pos=None) == 1
    assert step(p, pos=ctypes.c_void_p((1 << 20) + 2)) == 1      # int32 array misaligned
    assert step(p, V=None) == 1
    assert step(p, out=ctypes.c_void_p((1 << 20) + 4)) == 1
    assert step(p, scale=float("nan")) == 1
    assert step(p, ws=need - 1) == 3
    assert step(kvr.SelectParams(64, 65, 8)) == 1
