"""Helpers for the GPU parity tests: run the CUDA path through the C ABI and
the oracle on the same seeded inputs, unit by unit."""
import numpy as np
import torch

import oracle
import sparse_decode_attention_gb300 as kvr


def shape_of_cache(K, Hq=None):
    B, Hkv, cap, d = K.shape
    return kvr.Shape(B, Hq or Hkv, Hkv, d, cap, K.dtype)


def planes_to_bytes(codes, B, Hkv, cap, d):
    """Per-token code bytes [B, Hkv, cap, d/8] from the library's bit-plane
    tiles (test-side reading of the documented layout)."""
    raw = codes.detach().cpu().numpy() if isinstance(codes, torch.Tensor) else codes
    tiles = (cap + 1023) // 1024
    words = raw[:B * Hkv * tiles * d * 128].view(np.uint32).reshape(B * Hkv, tiles, d // 4, 32, 4)
    out = np.zeros((B * Hkv, tiles * 1024, d // 8), dtype=np.uint8)
    shifts = np.arange(32, dtype=np.uint32)
    for u in range(B * Hkv):
        # [tile, block, plane] -> bits [tile, block, token-in-block, plane]
        planes = words[u].transpose(0, 2, 1, 3).reshape(tiles, 32, d)
        bits = ((planes[:, :, None, :] >> shifts[None, None, :, None]) & 1).astype(np.uint8)
        bits = bits.reshape(tiles * 1024, d)
        out[u] = np.packbits(bits.reshape(-1, d // 8, 8), axis=-1, bitorder="little")[..., 0]
    return out.reshape(B, Hkv, tiles * 1024, d // 8)[:, :, :cap]


def encode_gpu(K, sgn, rows, pos0=0):
    B = K.shape[0]
    codes = kvr.codes_buffer(shape_of_cache(K), K.device)
    p0 = torch.full((B,), pos0, dtype=torch.int32, device=K.device)
    kvr.kvr_encode_keys(K, p0, rows, sgn, codes)
    return codes


def codes_bytes_gpu(codes, K):
    B, Hkv, cap, d = K.shape
    return planes_to_bytes(codes, B, Hkv, cap, d)


def select_gpu(q, K, codes, seq_len, sgn, params):
    """kvr_select (with coarse scores stored); outputs and workspace parts on the CPU."""
    B, Hkv, cap, d = K.shape
    params = kvr.SelectParams(params.C, params.k, params.W, params.lut,
                              params.flags | kvr.SELECT_STORE_COARSE,
                              V_prefetch=params.V_prefetch, rsq_records=params.rsq_records,
                              sink=params.sink, region_end=params.region_end)
    shape = kvr.Shape.of(K, q)
    ws = kvr.workspace(kvr.kvr_select_workspace_size(shape, params))
    ws.fill_(0xAB)  # stale contents must not matter
    out_idx = torch.full((B, Hkv, params.k), 7, dtype=torch.int32, device=K.device)
    out_cnt = torch.full((B, Hkv), 7, dtype=torch.int32, device=K.device)
    err = torch.zeros(1, dtype=torch.int32, device=K.device)
    kvr.kvr_select(q, K, codes, seq_len, sgn, params, out_idx, out_cnt, ws, err)
    bits = kvr.kvr_read_error(err)
    v = kvr.kvr_select_workspace_views(shape, params)
    U, C = B * Hkv, params.C
    cap_pad = (cap + 15) // 16 * 16
    wsc = ws.cpu()
    return dict(
        idx=out_idx.cpu().numpy(), count=out_cnt.cpu().numpy(), err=bits,
        coarse=wsc[v["coarse"]:v["coarse"] + U * cap_pad].numpy().reshape(U, cap_pad),
        cand=wsc[v["cand_idx"]:v["cand_idx"] + U * C * 4].view(torch.int32).numpy().reshape(U, C),
        cand_S=wsc[v["cand_score"]:v["cand_score"] + U * C * 4].view(torch.float32).numpy()
        .reshape(U, C),
        cand_count=wsc[v["cand_count"]:v["cand_count"] + U * 4].view(torch.int32).numpy(),
    )


def attend_gpu(q, K, V, idx, count, seq_len, W, scale):
    shape = kvr.Shape.of(K, q)
    ws = kvr.workspace(kvr.kvr_attend_workspace_size(shape, idx.shape[-1], W))
    ws.fill_(0xCD)
    out = torch.full(q.shape, float("nan"), dtype=torch.float32, device=K.device)
    err = torch.zeros(1, dtype=torch.int32, device=K.device)
    kvr.kvr_sparse_attend(q, K, V, idx, count, seq_len, W, scale, out, ws, err)
    bits = kvr.kvr_read_error(err)
    return out.cpu().numpy(), bits


def compare_select_unit(res, u, q_group, K_unit, codes_unit, N, sgn, params, check_diag=True):
    """Bit-exact comparison of one unit's selection with the oracle."""
    idx, cnt, dg = oracle.select_unit(q_group, K_unit, codes_unit, N, sgn, params.C, params.k,
                                      params.W, params.lut, diagnostics=True)
    b, h = divmod(u, res["idx"].shape[1])
    pool = max(0, N - params.W)
    Cp = min(params.C, pool)
    if check_diag:
        assert np.array_equal(res["coarse"][u, :pool].astype(np.int32), dg["coarse"]), \
            "coarse scores differ (unit %d)" % u
        assert res["cand_count"][u] == Cp
        assert np.array_equal(res["cand"][u, :Cp], dg["cand"]), "candidate sets differ (unit %d)" % u
        assert np.array_equal(res["cand_S"][u, :Cp].view(np.int32), dg["cand_S"].view(np.int32)), \
            "exact scores differ (unit %d)" % u
    assert res["count"][b, h] == cnt, "count differs (unit %d)" % u
    assert np.array_equal(res["idx"][b, h], idx), "top-k sets differ (unit %d)" % u
    return idx, cnt
