"""Seeded synthetic inputs for retrieval-based sparse decode attention.

This module only draws random numbers with the shapes, sizes and structure of
the long-context decode workloads the ParisKV and QEvict pages evaluate on
(Llama-3-8B-shaped layers, 128K and 1M contexts, drifting decode keys, a tiered
window cache). It holds none of the method's arithmetic: both the CUDA path
and the CPU oracle consume what it returns, and it imports neither.

Recipes (all seeded, torch.Generator on the requested device):
  * tiny: K, V ~ N(0, 1) fp32 with 4 seeded outlier channels scaled x8; q ~ N(0, 1).
  * low-rank (Llama-shaped): per (b, kv-head), K = Z U^T + 0.1 E with
    U ~ N(0, 1/r)^{d x r}, Z, E ~ N(0, 1); V drawn the same way with its own U.
    Planted keys sit at seeded pool positions with cosine 0.9 to the group's
    mean query direction q_hat: k = med||k|| (0.9 q_hat + sqrt(0.19) u_perp).
  * per-step queries: q_t = q_base + 0.1 N(0, 1).
  * drift: the key appended at step t is a draw of the prefill's law plus the
    mean 1.5 sigma_u (t+1)/T * u along a seeded unit direction u (sigma_u = std
    of the prefill keys along u); the step's queries are draws of the same
    low-rank law plus the same mean.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field, replace

import torch

DEFAULT_LUT = (3, 2, 1, 0, 0, 0, 0, 0, 0)
LINEAR_LUT = (8, 7, 6, 5, 4, 3, 2, 1, 0)
SRHT_SEED = 7


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    Hq: int
    Hkv: int
    d: int
    N: int
    dtype: str  # "f32" | "bf16"
    C: int = 0
    k: int = 0
    W: int = 0
    steps: int = 1
    rank: int = 0
    planted: int = 0
    seed: int = 1001
    lut: tuple = DEFAULT_LUT
    window: int = 64
    tier_frac: tuple = (0.25, 0.50, 0.25)
    extra: dict = field(default_factory=dict)

    @property
    def G(self) -> int:
        return self.Hq // self.Hkv

    def torch_dtype(self):
        return torch.float32 if self.dtype == "f32" else torch.bfloat16

    def with_(self, **kw) -> "Workload":
        return replace(self, **kw)


# The five workloads: a tiny correctness case, a Llama-3-8B-shaped 128K layer,
# a batched drifting decode, a million-token context and a tiered window cache.
TINY = Workload("tiny", B=1, Hq=4, Hkv=4, d=64, N=4096, dtype="f32", C=256, k=64, W=32,
                steps=16, seed=1001)
LLAMA_128K = Workload("llama3_8b_128k", B=1, Hq=32, Hkv=8, d=128, N=131072, dtype="bf16",
                      C=8192, k=2048, W=128, steps=200, rank=32, planted=64, seed=1002)
DRIFT = Workload("batched_drift", B=8, Hq=32, Hkv=8, d=128, N=32768, dtype="bf16", C=4096,
                 k=1024, W=128, steps=4096, rank=32, planted=0, seed=1003)
MILLION = Workload("million_token", B=1, Hq=32, Hkv=8, d=128, N=1 << 20, dtype="bf16",
                   C=16384, k=4096, W=256, rank=64, planted=256, seed=1004)
TIERED = Workload("tiered_window_cache", B=4, Hq=32, Hkv=8, d=128, N=131072, dtype="bf16",
                  steps=512, rank=32, planted=0, seed=1005, window=64)

ALL = {w.name: w for w in (TINY, LLAMA_128K, DRIFT, MILLION, TIERED)}


def gen(device, seed: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def srht_signs(d: int, seed: int = SRHT_SEED, device="cpu") -> torch.Tensor:
    """The seeded +-1 diagonal D of the rotation, int8 [d]."""
    g = gen("cpu", seed)
    s = torch.randint(0, 2, (d,), generator=g, dtype=torch.int64) * 2 - 1
    return s.to(torch.int8).to(device)


def _normal(shape, g, device, dtype=torch.float32):
    return torch.randn(shape, generator=g, device=device, dtype=dtype)


def _low_rank(n, d, r, g, device):
    U = _normal((d, r), g, device) / math.sqrt(r)
    Z = _normal((n, r), g, device)
    return Z @ U.T + 0.1 * _normal((n, d), g, device)


def make_cache(w: Workload, device="cpu", cap: int | None = None, seed: int | None = None,
               seq_len=None):
    """K, V [B, Hkv, cap, d] and q_base [B, Hq, d] in the workload's dtype.

    Rows [0, N) hold the context; rows beyond it (when cap > N) hold further
    keys of the same law for appending steps.
    """
    seed = w.seed if seed is None else seed
    cap = w.N if cap is None else cap
    g = gen(device, seed)
    B, Hkv, Hq, d = w.B, w.Hkv, w.Hq, w.d
    dt = w.torch_dtype()
    if w.rank == 0:
        K = _normal((B, Hkv, cap, d), g, device)
        V = _normal((B, Hkv, cap, d), g, device)
        q = _normal((B, Hq, d), g, device)
        ch = torch.randperm(d, generator=gen("cpu", seed + 17))[:4].to(device)
        K[..., ch] *= 8.0
        V[..., ch] *= 8.0
        return K.to(dt), V.to(dt), q.to(dt)
    K = torch.empty((B, Hkv, cap, d), device=device, dtype=dt)
    V = torch.empty((B, Hkv, cap, d), device=device, dtype=dt)
    q = _normal((B, Hq, d), g, device)
    G = w.G
    for b in range(B):
        for h in range(Hkv):
            kk = _low_rank(cap, d, w.rank, g, device)
            if w.planted:
                n_b = w.N if seq_len is None else int(seq_len[b])
                pool = max(1, n_b - w.W)
                qh = q[b, h * G:(h + 1) * G].mean(0)
                qh = qh / qh.norm()
                pos = torch.randperm(pool, generator=gen("cpu", seed * 131 + b * 17 + h))
                pos = pos[:min(w.planted, pool)].to(device)
                med = kk[:n_b].norm(dim=1).median()
                u = _normal((pos.numel(), d), g, device)
                u = u - (u @ qh)[:, None] * qh[None, :]
                u = u / u.norm(dim=1, keepdim=True)
                kk[pos] = med * (0.9 * qh[None, :] + math.sqrt(0.19) * u)
            K[b, h] = kk.to(dt)
            V[b, h] = _low_rank(cap, d, w.rank, g, device).to(dt)
    return K, V, q.to(dt)


def step_query(w: Workload, q_base: torch.Tensor, step: int, seed: int | None = None):
    """q_t = q_base + 0.1 N(0, 1), seeded per step."""
    seed = w.seed if seed is None else seed
    g = gen(q_base.device, seed * 7919 + step + 1)
    noise = _normal(q_base.shape, g, q_base.device)
    return (q_base.float() + 0.1 * noise).to(q_base.dtype)


def drift_direction(w: Workload, K: torch.Tensor, n_prefill: int, seed: int | None = None):
    """Seeded unit direction u per (b, kv-head) and sigma_u of the prefill keys along u."""
    seed = w.seed if seed is None else seed
    g = gen(K.device, seed + 4242)
    B, Hkv, _, d = K.shape
    u = _normal((B, Hkv, d), g, K.device)
    u = u / u.norm(dim=-1, keepdim=True)
    proj = torch.einsum("bhnd,bhd->bhn", K[:, :, :n_prefill].float(), u)
    return u, proj.std(dim=-1)


def drift_inputs(w: Workload, K: torch.Tensor, n_prefill: int, total: int,
                 seed: int | None = None):
    """Keys appended and queries of the drifting decode steps t = 0..total-1.

    K must hold rows [n_prefill, n_prefill + total) drawn by make_cache (the
    prefill's law); the key appended at step t is that row plus the drift mean
    1.5 sigma_u (t+1)/total u. The step's G queries per KV head are fresh draws
    of the same low-rank law plus the same mean. Returns k_new [B, Hkv, total,
    d] and q [total, B, Hq, d] in the workload's dtype.
    """
    seed = w.seed if seed is None else seed
    u, sigma = drift_direction(w, K, n_prefill, seed)
    dev = K.device
    B, Hkv, _, d = K.shape
    G, r = w.G, w.rank
    frac = torch.arange(1, total + 1, device=dev, dtype=torch.float32) / total
    shift = 1.5 * sigma[:, :, None, None] * frac[None, None, :, None] * u[:, :, None, :]
    k_new = (K[:, :, n_prefill:n_prefill + total].float() + shift).to(K.dtype)
    g = gen(dev, seed * 104729 + 1)
    Uq = _normal((B, Hkv, d, r), g, dev) / math.sqrt(r)
    q = _normal((B, Hkv, total * G, r), g, dev) @ Uq.transpose(-1, -2)
    q = q + 0.1 * _normal((B, Hkv, total * G, d), g, dev)
    q = q.view(B, Hkv, total, G, d) + shift[:, :, :, None, :]
    q = q.permute(2, 0, 1, 3, 4).reshape(total, B, Hkv * G, d)
    return k_new, q.to(w.torch_dtype()).contiguous()


def random_tier_plan(n_windows: int, frac=(0.25, 0.5, 0.25), seed: int = 0):
    """Seeded initial tiers of n_windows closed windows: 0 bf16, 1 INT2, 2 evicted."""
    g = gen("cpu", seed)
    perm = torch.randperm(n_windows, generator=g)
    n_bf = int(round(frac[0] * n_windows))
    n_q = int(round(frac[1] * n_windows))
    tiers = torch.full((n_windows,), 2, dtype=torch.int8)
    tiers[perm[:n_bf]] = 0
    tiers[perm[n_bf:n_bf + n_q]] = 1
    return tiers
