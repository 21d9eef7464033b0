"""Seeded synthetic inputs shaped like the decode workloads MagicPIG is evaluated on.

This module only draws random numbers: it holds no hashing, projection, counting or attention
arithmetic, so that the oracle and the CUDA path can both be fed from it without sharing any of
the method's code.

Geometry follows "MagicPIG: LSH Sampling for Efficient LLM Generation" (background section,
observations on the geometry of attention, items 1-3) and "MagicPIG: don't pick the tallest"
(section 4, "Where the keys live"): cached keys sit in a narrow cone around a stable mean
direction, queries point into the opposite cone, and the first token is an attention sink whose
score stands far above the rest.

Recipe per (sequence, KV head), with u a uniform random unit vector:
  mu        = 8 u                                  (shared offset of the key cone)
  k_i       ~ N(mu, I)                             i = 0..n-1
  q_h       = -4 u + N(0, 0.5^2 I)                 one per query head of the GQA group
  k_0       = mu + 12 qbar/|qbar|                  sink: q.(k_0 - mu) = 12 |q| = 12 sigma,
                                                   qbar the group's mean query
  v_i       ~ N(0, I)
  q_h      *= exp(N(0, s^2))                       only where a workload asks for log-normal
                                                   query norms
  k_i      += sqrt(a) xi_i v,  xi_i ~ N(0, 1)      only where a workload asks for a spread key
                                                   cone (i >= 1): covariance I + a v v^T with
                                                   a = A exp(N(0, s_a^2)) per (sequence, KV
                                                   head) and v = unit(qbar + 0.5 e), e a random
                                                   unit vector: a direction near the group's
                                                   queries, so the sample sizes differ by head
Hyperplanes W ~ N(0, 1) of shape [d, K*L], one matrix for every head and layer of a run (the
shared random projector of the system design section). Workloads stored in bf16 round W to bf16:
at (K, L) = (10, 150) that is the 128 x 1500 x 2 B = 384,000 B (about 400 KB) projector size the
system design section quotes.

Seeds: layer l of workload c draws from SEED_BASE + 1000 c + l; W from SEED_BASE + 1000 c + 999.
"""
from __future__ import annotations

import dataclasses
import math

import torch

SEED_BASE = 20241016


@dataclasses.dataclass(frozen=True)
class Workload:
    """Shape and distribution of one synthetic decode workload."""

    name: str
    index: int            # stable id used in seeds
    B: int                # sequences in the decode batch
    Hq: int               # query heads
    Hkv: int              # key/value heads (GQA: query head h reads KV head h // (Hq // Hkv))
    n: int                # cached tokens per sequence
    d: int                # head dimension
    K: int                # bits per hash table
    L: int                # hash tables
    n_sink: int           # exact-attention sink tokens at the start
    n_local: int          # exact-attention local window at the end
    layers: int = 1
    kv_dtype: torch.dtype = torch.bfloat16
    q_dtype: torch.dtype = torch.bfloat16
    w_dtype: torch.dtype = torch.bfloat16
    mu_norm: float = 8.0
    q_dir: float = 4.0
    q_noise: float = 0.5
    sink_sigmas: float = 12.0
    q_lognormal_sigma: float = 0.0
    key_spread: float = 0.0           # A of the spread key cone (0: isotropic keys)
    key_spread_sigma: float = 0.0     # s_a, the log-normal spread of a between heads

    @property
    def G(self) -> int:
        return self.Hq // self.Hkv

    @property
    def C(self) -> int:
        return self.K * self.L

    def replace(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


WORKLOADS: dict[str, Workload] = {
    # tiny single head, everything fp32, (K, L) = (8, 75)
    "tiny_f32_n4096": Workload(
        "tiny_f32_n4096", 0, B=1, Hq=1, Hkv=1, n=4096, d=128, K=8, L=75, n_sink=4, n_local=64,
        kv_dtype=torch.float32, q_dtype=torch.float32, w_dtype=torch.float32),
    # Llama-3.1-8B-shaped single layer, batch 4, 16K context
    "llama8b_b4_n16k": Workload(
        "llama8b_b4_n16k", 1, B=4, Hq=32, Hkv=8, n=16384, d=128, K=10, L=150, n_sink=4,
        n_local=64),
    # Llama-3.1-8B-shaped, 96K context, batch 1, all 32 layers back to back
    "llama8b_n96k_32layers": Workload(
        "llama8b_n96k_32layers", 2, B=1, Hq=32, Hkv=8, n=98304, d=128, K=10, L=150, n_sink=4,
        n_local=64, layers=32),
    # large-batch decode with log-normal query norms
    "llama8b_b32_n32k": Workload(
        "llama8b_b32_n32k", 3, B=32, Hq=32, Hkv=8, n=32768, d=128, K=10, L=150, n_sink=4,
        n_local=64, q_lognormal_sigma=0.3),
    # as llama8b_b32_n32k, and each head's keys spread along a direction near its queries
    # (covariance I + a v v^T, a = 16 exp(N(0, 0.3^2))): an added variant whose sample sizes
    # differ between heads
    "llama8b_b32_n32k_spread": Workload(
        "llama8b_b32_n32k_spread", 5, B=32, Hq=32, Hkv=8, n=32768, d=128, K=10, L=150, n_sink=4,
        n_local=64, q_lognormal_sigma=0.3, key_spread=16.0, key_spread_sigma=0.3),
    # Llama-3.1-70B-shaped (GQA group 8), 128K context, batch 2, 80 layers
    "llama70b_b2_n128k_80layers": Workload(
        "llama70b_b2_n128k_80layers", 4, B=2, Hq=64, Hkv=8, n=131072, d=128, K=10, L=150,
        n_sink=4, n_local=64, layers=80),
}


def small_workload(name: str = "case", index: int = 100, **kw) -> Workload:
    """A free-form workload for parity and edge-case tests (bf16 unless told otherwise)."""
    base = dict(B=1, Hq=4, Hkv=1, n=4096, d=128, K=10, L=150, n_sink=4, n_local=64)
    base.update(kw)
    return Workload(name, index, **base)


def layer_seed(wl: Workload, layer: int) -> int:
    return SEED_BASE + 1000 * wl.index + layer


def _gen(device, seed: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def make_hyperplanes(wl: Workload, device="cpu") -> torch.Tensor:
    """W ~ N(0, 1), shape [d, K*L], column j = t*K + b is bit b of table t; in wl.w_dtype."""
    g = _gen(device, SEED_BASE + 1000 * wl.index + 999)
    W = torch.randn(wl.d, wl.C, generator=g, device=device, dtype=torch.float32)
    return W.to(wl.w_dtype).contiguous()


def make_layer(wl: Workload, layer: int = 0, device="cpu") -> dict:
    """Keys, values [B, Hkv, n, d] and queries [B, Hq, d] of one layer (see module recipe)."""
    g = _gen(device, layer_seed(wl, layer))
    B, Hq, Hkv, n, d, G = wl.B, wl.Hq, wl.Hkv, wl.n, wl.d, wl.G
    f32 = torch.float32
    u = torch.randn(B, Hkv, d, generator=g, device=device, dtype=f32)
    u = u / u.norm(dim=-1, keepdim=True)
    mu = wl.mu_norm * u
    keys = torch.randn(B, Hkv, n, d, generator=g, device=device, dtype=f32)
    keys += mu[:, :, None, :]
    q = torch.randn(B, Hq, d, generator=g, device=device, dtype=f32) * wl.q_noise
    q -= wl.q_dir * u.repeat_interleave(G, dim=1)
    if wl.q_lognormal_sigma > 0:
        q *= torch.exp(wl.q_lognormal_sigma
                       * torch.randn(B, Hq, 1, generator=g, device=device, dtype=f32))
    qbar = q.view(B, Hkv, G, d).mean(dim=2)
    qbar = qbar / qbar.norm(dim=-1, keepdim=True).clamp_min(1e-30)
    if n > 0:
        keys[:, :, 0, :] = mu + wl.sink_sigmas * qbar
    values = torch.randn(B, Hkv, n, d, generator=g, device=device, dtype=f32)
    if wl.key_spread > 0 and n > 1:
        a = wl.key_spread * torch.exp(
            wl.key_spread_sigma * torch.randn(B, Hkv, 1, 1, generator=g, device=device, dtype=f32))
        e = torch.randn(B, Hkv, d, generator=g, device=device, dtype=f32)
        e = e / e.norm(dim=-1, keepdim=True)
        v = qbar + 0.5 * e
        v = v / v.norm(dim=-1, keepdim=True)
        xi = torch.randn(B, Hkv, n - 1, 1, generator=g, device=device, dtype=f32)
        keys[:, :, 1:, :] += a.sqrt() * xi * v[:, :, None, :]
    return {
        "keys": keys.to(wl.kv_dtype).contiguous(),
        "values": values.to(wl.kv_dtype).contiguous(),
        "q": q.to(wl.q_dtype).contiguous(),
    }


def kv_bytes_per_layer(wl: Workload) -> int:
    es = torch.empty((), dtype=wl.kv_dtype).element_size()
    return 2 * wl.B * wl.Hkv * wl.n * wl.d * es


def describe(wl: Workload) -> str:
    return (f"{wl.name}: B={wl.B} Hq={wl.Hq} Hkv={wl.Hkv} n={wl.n} d={wl.d} (K,L)=({wl.K},{wl.L})"
            f" T={wl.n_sink}+{wl.n_local} layers={wl.layers} kv={wl.kv_dtype} "
            f"KV/layer={kv_bytes_per_layer(wl) / 2**20:.1f} MiB, sink +{wl.sink_sigmas:g} sigma,"
            f" |mu|={wl.mu_norm:g}, exp(q) sigma={wl.q_lognormal_sigma:g}"
            f" ({math.prod([wl.B, wl.Hq, wl.layers])} query rows per step)")
