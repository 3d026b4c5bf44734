"""Seeded synthetic workloads for prompt KV-cache compression.

This module only synthesises inputs: the observation-window queries Q_obs,
the prompt keys K and values V, and the per-workload knobs (window, budgets,
mass threshold, channel-pruning ratio).  It contains none of the compression
arithmetic itself; both the CUDA path and the CPU oracle consume the bytes it
produces.

Shapes and distributions stand in for the models the method pages evaluate
(Llama-3-8B / Mistral-7B attention geometry: 32 query heads, 8 KV heads,
head dim 128).  No model weights or datasets are used.

Layouts (all contiguous):
  q  [L][H_q][W][D]   window queries of every query head
  k  [L][H_kv][T][D]  prompt keys
  v  [L][H_kv][T][D]  prompt values
Query head h belongs to KV head h // (H_q / H_kv).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, replace
from typing import List, Optional

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    n_layers: int
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    seq_len: int
    window: int
    dtype: str                      # "f32" or "bf16"
    # budget: either a uniform per-head budget (SnapKV) or a ZigZagKV total
    per_head_budget: Optional[int] = None
    total_budget: Optional[int] = None
    layer_floor: int = 0
    mass_num: int = 9
    mass_den: int = 10
    think_lambda: Optional[float] = None
    # generator knobs
    q_gen: str = "iid"              # "iid" or "mix"
    planted: int = 0                # keys per KV head planted as 3 x mean query
    outlier_channels: int = 0       # key channels per head scaled up
    outlier_scale: float = 8.0
    mix_rows: int = 64              # key rows mixed into each window query
    mix_weight: float = 0.7
    temperature: Optional[tuple] = None   # (lo, hi) log-uniform per layer

    @property
    def group(self) -> int:
        return self.n_q_heads // self.n_kv_heads

    @property
    def prefix_len(self) -> int:
        return self.seq_len - self.window

    def budget_args(self):
        """(total_budget, layer_floor) for the allocation call."""
        if self.total_budget is not None:
            return int(self.total_budget), int(self.layer_floor)
        return int(self.per_head_budget) * self.n_layers, int(self.per_head_budget)

    @property
    def k_max(self) -> int:
        """Row stride of the per-head index buffer: the largest budget one
        layer can receive (every other layer at its floor; the whole prefix at
        most)."""
        total, floor = self.budget_args()
        return int(max(0, min(self.prefix_len, total - (self.n_layers - 1) * floor)))

    @property
    def elt_size(self) -> int:
        return 4 if self.dtype == "f32" else 2

    @property
    def torch_dtype(self):
        return torch.float32 if self.dtype == "f32" else torch.bfloat16

    def scaled(self, **kw) -> "Workload":
        return replace(self, **kw)


# --- the five workloads ---------------------------------------------------

TINY = Workload(
    name="tiny_mha_T1024_D64_f32", n_layers=1, n_q_heads=4, n_kv_heads=4,
    head_dim=64, seq_len=1024, window=32, dtype="f32", per_head_budget=128,
    q_gen="iid", planted=4)

LLAMA3_8B_LAYER = Workload(
    name="llama3_8b_1layer_T16384", n_layers=1, n_q_heads=32, n_kv_heads=8,
    head_dim=128, seq_len=16384, window=128, dtype="bf16", per_head_budget=1024,
    q_gen="mix", outlier_channels=4)

ZIGZAG_32K = Workload(
    name="llama3_8b_zigzag_32L_T32768", n_layers=32, n_q_heads=32, n_kv_heads=8,
    head_dim=128, seq_len=32768, window=128, dtype="bf16",
    total_budget=32 * 2048, layer_floor=256, q_gen="mix", outlier_channels=4,
    temperature=(0.3, 3.0))

THINK_128K = Workload(
    name="llama3_8b_zigzag_think_32L_T131072", n_layers=32, n_q_heads=32,
    n_kv_heads=8, head_dim=128, seq_len=131072, window=128, dtype="bf16",
    total_budget=32 * 4096, layer_floor=512, think_lambda=0.4, q_gen="mix",
    outlier_channels=4)

WORKLOADS = {w.name: w for w in (TINY, LLAMA3_8B_LAYER, ZIGZAG_32K, THINK_128K)}


def ragged_mistral_batch(seed: int, n_prompts: int = 8, lo: int = 4096,
                         hi: int = 65536, ratio: float = 0.2) -> List[Workload]:
    """Eight Mistral-7B-shaped prompts with log-uniform lengths in [lo, hi].

    Each prompt keeps ratio*T prefix tokens per head on average over its 32
    layers (total = 32 * floor(ratio*T)); the per-layer floor is one eighth of
    that mean, the same floor-to-mean ratio as the 32K and 128K workloads.
    """
    g = torch.Generator().manual_seed(seed)
    u = torch.rand(n_prompts, generator=g, dtype=torch.float64)
    lens = torch.floor(torch.exp(math.log(lo) + u * (math.log(hi) - math.log(lo))))
    out = []
    for b, t in enumerate(lens.tolist()):
        t = int(t)
        mean_b = int(math.floor(ratio * t))
        out.append(Workload(
            name=f"mistral7b_ragged_p{b}_T{t}", n_layers=32, n_q_heads=32,
            n_kv_heads=8, head_dim=128, seq_len=t, window=64, dtype="bf16",
            total_budget=32 * mean_b, layer_floor=mean_b // 8, q_gen="mix",
            outlier_channels=4))
    return out


def seed_for(config_index: int, rep: int = 0) -> int:
    return 1000 * config_index + rep


# --- generators -------------------------------------------------------------

def _gen(device, seed):
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def make_inputs(wl: Workload, seed: int, device="cpu", with_v: bool = True):
    """Return dict(q=..., k=..., v=...) as contiguous tensors in wl's dtype.

    iid:  Q, K, V ~ N(0,1); `planted` keys per KV head at distinct seeded
          prefix positions are overwritten with 3 x (mean of that head's
          group window queries).
    mix:  K ~ N(0,1) with `outlier_channels` seeded channels per head scaled
          by `outlier_scale`; V ~ N(0,1).  Per KV head one seeded set of
          `mix_rows` distinct prefix positions R; each window query row is
          mix_weight * sum_r w_r k_r + (1-mix_weight) * eps with w ~ U(0,1)
          normalised to sum 1 and eps ~ N(0,1).  With `temperature`, every
          query of layer l is divided by tau_l, log-uniform in the range.
    Everything is drawn in fp32 and rounded once to the workload dtype.
    """
    L, Hq, Hkv, D, T, W = (wl.n_layers, wl.n_q_heads, wl.n_kv_heads,
                           wl.head_dim, wl.seq_len, wl.window)
    G, P = wl.group, wl.prefix_len
    dt = wl.torch_dtype
    g = _gen(device, seed)
    q = torch.empty((L, Hq, W, D), dtype=dt, device=device)
    k = torch.empty((L, Hkv, T, D), dtype=dt, device=device)
    v = torch.empty((L, Hkv, T, D), dtype=dt, device=device) if with_v else None
    taus = None
    planted = (torch.empty((L, Hkv, wl.planted), dtype=torch.int64, device=device)
               if wl.planted else None)
    if wl.temperature is not None:
        lo, hi = wl.temperature
        u = torch.rand(L, generator=g, device=device, dtype=torch.float64)
        taus = torch.exp(math.log(lo) + u * (math.log(hi) - math.log(lo))).float()
    for l in range(L):
        kl = torch.randn((Hkv, T, D), generator=g, device=device)
        if wl.outlier_channels:
            for h in range(Hkv):
                ch = torch.randperm(D, generator=g, device=device)[: wl.outlier_channels]
                kl[h][:, ch] *= wl.outlier_scale
        k[l].copy_(kl)
        del kl
        if with_v:
            v[l].copy_(torch.randn((Hkv, T, D), generator=g, device=device))
        if wl.q_gen == "iid":
            ql = torch.randn((Hq, W, D), generator=g, device=device)
        else:
            kf = k[l].float()
            ql = torch.empty((Hq, W, D), device=device)
            m = min(wl.mix_rows, P)
            for h in range(Hkv):
                rows = torch.randperm(P, generator=g, device=device)[:m]
                w = torch.rand((G * W, m), generator=g, device=device)
                w = w / w.sum(dim=1, keepdim=True)
                eps = torch.randn((G * W, D), generator=g, device=device)
                mixed = wl.mix_weight * (w @ kf[h][rows]) + (1.0 - wl.mix_weight) * eps
                ql[h * G:(h + 1) * G] = mixed.view(G, W, D)
            del kf
        if taus is not None:
            ql = ql / taus[l]
        if wl.planted:
            qm = ql.view(Hkv, G * W, D).mean(dim=1)          # [Hkv][D]
            for h in range(Hkv):
                pos = torch.randperm(P, generator=g, device=device)[: wl.planted]
                k[l, h, pos] = (3.0 * qm[h]).to(dt)
                planted[l, h] = pos
        q[l].copy_(ql)
    out = dict(q=q, k=k, v=v)
    if taus is not None:
        out["tau"] = taus
    if planted is not None:
        out["planted"] = planted
    return out
