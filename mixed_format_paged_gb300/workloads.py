"""Seeded synthetic workloads (shapes, tier layouts, K/V/q values).

This module only draws inputs; it contains none of the method's arithmetic,
so both the CUDA path (tests, bench) and the oracle may consume what it
produces.  The five workloads follow the configurations the library is
measured on (head shape of the Qwen3.6-27B profiles the Minima-KV pages
report: 24 query heads, 4 kv heads, d = 256, 16 full-attention layers;
the canary's two 59,008-token requests).  Recipes:

* K rows: N(0,1) plus 4 outlier channels per kv head offset by +-8 (seeded
  channel and sign; workload "cfg1" uses the same 4 channels for every head,
  offset +8).  V rows: N(0,1), or iid Student-t with 3 degrees of freedom
  ("cfg4", heavy-tailed value rows).  q: N(0,1), fp32 in "cfg1", bf16
  elsewhere; K/V fp32 in "cfg1", bf16 elsewhere.
* Tiers: the last W pages (including a partial tail page) are Recent;
  Anchors are drawn uniformly without replacement from the older pages
  (round(fraction * pages)), plus page 0 where the workload says so; every
  other page is Stale (TQ3).  Anchor selection by relevance is not defined on
  the pages, hence the seeded draw.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np
import torch

R, A, S = 1, 2, 3   # tier tags (mkv_tier values)


@dataclass
class Workload:
    name: str
    num_layers: int
    Hq: int
    Hkv: int
    D: int
    P: int
    lengths: list
    windows: list            # Recent window W per request (pages)
    anchors: list            # set of anchor page indices per request
    steps: int               # decode steps in a timed run
    kv_dtype: torch.dtype
    q_dtype: torch.dtype
    v_student_t: bool
    seed: int
    outlier_ch: np.ndarray = field(default=None)    # [Hkv, 4] channel ids
    outlier_off: np.ndarray = field(default=None)   # [Hkv, 4] offsets
    description: str = ""

    @property
    def n(self) -> int:
        return len(self.lengths)

    def npages(self, r: int, length: int | None = None) -> int:
        ln = self.lengths[r] if length is None else length
        return (ln + self.P - 1) // self.P

    def tier(self, r: int, page: int, length: int | None = None) -> int:
        npg = self.npages(r, length)
        if page >= npg - self.windows[r]:
            return R
        if page in self.anchors[r]:
            return A
        return S

    def tiers(self, r: int, length: int | None = None) -> list:
        return [self.tier(r, p, length) for p in range(self.npages(r, length))]

    def subset(self, idx) -> "Workload":
        """The same workload restricted to requests `idx` (in that order): a
        reduced-size case of the same shape, e.g. for a profiler capture."""
        idx = [int(i) for i in idx]
        w = Workload(f"{self.name}[{','.join(map(str, idx))}]", self.num_layers, self.Hq, self.Hkv, self.D, self.P,
                     [self.lengths[i] for i in idx], [self.windows[i] for i in idx],
                     [set(self.anchors[i]) for i in idx], self.steps, self.kv_dtype, self.q_dtype, self.v_student_t,
                     self.seed, self.outlier_ch, self.outlier_off,
                     f"requests {idx} of: {self.description}")
        return w

    def layout_classes(self) -> dict:
        """Request indices by tier layout: 'all_fp8' (every page Recent or
        Anchor), 'mostly_tq3' (at least 98 % of pages TQ3) and 'mixed'."""
        out = {"all_fp8": [], "mostly_tq3": [], "mixed": []}
        for r in range(self.n):
            t = self.tiers(r)
            stale = sum(1 for x in t if x == S)
            if stale == 0:
                out["all_fp8"].append(r)
            elif stale >= 0.98 * len(t):
                out["mostly_tq3"].append(r)
            else:
                out["mixed"].append(r)
        return out

    # ------------------------------------------------------------------ data
    def _gen(self, device, *key) -> torch.Generator:
        g = torch.Generator(device=device)
        h = self.seed
        for k in key:
            h = (h * 1000003 + int(k) + 0x9E3779B1) % (2 ** 63)
        g.manual_seed(h)
        return g

    def _kv(self, n_tok: int, g: torch.Generator, device):
        K = torch.randn((n_tok, self.Hkv, self.D), generator=g, device=device, dtype=torch.float32)
        ch = torch.as_tensor(self.outlier_ch, device=device, dtype=torch.long)
        off = torch.as_tensor(self.outlier_off, device=device, dtype=torch.float32)
        for h in range(self.Hkv):
            K[:, h, ch[h]] += off[h]
        if self.v_student_t:
            z = torch.randn((n_tok, self.Hkv, self.D), generator=g, device=device, dtype=torch.float32)
            c = torch.randn((3, n_tok, self.Hkv, self.D), generator=g, device=device, dtype=torch.float32)
            V = z / torch.sqrt((c * c).sum(0) / 3.0)
        else:
            V = torch.randn((n_tok, self.Hkv, self.D), generator=g, device=device, dtype=torch.float32)
        return K.to(self.kv_dtype), V.to(self.kv_dtype)

    def prefill_kv(self, layer: int, r: int, device="cpu"):
        """K, V [lengths[r], Hkv, D] of request r's initial context in `layer`."""
        return self._kv(self.lengths[r], self._gen(device, 1, layer, r), device)

    def step_kv(self, layer: int, step: int, device="cpu"):
        """K, V [n, Hkv, D]: the token each request appends at decode `step`."""
        return self._kv(self.n, self._gen(device, 2, layer, step), device)

    def query(self, layer: int, step: int, device="cpu") -> torch.Tensor:
        g = self._gen(device, 3, layer, step)
        return torch.randn((self.n, self.Hq, self.D), generator=g, device=device,
                           dtype=torch.float32).to(self.q_dtype)


def _outliers(rng, Hkv, D, same_for_all_heads):
    if same_for_all_heads:
        ch = np.sort(rng.choice(D, 4, replace=False))
        return np.tile(ch, (Hkv, 1)), np.full((Hkv, 4), 8.0)
    ch = np.stack([np.sort(rng.choice(D, 4, replace=False)) for _ in range(Hkv)])
    off = 8.0 * rng.choice([-1.0, 1.0], size=(Hkv, 4))
    return ch, off


def _draw_anchors(rng, npages, W, frac, page0):
    older = [p for p in range(npages - W) if not (page0 and p == 0)]
    k = int(round(frac * npages))
    k = min(k, len(older))
    chosen = set(int(x) for x in rng.choice(older, size=k, replace=False)) if k > 0 else set()
    if page0 and npages - W > 0:
        chosen.add(0)
    return chosen


def make(name: str) -> Workload:
    """Workloads 'cfg1' .. 'cfg5' (see the module docstring)."""
    idx = int(name.replace("cfg", ""))
    seed = 1000 + idx
    rng = np.random.default_rng(seed)
    if idx == 1:
        ch, off = _outliers(rng, 4, 256, True)
        return Workload("cfg1", 1, 24, 4, 256, 64, [4096], [8], [{0}], 1, torch.float32, torch.float32, False,
                        seed, ch, off, "1 request x 4,096 tokens, 1 layer, p=64; page 0 Anchor, last 8 Recent, "
                                       "55 TQ3; fp32 q/K/V, K +8 on 4 shared channels")
    if idx == 2:
        ch, off = _outliers(rng, 4, 256, False)
        lengths = [int(x) for x in rng.integers(8192, 32769, size=8)]
        anchors = [_draw_anchors(rng, (L + 63) // 64, 8, 0.02, True) for L in lengths]
        return Workload("cfg2", 16, 24, 4, 256, 64, lengths, [8] * 8, anchors, 64, torch.bfloat16, torch.bfloat16,
                        False, seed, ch, off, "8 requests, U[8192, 32768] tokens, 16 layers, p=64; W=8, page 0 + "
                                              "2% random Anchors; bf16")
    if idx == 3:
        ch, off = _outliers(rng, 4, 256, False)
        lengths = [59008, 59008]
        anchors = [_draw_anchors(rng, 922, 16, 0.03, False) for _ in lengths]
        return Workload("cfg3", 16, 24, 4, 256, 64, lengths, [16, 16], anchors, 256, torch.bfloat16,
                        torch.bfloat16, False, seed, ch, off,
                        "2 x 59,008 tokens, 16 layers, p=64; W=16, 3% random Anchors; 256 decode steps with "
                        "append + demotion")
    if idx == 4:
        ch, off = _outliers(rng, 4, 256, False)
        lengths = [int(math.floor(math.exp(x))) for x in rng.uniform(math.log(1024), math.log(65536), size=64)]
        windows, anchors = [], []
        for L in lengths:
            npg = (L + 63) // 64
            u = rng.uniform()
            if u < 0.125:
                windows.append(npg)
                anchors.append(set())
            elif u < 0.25 and npg >= 50:
                windows.append(1)
                anchors.append(set())
            else:
                windows.append(8)
                anchors.append(_draw_anchors(rng, npg, 8, 0.05, False))
        return Workload("cfg4", 16, 24, 4, 256, 64, lengths, windows, anchors, 64, torch.bfloat16, torch.bfloat16,
                        True, seed, ch, off, "64 ragged requests, log-uniform [1024, 65536] tokens, 16 layers, "
                                             "p=64; mixed layouts; Student-t(3) V rows")
    if idx == 5:
        ch, off = _outliers(rng, 4, 256, False)
        # staggered phases: request i sits i*8 tokens before a page boundary
        lengths = [131072 - 8 * i for i in range(16)]
        anchors = [_draw_anchors(rng, (L + 127) // 128, 8, 0.01, False) for L in lengths]
        return Workload("cfg5", 16, 24, 4, 256, 128, lengths, [8] * 16, anchors, 32, torch.bfloat16,
                        torch.bfloat16, False, seed, ch, off,
                        "16 x ~131,072 tokens (staggered), 16 layers, p=128; W=8, 1% Anchors; continuous append")
    raise ValueError(name)
