"""Drive an ``MkvPool`` through a workload: prefill, tier tagging, demotion
and decode steps.  Only calls the C ABI (through ``MkvPool``) and draws
inputs from ``workloads``; it computes nothing on cache data.

Tier policy (the pages name Recent, Anchor and Stale pages but give no
schedule): the last W pages of a request, including its partial tail page,
are Recent; when a request opens page n, page n - W leaves the window and is
demoted to TQ3, or re-tagged Anchor when it is one (Anchors stay FP8).
"""
from __future__ import annotations

import torch

from .pool import MkvPool
from .workloads import A, R, S, Workload


def pool_sizes(w: Workload, extra_steps: int | None = None):
    """FP8 / TQ3 slot counts needed to hold the workload (prefilled one
    request at a time) plus `extra_steps` decode steps."""
    steps = w.steps if extra_steps is None else extra_steps
    grow = (steps + w.P - 1) // w.P + 1
    npg = [w.npages(r) + grow for r in range(w.n)]
    fp8_steady = sum(min(npg[r], w.windows[r] + len(w.anchors[r]) + 1) for r in range(w.n))
    fp8 = fp8_steady + max(npg) + 2
    tq3 = sum(npg) + 2
    return fp8, tq3, max(npg)


def make_pool(w: Workload, device="cuda", extra_steps: int | None = None, seed: int = 0x5EED, host_only=False,
              max_batch: int | None = None):
    """A pool sized for the workload; max_batch (batch entries of one decode
    plan) defaults to the request count, larger for several query tokens."""
    fp8, tq3, maxp = pool_sizes(w, extra_steps)
    mb = max(w.n, max_batch or w.n)
    return MkvPool(w.num_layers, w.Hq, w.Hkv, w.D, w.P, fp8, tq3, max_seqs=mb, max_pages_per_seq=maxp,
                   max_batch=mb, rotation_seed=seed, device=device, host_only=host_only)


def prefill(pool: MkvPool, w: Workload, device="cuda", keep_raw: bool = False, layers=None):
    """Write every request's initial context into the pool, tag Anchors and
    demote Stale pages.  Returns the raw K/V per (layer, request) on the host
    when keep_raw (small workloads only)."""
    raw = {}
    layers = range(w.num_layers) if layers is None else layers
    for r in range(w.n):
        pool.extend([r], [w.lengths[r]])
        for layer in layers:
            K, V = w.prefill_kv(layer, r, device="cpu" if keep_raw else device)
            if keep_raw:
                raw[(layer, r)] = (K.clone(), V.clone())
            pool.append(layer, [r], [w.lengths[r]], K.to(device).contiguous(), V.to(device).contiguous())
        tiers = w.tiers(r)
        for p, t in enumerate(tiers):
            if t == A:
                pool.set_tier(r, p, 2)
        stale = [p for p, t in enumerate(tiers) if t == S]
        if stale:
            pool.demote([r] * len(stale), stale)
    return raw


class Stepper:
    """Decode steps: extend every request by one token, demote pages that left
    the Recent window, then per layer append the new token and decode."""

    def __init__(self, pool: MkvPool, w: Workload, device="cuda"):
        self.pool, self.w, self.device = pool, w, device
        self.lengths = list(w.lengths)
        self.ids = list(range(w.n))
        self.step_no = 0

    def pre_step(self):
        w = self.w
        ids = self.ids
        self.pool.extend(ids, [1] * len(ids))
        dem_s, dem_p = [], []
        for r in ids:
            self.lengths[r] += 1
            if (self.lengths[r] - 1) % w.P == 0:            # a new page was opened
                npg = (self.lengths[r] + w.P - 1) // w.P
                leaving = npg - 1 - w.windows[r]
                if leaving >= 0:
                    tier, _ = self.pool.page_info(r, leaving)
                    if leaving in w.anchors[r]:
                        if tier == R:
                            self.pool.set_tier(r, leaving, A)     # protected: stays FP8
                    elif tier != S:
                        dem_s.append(r)
                        dem_p.append(leaving)
        if dem_s:
            self.pool.demote(dem_s, dem_p)

    def layer(self, layer: int, k: torch.Tensor, v: torch.Tensor, q: torch.Tensor, out=None, lse=None):
        """Append the step's token and decode, in one library call."""
        return self.pool.append_decode(layer, self.ids, k, v, q, out, lse)

    def layer_separate(self, layer: int, k: torch.Tensor, v: torch.Tensor, q: torch.Tensor, out=None, lse=None):
        """The same through the two separate calls (append, then decode)."""
        self.pool.append(layer, self.ids, [1] * len(self.ids), k, v)
        return self.pool.decode(layer, self.ids, q, out, lse)
