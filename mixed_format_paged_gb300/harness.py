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


class RelevanceAnchors:
    """Relevance-based Anchor protection: which FP8 pages stay FP8 when they
    leave the Recent window.  The pages protect Anchor pages by "age and
    relevance" (insight.aitobox.com post, "执行摘要") and define neither; this
    policy is the library's own design.

    Age: the last W pages of a request are Recent (as in Stepper).
    Relevance: `observe(mass)` folds a decode step's attention mass per page
    (MkvPool.relevance, i.e. mkv_page_relevance) into a moving average per
    page, rho <- (1 - beta) rho + beta mass.  When page j leaves the Recent
    window (`decide`), with `older` the request's pages older than the window
    and budget = max(1, ceil(frac * older)) Anchors per request:
      * room in the budget: j becomes an Anchor if rho_j * older >= kappa,
        i.e. it draws at least kappa times an even share of the weight;
      * budget full: j replaces the weakest Anchor a if rho_j > (1 +
        hysteresis) rho_a and rho_j * older >= kappa; a is then released
        (back to an ordinary FP8 page, then demoted to TQ3);
      * otherwise j is demoted to TQ3.
    Ties go to the older page.  `decide` only returns actions; `apply` makes
    them through the C ABI (mkv_set_tier, mkv_demote_pages)."""

    def __init__(self, frac: float = 0.05, kappa: float = 2.0, beta: float = 0.25, hysteresis: float = 0.25):
        self.frac, self.kappa, self.beta, self.hysteresis = frac, kappa, beta, hysteresis
        self.rho = {}                     # (request, page) -> moving average of the mass
        self.anchors = {}                 # request -> set of Anchor pages chosen by the policy

    def observe(self, seq_ids, mass, npages):
        """mass: [n, >= max pages] (host array or tensor); npages: page count per request."""
        import numpy as np
        m = mass.detach().float().cpu().numpy() if hasattr(mass, "detach") else np.asarray(mass, dtype=np.float64)
        for b, r in enumerate(seq_ids):
            for j in range(int(npages[b])):
                key = (r, j)
                self.rho[key] = (1.0 - self.beta) * self.rho.get(key, 0.0) + self.beta * float(m[b, j])

    def decide(self, r: int, leaving: int, older: int):
        """Actions for page `leaving` of request r as it leaves the Recent
        window; `older` = the request's pages older than the window after
        this one left.  Returns a list of ("anchor", page), ("demote", page)
        and ("release", page)."""
        import math
        held = self.anchors.setdefault(r, set())
        budget = max(1, math.ceil(self.frac * older))
        rho = self.rho.get((r, leaving), 0.0)
        strong = rho * older >= self.kappa
        if strong and len(held) < budget:
            held.add(leaving)
            return [("anchor", leaving)]
        if strong and held:
            weakest = min(held, key=lambda a: (self.rho.get((r, a), 0.0), -a))
            if rho > (1.0 + self.hysteresis) * self.rho.get((r, weakest), 0.0):
                held.discard(weakest)
                held.add(leaving)
                return [("release", weakest), ("anchor", leaving)]
        return [("demote", leaving)]

    def apply(self, pool, r: int, actions):
        demote = []
        for act, page in actions:
            if act == "anchor":
                pool.set_tier(r, page, A)
            elif act == "release":
                pool.set_tier(r, page, R)      # an ordinary FP8 page again, then demoted
                demote.append(page)
            else:
                demote.append(page)
        if demote:
            pool.demote([r] * len(demote), demote)


class RelevanceStepper(Stepper):
    """Stepper whose Anchors come from RelevanceAnchors instead of the
    workload's seeded draw: at each page roll-over the leaving page is
    anchored, demoted, or swapped with the weakest Anchor; after the decode
    of `layer` (every `every` steps) the step's attention mass per page is
    observed."""

    def __init__(self, pool: MkvPool, w: Workload, policy: RelevanceAnchors, layer: int = 0, every: int = 1,
                 device="cuda"):
        super().__init__(pool, w, device)
        self.policy, self.obs_layer, self.every = policy, layer, every

    def pre_step(self):
        w = self.w
        ids = self.ids
        self.pool.extend(ids, [1] * len(ids))
        for r in ids:
            self.lengths[r] += 1
            if (self.lengths[r] - 1) % w.P == 0:            # a new page was opened
                npg = (self.lengths[r] + w.P - 1) // w.P
                leaving = npg - 1 - w.windows[r]
                if leaving >= 0:
                    tier, _ = self.pool.page_info(r, leaving)
                    if tier == R:
                        self.policy.apply(self.pool, r, self.policy.decide(r, leaving, leaving + 1))
        self.step_no += 1

    def layer(self, layer: int, k: torch.Tensor, v: torch.Tensor, q: torch.Tensor, out=None, lse=None):
        out, lse = super().layer(layer, k, v, q, out, lse)
        if layer == self.obs_layer and self.step_no % self.every == 0:
            mass = self.pool.relevance(layer, self.ids, q, lse)
            self.policy.observe(self.ids, mass, [self.pool.seq_info(r)[1] for r in self.ids])
        return out, lse
