"""CPU tests of the C-ABI library: it loads, exports every symbol the header
declares, and its host logic (pool bookkeeping, tier transitions, errors,
decode planning, accounting) behaves as specified.  No GPU work: pools are
created with MKV_POOL_HOST_ONLY."""
import ctypes
import os
import re
import subprocess

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="session")
def mkv():
    lib_path = os.path.join(ROOT, "mixed_format_paged_gb300", "libmkv.so")
    if not os.path.exists(lib_path):
        from mixed_format_paged_gb300 import build as b
        b.build()
    import mixed_format_paged_gb300 as m
    return m


def _declared_symbols():
    src = open(os.path.join(ROOT, "include", "mkv.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(mkv_[a-z0-9_]+)\s*\(", src)))


def test_library_exports_every_declared_symbol(mkv):
    declared = _declared_symbols()
    assert len(declared) >= 19
    lib = mkv.binding.lib()
    for name in declared:
        assert hasattr(lib, name), name
    out = subprocess.run(["nm", "-D", "--defined-only", mkv.binding.LIB_PATH], capture_output=True, text=True).stdout
    exported = set(re.findall(r"\bT (mkv_[a-z0-9_]+)", out))
    assert set(declared) <= exported
    assert set(mkv.binding.EXPORTED) == set(declared)


def test_codebook_matches_oracle(mkv):
    from oracle.codebook import tq3_codebook
    lv, th = mkv.mkv_tq3_codebook()
    L, T = tq3_codebook()
    assert np.array_equal(np.array(lv, dtype=np.float64), L)
    assert np.array_equal(np.array(th, dtype=np.float64), T)


def _host_pool(mkv, **kw):
    args = dict(num_layers=2, num_q_heads=24, num_kv_heads=4, head_dim=256, page_size=64, fp8_slots=12,
                tq3_slots=6, max_seqs=4, max_pages_per_seq=16, max_batch=4, rotation_seed=99)
    args.update(kw)
    return mkv.MkvPool(host_only=True, **args)


def test_rotation_signs_match_oracle(mkv):
    from oracle.rotation import rotation_signs
    for seed in (0, 99, 2 ** 63 + 5):
        p = _host_pool(mkv, rotation_seed=seed)
        assert np.array_equal(np.array(p.rotation_signs(), dtype=np.float64), rotation_signs(seed, 256))


def test_required_bytes_closed_form(mkv):
    cfg = mkv.PoolConfig(16, 24, 4, 256, 64, 100, 300, 8, 600, 8, 0, 0, 1)
    nbytes = mkv.mkv_pool_required_bytes(cfg)
    arenas = 16 * 100 * 132096 + 16 * 300 * 50176
    assert arenas <= nbytes <= arenas + 64 * 2 ** 20
    # no dense shadow: the non-arena part does not grow with context length
    cfg2 = mkv.PoolConfig(16, 24, 4, 256, 64, 100, 300, 8, 600, 8, 0, 0, 1)
    cfg2.fp8_slots, cfg2.tq3_slots = 1000, 3000
    extra1 = nbytes - arenas
    extra2 = mkv.mkv_pool_required_bytes(cfg2) - (16 * 1000 * 132096 + 16 * 3000 * 50176)
    assert abs(extra1 - extra2) < 512


def test_config_validation(mkv):
    bad = [dict(head_dim=128), dict(page_size=32), dict(num_q_heads=25), dict(num_q_heads=72)]
    for b in bad:
        with pytest.raises(mkv.MkvError) as e:
            _host_pool(mkv, **b)
        assert e.value.status in (1, 2)


def test_extend_all_or_nothing_and_release(mkv):
    p = _host_pool(mkv)
    p.extend([0, 1], [64 * 5, 64 * 4 + 1])           # 5 + 5 pages = 10 of 12 FP8 slots
    assert p.seq_info(0) == (320, 5) and p.seq_info(1) == (257, 5)
    with pytest.raises(mkv.MkvError) as e:
        p.extend([2, 3], [64, 64 * 2])               # needs 3 slots, 2 free
    assert e.value.status == 3
    assert p.seq_info(2) == (0, 0) and p.seq_info(3) == (0, 0)
    with pytest.raises(mkv.MkvError):
        p.extend([0, 0], [1, 1])                     # repeated id
    with pytest.raises(mkv.MkvError):
        p.extend([7], [1])                           # bad id
    with pytest.raises(mkv.MkvError):
        p.extend([2], [64 * 17])                     # beyond max_pages_per_seq
    st = p.stats()
    assert st.fp8_slots_free == 2 and st.recent_pages == 10
    p.release(0)
    assert p.seq_info(0) == (0, 0) and p.stats().fp8_slots_free == 7


def test_tier_transitions(mkv):
    p = _host_pool(mkv)
    p.extend([0], [64 * 6 + 10])                     # 7 pages, tail partial
    p.set_tier(0, 0, 2)
    assert p.page_info(0, 0)[0] == 2
    with pytest.raises(mkv.MkvError) as e:
        p.demote([0], [0])                           # Anchor
    assert e.value.status == 4
    with pytest.raises(mkv.MkvError) as e:
        p.demote([0], [6])                           # partial tail page
    assert e.value.status == 4
    with pytest.raises(mkv.MkvError) as e:
        p.demote([0, 0], [2, 2])                     # listed twice
    assert e.value.status == 4
    with pytest.raises(mkv.MkvError) as e:
        p.set_tier(0, 1, 3)                          # STALE only through demotion
    assert e.value.status == 4
    free_fp8 = p.stats().fp8_slots_free
    p.demote([0, 0, 0], [1, 2, 3])
    st = p.stats()
    assert st.stale_pages == 3 and st.fp8_slots_free == free_fp8 + 3 and st.tq3_slots_free == 3
    with pytest.raises(mkv.MkvError) as e:
        p.demote([0], [2])                           # already TQ3
    assert e.value.status == 4
    with pytest.raises(mkv.MkvError) as e:
        p.set_tier(0, 2, 2)                          # TQ3 page cannot become Anchor
    assert e.value.status == 4
    # OUT_OF_PAGES is all-or-nothing: 3 TQ3 slots left, ask for 4
    p.set_tier(0, 0, 1)
    with pytest.raises(mkv.MkvError) as e:
        p.demote([0, 0, 0, 0], [0, 4, 5, 6 - 1])
    assert e.value.status in (3, 4)
    assert p.stats().stale_pages == 3
    # appending into a TQ3 page is refused
    with pytest.raises(mkv.MkvError) as e:
        p.append(0, [0], [64 * 6 + 10], _FakeTensor(), _FakeTensor())
    assert e.value.status in (1, 4)
    p.release(0)
    st = p.stats()
    assert st.tq3_slots_free == 6 and st.fp8_slots_free == 12


class _FakeTensor:
    """Stands in for a device tensor in host-only calls (never dereferenced)."""
    dtype = None

    def __init__(self):
        import torch
        self.dtype = torch.float32

    def is_contiguous(self):
        return True

    def data_ptr(self):
        return 0x1000


def test_stats_accounting(mkv):
    from oracle.accounting import bytes_per_token_layer
    p = _host_pool(mkv, num_layers=16, fp8_slots=20, tq3_slots=20)
    p.extend([0], [64 * 10])
    p.demote([0] * 6, list(range(6)))
    st = p.stats()
    fp8_tok, tq3_tok = 4 * 64, 6 * 64
    exp = 16 * (fp8_tok * bytes_per_token_layer("fp8") + tq3_tok * bytes_per_token_layer("tq3"))
    assert st.fp8_bytes + st.tq3_bytes == exp
    assert abs(st.kv_bytes_per_live_token - exp / 640) < 1e-9


def _check_plan_covers(mkv, pool, ids, lengths, tiers_of):
    plan = pool.plan(ids)
    H = 4
    for b, r in enumerate(ids):
        tiers = tiers_of(r)
        fp8_pages = [i for i, t in enumerate(tiers) if t != 3]
        tq3_pages = [i for i, t in enumerate(tiers) if t == 3]
        for kvh in range(H):
            mine = [c for c in plan if c[0] == b and c[1] == kvh]
            f = sorted((c[3], c[4]) for c in mine if c[2] == 1)
            t = sorted((c[3], c[4]) for c in mine if c[2] == 3)
            # chunk entry ranges cover each tier's page list in order; a page
            # may be cut between two consecutive chunks (block granularity)
            for ranges, pages in ((f, fp8_pages), (t, tq3_pages)):
                if not pages:
                    assert not ranges
                    continue
                pos = [a for a, _ in ranges]
                assert pos == sorted(pos)
                assert all(n >= 1 for _, n in ranges)
                for (a, n), (a2, _) in zip(ranges, ranges[1:]):
                    assert a2 in (a + n - 1, a + n)
                first, (la, ln) = ranges[0][0], ranges[-1]
                assert la + ln - first == len(pages)
            assert sum(c[5] for c in mine) == lengths[b]
    return plan


def test_plan_covers_every_page_once(mkv):
    from mixed_format_paged_gb300 import workloads
    from mixed_format_paged_gb300.harness import make_pool
    for name in ("cfg1", "cfg2", "cfg4"):
        w = workloads.make(name)
        w.num_layers = 1
        pool = make_pool(w, host_only=True, extra_steps=0)
        for r in range(w.n):
            pool.extend([r], [w.lengths[r]])
            tiers = w.tiers(r)
            for pg, t in enumerate(tiers):
                if t == 2:
                    pool.set_tier(r, pg, 2)
            stale = [pg for pg, t in enumerate(tiers) if t == 3]
            if stale:
                pool.demote([r] * len(stale), stale)
        ids = list(range(w.n))
        plan = _check_plan_covers(mkv, pool, ids, w.lengths, w.tiers)
        # balance: a host-only pool plans for up to 152 CTAs (24 blocks each at
        # least); no chunk is larger than
        # one CTA's share of the estimated work (blocks of 32 TQ3 / 16 FP8
        # tokens with a fixed cost each, and a fixed cost per chunk) plus one
        # warp-round of blocks; there are at most a few chunks per CTA
        def cost(c):
            bt, per_tok = (32, 1.0) if c[2] == 3 else (16, 1.45)
            return c[5] * per_tok + 8.0 * -(-c[5] // bt) + 630.0
        nblk = sum(-(-c[5] // (32 if c[2] == 3 else 16)) for c in plan)
        share = sum(cost(c) for c in plan) / max(1, min(152, nblk // 24))
        assert max(cost(c) for c in plan) <= share + 12 * 40.0
        assert len(plan) <= w.n * 4 * 2 + 4 * 1024


def test_decode_argument_errors(mkv):
    p = _host_pool(mkv)
    p.extend([0], [100])
    q = _FakeTensor()
    with pytest.raises(mkv.MkvError):
        mkv.mkv_decode_attention(p.handle, 0, [1], q, 0, q, q)        # empty sequence
    with pytest.raises(mkv.MkvError):
        mkv.mkv_decode_attention(p.handle, 5, [0], q, 0, q, q)        # bad layer
    with pytest.raises(mkv.MkvError):
        mkv.mkv_decode_attention(p.handle, 0, [0, 0], q, 0, q, q)     # repeated id
    with pytest.raises(mkv.MkvError):
        mkv.mkv_decode_attention(p.handle, 0, [0], None, 0, q, q)     # NULL q
    mkv.mkv_decode_attention(p.handle, 0, [0], q, 0, q, q)            # host-only: validates, no launch


def test_decode_multi_argument_errors(mkv):
    p = _host_pool(mkv)                                # P = 64, max_batch 4
    p.extend([0, 1], [64 * 3 + 2, 40])
    p.demote([0], [2])                                 # page 2 TQ3, tail page 3 holds 2 tokens
    q = _FakeTensor()
    call = lambda ids, nq: mkv.mkv_decode_attention_multi(p.handle, 0, ids, nq, q, 0, q, q)
    call([0, 1], 2)                                    # host-only: validates and plans, no launch
    call([1], 4)
    for ids, nq in (([0], 0), ([0, 1], 3), ([1], 41), ([1], 5)):   # nq < 1; 2 x 3 and 5 > max_batch
        with pytest.raises(mkv.MkvError) as e:
            call(ids, nq)
        assert e.value.status == 1
    with pytest.raises(mkv.MkvError) as e:
        call([0], 3)                                   # the first query token sits in TQ3 page 2
    assert e.value.status == 4


def test_selftest_wait_timeout_arguments(mkv):
    p = _host_pool(mkv)
    for bad in (0, -5, 4_000_000_001):
        with pytest.raises(mkv.MkvError) as e:
            p.selftest_wait_timeout(bad)
        assert e.value.status == 1
    with pytest.raises(mkv.MkvError) as e:
        p.selftest_wait_timeout(1000)                  # host-only pool: no device error word
    assert e.value.status == 2


def _blocks_of(layouts, P, H=4):
    """The planner's work units for requests given as (tokens, tiers per page):
    per (request, kv head, tier) group, TQ3 before FP8, blocks of 32 TQ3 / 16
    FP8 tokens page by page, each with its integer cost: tokens x (20 TQ3 |
    29 FP8) + 160.  Returns [(group key, [block costs])] in plan order."""
    groups = []
    for b, (n, tiers) in enumerate(layouts):
        nv = [min(P, n - i * P) for i in range(len(tiers))]
        for kvh in range(H):
            for fmt in (3, 1):
                pages = [nv[i] for i, t in enumerate(tiers) if (t == 3) == (fmt == 3)]
                if not pages:
                    continue
                bt, rate = (32, 20) if fmt == 3 else (16, 29)
                bpp = P // bt
                nblk = (len(pages) - 1) * bpp + -(-pages[-1] // bt)
                groups.append(((b, kvh, fmt), [max(0, min(bt, pages[k // bpp] - (k % bpp) * bt)) * rate + 160
                                              for k in range(nblk)]))
    return groups


PIECE = 63000


def _piece_cost(costs):
    """A piece of blocks with these costs, in the planner's model: rounds of
    12 blocks from the piece's first, each costing its slowest block x
    (24 + 3 n) for n blocks, plus 63000 for the piece."""
    return PIECE + sum(max(costs[i:i + 12]) * (24 + 3 * len(costs[i:i + 12])) for i in range(0, len(costs), 12))


def _plan_cta_costs(plan, groups):
    cost = dict(groups)
    ctas = {}
    for b, kvh, tier, _, _, _, cta, blk0, nblk in plan:
        ctas[cta] = ctas.get(cta, 0) + _piece_cost(cost[(b, kvh, tier)][blk0:blk0 + nblk])
    return ctas


def test_plan_minimises_the_largest_cta(mkv):
    """The split is contiguous over the block sequence and its largest CTA
    cost equals the optimum of an exhaustive dynamic programme over every
    cut point (any block), in the planner's integer cost model."""
    P = 64
    layouts = [(64 * 30 + 17, [2] + [3] * 21 + [1] * 9), (64 * 12, [3] * 9 + [1] * 3),
               (64 * 5 + 1, [1] * 6), (64 * 18 + 40, [2, 3, 3, 2] + [3] * 11 + [1] * 4)]
    p = _host_pool(mkv, num_layers=1, fp8_slots=64, tq3_slots=64, max_seqs=4, max_pages_per_seq=40)
    for r, (n, tiers) in enumerate(layouts):
        p.extend([r], [n])
        for pg, t in enumerate(tiers):
            if t == 2:
                p.set_tier(r, pg, 2)
        stale = [pg for pg, t in enumerate(tiers) if t == 3]
        p.demote([r] * len(stale), stale)
    plan = p.plan(list(range(len(layouts))))
    groups = _blocks_of(layouts, P)
    first = {}
    blocks = []                                        # (group key, block cost) in plan order
    for key, costs in groups:
        first[key] = len(blocks)
        blocks += [(key, c) for c in costs]
    # the split as block ranges, CTA by CTA, contiguous and covering every block once
    seq = sorted((cta, first[(b, kvh, tier)] + blk0, nblk) for b, kvh, tier, _, _, _, cta, blk0, nblk in plan)
    assert [c for c, _, _ in seq] == sorted(c for c, _, _ in seq)
    assert seq[0][1] == 0 and seq[-1][1] + seq[-1][2] == len(blocks)
    assert all(a[1] + a[2] == b[1] for a, b in zip(seq, seq[1:])), "CTAs hold contiguous runs of blocks"
    assert any(blk0 % 12 for *_, blk0, _ in plan), "cuts are not held to round boundaries"
    got = max(_plan_cta_costs(plan, groups).values())
    # exhaustive optimum over all cut points: C[i, j] = cost of blocks i..j-1
    # as one CTA, f_k[j] = min_i max(f_{k-1}[i], C[i, j])
    R = len(blocks)
    C = np.full((R + 1, R + 1), np.inf)
    for i in range(R):
        acc, start, key = 0, i, blocks[i][0]
        for j in range(i, R):
            if blocks[j][0] != key:                    # a new piece
                acc += _piece_cost([c for _, c in blocks[start:j]])
                start, key = j, blocks[j][0]
            C[i, j + 1] = acc + _piece_cost([c for _, c in blocks[start:j + 1]])
    kmax = max(1, min(152, R // 24))
    f = C[0].copy()
    best = f[R]
    for _ in range(kmax - 1):
        f = np.min(np.maximum(f[:, None], C), axis=0)
        best = min(best, f[R])
    assert len({c for *_, c, _, _ in plan}) <= kmax
    assert got == best, (got, best)


def test_multi_query_plan_covers_each_prefix(mkv):
    """mkv_plan_decode_multi: query tokens go in pairs; batch entry
    b * ceil(nq / 2) + j reads request b up to its query token
    min(2j + 1, nq - 1), per kv head and tier exactly once."""
    P = 64
    layouts = [(64 * 9 + 3, [2, 3, 3, 3, 3, 1, 1, 1, 1, 1]), (64 * 4, [3, 3, 1, 1]), (5, [1])]
    p = _host_pool(mkv, num_layers=1, fp8_slots=64, tq3_slots=64, max_seqs=16, max_batch=16, max_pages_per_seq=40)
    for r, (n, tiers) in enumerate(layouts):
        p.extend([r], [n])
        for pg, t in enumerate(tiers):
            if t == 2:
                p.set_tier(r, pg, 2)
        stale = [pg for pg, t in enumerate(tiers) if t == 3]
        if stale:
            p.demote([r] * len(stale), stale)
    nq = 5
    npair = (nq + 1) // 2
    plan = p.plan([0, 1, 2], nq=nq)
    assert {c[0] for c in plan} == set(range(3 * npair))
    for b, (n, tiers) in enumerate(layouts):
        for j in range(npair):
            visible = n - nq + 1 + min(2 * j + 1, nq - 1)
            tq3 = sum(min(P, visible - pg * P) for pg, t in enumerate(tiers) if t == 3 and pg * P < visible)
            fp8 = visible - tq3
            for kvh in range(4):
                mine = [c for c in plan if c[0] == b * npair + j and c[1] == kvh]
                assert sum(c[5] for c in mine if c[2] == 3) == tq3
                assert sum(c[5] for c in mine if c[2] == 1) == fp8
    # nq = 1 is the decode plan
    assert p.plan([0, 1, 2], nq=1) == p.plan([0, 1, 2])
    with pytest.raises(mkv.MkvError):
        p.plan([0, 1, 2], nq=6)                        # request 2 holds 5 tokens


def test_paired_plan_fits_a_full_batch(mkv):
    """A paired piece writes two partial states: a batch at max_batch with an
    odd nq (every request's FP8 and TQ3 groups in every kv head) plans
    without running out of partial-state room."""
    n, nq = 100, 3
    p = _host_pool(mkv, num_layers=1, fp8_slots=3 * n, tq3_slots=n, max_seqs=n * nq, max_batch=n * nq,
                   max_pages_per_seq=4)
    ids = list(range(n))
    for r in ids:
        p.extend([r], [64 * 2 + 7 + r % 5])
    p.demote(ids, [0] * n)
    plan = p.plan(ids, nq=nq)
    npair = (nq + 1) // 2
    assert {c[0] for c in plan} == set(range(n * npair))
    assert sum(1 for c in plan if c[2] == 3) >= n * npair * 4        # every entry's TQ3 group, per kv head


def test_inject_plan_slot_needs_a_device_plan(mkv):
    p = _host_pool(mkv)
    with pytest.raises(mkv.MkvError) as e:
        mkv.binding.mkv_inject_plan_slot(p.handle, 0, 5)
    assert e.value.status == 2                         # host-only pool


def test_missing_library_fails_loudly(mkv, monkeypatch):
    """No CPU or dense fallback: without libmkv.so every call raises."""
    monkeypatch.setattr(mkv.binding, "_lib", None)
    monkeypatch.setattr(mkv.binding, "LIB_PATH", os.path.join(ROOT, "no_such_dir", "libmkv.so"))
    with pytest.raises(ImportError):
        mkv.binding.lib()
    with pytest.raises(ImportError):
        _host_pool(mkv)


def _reference_split(groups, max_cta):
    """The plain split the planner computes: a greedy fill that gives each CTA
    the longest run of blocks that fits the bound (a round at a time, then
    block by block within the round that does not fit), and the smallest
    integer bound that fits in max_cta CTAs.  Returns the pieces
    (group key, CTA, first block, blocks)."""
    lo = max(PIECE + 27 * costs[0] for _, costs in groups)
    hi = sum(PIECE + 60 * costs[0] * -(-len(costs) // 12) for _, costs in groups)

    def fill(bound, pieces=None):
        n_cta, acc = 0, 0
        for key, costs in groups:
            b = 0
            while b < len(costs):
                def longest(budget):
                    used, e = 0, b
                    while e < len(costs):
                        n = min(12, len(costs) - e)
                        full = costs[e] * (24 + 3 * n)
                        if used + full <= budget:
                            used, e = used + full, e + n
                            continue
                        k = 0
                        while k + 1 < n and used + costs[e] * (24 + 3 * (k + 1)) <= budget:
                            k += 1
                        return e + k, used + (costs[e] * (24 + 3 * k) if k else 0)
                    return e, used
                e, c = longest(bound - acc - PIECE) if n_cta and acc + PIECE < bound else (b, 0)
                if e == b:
                    n_cta, acc = n_cta + 1, 0
                    e, c = longest(bound - PIECE)
                if pieces is not None:
                    pieces.append((key, n_cta - 1, b, e - b))
                acc += PIECE + c
                b = e
        return n_cta
    if fill(lo) > max_cta:
        while hi - lo > 1:
            mid = lo + (hi - lo) // 2
            if fill(mid) <= max_cta:
                hi = mid
            else:
                lo = mid
        lo = hi
    pieces = []
    fill(lo, pieces)
    return pieces


def test_plan_split_matches_reference(mkv):
    """The planner takes whole rounds of full blocks in O(1) per CTA; on all
    five workloads its split must equal the plain round-by-round, then
    block-by-block, algorithm's."""
    from mixed_format_paged_gb300 import workloads
    from mixed_format_paged_gb300.harness import make_pool
    for name in ("cfg1", "cfg2", "cfg3", "cfg4", "cfg5"):
        w = workloads.make(name)
        w.num_layers = 1
        pool = make_pool(w, host_only=True, extra_steps=0)
        layouts = []
        for r in range(w.n):
            pool.extend([r], [w.lengths[r]])
            tiers = w.tiers(r)
            for pg, t in enumerate(tiers):
                if t == 2:
                    pool.set_tier(r, pg, 2)
            stale = [pg for pg, t in enumerate(tiers) if t == 3]
            if stale:
                pool.demote([r] * len(stale), stale)
            layouts.append((w.lengths[r], tiers))
        plan = pool.plan(list(range(w.n)))
        groups = _blocks_of(layouts, w.P)
        max_cta = max(1, min(152, sum(len(c) for _, c in groups) // 24))
        exp = [(key[0], key[1], key[2], cta, b0, nb) for key, cta, b0, nb in _reference_split(groups, max_cta)]
        got = [(b, kvh, tier, cta, blk0, nblk) for b, kvh, tier, _, _, _, cta, blk0, nblk in plan]
        assert got == exp, name
