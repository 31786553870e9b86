"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle.

Criteria (the library's spec, include/mkv.h):
* FP8 codes and scales: bit-exact (the quantiser decides in IEEE fp32 on both
  sides).
* TQ3 codes: bit-exact except where the oracle's fp64 pre-decision value lies
  within 1e-6 (relative) of a threshold; such codes must be <= 0.01 %.  TQ3
  scales: exact except at fp16 rounding ties (same 1e-6 rule).  Codes are
  compared by re-encoding with the oracle given the GPU's FP8 bytes and fp16
  scale, so a scale tie cannot cascade.
* decode: max|out - out_oracle| <= 2e-3 * max|out_oracle| per request and
  |lse - lse_oracle| <= 1e-4, with the oracle reading the GPU's stored pages;
  an end-to-end check from raw inputs runs on the small workload.
"""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

OUT_TOL = 2e-3
LSE_TOL = 1e-4


@pytest.fixture(scope="module")
def mkv():
    import os
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    if not os.path.exists(os.path.join(root, "mixed_format_paged_gb300", "libmkv.so")):
        from mixed_format_paged_gb300 import build as b
        b.build()
    import mixed_format_paged_gb300 as m
    assert torch.cuda.is_available()
    return m


DEV = "cuda:0"


def _export(pool, layer, r):
    pages = []
    for p in range(pool.seq_info(r)[1]):
        b, tier, nv = pool.export_page(layer, r, p)
        pages.append((tier, np.frombuffer(b, dtype=np.uint8).copy(), nv))
    return pages


def _check_decode(pool, layer, ids, q, out, lse, seed, D=256):
    from oracle.paged import decode_attention_streaming
    H, P = pool.num_kv_heads, pool.page_size
    worst = (0.0, 0.0)
    for b, r in enumerate(ids):
        pages = _export(pool, layer, r)
        ro, rl = decode_attention_streaming(q[b].double().cpu().numpy(), pages, P, H, D, seed)
        o = out[b].double().cpu().numpy()
        l_ = lse[b].double().cpu().numpy()
        eo = np.abs(o - ro).max() / np.abs(ro).max()
        el = np.abs(l_ - rl).max()
        assert eo <= OUT_TOL, f"request {r}: relative out error {eo:.3e}"
        assert el <= LSE_TOL, f"request {r}: lse error {el:.3e}"
        worst = (max(worst[0], eo), max(worst[1], el))
    return worst


def _tq3_check(fp8_page, tq3_page, P, H, D, seed):
    """Return (#code mismatches, #codes) after the boundary exemption; raise on
    a non-exempt mismatch."""
    from oracle import layout
    from oracle.paged import fp8_page_dequant
    from oracle.tq3 import boundary_distance, fp16_tie_distance, tq3_encode_rows, tq3_sigma_raw
    Kh, Vh = fp8_page_dequant(fp8_page, P, H, D)
    kc, ks, vc, vs = layout.unpack_tq3_page(tq3_page, P, H, D)
    mism = 0
    for X, codes, sig in ((Kh, kc, ks), (Vh, vc, vs)):
        raw = tq3_sigma_raw(X)
        _, s_or, _ = tq3_encode_rows(X, seed)
        bad_s = sig != s_or
        far_s = int(np.sum(fp16_tie_distance(raw[bad_s]) > 1e-6))
        assert far_s == 0, (f"{far_s} TQ3 scale mismatches away from an fp16 tie "
                            f"({int(bad_s.sum())} mismatches of {sig.size} scales)")
        ref, _, u = tq3_encode_rows(X, seed, sigma=sig)
        diff = codes != ref
        far = int(np.sum(boundary_distance(u[diff]) > 1e-6)) if diff.any() else 0
        assert far == 0, (f"{far} TQ3 code mismatches away from a threshold "
                          f"({int(diff.sum())} mismatches of {codes.size} codes)")
        mism += int(diff.sum())
    return mism, 2 * Kh.size


def _small_pool(mkv, P=64, layers=1, fp8=64, tq3=64, nseq=8, maxp=32, seed=4321):
    return mkv.MkvPool(layers, 24, 4, 256, P, fp8, tq3, max_seqs=nseq, max_pages_per_seq=maxp, max_batch=nseq,
                       rotation_seed=seed, device=DEV)


def _kv(n, dtype, g, outlier=True):
    K = torch.randn(n, 4, 256, generator=g)
    V = torch.randn(n, 4, 256, generator=g)
    if outlier:
        K[..., 5] += 8.0
        K[..., 200] -= 8.0
    return K.to(dtype), V.to(dtype)


# ------------------------------------------------------------------ append
@pytest.mark.parametrize("P", [64, 128])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_append_fp8_bit_exact(mkv, P, dtype):
    from oracle.paged import encode_fp8_page
    g = torch.Generator().manual_seed(1)
    pool = _small_pool(mkv, P=P)
    n0 = 2 * P + 37
    K, V = _kv(n0 + 2, dtype, g)
    K[3] = 0.0                                   # an all-zero row (scale 0)
    V[4, 1] = torch.tensor(1e-30).to(dtype)      # tiny values
    pool.extend([0], [n0])
    pool.append(0, [0], [n0], K[:n0].to(DEV), V[:n0].to(DEV))
    for t in (n0, n0 + 1):                       # two single-token appends
        pool.extend([0], [1])
        pool.append(0, [0], [1], K[t:t + 1].to(DEV).contiguous(), V[t:t + 1].to(DEV).contiguous())
    torch.cuda.synchronize()
    pages = _export(pool, 0, 0)
    Kf, Vf = K.float().numpy(), V.float().numpy()
    for p, (tier, b, nv) in enumerate(pages):
        exp = encode_fp8_page(Kf[p * P: p * P + nv], Vf[p * P: p * P + nv], P)
        assert np.array_equal(b, exp), f"page {p}: {int((b != exp).sum())} bytes differ"
    pool.check_device_errors()


# ------------------------------------------------------------------ demote
@pytest.mark.parametrize("P", [64, 128])
def test_demote_tq3_codes(mkv, P):
    g = torch.Generator().manual_seed(2)
    pool = _small_pool(mkv, P=P, layers=2)
    n = 6 * P
    pool.extend([0], [n])
    for layer in range(2):
        K, V = _kv(n, torch.bfloat16, g)
        if layer == 1:
            V = (V.float() * torch.linspace(0.01, 30, n)[:, None, None]).to(torch.bfloat16)
        pool.append(layer, [0], [n], K.to(DEV), V.to(DEV))
    torch.cuda.synchronize()
    before = {(l_, p): _export(pool, l_, 0)[p][1] for l_ in range(2) for p in range(6)}
    pool.demote([0] * 4, [0, 2, 3, 4])
    torch.cuda.synchronize()
    total_m, total = 0, 0
    for l_ in range(2):
        after = _export(pool, l_, 0)
        for p in (0, 2, 3, 4):
            assert after[p][0] == 3
            m, t = _tq3_check(before[(l_, p)], after[p][1], P, 4, 256, 4321)
            total_m += m
            total += t
        for p in (1, 5):
            assert np.array_equal(after[p][1], before[(l_, p)])      # untouched FP8 pages
    assert total_m <= 1e-4 * total, f"{total_m} exempted TQ3 code mismatches of {total} codes"
    pool.check_device_errors()


# ------------------------------------------------------------------ decode
@pytest.mark.parametrize("P", [64, 128])
@pytest.mark.parametrize("qdtype", [torch.float32, torch.bfloat16])
def test_decode_mixed_layouts(mkv, P, qdtype):
    g = torch.Generator().manual_seed(3)
    pool = _small_pool(mkv, P=P, fp8=96, tq3=96, maxp=24)
    # request layouts: (tokens, anchors, stale pages)
    specs = [
        (1, [], []),                                   # a single token
        (P, [], []),                                   # one full FP8 page
        (5 * P + 1, [0], [1, 2, 3]),                   # tail of 1 token
        (9 * P + 33, [], list(range(8))),              # mostly TQ3
        (3 * P + 5, [0, 1, 2], []),                    # all FP8 with Anchors
        (12 * P, [4], [0, 1, 2, 3, 5, 6, 7, 8, 9, 10]),  # full tail page, TQ3 around an Anchor
    ]
    for r, (n, anc, st) in enumerate(specs):
        K, V = _kv(n, torch.bfloat16, g)
        pool.extend([r], [n])
        pool.append(0, [r], [n], K.to(DEV), V.to(DEV))
        for a in anc:
            pool.set_tier(r, a, 2)
        if st:
            pool.demote([r] * len(st), st)
    ids = list(range(len(specs)))
    q = torch.randn(len(ids), 24, 256, generator=g).to(qdtype)
    out, lse = pool.decode(0, ids, q.to(DEV))
    torch.cuda.synchronize()
    pool.check_device_errors()
    _check_decode(pool, 0, ids, q.float(), out, lse, 4321)
    # a sub-batch in another order gives the same rows (up to the parity
    # tolerance: another batch is split differently, and P is rounded to fp16
    # relative to each split's running max)
    out2, lse2 = pool.decode(0, [5, 2], q[[5, 2]].to(DEV).contiguous())
    torch.cuda.synchronize()
    for i, r in enumerate([5, 2]):
        ref = out[r].double()
        assert (out2[i].double() - ref).abs().max() <= OUT_TOL * ref.abs().max()
        assert (lse2[i].double() - lse[r].double()).abs().max() <= LSE_TOL


def test_decode_repeatable(mkv):
    g = torch.Generator().manual_seed(4)
    pool = _small_pool(mkv)
    K, V = _kv(700, torch.bfloat16, g)
    pool.extend([0], [700])
    pool.append(0, [0], [700], K.to(DEV), V.to(DEV))
    pool.demote([0] * 5, [0, 1, 2, 3, 4])
    q = torch.randn(1, 24, 256, generator=g).to(torch.bfloat16).to(DEV)
    a = pool.decode(0, [0], q)
    b = pool.decode(0, [0], q)
    torch.cuda.synchronize()
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


# ------------------------------------------------------------------ workload cfg1 end to end
def test_cfg1_end_to_end(mkv):
    from mixed_format_paged_gb300 import workloads
    from mixed_format_paged_gb300.harness import make_pool, prefill
    from oracle.paged import TIER_STALE, decode_attention, demote_page, encode_fp8_page
    w = workloads.make("cfg1")
    pool = make_pool(w, device=DEV, extra_steps=0, seed=777)
    raw = prefill(pool, w, device=DEV, keep_raw=True)
    q = w.query(0, 0)
    out, lse = pool.decode(0, [0], q.to(DEV))
    torch.cuda.synchronize()
    pool.check_device_errors()
    pages = _export(pool, 0, 0)
    tiers = [t for t, _, _ in pages]
    assert tiers.count(TIER_STALE) == 55 and tiers[0] == 2 and tiers[56:] == [1] * 8
    # codecs: FP8 pages bit-exact; TQ3 pages within the boundary exemption
    K, V = (x.float().numpy() for x in raw[(0, 0)])
    mism = total = 0
    oracle_pages = []
    for p, (tier, b, nv) in enumerate(pages):
        f8 = encode_fp8_page(K[p * 64:(p + 1) * 64], V[p * 64:(p + 1) * 64], 64)
        if tier == TIER_STALE:
            m, t = _tq3_check(f8, b, 64, 4, 256, 777)
            mism += m
            total += t
            oracle_pages.append((tier, demote_page(f8, 64, 4, 256, 777)[0], nv))
        else:
            assert np.array_equal(b, f8)
            oracle_pages.append((tier, f8, nv))
    assert mism <= 1e-4 * total, f"{mism} exempted TQ3 code mismatches of {total} codes"
    # decode against the stored pages
    _check_decode(pool, 0, [0], q, out, lse, 777)
    # end to end from the raw fp32 inputs (oracle encodes every page itself)
    ro, rl = decode_attention(q[0].double().numpy(), oracle_pages, 64, 4, 256, 777)
    o = out[0].double().cpu().numpy()
    assert np.abs(o - ro).max() <= OUT_TOL * np.abs(ro).max()
    assert np.abs(lse[0].double().cpu().numpy() - rl).max() <= LSE_TOL


# ------------------------------------------------------------------ decode steps with demotion
def test_decode_steps_with_demotion(mkv):
    from mixed_format_paged_gb300 import workloads
    from mixed_format_paged_gb300.harness import Stepper, make_pool, prefill
    w = workloads.make("cfg3")
    w.lengths = [64 * 20 - 3, 64 * 31 - 1]      # short, both about to roll over
    w.anchors = [{2, 5}, {1}]
    w.num_layers = 2
    w.steps = 70
    pool = make_pool(w, device=DEV, seed=31)
    prefill(pool, w, device=DEV)
    st = Stepper(pool, w, device=DEV)
    for step in range(w.steps):
        st.pre_step()
        for layer in range(w.num_layers):
            k, v = w.step_kv(layer, step)
            q = w.query(layer, step)
            out, lse = st.layer(layer, k.to(DEV), v.to(DEV), q.to(DEV))
        if step in (0, 3, 69):
            torch.cuda.synchronize()
            _check_decode(pool, w.num_layers - 1, st.ids, q.float(), out, lse, 31)
    pool.check_device_errors()
    for r in range(2):
        tiers = [pool.page_info(r, p)[0] for p in range(pool.seq_info(r)[1])]
        npg = len(tiers)
        assert all(t != 3 for t in tiers[npg - w.windows[r]:])
        assert all(tiers[a] == 2 for a in w.anchors[r])
        assert sum(t == 3 for t in tiers) == npg - w.windows[r] - len(w.anchors[r])


# ------------------------------------------------------------------ full-size workloads, sampled
@pytest.mark.parametrize("name", ["cfg2", "cfg3", "cfg4", "cfg5"])
def test_full_size_sampled(mkv, name):
    from mixed_format_paged_gb300 import workloads
    from mixed_format_paged_gb300.harness import Stepper, make_pool, prefill
    w = workloads.make(name)
    rng = np.random.default_rng(5)
    layers = [0, w.num_layers - 1]
    pool = make_pool(w, device=DEV, extra_steps=2, seed=99)
    prefill(pool, w, device=DEV, layers=layers)
    st = Stepper(pool, w, device=DEV)
    st.pre_step()
    outs = {}
    for layer in layers:
        k, v = w.step_kv(layer, 0)
        q = w.query(layer, 0)
        outs[layer] = (q,) + tuple(x.clone() for x in st.layer(layer, k.to(DEV), v.to(DEV), q.to(DEV)))
    torch.cuda.synchronize()
    pool.check_device_errors()
    nsample = 2 if name == "cfg5" else 3
    for layer in layers:
        q, out, lse = outs[layer]
        rs = sorted(rng.choice(w.n, size=min(nsample, w.n), replace=False).tolist())
        if name == "cfg4":
            # the two extreme layout classes, whatever the draw picked
            cls = w.layout_classes()
            assert cls["all_fp8"] and cls["mostly_tq3"]
            rs = sorted(set(rs) | {cls["all_fp8"][layer % len(cls["all_fp8"])],
                                   cls["mostly_tq3"][layer % len(cls["mostly_tq3"])]})
        from oracle.paged import decode_attention_streaming
        for r in rs:
            pages = _export(pool, layer, r)
            kvh = [int(rng.integers(0, 4))]
            ro, rl = decode_attention_streaming(q[r].double().numpy(), pages, w.P, 4, 256, 99, kv_heads=kvh)
            sl = slice(kvh[0] * 6, kvh[0] * 6 + 6)
            o = out[r].double().cpu().numpy()[sl]
            assert np.abs(o - ro[sl]).max() <= OUT_TOL * np.abs(ro[sl]).max()
            assert np.abs(lse[r].double().cpu().numpy()[sl] - rl[sl]).max() <= LSE_TOL
    # a property that holds at any size: every live page is addressable and the
    # workspace does not depend on context length
    s = pool.stats()
    assert s.live_tokens == sum(st.lengths)
    assert s.workspace_bytes < 64 * 2 ** 20


# ------------------------------------------------------------------ fused append + decode
def test_append_decode_matches_separate_calls(mkv):
    """mkv_append_decode (append fused into the decode kernel) gives the
    same page bytes and the same outputs as mkv_append_tokens + mkv_decode_attention."""
    g = torch.Generator().manual_seed(21)
    pools = [_small_pool(mkv, P=64, layers=2, fp8=64, tq3=64, maxp=24, seed=77) for _ in range(2)]
    lens = [64 * 6 + 63, 64 * 3, 1]
    data = [(torch.randn(n, 4, 256, generator=g).to(torch.bfloat16), torch.randn(n, 4, 256, generator=g).to(torch.bfloat16))
            for n in lens]
    for pool in pools:
        for r, n in enumerate(lens):
            pool.extend([r], [n])
            for layer in range(2):
                pool.append(layer, [r], [n], data[r][0].to(DEV), data[r][1].to(DEV))
        pool.demote([0, 0, 0], [1, 2, 3])
    ids = [0, 1, 2]
    for step in range(3):
        k = torch.randn(3, 4, 256, generator=g).to(torch.bfloat16).to(DEV)
        v = torch.randn(3, 4, 256, generator=g).to(torch.bfloat16).to(DEV)
        q = torch.randn(3, 24, 256, generator=g).to(torch.bfloat16).to(DEV)
        outs = []
        for i, pool in enumerate(pools):
            pool.extend(ids, [1, 1, 1])
            res = []
            for layer in range(2):
                if i == 0:
                    o, l_ = pool.append_decode(layer, ids, k, v, q)
                else:
                    pool.append(layer, ids, [1, 1, 1], k, v)
                    o, l_ = pool.decode(layer, ids, q)
                res.append((o.clone(), l_.clone()))
            outs.append(res)
        torch.cuda.synchronize()
        for layer in range(2):
            assert torch.equal(outs[0][layer][0], outs[1][layer][0])
            assert torch.equal(outs[0][layer][1], outs[1][layer][1])
    for layer in range(2):
        for r in ids:
            a = _export(pools[0], layer, r)
            b = _export(pools[1], layer, r)
            assert all(np.array_equal(x[1], y[1]) for x, y in zip(a, b))
    _check_decode(pools[0], 1, ids, q.float(), outs[0][1][0], outs[0][1][1], 77)
    for pool in pools:
        pool.check_device_errors()


# ------------------------------------------------------------------ page relevance
@pytest.mark.parametrize("P", [64, 128])
@pytest.mark.parametrize("qdtype", [torch.float32, torch.bfloat16])
def test_page_relevance_matches_oracle(mkv, P, qdtype):
    """mkv_page_relevance against oracle.paged.page_attention_mass on the
    GPU's stored pages.  It normalises with the decode call's lse, whose
    error is <= 1e-4, so each mass carries a relative error of about 1e-4."""
    from oracle.paged import page_attention_mass
    g = torch.Generator().manual_seed(41)
    pool = _small_pool(mkv, P=P, fp8=96, tq3=96, maxp=24)
    specs = [(5 * P + 9, [0], [1, 2, 3]), (9 * P + 33, [], list(range(8))), (2 * P + 1, [0], [])]
    for r, (n, anc, st) in enumerate(specs):
        K, V = _kv(n, torch.bfloat16, g)
        if r == 1:
            K[3 * P: 3 * P + 5] *= 3.0                 # a few loud keys: one page draws most of the weight
        pool.extend([r], [n])
        pool.append(0, [r], [n], K.to(DEV), V.to(DEV))
        for a in anc:
            pool.set_tier(r, a, 2)
        if st:
            pool.demote([r] * len(st), st)
    ids = [0, 1, 2]
    q = torch.randn(3, 24, 256, generator=g).to(qdtype)
    out, lse = pool.decode(0, ids, q.to(DEV))
    mass = pool.relevance(0, ids, q.to(DEV), lse)
    torch.cuda.synchronize()
    pool.check_device_errors()
    m = mass.double().cpu().numpy()
    for b, r in enumerate(ids):
        pages = _export(pool, 0, r)
        ref = page_attention_mass(q[b].double().numpy(), pages, P, 4, 256, 4321)
        got = m[b, :len(pages)]
        assert np.all(np.abs(got - ref) <= 3e-4 * ref + 1e-7), (r, np.abs(got - ref).max())
        assert abs(got.sum() - 1.0) <= 3e-4
        assert np.all(m[b, len(pages):] == 0.0)        # entries past the sequence stay untouched
        top = np.sort(ref)[::-1]
        if top[0] > 1.01 * top[1]:
            assert got.argmax() == ref.argmax()         # the same most relevant page


def test_relevance_stepper_anchors_the_attended_page(mkv):
    """RelevanceStepper end to end: the page whose keys line up with every
    query draws most of the attention mass (mkv_page_relevance), so when it
    leaves the Recent window it becomes an Anchor and stays FP8; the next
    page to leave draws little and goes to TQ3.  Decode still matches the
    oracle on the resulting mixed layout."""
    from mixed_format_paged_gb300 import workloads
    from mixed_format_paged_gb300.harness import RelevanceAnchors, RelevanceStepper, make_pool
    g = torch.Generator().manual_seed(53)
    w = workloads.make("cfg3")
    w.lengths, w.windows, w.anchors, w.num_layers, w.steps = [64 * 6 - 2], [3], [set()], 1, 70
    pool = make_pool(w, device=DEV, seed=53)
    u = torch.randn(256, generator=g)
    u /= u.norm()
    K = torch.randn(w.lengths[0], 4, 256, generator=g)
    V = torch.randn(w.lengths[0], 4, 256, generator=g)
    K[3 * 64: 4 * 64] = 6.0 * u                          # page 3: q.k / 16 = 3 for every token
    pool.extend([0], [w.lengths[0]])
    pool.append(0, [0], [w.lengths[0]], K.to(torch.bfloat16).to(DEV), V.to(torch.bfloat16).to(DEV))
    pool.demote([0, 0, 0], [0, 1, 2])
    pol = RelevanceAnchors(frac=0.05, kappa=2.0, beta=1.0)
    st = RelevanceStepper(pool, w, pol, layer=0, device=DEV)
    for step in range(w.steps):
        st.pre_step()
        k = torch.randn(1, 4, 256, generator=g).to(torch.bfloat16)
        v = torch.randn(1, 4, 256, generator=g).to(torch.bfloat16)
        q = (8.0 * u + 0.1 * torch.randn(1, 24, 256, generator=g)).to(torch.bfloat16)
        out, lse = st.layer(0, k.to(DEV), v.to(DEV), q.to(DEV))
    torch.cuda.synchronize()
    pool.check_device_errors()
    tiers = [pool.page_info(0, p)[0] for p in range(pool.seq_info(0)[1])]
    assert tiers[:5] == [3, 3, 3, 2, 3], tiers           # page 3 anchored, page 4 demoted
    assert all(t == 1 for t in tiers[5:])
    assert pol.anchors[0] == {3} and pol.rho[(0, 3)] > 0.5
    _check_decode(pool, 0, [0], q.float(), out, lse, 53)


# ------------------------------------------------------------------ step graph
@pytest.mark.parametrize("P", [64, 128])
@pytest.mark.parametrize("append", [True, False])
def test_step_graph_matches_per_layer_calls(mkv, append, P):
    """mkv_step_graph_*: one recorded launch per step over every layer gives,
    bit for bit, what the per-layer calls give -- through re-plans (the
    batch grows every step) and a demotion between steps -- and the oracle
    agrees with it."""
    g = torch.Generator().manual_seed(31)
    L = 3
    pools = [_small_pool(mkv, P=P, layers=L, fp8=64, tq3=64, maxp=24, seed=79) for _ in range(2)]
    lens = [P * 5 + P - 2, P * 3 + 1, 7]              # request 0 opens a new page during the steps
    data = [[(torch.randn(n, 4, 256, generator=g).to(torch.bfloat16), torch.randn(n, 4, 256, generator=g).to(torch.bfloat16))
             for _ in range(L)] for n in lens]
    for pool in pools:
        for r, n in enumerate(lens):
            pool.extend([r], [n])
            for layer in range(L):
                pool.append(layer, [r], [n], data[r][layer][0].to(DEV), data[r][layer][1].to(DEV))
        pool.set_tier(0, 0, 2)
        pool.demote([0, 0, 1], [1, 2, 0])
    ids = [0, 1, 2]
    n = len(ids)
    # fixed buffers of the graph path
    qb = [torch.empty(n, 24, 256, dtype=torch.bfloat16, device=DEV) for _ in range(L)]
    kb = [torch.empty(n, 4, 256, dtype=torch.bfloat16, device=DEV) for _ in range(L)] if append else None
    vb = [torch.empty(n, 4, 256, dtype=torch.bfloat16, device=DEV) for _ in range(L)] if append else None
    ob = [torch.empty(n, 24, 256, dtype=torch.float32, device=DEV) for _ in range(L)]
    lb = [torch.empty(n, 24, dtype=torch.float32, device=DEV) for _ in range(L)]
    graph = None
    for step in range(3):
        ks = [torch.randn(n, 4, 256, generator=g).to(torch.bfloat16).to(DEV) for _ in range(L)]
        vs = [torch.randn(n, 4, 256, generator=g).to(torch.bfloat16).to(DEV) for _ in range(L)]
        qs = [torch.randn(n, 24, 256, generator=g).to(torch.bfloat16).to(DEV) for _ in range(L)]
        if step == 2:
            for pool in pools:
                pool.demote([0], [3])               # page 3 of request 0 leaves the Recent window
        # per-layer calls
        pools[0].extend(ids, [1] * n)
        ref = []
        for layer in range(L):
            if append:
                o, l_ = pools[0].append_decode(layer, ids, ks[layer], vs[layer], qs[layer])
            else:
                pools[0].append(layer, ids, [1] * n, ks[layer], vs[layer])
                o, l_ = pools[0].decode(layer, ids, qs[layer])
            ref.append((o.clone(), l_.clone()))
        # the graph
        pools[1].extend(ids, [1] * n)
        for layer in range(L):
            qb[layer].copy_(qs[layer])
            if append:
                kb[layer].copy_(ks[layer])
                vb[layer].copy_(vs[layer])
            else:
                pools[1].append(layer, ids, [1] * n, ks[layer], vs[layer])
        if graph is None:
            graph = pools[1].step_graph(ids, qb, ob, lb, k=kb, v=vb)
        graph.launch()
        torch.cuda.synchronize()
        for layer in range(L):
            assert torch.equal(ref[layer][0], ob[layer]), (step, layer)
            assert torch.equal(ref[layer][1], lb[layer]), (step, layer)
    for layer in range(L):
        for r in ids:
            a = _export(pools[0], layer, r)
            b = _export(pools[1], layer, r)
            assert all(np.array_equal(x[1], y[1]) for x, y in zip(a, b))
    _check_decode(pools[1], L - 1, ids, qs[L - 1].float(), ob[L - 1], lb[L - 1], 79)
    graph.close()
    for pool in pools:
        pool.check_device_errors()


# ------------------------------------------------------------------ materialising export
@pytest.mark.parametrize("P", [64, 128])
def test_dequantize_pages_matches_oracle(mkv, P):
    from oracle.paged import TIER_STALE, fp8_page_dequant, tq3_page_dequant
    g = torch.Generator().manual_seed(31)
    pool = _small_pool(mkv, P=P, layers=2, seed=555)
    n = 5 * P + 19
    pool.extend([0], [n])
    for layer in range(2):
        K, V = _kv(n, torch.bfloat16, g)
        pool.append(layer, [0], [n], K.to(DEV), V.to(DEV))
    pool.set_tier(0, 4, 2)
    pool.demote([0, 0, 0], [0, 2, 3])
    k32, v32 = pool.dequantize(1, 0, 0, 6)
    kb, vb = pool.dequantize(1, 0, 1, 4, dtype=torch.bfloat16)
    torch.cuda.synchronize()
    pages = _export(pool, 1, 0)
    for pg, (tier, b, nv) in enumerate(pages):
        if tier == TIER_STALE:
            Kr, Vr = tq3_page_dequant(b, P, 4, 256, 555)
            tol = 1e-5
        else:
            Kr, Vr = fp8_page_dequant(b, P, 4, 256)
            tol = 0.0
        kg = k32[pg * P:(pg + 1) * P].double().cpu().numpy()
        vg = v32[pg * P:(pg + 1) * P].double().cpu().numpy()
        for got, ref in ((kg, Kr), (vg, Vr)):
            assert np.abs(got[:nv] - ref[:nv]).max() <= tol * max(1.0, np.abs(ref[:nv]).max())
            assert np.all(got[nv:] == 0.0)
    # bf16 output is the fp32 result rounded to nearest even
    assert torch.equal(kb, k32[P:5 * P].to(torch.bfloat16)) and torch.equal(vb, v32[P:5 * P].to(torch.bfloat16))
    pool.check_device_errors()


# ------------------------------------------------------------------ several query tokens per request
@pytest.mark.parametrize("P", [64, 128])
@pytest.mark.parametrize("qdtype", [torch.float32, torch.bfloat16])
def test_decode_multi_query_causal(mkv, P, qdtype):
    """mkv_decode_attention_multi: query token i of each request attends to the
    request's tokens up to its own position (oracle: causal attention over the
    stored pages)."""
    from oracle.paged import decode_attention_multi
    g = torch.Generator().manual_seed(23)
    pool = _small_pool(mkv, P=P, fp8=96, tq3=96, nseq=32, maxp=24)   # 4 requests x 8 query tokens
    # (tokens, anchors, stale pages): tails of 1, 5 and P tokens, so that the
    # query tokens of some requests start in the page before the tail
    specs = [(4 * P + 5, [0], [1, 2]), (9, [], []), (6 * P + 1, [], [0, 1, 2, 3]), (3 * P, [1], [0])]
    for r, (n, anc, st) in enumerate(specs):
        K, V = _kv(n, torch.bfloat16, g)
        pool.extend([r], [n])
        pool.append(0, [r], [n], K.to(DEV), V.to(DEV))
        for a in anc:
            pool.set_tier(r, a, 2)
        if st:
            pool.demote([r] * len(st), st)
    ids = list(range(len(specs)))
    for nq in (1, 2, 3, 8):
        q = torch.randn(len(ids), nq, 24, 256, generator=g).to(qdtype)
        out, lse = pool.decode_multi(0, ids, q.to(DEV))
        torch.cuda.synchronize()
        pool.check_device_errors()
        for b, r in enumerate(ids):
            ro, rl = decode_attention_multi(q[b].double().numpy(), _export(pool, 0, r), P, 4, 256, 4321)
            o = out[b].double().cpu().numpy()
            l_ = lse[b].double().cpu().numpy()
            for i in range(nq):
                assert np.abs(o[i] - ro[i]).max() <= OUT_TOL * np.abs(ro[i]).max(), (nq, r, i)
                assert np.abs(l_[i] - rl[i]).max() <= LSE_TOL, (nq, r, i)
        if nq == 1:
            # one query token is the decode step itself (same plan, same bits)
            o1, l1 = pool.decode(0, ids, q[:, 0].contiguous().to(DEV))
            torch.cuda.synchronize()
            assert torch.equal(o1, out[:, 0]) and torch.equal(l1, lse[:, 0])
        else:
            # paired entries merge in a fixed order too: a second call repeats every bit
            o2, l2 = pool.decode_multi(0, ids, q.to(DEV))
            torch.cuda.synchronize()
            assert torch.equal(o2, out) and torch.equal(l2, lse)
    # a query token in a TQ3 page is refused; so are too many query tokens
    with pytest.raises(mkv.MkvError):
        pool.decode_multi(0, [2], torch.randn(1, 3 * P, 24, 256).to(DEV))
    with pytest.raises(mkv.MkvError):
        pool.decode_multi(0, [1], torch.randn(1, 10, 24, 256).to(DEV))


def _prefix(pages, P, visible):
    """The exported pages cut to their first `visible` tokens."""
    out = []
    for i, (tier, b, nv) in enumerate(pages):
        if i * P >= visible:
            break
        out.append((tier, b, min(nv, visible - i * P)))
    return out


@pytest.mark.parametrize("name", ["cfg3", "cfg5"])
def test_multi_query_full_size_sampled(mkv, name):
    """Paired multi-query decode at full context length (one layer, nq = 4
    query tokens appended to each request): the 2 x 59,008-token workload
    (P = 64), and two requests of the 16 x 131K-token one (P = 128).  Query
    tokens 0 and 3 of a sampled (request, kv head), each against the oracle
    over its own causal prefix of the stored pages."""
    from mixed_format_paged_gb300 import workloads
    from mixed_format_paged_gb300.harness import make_pool, prefill
    from oracle.paged import decode_attention_streaming
    w = workloads.make(name)
    if w.n > 2:
        w = w.subset([0, 1])
    nq = 4
    pool = make_pool(w, device=DEV, extra_steps=nq + 2, seed=77, max_batch=w.n * nq)
    prefill(pool, w, device=DEV, layers=[0])
    ids = list(range(w.n))
    g = torch.Generator().manual_seed(41)
    pool.extend(ids, [nq] * w.n)
    K, V = _kv(w.n * nq, torch.bfloat16, g)
    pool.append(0, ids, [nq] * w.n, K.to(DEV), V.to(DEV))
    q = torch.randn(w.n, nq, 24, 256, generator=g).to(torch.bfloat16)
    out, lse = pool.decode_multi(0, ids, q.to(DEV))
    torch.cuda.synchronize()
    pool.check_device_errors()
    rng = np.random.default_rng(8)
    r = int(rng.integers(0, w.n))
    kvh = int(rng.integers(0, 4))
    pages = _export(pool, 0, r)
    T = sum(nv for _, _, nv in pages)
    sl = slice(kvh * 6, kvh * 6 + 6)
    for i in (0, nq - 1):
        ro, rl = decode_attention_streaming(q[r, i].double().numpy(), _prefix(pages, w.P, T - nq + i + 1), w.P, 4,
                                            256, 77, kv_heads=[kvh])
        o = out[r, i].double().cpu().numpy()[sl]
        assert np.abs(o - ro[sl]).max() <= OUT_TOL * np.abs(ro[sl]).max(), (r, kvh, i)
        assert np.abs(lse[r, i].double().cpu().numpy()[sl] - rl[sl]).max() <= LSE_TOL, (r, kvh, i)


# ------------------------------------------------------------------ failure detection without a fault
def test_wait_timeout_is_reported_and_context_stays_usable(mkv):
    """A bounded wait that runs out (an mbarrier nothing arrives on) records
    the timeout in the pool's error word; mkv_check_device_errors reports
    MKV_ERR_DEVICE_CHECK once and clears it, and decode still matches the oracle."""
    g = torch.Generator().manual_seed(29)
    pool = _small_pool(mkv)
    K, V = _kv(3 * 64 + 7, torch.bfloat16, g)
    pool.extend([0], [3 * 64 + 7])
    pool.append(0, [0], [3 * 64 + 7], K.to(DEV), V.to(DEV))
    pool.demote([0], [1])
    pool.check_device_errors()
    pool.selftest_wait_timeout(2_000_000)              # ~1 ms at 2 GHz
    with pytest.raises(mkv.MkvError) as e:
        pool.check_device_errors()
    assert e.value.status == 6                         # MKV_ERR_DEVICE_CHECK
    pool.check_device_errors()                         # cleared
    q = torch.randn(1, 24, 256, generator=g).to(torch.bfloat16)
    out, lse = pool.decode(0, [0], q.to(DEV))
    torch.cuda.synchronize()
    pool.check_device_errors()
    _check_decode(pool, 0, [0], q.float(), out, lse, 4321)


def test_corrupt_plan_entry_is_caught(mkv):
    """A page entry injected with a slot outside the arena (host-side fault
    injection) is caught by the decode kernel's slot check: no copy, an error
    word, MKV_ERR_DEVICE_CHECK on the next check, no fault.  A replanned
    decode is right again."""
    from mixed_format_paged_gb300 import binding as B
    g = torch.Generator().manual_seed(31)
    pool = _small_pool(mkv)
    n = 5 * 64 + 9
    K, V = _kv(n, torch.bfloat16, g)
    pool.extend([0], [n])
    pool.append(0, [0], [n], K.to(DEV), V.to(DEV))
    pool.demote([0], [1, 2])
    q = torch.randn(1, 24, 256, generator=g).to(torch.bfloat16)
    for entry, slot in ((0, 1 << 20), (4, -7)):       # an FP8 entry, then a TQ3 entry
        pool.decode(0, [0], q.to(DEV))                 # plans and uploads
        torch.cuda.synchronize()
        pool.check_device_errors()
        B.mkv_inject_plan_slot(pool.handle, entry, slot)
        pool.decode(0, [0], q.to(DEV))                 # same batch: the injected plan
        torch.cuda.synchronize()
        with pytest.raises(mkv.MkvError) as e:
            pool.check_device_errors()
        assert e.value.status == 6
        pool.plan([0])                                 # drops the device plan: the next decode replans
    out, lse = pool.decode(0, [0], q.to(DEV))
    torch.cuda.synchronize()
    pool.check_device_errors()
    _check_decode(pool, 0, [0], q.float(), out, lse, 4321)
