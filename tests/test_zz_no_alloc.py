"""GPU test of mkv_decode_attention_noalloc, the decode entry point that keeps
its scratch in a fixed array compiled into the library.  It exists for
callers that may not allocate device memory during a call (a framework
allocator that owns the whole device, or a step that must not trigger
cudaMalloc).  The test calls it twice in a row through the C ABI and checks
both results against mkv_decode_attention, with the tolerances of the other
parity tests; it also checks that a batch too large for the fixed scratch is
refused.  It lives in its own file so that it runs after every other test,
and it also passes when run alone in a fresh process."""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


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


def _mixed_pool(mkv):
    g = torch.Generator().manual_seed(11)
    pool = mkv.MkvPool(2, 24, 4, 256, 64, 64, 64, max_seqs=4, max_pages_per_seq=24, max_batch=4,
                       rotation_seed=5, device=DEV)
    specs = [(7 * 64 + 9, [0], [1, 2, 3, 4]), (3 * 64, [], []), (12 * 64 + 1, [3], [0, 1, 2, 4, 5, 6, 7, 8, 9])]
    for r, (n, anc, st) in enumerate(specs):
        pool.extend([r], [n])
        for layer in range(2):
            K = torch.randn(n, 4, 256, generator=g)
            K[..., 9] += 8.0
            V = torch.randn(n, 4, 256, generator=g)
            pool.append(layer, [r], [n], K.to(torch.bfloat16).to(DEV), V.to(torch.bfloat16).to(DEV))
        for a in anc:
            pool.set_tier(r, a, 2)
        if st:
            pool.demote([r] * len(st), st)
    q = torch.randn(len(specs), 24, 256, generator=g).to(torch.bfloat16).to(DEV)
    return pool, list(range(len(specs))), q


def test_noalloc_matches_decode_twice(mkv):
    pool, ids, q = _mixed_pool(mkv)
    B = mkv.binding
    for layer in (1, 0):
        ref_o, ref_l = pool.decode(layer, ids, q)
        torch.cuda.synchronize()
        for _ in range(2):
            out = torch.full_like(ref_o, float("nan"))
            lse = torch.full_like(ref_l, float("nan"))
            B.mkv_decode_attention_noalloc(pool.handle, layer, ids, q, B.MKV_BF16, out, lse,
                                           torch.cuda.current_stream())
            torch.cuda.synchronize()
            for b in range(len(ids)):
                ro = ref_o[b].double().cpu().numpy()
                assert np.abs(out[b].double().cpu().numpy() - ro).max() <= 2e-3 * np.abs(ro).max()
                assert np.abs(lse[b].double().cpu().numpy() - ref_l[b].double().cpu().numpy()).max() <= 1e-4
    pool.check_device_errors()


def test_noalloc_refuses_batches_beyond_its_scratch(mkv):
    # 400 one-page sequences need one partial state per (sequence, kv head):
    # 1,600 x 6 x 258 x 4 B > 8 MiB.
    n = 400
    pool = mkv.MkvPool(1, 24, 4, 256, 64, n, 1, max_seqs=n, max_pages_per_seq=1, max_batch=n,
                       rotation_seed=3, device=DEV)
    ids = list(range(n))
    pool.extend(ids, [5] * n)
    k = torch.randn(5 * n, 4, 256, device=DEV).to(torch.bfloat16)
    pool.append(0, ids, [5] * n, k, k)
    q = torch.randn(n, 24, 256, device=DEV).to(torch.bfloat16)
    out = torch.empty(n, 24, 256, device=DEV)
    lse = torch.empty(n, 24, device=DEV)
    B = mkv.binding
    with pytest.raises(mkv.MkvError) as e:
        B.mkv_decode_attention_noalloc(pool.handle, 0, ids, q, B.MKV_BF16, out, lse, torch.cuda.current_stream())
    assert e.value.status == 7
    # the regular entry point still serves the same batch from the pool workspace
    pool.decode(0, ids, q, out, lse)
    torch.cuda.synchronize()
    assert torch.isfinite(out).all() and torch.isfinite(lse).all()
