"""CPU tests of the seeded workload generator and of bench.py's JSON contract
(the reference arm, which times the oracle, runs without a GPU)."""
import json
import os
import subprocess
import sys

import numpy as np
import torch

from mixed_format_paged_gb300 import workloads

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_cfg1_layout_matches_its_description():
    w = workloads.make("cfg1")
    t = w.tiers(0)
    assert w.lengths == [4096] and len(t) == 64
    assert t[0] == workloads.A and t[56:] == [workloads.R] * 8 and t[1:56] == [workloads.S] * 55
    assert w.kv_dtype == torch.float32 and w.q_dtype == torch.float32


def test_workload_shapes_and_layouts():
    w2 = workloads.make("cfg2")
    assert w2.n == 8 and all(8192 <= L <= 32768 for L in w2.lengths) and w2.num_layers == 16
    for r in range(8):
        t = w2.tiers(r)
        assert t[0] == workloads.A                       # page 0 is an Anchor
        assert t[-8:] == [workloads.R] * 8
        assert abs(sum(x == workloads.A for x in t) - 1 - round(0.02 * len(t))) <= 1
    w3 = workloads.make("cfg3")
    assert w3.lengths == [59008, 59008] and [w3.npages(r) for r in range(2)] == [922, 922]
    assert all(len(a) == 28 for a in w3.anchors)
    w4 = workloads.make("cfg4")
    assert w4.n == 64 and all(1024 <= L <= 65536 for L in w4.lengths) and w4.v_student_t
    kinds = [(wi, len(a)) for wi, a in zip(w4.windows, w4.anchors)]
    assert any(wi == 1 for wi, _ in kinds) and any(wi == w4.npages(r) for r, (wi, _) in enumerate(kinds))
    w5 = workloads.make("cfg5")
    assert w5.n == 16 and w5.P == 128 and all(abs(L - 131072) <= 128 for L in w5.lengths)
    assert all(len(a) == 10 for a in w5.anchors)


def test_generator_is_deterministic_and_has_outliers():
    w = workloads.make("cfg2")
    w.lengths = [200] + w.lengths[1:]
    k1, v1 = w.prefill_kv(3, 0)
    k2, v2 = w.prefill_kv(3, 0)
    assert torch.equal(k1, k2) and torch.equal(v1, v2)
    k3, _ = w.prefill_kv(4, 0)
    assert not torch.equal(k1, k3)
    kf = k1.float()
    for h in range(4):
        ch = w.outlier_ch[h]
        means = kf[:, h, ch].mean(0).numpy()
        assert np.all(np.abs(np.abs(means) - 8.0) < 0.5)
    assert torch.equal(w.query(1, 5), w.query(1, 5))


def test_student_t_values_are_heavy_tailed():
    w = workloads.make("cfg4")
    w.lengths = [4096] + w.lengths[1:]
    _, v = w.prefill_kv(0, 0)
    x = v.float().flatten().numpy()
    kurt = np.mean((x - x.mean()) ** 4) / np.var(x) ** 2
    assert kurt > 6.0                                   # Gaussian is 3


def test_bench_reference_arm_prints_one_json_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "2",
                        "--warmup", "1"], capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr
    lines = [l for l in r.stdout.splitlines() if l.strip().startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["value"] > 0 and d["e2e"]["h2d_bytes_per_step"] == 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["config"]["workload"].startswith("cfg5")
