"""Host helpers of bench.py that need no GPU, and its reference arm (the
oracle on the host cores), which runs end to end here.

The end-to-end measurement moves a step's x, y and row -> adapter ids in one
copy: they live in one byte buffer as views at 256-byte-aligned offsets (the
C ABI wants 16-byte-aligned rows).  The views must hold the original values,
not overlap, and together span the buffer.
"""
import pytest
import torch

import bench


def test_packed_views_hold_the_tensors_without_overlap():
    X = torch.randn(3, 40, dtype=torch.float16)
    Y = torch.randn(3, 24, dtype=torch.float32)
    ra = torch.tensor([2, -1, 0], dtype=torch.int32)
    buf, (x, y, r) = bench._packed([X, Y, ra], "cpu")
    assert torch.equal(x, X) and torch.equal(y, Y) and torch.equal(r, ra)
    base = buf.data_ptr()
    spans = sorted((v.data_ptr() - base, v.data_ptr() - base + v.nbytes) for v in (x, y, r))
    assert all(lo % 256 == 0 for lo, _ in spans)
    assert all(spans[i][1] <= spans[i + 1][0] for i in range(len(spans) - 1))
    assert spans[-1][1] == buf.nbytes
    # writing through the buffer is seen by the views (one copy moves all three)
    buf.zero_()
    assert not x.any() and not y.any() and not r.any()


def test_parallel_oracle_is_the_one_call_oracle():
    """The all-core CPU baseline runs the unmodified oracle on ranges of rows
    from several threads; the result must be the single call's, bit for bit,
    however the positions are cut (ranges inside a segment, across segments,
    more ranges than rows)."""
    from concurrent.futures import ThreadPoolExecutor

    import numpy as np

    import oracle

    rng = np.random.default_rng(3)
    T, L, H1, H2, r = 50, 6, 32, 24, 4
    ra = rng.integers(-1, L, T).astype(np.int32)
    X = rng.standard_normal((T, H1))
    A = rng.standard_normal((L, H1, r))
    B = rng.standard_normal((L, r, H2))
    Y = rng.standard_normal((T, H2))
    o = oracle.default()
    perm, sp, ix = o.build_segments(ra, L)
    ref = o.sgmv_apply(Y, X, A, B, sp, ix, 0.5, perm=perm, widened=True)
    with ThreadPoolExecutor(4) as pool:
        for n in (1, 3, 7, 50, 80):
            tasks = bench.oracle_tasks(perm, sp, ix, n)
            rows = np.concatenate([t[0] for t in tasks])
            assert np.array_equal(np.sort(rows), np.arange(T))  # every row once
            got = bench.oracle_apply_parallel(o, pool, Y, X, A, B, perm, sp, ix, 0.5, n)
            assert np.array_equal(got, ref)


def test_rotation_copies():
    assert bench.rotation_copies(9_175_040, 126 << 20) == 29
    assert bench.rotation_copies(300 << 20, 126 << 20) == 2
    assert bench.rotation_copies(90_000, 126 << 20) == 256   # capped: stays in L2


def test_default_workload_is_the_full_stack():
    args = bench.parse_args([])
    assert args.workload == "llama7b-stack" and args.gpus == 1 and args.warmup >= 3


@pytest.mark.parametrize("grouped", [True, False])
def test_stack_launch_groups_cover_every_projection_once(grouped):
    """Each layer's seven projections appear once, in layer order; a grouped
    launch only joins projections that read the same rows and have the same
    shapes (q, k, v; gate, up), never o or down (they read other rows)."""
    import bench
    from rank_gemv_gb300 import workloads as wl

    launches = bench.stack_launch_groups(grouped)
    assert len(launches) == wl.LLAMA7B_LAYERS * (4 if grouped else 7)
    seen = [(layer, k) for layer, g in launches for k in g]
    assert seen == [(layer, k) for layer in range(wl.LLAMA7B_LAYERS) for k in range(7)]
    same_rows = [{0, 1, 2}, {4, 5}]
    for _, g in launches:
        assert 1 <= len(g) <= 4
        if len(g) > 1:
            assert any(set(g) <= s for s in same_rows)
            assert len({wl.LLAMA7B_PROJ[k][1:] for k in g}) == 1


def test_reference_arm_prints_one_contract_line():
    """`bench.py --impl reference` (the oracle on the host cores) prints one
    JSON line with the arm's keys, the same metric and unit as the GPU arm,
    and an end-to-end figure that copies nothing."""
    import json
    import os
    import subprocess
    import sys

    out = subprocess.run([sys.executable, os.path.join(bench.ROOT, "bench.py"), "--impl", "reference",
                          "--steps", "3", "--warmup", "3", "--workload", "tiny"],
                         capture_output=True, text=True, timeout=600, check=True).stdout
    lines = [ln for ln in out.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["steps"] == 3 and d["warmup"] == 3
    assert d["metric"] == bench.METRIC and d["unit"] == "rows/s" and d["higher_is_better"]
    assert d["value"] > 0 and d["config"]["workload"] == "tiny"
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"] == {"value": d["value"], "unit": "rows/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}


def test_reference_arm_runs_on_rank_zero_only():
    """Under a two-rank launch only rank 0 runs the oracle and prints; rank 1
    exits at once with status 0 and prints nothing."""
    import os
    import subprocess
    import sys

    env = dict(os.environ, RANK="1", LOCAL_RANK="1", WORLD_SIZE="2")
    res = subprocess.run([sys.executable, os.path.join(bench.ROOT, "bench.py"), "--impl",
                          "reference", "--steps", "3", "--warmup", "3", "--workload", "tiny"],
                         capture_output=True, text=True, timeout=600, env=env)
    assert res.returncode == 0
    assert not [ln for ln in res.stdout.splitlines() if ln.startswith("{")]
