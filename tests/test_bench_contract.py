"""bench.py's command-line contract on CPU: the reference arm (the C oracle on
the host cores) prints one JSON line with the metric, unit and keys the
driver reads; the product arm has no CPU path and fails loudly without a GPU."""
import json
import os
import subprocess
import sys

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run(*args, timeout=600):
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], cwd=ROOT, capture_output=True,
                          text=True, timeout=timeout)


def test_reference_arm_prints_one_contract_line():
    sys.path.insert(0, ROOT)
    import bench
    r = _run("--impl", "reference", "--workload", "int8_pth_tiny", "--steps", "3", "--warmup", "3")
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    d = json.loads(lines[-1])
    assert d["metric"] == bench.METRIC and d["unit"] == "GB/s" and d["impl"] == "reference"
    assert d["value"] > 0 and d["higher_is_better"] is True and d["steps"] == 3 and d["warmup"] == 3
    assert d["n_gpus"] == 1 and d["scaling"] == "weak" and d["vs_baseline"] is None
    assert d["config"]["workload"] == "int8_pth_tiny"
    import workloads as wl
    assert d["config"] == bench.config_of(wl.WORKLOADS["int8_pth_tiny"])   # the product arm's config, too
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] == 1
    assert d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"] == {"value": d["value"], "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the behaviour without a GPU")
def test_product_arm_has_no_cpu_fallback():
    r = _run("--workload", "int8_pth_tiny", "--steps", "3", "--warmup", "3", "--no-cpu-baseline", timeout=300)
    assert r.returncode != 0
    assert not any(l.startswith("{") for l in r.stdout.splitlines())


def test_suite_names_resolve_and_cover_every_configuration():
    sys.path.insert(0, ROOT)
    import bench
    import workloads as wl
    names = set(bench.SUITE)
    assert set(wl.WORKLOADS) <= names and set(bench.VARIANTS) <= names and set(bench.SPEC_VARIANTS) <= names
    for n in bench.SUITE:
        w = bench.workload_by_name(n)
        assert w.name == n and bench.base_of(n) in wl.WORKLOADS
        lay = wl.paged_layout(w)
        assert bench.config_of(w, lay)["workload"] == n


def test_decode_kernel_named_per_workload():
    """The roofline names the kernel that runs: tcgen05 for the 4-bit modes with
    several queries, the KVarN kernel for KVarN (one or several queries), else
    the mma.sync kernel."""
    import bench
    assert bench.decode_kernel_of(bench.workload_by_name("nvfp4_b32_s32768")) == "decode_kernel"
    assert bench.decode_kernel_of(bench.workload_by_name("nvfp4_b32_s32768:spec4")) == "umma_decode_kernel"
    assert bench.decode_kernel_of(bench.workload_by_name("kvarn_b16_s16384:spec4")) == "kvarn_decode_kernel"
    assert bench.decode_kernel_of(bench.workload_by_name("pth_b64_u1k_32k:int4")) == "decode_kernel"
    for k in ("decode_kernel", "kvarn_decode_kernel", "umma_decode_kernel"):
        assert len(bench.kernel_sources_hash(k)) == 16


def test_launch_count_follows_the_plan():
    """A decode step launches the write and the decode, plus the split combine
    only when the plan asks for workspace (splits merged inside a thread-block
    cluster need none and launch no combine)."""
    import types
    import bench
    cases = [((1, 4096, 0), 2, ""), ((7, 4688, 1 << 20), 3, " + its split combine"),
             ((4, 1024, 0), 2, " (splits merged in a thread-block cluster)")]
    for plan, launches, label in cases:
        gw = types.SimpleNamespace(plan=plan)
        assert bench.GpuWorkload.launches_per_step(gw) == launches
        assert bench.GpuWorkload.split_merge(gw) == label
