"""bench.py's host-side parts, on the CPU: the reference arm's JSON line (the fp64 oracle timed on the host), the
clock-sample summary that decides whether a timed run is kept, and the source hash that ties the committed ncu
traffic figure to the attention kernel it was measured on (bench.py reports no traffic once the hash differs)."""
import importlib.util
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    spec = importlib.util.spec_from_file_location("bench_under_test", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def test_reference_arm_prints_one_contract_line():
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "2", "--warmup", "1"], cwd=ROOT,
                       capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    b = _bench()
    assert d["impl"] == "reference" and d["metric"] == b.METRIC and d["unit"] == "GB/s"
    assert d["higher_is_better"] is True and d["steps"] == 2 and d["warmup"] == 1 and d["n_gpus"] == 1
    assert d["value"] > 0 and d["ms_per_step"] > 0 and d["dtype"] == "f64"
    assert d["config"]["workload"] == "llama3_8b_gqa_paged_decode"
    cpu = d["cpu_baseline"]
    assert cpu["kind"] == "oracle" and cpu["cores"] >= 1 and cpu["value"] == d["value"] and cpu["sample"]
    assert d["e2e"] == {"value": d["value"], "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}


def test_clock_summary_keeps_only_the_timed_window_and_reports_throttle_reasons():
    b = _bench()
    c = b.ClockSampler(0)
    c.t0, c.t1 = 10.0, 20.0
    row = "0, {sm}, 2070, 900.0, 0x0, {hw}, Not Active, Not Active, {pc}"
    c.lines = [(9.0, row.format(sm=300, hw="Not Active", pc="Not Active")),      # before the timed region
               (11.0, row.format(sm=2070, hw="Not Active", pc="Not Active")),
               (12.0, row.format(sm=2040, hw="Not Active", pc="Active")),
               (13.0, row.format(sm=2070, hw="Active", pc="Not Active")),
               (30.0, row.format(sm=100, hw="Not Active", pc="Not Active"))]     # after it
    s = c.summary()
    assert s["samples"] == 3 and s["sm_mhz"] == 2070.0 and s["sm_max_mhz"] == 2070.0
    assert s["reasons"] == ["hw_slowdown", "sw_power_cap"]
    assert s["samples_in_timed_region"] == 3
    assert b.ClockSampler(0).summary()["reasons"] == ["unsampled"]
    # with a clock window after the timed region (mark t2) its samples count too, and the ones inside the
    # timed region are told apart
    c.t2 = 25.0
    c.lines.insert(4, (22.0, row.format(sm=2055, hw="Not Active", pc="Not Active")))
    s = c.summary()
    assert s["samples"] == 4 and s["samples_in_timed_region"] == 3 and s["window_s"] == 15.0


def test_attention_source_hash_spans_the_attention_kernel():
    b = _bench()
    src = open(b.DECODE_SRC).read()
    a = src.index("// ============================================================================= 2. attention")
    e = src.index("// ============================================================================= 3. partition merge")
    assert e > a and "attend_kernel" in src[a:e] and "partition_reduce_kernel(" not in src[a:e]
    h = b.attend_source_sha256()
    assert len(h) == 64
    # the hash moves with the attention section, not only with the device header
    import hashlib
    assert h == hashlib.sha256((src[a:e] + open(b.DEVICE_HDR).read()).encode()).hexdigest()
    assert h != hashlib.sha256(open(b.DEVICE_HDR).read().encode()).hexdigest()


def test_every_measure_choice_has_its_function():
    """Each --measure choice and each leg of the default line resolves to a function (a missing one would only
    surface on a GPU machine)."""
    b = _bench()
    import inspect
    src = inspect.getsource(b.main)
    for name in ("run_ours", "run_reference", "run_swap", "run_prefill", "run_configs", "run_vmm", "measure_swap",
                 "measure_vmm", "measure_prefill", "measure_workloads", "measure_cache_ops", "run_e2e"):
        assert callable(getattr(b, name, None)), name
    for choice in ("swap", "prefill", "configs", "vmm"):
        assert f'"{choice}"' in src
