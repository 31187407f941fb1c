"""Host logic of bench.py (no GPU): algorithmic bytes and flops, the choice of
roofline, the traffic lookup keyed by the kernel source, GPU ids for the clock
sampler, and the fields of the JSON line."""
import json
import os
import sys
import types

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import bench  # noqa: E402
import workloads as wl  # noqa: E402

PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
         "source": "test"}


def test_expert_bytes_from_the_format():
    # decode layer: gate, up and down each hold 7168 x 2048 int4 values (half a
    # byte each) and one bf16 scale per 32 of them
    w = wl.WORKLOADS["decode"]
    int4 = 3 * 7168 * 2048 // 2
    scales = 3 * 7168 * 2048 // 32 * 2
    assert int4 == 22_020_096 and scales == 2_752_512
    assert bench.expert_bytes(w) == int4 + scales == 24_772_608
    # latent experts read the latent width 3584 with I = 1024
    assert bench.expert_bytes(wl.WORKLOADS["latent"]) == 3 * 3584 * 1024 * 9 // 16


def test_roofline_decode_is_hbm_bound():
    w = wl.WORKLOADS["decode"]
    active, ms = 181, 0.942
    r = bench.roofline(w, ms, active, PEAKS)
    rows = 32 * 8
    act = rows * 7168 * 2 + 2 * rows * 2048 * 2 + rows * 7168 * 2
    assert r["bound"] == "hbm" and r["unit"] == "GB/s"
    assert r["algorithmic_bytes"] == active * 24_772_608 + act
    assert r["achieved"] == pytest.approx(r["algorithmic_bytes"] / (ms * 1e-3) / 1e9)
    assert r["frac"] == pytest.approx(r["achieved"] / 6800.0)
    assert r["peak_source"] == "test" and r["active_experts"] == active


# active experts as the workloads route them: prefill's 16 dead experts get no
# token, exact mode sends every token to the same 8
@pytest.mark.parametrize("name,active,bound", [("prefill", 368, "tensor"), ("exact", 8, "tensor"),
                                               ("latent", 384, "hbm")])
def test_roofline_bound_follows_intensity(name, active, bound):
    w = wl.WORKLOADS[name]
    r = bench.roofline(w, 1.0, active, PEAKS)
    flops = 2.0 * w.T * w.k * 3 * w.D * w.I
    assert r["algorithmic_flops"] == flops
    assert r["bound"] == bound
    if bound == "tensor":
        assert r["achieved"] == pytest.approx(flops / 1e-3 / 1e12)
        assert r["peak"] == 1700.0  # the sustained figure: the call is timed inside a loop
    # the ridge: flops per byte of the measured pair
    assert (flops / r["algorithmic_bytes"] >= 1700e12 / 6800e9) == (bound == "tensor")


def test_prefill_flops_match_the_stated_total():
    w = wl.WORKLOADS["prefill"]
    assert bench.roofline(w, 1.0, 368, PEAKS)["algorithmic_flops"] == pytest.approx(5.772e12,
                                                                                    rel=1e-3)


def test_traffic_is_reported_only_for_the_profiled_source():
    h = bench._source_hash()
    with open(os.path.join(ROOT, "profiles", "traffic.txt")) as f:
        rows = [l.split() for l in f if l.strip() and not l.startswith("#")]
    for name, src, nbytes in rows:
        got = bench._profiled_traffic(name)
        assert got == (float(nbytes) if src == h else None)
    assert bench._profiled_traffic("no_such_workload") is None


def test_visible_gpu_id():
    assert bench.visible_gpu_id("0,1", 1, 0) == "1"
    assert bench.visible_gpu_id("GPU-3f1e, GPU-77aa", 0, 5) == "GPU-3f1e"
    assert bench.visible_gpu_id(None, 0, 3) == "3"
    assert bench.visible_gpu_id("", 0, 2) == "2"
    assert bench.visible_gpu_id("4", 1, 0) == "0"   # fewer entries than ranks: current device


def test_peaks_are_positive_with_a_source():
    p = bench._peaks()
    assert p["source"] in ("measured", "fallback")
    assert p["hbm_gbs"] > 0 and p["bf16_tflops"] > 0 and p["bf16_tflops_sustained"] > 0


def _entry(w, ms, active):
    roof = bench.roofline(w, ms, active, PEAKS)
    e2e = {"value": 1.0, "unit": "tokens/s", "h2d_bytes_per_step": 1, "d2h_bytes_per_step": 1}
    clocks = {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": []}
    return {"value": w.T / ms * 1e3, "ms_per_step": ms, "roofline": roof, "e2e": e2e,
            "gpu_launches": 12, "clocks": clocks, "config": bench._config(w, 1, roof)}


def test_json_line_has_the_contract_fields(capsys):
    args = types.SimpleNamespace(steps=5, warmup=3)
    head = _entry(wl.WORKLOADS["prefill"], 5.7, 368)
    others = {"decode": _entry(wl.WORKLOADS["decode"], 0.99, 181),
              "exact": _entry(wl.WORKLOADS["exact"], 0.7, 8)}
    cpu = {"value": 0.3, "unit": "tokens/s", "cores": 4, "kind": "oracle", "sample": "s"}
    bench._report(args, 1, head, others, cpu)
    line = json.loads(capsys.readouterr().out.strip())
    for key in ["metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "roofline", "cpu_baseline", "e2e", "gpu_launches", "clocks", "workloads"]:
        assert key in line, key
    assert line["config"]["workload"] == "prefill" and line["higher_is_better"] is True
    assert line["scaling"] == "weak" and line["vs_baseline"] is None and line["steps"] == 5
    for key in ["bound", "achieved", "peak", "unit", "frac", "traffic"]:
        assert key in line["roofline"], key
    assert set(line["workloads"]) == {"decode", "exact"}
    for name, entry in line["workloads"].items():
        assert entry["config"]["workload"] == name
        for key in ["value", "ms_per_step", "roofline", "e2e", "clocks", "gpu_launches"]:
            assert key in entry, (name, key)


def test_bench_defaults_to_the_largest_workload():
    """The headline line is the prefill workload, the largest configuration;
    the other three are reported beside it."""
    args = bench._parser().parse_args([])
    assert args.config == "prefill"
    assert max(wl.WORKLOADS.values(), key=lambda w: w.T * w.k).name == "prefill"
    assert set(args.workloads.split(",")) == {"decode", "latent", "exact"}


def test_cpu_baseline_times_oracle_arithmetic_only(monkeypatch):
    """The sampler generates the expert weights of the pairs it is about to
    time before the clock starts: inside run() nothing is generated."""
    w = wl.workload("tiny", name="tiny")
    sampler = bench.OracleSampler(w)
    n = 5
    sampler.prepare(n)

    def no_generation(*a, **k):
        raise AssertionError("expert weights generated inside the timed region")

    monkeypatch.setattr(sampler.oi, "expert_arrays", no_generation)
    dt = sampler.run(n)
    assert dt > 0 and sampler.pair == n
