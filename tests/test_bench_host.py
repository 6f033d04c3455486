"""Host-side logic of bench.py on the CPU: the FLOP accounting behind the
metric, the whole-job aggregation over ranks (two gloo ranks), and the
reference arm's rank rule.  Nothing here needs a GPU."""
import importlib.util
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from synth import SHAPES

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    spec = importlib.util.spec_from_file_location("bench_under_test", os.path.join(ROOT, "bench.py"))
    m = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(m)
    return m


# Algorithmic FLOPs of one FINE step per workload, counted by hand from the
# block's GEMMs and the causal attention products: FFN 14·M·H·F; attention
# 30·M·H² + 9·B·S²·H (forward 8·M·H² + 2·B·S²·H, recompute 6·M·H² + 2·B·S²·H,
# backward 16·M·H² + 5·B·S²·H).
@pytest.mark.parametrize("name,gflop", [("ffn_bf16_h1024", 240.52), ("attn_bf16_h2048", 592.71),
                                        ("layer_bf16_h4096", 12437.5), ("stack4_bf16_h2560", 40030.0)])
def test_fine_flop_counts(name, gflop):
    b = _bench()
    assert b.flops_fine(SHAPES[name]) / 1e9 == pytest.approx(gflop, rel=2e-4)


def test_modes_are_credited_with_what_they_execute():
    b = _bench()
    s = SHAPES["layer_bf16_h4096"]
    M, H, F, B, S = s.rows, s.hidden, s.ffn, s.batch, s.seq
    fine = b.flops_fine(s, "fine")
    none = b.flops_fine(s, "none")
    sel = b.flops_fine(s, "selective")
    assert b.flops_fine(s, "full") == fine          # FULL's extra work is not credited
    assert fine - none == 2 * M * H * F + 6 * M * H * H + 2 * B * S * S * H   # the recompute
    assert sel - none == 2 * B * S * S * H          # the attention operation again
    f = SHAPES["ffn_bf16_h1024"]
    assert b.flops_fine(f, "selective") == b.flops_fine(f, "none")


def test_traffic_is_reported_only_for_a_captured_workload():
    b = _bench()
    for name in SHAPES:
        t = b.recorded_traffic(name)
        rec = b.NCU_TRAFFIC.get(name)
        if rec is None:
            assert t is None, name
        else:   # the capture's bytes while the GEMM sources hash to the captured ones
            assert t in (None, rec["bytes_per_launch"])
            assert (t is None) == (b.kernel_source_sha() != rec["source_sha256"])


def test_roofline_entries_aggregate_the_gemm_launches():
    b = _bench()
    pk = {"bf16_tflops": 2000.0, "hbm_gbs": 7000.0, "source": "measured"}
    rows = [{"kernel": "a", "shape": "1", "family": "gemm", "algorithmic": 2e12, "avg_us": 1e3,
             "frac": 1.0},
            {"kernel": "b", "shape": "2", "family": "gemm", "algorithmic": 1e12, "avg_us": 2e3,
             "frac": 0.25},
            {"kernel": "c", "shape": "3", "family": "attn_bwd", "algorithmic": 1e12,
             "avg_us": 1e3, "frac": 0.5},
            {"kernel": "d", "shape": "4", "family": "hbm", "algorithmic": 1e9, "avg_us": 1.0,
             "frac": 0.1}]
    out = b.roofline_entries(rows, pk, "no_such_workload")
    r = out["roofline"]
    assert r["achieved"] == pytest.approx(3e12 / 3e-3 / 1e12)   # 1000 TFLOP/s
    assert r["frac"] == pytest.approx(0.5)
    assert r["algorithmic_flops_per_launch"] == pytest.approx(1.5e12)
    assert r["avg_launch_s"] == pytest.approx(1.5e-3)
    assert r["traffic"] is None and r["bound"] == "tensor" and len(r["launches"]) == 2
    assert out["roofline_attention_bwd"]["frac"] == pytest.approx(0.5)
    assert "fp8_gemm" not in out
    rows.append({"kernel": "q", "shape": "5", "family": "mx", "bound": "hbm", "algorithmic": 1e9,
                 "avg_us": 1.0, "achieved": 1e3, "frac": 0.2})
    rows.append({"kernel": "mxg", "shape": "6", "family": "mx", "bound": "tensor",
                 "algorithmic": 4e12, "avg_us": 1e3, "achieved": 4000.0, "peak": 4000.0,
                 "frac": 1.0})
    out = b.roofline_entries(rows, pk, "no_such_workload")
    assert out["fp8_gemm"]["frac"] == 1.0 and len(out["fp8_gemm"]["quantize"]) == 1
    assert out["roofline"]["frac"] == pytest.approx(0.5)   # the MX rows are not in the bf16 GEMM family


def test_clock_summary_keeps_only_samples_inside_the_timed_regions():
    b = _bench()
    c = b.ClockSampler(0)
    c.samples = [(1.0, 1000.0, 2070.0, 0x1), (2.0, 2000.0, 2070.0, 0x4), (3.0, 2050.0, 2070.0, 0x0),
                 (4.0, 900.0, 2070.0, 0x20), (5.0, 1990.0, 2070.0, 0x0)]
    c.windows = [[1.5, 3.5], [4.5, 5.5]]
    sm = c.summary()
    assert sm["samples"] == 3 and sm["sm_mhz"] == 2000.0
    assert sm["reasons"] == ["sw_power_cap"]   # the thermal sample lies outside the regions
    c.windows = [[10.0, 11.0]]
    assert c.summary()["reasons"] == ["unsampled"]


@pytest.mark.parametrize("name", sorted(SHAPES))
@pytest.mark.parametrize("seconds", [0.01, 0.5, 5.0, 1e6])
def test_oracle_sample_is_the_largest_that_fits(name, seconds):
    b = _bench()
    shape, rate = SHAPES[name], 2e11
    s = b.oracle_sample(shape, "fine", seconds, rate)
    s.validate()
    assert s.batch % shape.sub_batches == 0 and s.batch <= shape.batch and s.seq <= shape.seq
    cost = lambda t: b.flops_fine(t) / rate
    if s.seq > 8:
        assert cost(s) <= seconds
    if s.seq < shape.seq:     # halved from a length that did not fit, one sub-batch's worth
        assert s.batch == shape.sub_batches and cost(s.replace(seq=2 * s.seq)) > seconds
    elif s.batch < shape.batch:
        assert cost(s.replace(batch=s.batch + shape.sub_batches)) > seconds
    if seconds == 1e6:
        assert s == shape


def test_whole_job_throughput_is_total_work_over_slowest_rank():
    b = _bench()
    assert b.whole_job_tflops(2e12, 4, 0.5) == pytest.approx(16.0)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        b = _bench()
        t = b.max_over_ranks(0.010 * (rank + 1), "cpu")   # rank r took (r + 1) * 10 ms
        out[rank] = b.whole_job_tflops(1e12, world, t)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_the_slowest_step():
    world, port = 2, _free_port()
    out = mp.Manager().dict()
    mp.spawn(_rank, args=(world, port, out), nprocs=world, join=True)
    # both ranks see the slowest rank's 20 ms: 2 replicas x 1 TFLOP / 0.02 s
    assert out[0] == pytest.approx(100.0) and out[1] == pytest.approx(100.0)


def test_single_process_max_is_the_value_itself():
    assert _bench().max_over_ranks(0.25, "cpu") == 0.25


def test_reference_arm_runs_on_rank_zero_only(monkeypatch, capsys):
    b = _bench()
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")

    class Args:
        steps, warmup, recompute, workload = 1, 0, "fine", "ffn_bf16_h1024"

    assert b.run_reference(Args, SHAPES["ffn_bf16_h1024"]) is None
    assert capsys.readouterr().out == ""   # no line from a non-zero rank


def test_reference_arm_prints_the_contract_line():
    """bench.py --impl reference end to end (the oracle on this host): one JSON
    line with the contract's keys, the oracle's own numbers in value, e2e and
    cpu_baseline."""
    import json
    import subprocess
    import sys
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--workload", "ffn_f32_h256", "--steps", "2", "--warmup", "1"],
                       capture_output=True, text=True, timeout=600, cwd=ROOT,
                       env={**os.environ, "RANK": "0", "WORLD_SIZE": "1"})
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for k in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
              "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
              "cpu_baseline", "e2e"):
        assert k in d, k
    assert d["impl"] == "reference" and d["unit"] == "TFLOP/s" and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"] == {"value": d["value"], "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}
    assert d["config"]["workload"] == "ffn_f32_h256" and d["steps"] == 2
