"""bench.py's reference arm (the fp64 CPU oracle on the host cores) keeps
the benchmark's output contract: one JSON line from rank 0 with the metric,
the throughput, the run shape, the CPU-baseline record and an end-to-end
record with no host/device copies; under torchrun the other ranks print
nothing and exit 0.  Runs without a GPU."""
import json
import os
import socket
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
ARGS = ["--impl", "reference", "--steps", "1", "--warmup", "0", "--ref-seqs", "1"]
KEYS = ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
        "vs_baseline", "dtype", "data", "config")


def _json_lines(out: str):
    return [json.loads(l) for l in out.splitlines() if l.startswith("{")]


def _check_line(d: dict, n_gpus: int):
    for k in KEYS:
        assert k in d, k
    assert d["impl"] == "reference"
    assert d["n_gpus"] == n_gpus and d["steps"] == 1 and d["warmup"] == 0
    assert d["value"] > 0 and d["ms_per_step"] > 0 and d["higher_is_better"] is True
    assert d["data"] == "synthetic" and "workload" in d["config"]
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["sample"] and cb["value"] == d["value"]
    e2e = d["e2e"]
    assert e2e["value"] == d["value"] and e2e["unit"] == d["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0


def test_reference_arm_prints_one_contract_line():
    r = subprocess.run([sys.executable, "bench.py"] + ARGS, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = _json_lines(r.stdout)
    assert len(lines) == 1
    _check_line(lines[0], 1)


def test_reference_arm_under_torchrun_prints_from_rank_0_only():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py", "--gpus", "2"] + ARGS
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = _json_lines(r.stdout)
    assert len(lines) == 1
    _check_line(lines[0], 2)


def _bench_module():
    import importlib.util
    spec = importlib.util.spec_from_file_location("bench_under_test", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def test_clock_record_from_nvidia_smi_samples():
    """The clock record: median SM clock, the highest max clock, and every
    throttle reason seen active in any sample; lines that are not samples
    (short, or with fields nvidia-smi could not read) are skipped."""
    B = _bench_module()
    cs = B.ClockSampler(0)
    cs.lines = [
        "0, 2070, 2070, 900.1, 0x0, Not Active, Not Active, Not Active, Not Active",
        "0, 1980, 2070, 1390.0, 0x4, Not Active, Not Active, Not Active, Active",
        "0, 2070, 2070, 950.0, 0x0, Not Active, Not Active, Not Active, Not Active",
        "0, [N/A], 2070, 0, 0x0, Not Active, Not Active, Not Active, Not Active",
        "garbage",
        "",
    ]
    s = cs.summary()
    assert s == {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"], "samples": 3}
    cs.lines.append("0, 1200, 2070, 700.0, 0x8, Active, Not Active, Active, Not Active")
    s = cs.summary()
    assert s["reasons"] == ["hw_slowdown", "sw_power_cap", "sw_thermal_slowdown"] and s["samples"] == 4
    assert s["sm_mhz"] == 2025.0
    cs.lines = []
    assert cs.summary() == {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}


def test_decode_algorithmic_bytes():
    """The roofline's numerator for a decode call: the 16K decode's
    437 796 992 B (the figure its DRAM-traffic capture is compared with);
    per closed tile one record per KV head of the size the C library gives a
    block (every preset); 512 B per raw open-tile token and KV head."""
    from bit_kv_cache_quantize_gb300 import build as Bld, inputs as I, kvarn as K
    B = _bench_module()
    w = I.qwen3_32b()
    assert B.decode_bytes(w.seq_lens, w) == 437_796_992
    Bld.build()
    for kb, vb in ((4, 2), (2, 2), (4, 4)):
        w = I.qwen3_32b()
        w.k_bits, w.v_bits = kb, vb
        cfg = K.make_config(w.num_kv_heads, w.num_q_heads, 1, w.dtype, k_bits=kb, v_bits=vb)
        one = B.decode_bytes([128], w) - B.decode_bytes([0], w)
        assert one == K.kvarn_block_bytes(cfg) + 4, (kb, vb)
        assert B.decode_bytes([128 + 5], w) - B.decode_bytes([128], w) == 5 * w.num_kv_heads * 2 * 128 * 2
