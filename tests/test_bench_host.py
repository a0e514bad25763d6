"""Host-side checks of bench.py's accounting (no GPU): the algorithmic bytes of
one step against hand-computed figures, and the argument rules."""
import numpy as np
import pytest

import bench
from session_decode_step_dsb_gb300 import workloads


def test_step_bytes_llama68m_by_hand():
    ms = workloads.LLAMA68M
    lens = np.array([128, 2048])
    total, weights, kv = bench.step_bytes(ms, 2, 1, lens)
    # q8_0 rows of 768 columns: 24 blocks x 34 B = 816 B; of 3072 columns: 3264 B
    per_layer = 2304 * 816 + 768 * 816 + 6144 * 816 + 768 * 3264
    assert per_layer == 10_027_008
    assert weights == 2 * per_layer + 32000 * 816 == 46_166_016
    # K and V, fp16, 12 kv heads x 64 dims, once per layer
    assert kv == 2 * (128 + 2048) * 12 * 64 * 2 * 2
    # embedding rows (q8_0) and float32 logits of the two tokens
    assert total == weights + kv + 2 * (816 + 4 * 32000)


def test_step_bytes_qwen_gqa_reads_each_kv_head_once():
    ms = workloads.QWEN3_14B
    lens = np.array([1, 4096])
    _, _, kv = bench.step_bytes(ms, 2, 1, lens)
    assert kv == 40 * 4097 * 8 * 128 * 2 * 2   # 8 kv heads, not 40 query heads


def test_warmup_below_three_is_rejected():
    with pytest.raises(SystemExit):
        bench.main(["--warmup", "2"])


def test_cpu_all_cores_runs_every_process():
    """The all-core oracle run starts its spawned processes together and
    counts every process's steps (bounded: two processes, half a second)."""
    r = bench.cpu_all_cores("llama-68m", 2, 1, budget_s=0.5, max_workers=2)
    assert r["cores"] == min(2, r["host_cores"])
    assert r["value"] > 0 and r["unit"] == "tokens/s"
    assert "oracle steps over" in r["sample"]
    assert bench._cpu_model().endswith(")")


def test_clock_summary_keeps_the_samples_inside_the_region(tmp_path):
    """Samples stamped before or after the timed region are left out; a
    throttle reason seen only outside it does not count."""
    import datetime
    c = bench.ClockSampler(0)
    c.path = str(tmp_path / "clocks.csv")
    c.t_start = datetime.datetime(2026, 1, 2, 10, 0, 0, 100000)
    c.t_end = datetime.datetime(2026, 1, 2, 10, 0, 0, 200000)
    rows = [("10:00:00.050", 1400, "Active"), ("10:00:00.120", 2070, "Not Active"),
            ("10:00:00.140", 2060, "Not Active"), ("10:00:00.260", 1000, "Active")]
    with open(c.path, "w") as f:
        for t, mhz, hw in rows:
            f.write(f"2026/01/02 {t}, 0, {mhz}, 2070, 800.5, 0x0, {hw}, Not Active, Not Active, Not Active\n")
    s = c.summary()
    assert s["samples"] == 2 and s["in_region"] and s["sm_mhz"] == 2065 and s["reasons"] == []


def test_clock_summary_falls_back_to_every_sample(tmp_path):
    import datetime
    c = bench.ClockSampler(0)
    c.path = str(tmp_path / "clocks.csv")
    c.t_start = datetime.datetime(2026, 1, 2, 10, 0, 1)
    c.t_end = datetime.datetime(2026, 1, 2, 10, 0, 1, 5000)
    with open(c.path, "w") as f:
        f.write("2026/01/02 10:00:00.900, 0, 2070, 2070, 700, 0x0, Not Active, Not Active, Not Active, Active\n")
    s = c.summary()
    assert s["samples"] == 1 and not s["in_region"] and s["reasons"] == ["sw_power_cap"]
