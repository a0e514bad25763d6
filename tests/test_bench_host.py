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
