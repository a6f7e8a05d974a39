"""The byte accounting behind bench.py's HBM figures, against counts derived by
hand from the block's shapes (every weight byte once, plus the K and V rows
each token attends to), and the roofline helpers.  CPU only."""

import pytest

import bench
from decode_attention_block_gb300 import synth

# bf16 weights of one layer: q_k_v_proj (6144 x 2560) + g_proj (16 x 2560) +
# o_proj (2560 x 4096) + input_layernorm (2560), two bytes each
LAYER_BF16 = 2 * (6144 * 2560 + 16 * 2560 + 2560 * 4096 + 2560)
ROW_BF16 = 2 * 4 * 256 * 2           # one cache row of K and V: 4 KV heads x 256 dims, bf16


def test_layer_weight_bytes():
    assert LAYER_BF16 == 52_515_840
    wl = synth.workloads()["full+sliding_bf16_b1_pos700"]
    assert wl.weight_bytes_per_layer() == LAYER_BF16


@pytest.mark.parametrize("name,want", [
    # one sliding layer in fp32, 41 rows read (positions 0..40)
    ("sliding_f32_b1_pos40", 2 * LAYER_BF16 + 41 * 2 * ROW_BF16),
    # full layer reads 701 rows, the wrapped sliding layer its window of 512
    ("full+sliding_bf16_b1_pos700", 2 * LAYER_BF16 + 701 * ROW_BF16 + 512 * ROW_BF16),
    # 36 layers: 9 full at context 8192 (8193 rows), 27 sliding (512 rows)
    ("stack36_bf16_b1_ctx8192", 36 * LAYER_BF16 + 9 * 8193 * ROW_BF16 + 27 * 512 * ROW_BF16),
    # 8 sequences at 131072: the full layer's 131073 rows and the window of 512 each
    ("full+sliding_bf16_b8_ctx131072", 2 * LAYER_BF16 + 8 * 131073 * ROW_BF16 + 8 * 512 * ROW_BF16),
])
def test_step_bytes_match_hand_counts(name, want):
    wl = synth.workloads()[name]
    sb = bench.step_bytes(wl)
    assert sb["total"] == want
    per = sb["per_kernel"]
    assert per["qkv_gate"] + per["gate_oproj"] + per["attention"] == sb["total"]


def test_hand_counts_are_the_published_totals():
    # the totals quoted for these workloads
    assert 2 * LAYER_BF16 + 701 * ROW_BF16 + 512 * ROW_BF16 == 110_000_128
    assert 36 * LAYER_BF16 + 9 * 8193 * ROW_BF16 + 27 * 512 * ROW_BF16 == 2_249_220_096
    assert 2 * LAYER_BF16 + 8 * 131073 * ROW_BF16 + 8 * 512 * ROW_BF16 == 4_416_808_960


def test_ragged_batch_counts_each_sequence_window():
    wl = synth.workloads()["full+sliding_bf16_b64_ctx512-32768"]
    want = 2 * LAYER_BF16 + sum(p + 1 for p in wl.positions) * ROW_BF16 + 64 * 512 * ROW_BF16
    assert bench.step_bytes(wl)["total"] == want


def test_attention_bytes_split_by_layer_class():
    wl = synth.workloads()["full+sliding_bf16_b8_ctx131072"]
    per = bench.step_bytes(wl)["per_kernel"]
    # the full layer's attention alone: 8 sequences x 131073 rows
    assert per["attention_full"] == 8 * 131073 * ROW_BF16 == 4_295_000_064
    assert per["attention_sliding"] == 8 * 512 * ROW_BF16
    assert per["attention_full"] + per["attention_sliding"] == per["attention"]
    assert bench.stage_layers(wl, "attention_full") == [0]
    assert bench.stage_layers(wl, "attention_sliding") == [1]
    assert bench.stage_layers(wl, "qkv_rope") == [0, 1]


def test_default_workload_is_the_largest_single_gpu_config():
    wls = synth.workloads()
    sizes = {n: bench.step_bytes(w)["total"] for n, w in wls.items()}
    assert bench.DEFAULT_WORKLOAD == max(sizes, key=sizes.get)
    assert bench.TARGET_WORKLOAD in wls


def test_attention_traffic_scales_with_the_rows_read():
    t, src = bench.measured_traffic("some_other_workload", "attention_full", 1_000_000)
    assert t == int(1_000_000 * bench.ATTN_TRAFFIC_RATIO) and "scaled" in src
    assert 1.0 <= bench.ATTN_TRAFFIC_RATIO < 1.02
    t, src = bench.measured_traffic("full+sliding_bf16_b64_ctx512-32768", "attention_full", 1_000_000)
    assert t == int(1_000_000 * bench.ATTN_RAGGED_TRAFFIC_RATIO) and "16 sequences" in src
    assert 1.0 <= bench.ATTN_RAGGED_TRAFFIC_RATIO < 1.02
    # the capture's algorithmic bytes: the rows its 16 sequences read
    wl = synth.workloads()["full_bf16_b16_ctx512-32768"]
    assert bench.step_bytes(wl)["per_kernel"]["attention_full"] == 1_111_035_904
    assert wl.positions == synth.workloads()["full+sliding_bf16_b64_ctx512-32768"].positions[:16]
    t, src = bench.measured_traffic("full+sliding_bf16_b1_pos700", "qkv_rope", 0)
    assert t == bench.TRAFFIC[("full+sliding_bf16_b1_pos700", "qkv_rope")]
    assert bench.measured_traffic("x", "gate_oproj", 1)[0] is None


def test_whole_job_tokens_per_second():
    # 4 sequences per rank, 2 ranks, 100 steps in 50 ms (max over ranks)
    assert bench.job_tokens_per_s(4, 2, 100, 50.0) == pytest.approx(4 * 2 * 100 / 0.05)
