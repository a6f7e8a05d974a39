"""The attention entry point that allocates nothing.

Callers that cannot allocate device memory (a host whose own memory pool owns
the device, a loop that must not allocate mid-run) call
spark_dbg_attention_noalloc, whose scratch is a fixed array inside the
library.  This file checks, through the C ABI, that it returns what the
workspace-based spark_dbg_attention returns, on two calls in a row (the array
keeps the previous call's contents), that it agrees with the oracle's
attention directly, that a clean call leaves the array's error word at zero,
and that it refuses a problem larger than its array.  It is collected last,
so a failure here leaves the rest of the suite already run.
"""

import numpy as np
import pytest
import torch

import oracle
from decode_attention_block_gb300 import build_lib, synth
from helpers import assert_close

pytestmark = pytest.mark.gpu

Q_DIM = 16 * 256


@pytest.fixture(scope="module")
def B():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    build_lib.build()
    from decode_attention_block_gb300 import binding
    binding.load()
    return binding


def _inputs(positions, is_full, seed):
    ring = 0 if is_full else 512
    wl = synth.Workload("noalloc", "", "bf16", positions, [synth.LayerSpec(is_full, ring)], seed=seed)
    kc, vc = synth.make_cache(wl, 0, "cuda")
    g = torch.Generator(device="cuda")
    g.manual_seed(seed + 1)
    q = torch.randn((len(positions), Q_DIM), generator=g, device="cuda")
    return ring, kc, vc, q


@pytest.mark.parametrize("is_full,positions", [(True, [3000, 9, 700, 131]), (False, [700, 40, 131072])])
def test_noalloc_matches_workspace_entry_on_two_calls(B, is_full, positions):
    ring, kc, vc, q = _inputs(positions, is_full, 900)
    geom = B.spark_geom_default()
    cls = B.SPARK_FULL if is_full else B.SPARK_SLIDING
    kv = B.KvLayer(kc, vc, ring)
    ws = B.make_workspace(geom, len(positions))
    want = torch.empty((len(positions), Q_DIM), device="cuda")
    B.spark_dbg_attention(geom, q, kv, cls, positions, want, ws)
    torch.cuda.synchronize()
    want_np = want.cpu().numpy()
    for call in range(2):
        got = torch.full((len(positions), Q_DIM), float("nan"), device="cuda")
        B.spark_dbg_attention_noalloc(geom, q, kv, cls, positions, got)
        torch.cuda.synchronize()
        assert_close(got.cpu().numpy(), want_np, f"no-alloc call {call}")
    assert B.spark_dbg_attention_noalloc_error_word() == 0


@pytest.mark.parametrize("is_full,positions", [
    (True, [20000, 0, 1023]),           # a long group (two CTAs per SM), a single row, a short one
    (False, [700, 511, 131072]),        # wrapped rings and a window that just fills
])
def test_noalloc_matches_the_oracle(B, is_full, positions):
    ring, kc, vc, q = _inputs(positions, is_full, 910)
    geom = B.spark_geom_default()
    got = torch.full((len(positions), Q_DIM), float("nan"), device="cuda")
    B.spark_dbg_attention_noalloc(geom, q, B.KvLayer(kc, vc, ring),
                                  B.SPARK_FULL if is_full else B.SPARK_SLIDING, positions, got)
    torch.cuda.synchronize()
    assert B.spark_dbg_attention_noalloc_error_word() == 0
    og = oracle.OracleGeometry()
    k_np, v_np = synth.to_numpy(kc), synth.to_numpy(vc)
    q64 = q.cpu().double().numpy()
    for b, p in enumerate(positions):
        seq_len, kv_start, active = oracle.window_params(p, is_full, og.window, ring)
        slots = np.array([oracle.read_slot(j, active) for j in range(kv_start, seq_len)], dtype=np.int64)
        want = oracle.attention_decode(q64[b].reshape(og.n_q, og.head_dim),
                                       oracle.cache_rows_to_f64(k_np[b][slots]),
                                       oracle.cache_rows_to_f64(v_np[b][slots]), og.scale, og.n_kv)
        assert_close(got[b].cpu().double().numpy(), want.reshape(-1), f"sequence {b} at {p}")


def test_noalloc_refuses_more_than_its_scratch(B):
    positions = [5] * 65                    # 65 sequences x 4 KV heads > 256 groups
    wl = synth.Workload("noalloc", "", "bf16", positions, [synth.LayerSpec(True)], seed=902)
    kc, vc = synth.make_cache(wl, 0, "cuda")
    q = torch.zeros((len(positions), Q_DIM), device="cuda")
    a = torch.zeros_like(q)
    geom = B.spark_geom_default()
    with pytest.raises(B.SparkError) as exc:
        B.spark_dbg_attention_noalloc(geom, q, B.KvLayer(kc, vc, 0), B.SPARK_FULL, positions, a)
    assert exc.value.status == -4
