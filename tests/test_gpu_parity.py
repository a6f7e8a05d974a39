"""Parity of the CUDA path (through the C ABI) with the CPU oracle.

Every stage is checked on its own with inputs drawn by the seeded generators
(so a stage's input never comes from another CUDA stage), then the whole block
end to end on each workload, at the sizes the oracle finishes in seconds and
at full size on sampled sequences.  Cache-row placement is bit-exact: after a
call exactly the slot of each sequence's position has changed.
"""

import numpy as np
import pytest
import torch

import oracle
from decode_attention_block_gb300 import build_lib, synth
from helpers import MAX_ABS, REL_L2, assert_close, err_stats, np_weights, oracle_geom

pytestmark = pytest.mark.gpu

D = 256
N_Q, N_KV = 16, 4
Q_DIM, KV_DIM = N_Q * D, N_KV * D
QKVG_LD = Q_DIM + 2 * KV_DIM + N_Q


@pytest.fixture(scope="module")
def B():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    build_lib.build()
    from decode_attention_block_gb300 import binding
    binding.load()
    return binding


class SeqCaches:
    """Per-sequence host copies of a cache, indexable like [batch][rows]."""

    def __init__(self, rows: dict, dtype):
        self.rows = rows
        self.dtype = dtype

    def __getitem__(self, b):
        return self.rows[b]


def f64(x):
    return oracle.cache_rows_to_f64(np.asarray(x)) if np.asarray(x).dtype == np.uint16 \
        else np.asarray(x, dtype=np.float64)


def _gen(seed):
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    return g


def assert_only_slot_changed(before: torch.Tensor, after: torch.Tensor, b: int, slot: int, what: str):
    assert torch.equal(before[b, :slot], after[b, :slot]), f"{what}: rows below slot {slot} changed"
    assert torch.equal(before[b, slot + 1:], after[b, slot + 1:]), f"{what}: rows above slot {slot} changed"


# ---------------------------------------------------------------------------
# stage 1: RMSNorm + q_k_v_proj + g_proj + split + rope + cache-row write
# ---------------------------------------------------------------------------

SLOT_POSITIONS = [0, 40, 511, 512, 513, 700, 1023, 1024]


def _qkv_oracle(wl, w_np, h_np, positions, is_full):
    r, theta = oracle.rope_params_for(is_full, 64, 256, 5e6, 1e4)
    norm_w, qkv_w, g_w = f64(w_np["norm_w"]), f64(w_np["qkv_w"]), f64(w_np["g_w"])
    out = []
    for b, p in enumerate(positions):
        x = oracle.rms_norm(h_np[b], norm_w, 1e-6)
        qkv = oracle.project(qkv_w, x)
        g = oracle.project(g_w, x)
        q = oracle.rope_neox(qkv[:Q_DIM].reshape(N_Q, D), p, r, theta)
        k = oracle.rope_neox(qkv[Q_DIM:Q_DIM + KV_DIM].reshape(N_KV, D), p, r, theta)
        v = qkv[Q_DIM + KV_DIM:].reshape(N_KV, D)
        out.append({"q": q, "k": k, "v": v, "g": g, "qkv": qkv})
    return out


def _assert_row_close(got: torch.Tensor, want_f64: np.ndarray, what: str):
    """A written cache row against the oracle's value: the kernel rounds its
    fp32 result, so compare as floats, and nearly every element must round to
    the oracle's own rounding of the exact value."""
    g = f64(synth.to_numpy(got))
    assert_close(g, want_f64, what)
    if got.dtype == torch.bfloat16:
        same = synth.to_numpy(got) == oracle.f64_to_bf16_bits(want_f64)
        assert np.mean(same) > 0.97, f"{what}: only {np.mean(same):.3f} bit-identical"


PATHS = {"auto": 0, "gemv": 1, "mma": 2}


def _run_qkv_case(B, is_full, dtype, positions, path, seed):
    batch = len(positions)
    ring = 0 if is_full else 512
    wl = synth.Workload("t", "", dtype, positions, [synth.LayerSpec(is_full, ring)], seed=seed)
    w = synth.make_weights(wl, 0, "cuda")
    h = synth.make_h(wl, "cuda")
    kc, vc = synth.make_cache(wl, 0, "cuda")
    kc0, vc0 = kc.clone(), vc.clone()
    q_rot = torch.full((batch, Q_DIM), float("nan"), device="cuda")
    g_log = torch.full((batch, N_Q), float("nan"), device="cuda")
    geom = B.spark_geom_default()
    ws = B.make_workspace(geom, batch)
    cls = B.SPARK_FULL if is_full else B.SPARK_SLIDING
    B.spark_dbg_qkv_rope(geom, h, B.LayerWeights(**w), B.KvLayer(kc, vc, ring), cls, positions, q_rot, g_log,
                         ws, PATHS[path])
    torch.cuda.synchronize()
    assert B.spark_attn_error_word(ws) == 0
    want = _qkv_oracle(wl, np_weights(w), synth.to_numpy(h).astype(np.float64), positions, is_full)
    got_q, got_g = q_rot.cpu().numpy(), g_log.cpu().numpy()
    for b, p in enumerate(positions):
        # tighter than the block tolerance: an fp32 rope angle at 131072 would miss by ~1e-2
        assert_close(got_q[b], want[b]["q"].reshape(-1), f"q b={b} p={p}", max_abs=2e-3, rel_l2=2e-4)
        assert_close(got_g[b], want[b]["g"], f"g b={b} p={p}", max_abs=2e-3, rel_l2=2e-4)
        slot = oracle.write_slot(p, ring)
        _assert_row_close(kc[b, slot], want[b]["k"], f"k row b={b} p={p}")
        _assert_row_close(vc[b, slot], want[b]["v"], f"v row b={b} p={p}")
        assert_only_slot_changed(kc0, kc, b, slot, f"K b={b} p={p}")
        assert_only_slot_changed(vc0, vc, b, slot, f"V b={b} p={p}")
    return q_rot, g_log, kc, vc


@pytest.mark.parametrize("path", ["auto", "mma"])
@pytest.mark.parametrize("is_full", [True, False])
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("positions", [SLOT_POSITIONS, [131072], [3, 700, 9]])
def test_qkv_rope_and_cache_slots(B, is_full, dtype, positions, path):
    if path == "mma" and dtype == "f32":
        pytest.skip("the tensor-core path takes bf16 weights")
    _run_qkv_case(B, is_full, dtype, positions, path, seed=300 + len(positions))


def _ragged_positions(n, seed, hi=140000):
    """n seeded positions in [0, hi), the first ones the ring's edge cases."""
    rng = np.random.default_rng(seed)
    pos = [int(p) for p in rng.integers(0, hi, size=n)]
    edges = [0, 1, 511, 512, 513, 131072]
    k = min(n, len(edges))
    pos[:k] = edges[:k]
    return pos


@pytest.mark.parametrize("is_full", [True, False])
@pytest.mark.parametrize("batch", [5, 8, 64, 130, 300])
def test_qkv_rope_tensor_core_batches(B, is_full, batch):
    """The batched path: padding to 8 sequences, split-K tiles, and more than
    128 sequences (chunks of 128 in one launch, the last one partial)."""
    positions = _ragged_positions(batch, 700 + batch)
    if is_full:
        positions = [p % 2048 for p in positions]   # a linear cache holds every position
    _run_qkv_case(B, is_full, "bf16", positions, "auto", seed=310 + batch)


def test_qkv_rope_paths_agree_and_repeat(B):
    """GEMV and tensor-core paths give the same projections (up to fp32
    rounding order), and the tensor-core path gives bit-identical results call
    after call on one workspace (its split-K tickets are reset)."""
    positions = [5, 700, 131072, 40, 9, 513, 77]
    wl = synth.Workload("t", "", "bf16", positions, [synth.LayerSpec(False, 512)], seed=320)
    w = B.LayerWeights(**synth.make_weights(wl, 0, "cuda"))
    h = synth.make_h(wl, "cuda")
    geom = B.spark_geom_default()
    ws = B.make_workspace(geom, len(positions))
    res = []
    for path in (1, 2, 2, 2):
        kc, vc = synth.make_cache(wl, 0, "cuda")
        q = torch.empty((len(positions), Q_DIM), device="cuda")
        g = torch.empty((len(positions), N_Q), device="cuda")
        B.spark_dbg_qkv_rope(geom, h, w, B.KvLayer(kc, vc, 512), B.SPARK_SLIDING, positions, q, g, ws, path)
        res.append((q, g, kc, vc))
    torch.cuda.synchronize()
    assert B.spark_attn_error_word(ws) == 0
    ma, rel = err_stats(res[1][0].cpu().numpy(), res[0][0].cpu().numpy())
    assert ma < 2e-4 and rel < 2e-5, (ma, rel)
    ma, rel = err_stats(res[1][1].cpu().numpy(), res[0][1].cpu().numpy())
    assert ma < 2e-4 and rel < 2e-5, (ma, rel)
    for r in res[2:]:
        for x, y in zip(r, res[1]):
            assert torch.equal(x, y)


def test_rope_class_selection_reaches_the_kernel(B):
    """The full class rotates only dims [0, 64) of each head at theta 5e6; the
    sliding class rotates all 256 at theta 1e4: swapping them must show."""
    positions = [700]
    wl = synth.Workload("t", "", "bf16", positions, [synth.LayerSpec(True)], seed=303)
    w = synth.make_weights(wl, 0, "cuda")
    h = synth.make_h(wl, "cuda")
    geom = B.spark_geom_default()
    got = {}
    for is_full in (True, False):
        spec = synth.LayerSpec(is_full, 0 if is_full else 512)
        wl2 = synth.Workload("t", "", "bf16", positions, [spec], seed=304)
        kc, vc = synth.make_cache(wl2, 0, "cuda")
        q_rot = torch.empty((1, Q_DIM), device="cuda")
        g_log = torch.empty((1, N_Q), device="cuda")
        B.spark_dbg_qkv_rope(geom, h, B.LayerWeights(**w), B.KvLayer(kc, vc, spec.ring_capacity),
                             B.SPARK_FULL if is_full else B.SPARK_SLIDING, positions, q_rot, g_log,
                             B.make_workspace(geom, 1))
        got[is_full] = q_rot.view(N_Q, D).cpu().numpy()
    proj = _qkv_oracle(wl, np_weights(w), synth.to_numpy(h).astype(np.float64), positions, True)[0]["qkv"]
    proj_q = proj[:Q_DIM].reshape(N_Q, D)
    assert_close(got[True][:, 64:], proj_q[:, 64:], "full class passes dims 64.. through",
                 max_abs=1e-3, rel_l2=1e-4)
    assert np.max(np.abs(got[False][:, 64:] - proj_q[:, 64:])) > 0.1
    assert np.max(np.abs(got[True][:, :64] - got[False][:, :64])) > 0.1


# ---------------------------------------------------------------------------
# stage 2: split-K GQA decode attention
# ---------------------------------------------------------------------------

ATTN_CASES = [
    # id, is_full, ring, capacity (None: max position + 1), positions, n_ctas, dtype
    ("single_row", True, 0, None, [0], 0, "bf16"),
    ("full_p40", True, 0, None, [40], 0, "bf16"),
    ("full_p700_f32", True, 0, None, [700], 0, "f32"),
    ("sliding_ring_wrapped", False, 512, 512, [700], 0, "bf16"),
    ("sliding_ring_unwrapped", False, 512, 512, [40], 0, "f32"),
    ("sliding_linear_window", False, 0, 2048, [1500], 0, "bf16"),
    ("full_ragged", True, 0, None, [5, 700, 3000], 0, "bf16"),
    ("sliding_ring_edges", False, 512, 512, [0, 511, 512, 513, 1024, 131072], 0, "bf16"),
    ("split1", True, 0, None, [3000], 1, "bf16"),
    ("split2", True, 0, None, [3000], 2, "bf16"),
    ("split7", True, 0, None, [3000], 7, "bf16"),
    ("split64_ragged", True, 0, None, [5, 700, 3000, 17, 1], 64, "bf16"),
    ("split1000_ragged", True, 0, None, [5, 700, 3000, 17, 1], 1000, "bf16"),
    ("big_batch_bucket", False, 512, 512, list(range(0, 2000, 10)), 0, "bf16"),
    # long equal histories at small batch
    ("split_clusters_b1", True, 0, None, [8192], 0, "bf16"),
    ("split_clusters_b2", True, 0, None, [5000, 5000], 0, "bf16"),
    ("split_clusters_b4", True, 0, None, [2000] * 4, 0, "bf16"),
    ("split_clusters_f32", True, 0, None, [4000], 0, "f32"),
    # cluster mode at every cluster size the planner picks for short histories:
    # batch 1 takes up to 16 CTAs of ~32 rows (70 rows: 3, 150: 5, 200: 7,
    # 300: 10, 450: 15), larger batches up to 8 of ~64 (2 x 300: 5, ragged
    # 3 x up to 130: 3); the merge then has idle lanes in its shuffle groups
    ("cluster_b1_r70", True, 0, None, [69], 0, "bf16"),
    ("cluster_b1_r150", True, 0, None, [149], 0, "bf16"),
    ("cluster_b1_r200_f32", True, 0, None, [199], 0, "f32"),
    ("cluster_b1_r300", True, 0, None, [299], 0, "bf16"),
    ("cluster_b1_r450", True, 0, None, [449], 0, "bf16"),
    ("cluster_b2_r300", True, 0, None, [299, 299], 0, "bf16"),
    ("cluster_b3_ragged", True, 0, None, [129, 100, 60], 0, "bf16"),
    # equal groups that nearly fill the GPU: one CTA per (sequence, KV head), no merge
    ("whole_groups_b64_ring", False, 512, 512, [700] * 64, 0, "bf16"),
    ("whole_groups_b30_full", True, 0, None, [299] * 30, 0, "bf16"),
]


def _attention_oracle(q, kc_np, vc_np, positions, is_full, ring, window=512):
    out = []
    for b, p in enumerate(positions):
        seq_len, kv_start, active = oracle.window_params(p, is_full, window, ring)
        slots = [oracle.read_slot(j, active) for j in range(kv_start, seq_len)]
        out.append(oracle.attention_decode(q[b].reshape(N_Q, D), f64(kc_np[b][slots]),
                                           f64(vc_np[b][slots]), 1 / 16, N_KV).reshape(-1))
    return np.stack(out)


@pytest.mark.parametrize("case", ATTN_CASES, ids=[c[0] for c in ATTN_CASES])
def test_attention_matches_oracle(B, case):
    _, is_full, ring, cap, positions, n_ctas, dtype = case
    batch = len(positions)
    wl = synth.Workload("t", "", dtype, positions, [synth.LayerSpec(is_full, ring)], seed=400 + batch)
    if cap is not None and ring == 0:
        wl.positions = positions
        kc, vc = synth.make_cache(wl, 0, "cuda")
        extra = cap - kc.shape[1]
        if extra > 0:
            pad = torch.randn((batch, extra, N_KV, D), generator=_gen(401), device="cuda").to(kc.dtype)
            kc = torch.cat([kc, pad], 1).contiguous()
            vc = torch.cat([vc, pad.flip(0)], 1).contiguous()
    else:
        kc, vc = synth.make_cache(wl, 0, "cuda")
    q = torch.randn((batch, Q_DIM), generator=_gen(402), device="cuda")
    a = torch.full((batch, Q_DIM), float("nan"), device="cuda")
    geom = B.spark_geom_default()
    ws = B.make_workspace(geom, batch)
    B.spark_dbg_attention(geom, q, B.KvLayer(kc, vc, ring), B.SPARK_FULL if is_full else B.SPARK_SLIDING,
                          positions, a, ws, n_ctas=n_ctas)
    assert B.spark_attn_error_word(ws) == 0
    got = a.cpu().numpy()
    want = _attention_oracle(q.cpu().numpy().astype(np.float64), synth.to_numpy(kc), synth.to_numpy(vc),
                             positions, is_full, ring)
    assert_close(got, want, "attention")
    if positions == [0]:
        # one row: softmax weight 1, the output is that row's v, exactly
        v0 = vc[0, 0].float().cpu().numpy()
        for h in range(N_Q):
            assert np.array_equal(got[0, h * D:(h + 1) * D], v0[h // 4])


def test_attention_split_count_invariance_and_reuse(B):
    """The result does not depend on how many CTAs share the rows, and the
    merge tickets are reset so a workspace serves call after call."""
    positions = [3000, 9, 4097]
    wl = synth.Workload("t", "", "bf16", positions, [synth.LayerSpec(True)], seed=410)
    kc, vc = synth.make_cache(wl, 0, "cuda")
    q = torch.randn((3, Q_DIM), generator=_gen(411), device="cuda")
    geom = B.spark_geom_default()
    ws = B.make_workspace(geom, 3)
    results = []
    for n in (1, 2, 7, 64, 0, 64, 1000, 3):
        a = torch.empty((3, Q_DIM), device="cuda")
        B.spark_dbg_attention(geom, q, B.KvLayer(kc, vc, 0), B.SPARK_FULL, positions, a, ws, n_ctas=n)
        results.append(a.cpu().numpy())
    assert B.spark_attn_error_word(ws) == 0
    for r in results[1:]:
        ma, _ = err_stats(r, results[0])
        assert ma < 1e-5
    ws_host = ws.cpu()
    assert int(ws_host[256:256 + 4 * 3 * 4].view(torch.int32).abs().sum()) == 0   # tickets back at 0


def test_equal_long_histories_reuse_and_split_invariance(B):
    """Equal long histories at batch 2: the default grid gives the result of an
    explicit 152-CTA split, call after call on one workspace, with the merge
    tickets back at 0."""
    positions = [6000, 6000]
    wl = synth.Workload("t", "", "bf16", positions, [synth.LayerSpec(True)], seed=412)
    kc, vc = synth.make_cache(wl, 0, "cuda")
    q = torch.randn((2, Q_DIM), generator=_gen(413), device="cuda")
    geom = B.spark_geom_default()
    ws = B.make_workspace(geom, 2)
    results = []
    for n in (0, 0, 152, 0):
        a = torch.empty((2, Q_DIM), device="cuda")
        B.spark_dbg_attention(geom, q, B.KvLayer(kc, vc, 0), B.SPARK_FULL, positions, a, ws, n_ctas=n)
        results.append(a.cpu().numpy())
    assert B.spark_attn_error_word(ws) == 0
    for r in results[1:]:
        ma, _ = err_stats(r, results[0])
        assert ma < 1e-5
    assert np.array_equal(results[0], results[1]) and np.array_equal(results[0], results[3])
    ws_host = ws.cpu()
    assert int(ws_host[256:256 + 4 * 2 * 4].view(torch.int32).abs().sum()) == 0   # tickets back at 0


# ---------------------------------------------------------------------------
# stage 3: head gate + o_proj + residual
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("dtype,batch,path", [("bf16", 1, "auto"), ("bf16", 2, "auto"), ("bf16", 5, "auto"), ("f32", 2, "auto"),
                                              ("bf16", 4, "auto"), ("bf16", 1, "mma"), ("bf16", 4, "gemv"),
                                              ("bf16", 64, "auto"), ("bf16", 130, "auto")])
def test_gate_oproj_matches_oracle(B, dtype, batch, path):
    wl = synth.Workload("t", "", dtype, [0] * batch, [synth.LayerSpec(True)], seed=500 + batch)
    w = synth.make_weights(wl, 0, "cuda")
    h = synth.make_h(wl, "cuda")
    a = torch.randn((batch, Q_DIM), generator=_gen(501), device="cuda")
    g_log = torch.randn((batch, N_Q), generator=_gen(502), device="cuda") * 2
    out = torch.empty_like(h)
    geom = B.spark_geom_default()
    ws = B.make_workspace(geom, batch)
    B.spark_dbg_gate_oproj(geom, a, g_log, h, B.LayerWeights(**w), out, ws, PATHS[path])
    # in place: out aliases h
    h2 = h.clone()
    B.spark_dbg_gate_oproj(geom, a, g_log, h2, B.LayerWeights(**w), h2, ws, PATHS[path])
    torch.cuda.synchronize()
    assert B.spark_attn_error_word(ws) == 0
    assert torch.equal(out, h2)
    wo = f64(np_weights(w)["o_w"])
    an, gn, hn = a.cpu().numpy(), g_log.cpu().numpy(), h.cpu().numpy().astype(np.float64)
    for b in range(batch):
        gated = oracle.head_gate(an[b].reshape(N_Q, D), gn[b].astype(np.float64))
        o = oracle.project(wo, gated.reshape(-1))
        # GEMV and GEMM both accumulate fp32 products of the exact bf16 weights
        assert_close(out[b].cpu().numpy() - hn[b], o, f"o b={b}", max_abs=2e-3, rel_l2=2e-4)


# ---------------------------------------------------------------------------
# the whole block, end to end through spark_attn_decode
# ---------------------------------------------------------------------------

def run_workload_parity(B, wl: synth.Workload, sample=None, layers=None):
    """Decode one step through every layer of the workload (each layer's input
    is the previous layer's output), on the GPU and in the oracle, and compare
    each layer's contribution o = out - in, the written cache rows, and the
    untouched rest of the caches."""
    seqs = list(range(wl.batch)) if sample is None else list(sample)
    geom = B.spark_geom_default()
    ws = B.make_workspace(geom, wl.batch)
    ogeom = oracle_geom(wl)
    cur = synth.make_h(wl, "cuda")
    cur_np = {b: synth.to_numpy(cur[b]).astype(np.float64) for b in seqs}
    h0 = {b: cur_np[b].copy() for b in seqs}
    worst = (0.0, 0.0)
    for li in (range(len(wl.layers)) if layers is None else layers):
        spec = wl.layers[li]
        w = synth.make_weights(wl, li, "cuda")
        kc, vc = synth.make_cache(wl, li, "cuda")
        kc0, vc0 = kc.clone(), vc.clone()
        k_np = SeqCaches({b: synth.to_numpy(kc[b]) for b in seqs}, np.uint16 if wl.dtype == "bf16" else np.float32)
        v_np = SeqCaches({b: synth.to_numpy(vc[b]) for b in seqs}, k_np.dtype)
        out = torch.empty_like(cur)
        cls = B.SPARK_FULL if spec.is_full else B.SPARK_SLIDING
        B.spark_attn_decode(geom, cur, B.LayerWeights(**w), B.KvLayer(kc, vc, spec.ring_capacity), cls,
                            wl.positions, out, ws)
        torch.cuda.synchronize()
        h_in = np.zeros((wl.batch, wl.hidden))
        for b in seqs:
            h_in[b] = cur_np[b]
        res = oracle.decode_step(ogeom, h_in, np_weights(w), k_np, v_np, spec.is_full, wl.positions,
                                 spec.ring_capacity, sequences=seqs)
        got_out = out.cpu().numpy().astype(np.float64)
        got_in = cur.cpu().numpy().astype(np.float64)
        for i, b in enumerate(seqs):
            ma, rel = assert_close(got_out[b] - got_in[b], res["o"][i], f"layer {li} o b={b}")
            worst = (max(worst[0], ma), max(worst[1], rel))
            slot = res["slot"][i]
            # the rows are projections of the layer input, computed in fp32 here
            # and fp64 there, then rounded: compared as float outputs
            assert_close(f64(synth.to_numpy(kc[b, slot])), f64(res["k_row"][i]), f"layer {li} k row b={b}")
            assert_close(f64(synth.to_numpy(vc[b, slot])), f64(res["v_row"][i]), f"layer {li} v row b={b}")
            cur_np[b] = res["out"][i]
        for b in range(wl.batch):
            slot = oracle.write_slot(wl.positions[b], spec.ring_capacity)
            assert_only_slot_changed(kc0, kc, b, slot, f"layer {li} K b={b}")
            assert_only_slot_changed(vc0, vc, b, slot, f"layer {li} V b={b}")
        cur = out
        del kc, vc, kc0, vc0
    assert B.spark_attn_error_word(ws) == 0
    got_final = cur.cpu().numpy().astype(np.float64)
    for b in seqs:
        assert_close(got_final[b] - h0[b], cur_np[b] - h0[b], f"stack output b={b}")
    return worst


WORKLOADS = synth.workloads()


def test_decode_sliding_f32_b1_pos40(B):
    run_workload_parity(B, WORKLOADS["sliding_f32_b1_pos40"])


def test_decode_full_sliding_bf16_b1_pos700(B):
    wl = WORKLOADS["full+sliding_bf16_b1_pos700"]
    run_workload_parity(B, wl)                 # full then sliding, chained
    run_workload_parity(B, wl, layers=[1])     # the sliding layer alone on the same h


def test_decode_stack36_bf16_b1_ctx8192(B):
    run_workload_parity(B, WORKLOADS["stack36_bf16_b1_ctx8192"])


def test_decode_ragged_b64(B):
    wl = WORKLOADS["full+sliding_bf16_b64_ctx512-32768"]
    pos = np.array(wl.positions)
    sample = sorted({int(pos.argmin()), int(pos.argmax()), 7, 31, 50})
    run_workload_parity(B, wl, sample=sample)


def test_decode_long_context_b8_ctx131072(B):
    run_workload_parity(B, WORKLOADS["full+sliding_bf16_b8_ctx131072"], sample=[0, 5])


def test_decode_short_history_b1(B):
    """One sequence at position 10 (11 rows): attention holds a handful of SMs,
    so o_proj's grid is cut to the SMs left free (148 CTAs of 17-18 rows)."""
    wl = synth.Workload("b1_short", "", "bf16", [10], [synth.LayerSpec(True, 0), synth.LayerSpec(False, 512)],
                        seed=605)
    run_workload_parity(B, wl)


def test_decode_position_zero_and_small_batch_edges(B):
    wl = synth.Workload("edges", "", "bf16", [0, 1, 2, 513], [synth.LayerSpec(True, 0), synth.LayerSpec(False, 512)],
                        seed=600)
    run_workload_parity(B, wl)


def test_zero_o_proj_returns_h_exactly(B):
    wl = synth.Workload("t", "", "bf16", [100, 3], [synth.LayerSpec(True)], seed=610)
    w = synth.make_weights(wl, 0, "cuda")
    w["o_w"].zero_()
    kc, vc = synth.make_cache(wl, 0, "cuda")
    h = synth.make_h(wl, "cuda")
    out = torch.empty_like(h)
    geom = B.spark_geom_default()
    ws = B.make_workspace(geom, 2)
    B.spark_attn_decode(geom, h, B.LayerWeights(**w), B.KvLayer(kc, vc, 0), B.SPARK_FULL, wl.positions, out, ws)
    torch.cuda.synchronize()
    assert torch.equal(out, h)


# ---------------------------------------------------------------------------
# the whole stack in one call (one persistent kernel, or the per-layer path)
# ---------------------------------------------------------------------------

def run_stack_parity(B, wl: synth.Workload, sample=None):
    """spark_attn_decode_stack over every layer of the workload against the
    oracle run layer after layer (each layer's input is its own previous
    output), and against the per-layer C entry point."""
    seqs = list(range(wl.batch)) if sample is None else list(sample)
    geom = B.spark_geom_default()
    ws = B.make_workspace(geom, wl.batch)
    ogeom = oracle_geom(wl)
    h = synth.make_h(wl, "cuda")
    layers = []
    for li, spec in enumerate(wl.layers):
        w = synth.make_weights(wl, li, "cuda")
        kc, vc = synth.make_cache(wl, li, "cuda")
        layers.append((spec, w, kc, vc, kc.clone(), vc.clone()))
    # oracle chain, from the caches as they are before any call
    cur = {b: synth.to_numpy(h[b]).astype(np.float64) for b in seqs}
    h0 = {b: cur[b].copy() for b in seqs}
    want_rows = []
    for spec, w, kc, vc, _, _ in layers:
        k_np = SeqCaches({b: synth.to_numpy(kc[b]) for b in seqs}, np.uint16 if wl.dtype == "bf16" else np.float32)
        v_np = SeqCaches({b: synth.to_numpy(vc[b]) for b in seqs}, k_np.dtype)
        h_in = np.zeros((wl.batch, wl.hidden))
        for b in seqs:
            h_in[b] = cur[b]
        res = oracle.decode_step(ogeom, h_in, np_weights(w), k_np, v_np, spec.is_full, wl.positions,
                                 spec.ring_capacity, sequences=seqs)
        want_rows.append(res)
        for i, b in enumerate(seqs):
            cur[b] = res["out"][i]
    # the stack call
    out = torch.empty_like(h)
    B.spark_attn_decode_stack(geom, h, [B.LayerWeights(**w) for _, w, *_ in layers],
                              [B.KvLayer(kc, vc, spec.ring_capacity) for spec, _, kc, vc, _, _ in layers],
                              [B.SPARK_FULL if spec.is_full else B.SPARK_SLIDING for spec, *_ in layers],
                              wl.positions, out, ws)
    torch.cuda.synchronize()
    assert B.spark_attn_error_word(ws) == 0
    got = out.cpu().numpy().astype(np.float64)
    for b in seqs:
        assert_close(got[b] - h0[b], cur[b] - h0[b], f"stack output b={b}")
    for li, (spec, w, kc, vc, kc0, vc0) in enumerate(layers):
        res = want_rows[li]
        for i, b in enumerate(seqs):
            slot = res["slot"][i]
            assert_close(f64(synth.to_numpy(kc[b, slot])), f64(res["k_row"][i]), f"layer {li} k row b={b}")
            assert_close(f64(synth.to_numpy(vc[b, slot])), f64(res["v_row"][i]), f"layer {li} v row b={b}")
        for b in range(wl.batch):
            slot = oracle.write_slot(wl.positions[b], spec.ring_capacity)
            assert_only_slot_changed(kc0, kc, b, slot, f"layer {li} K b={b}")
            assert_only_slot_changed(vc0, vc, b, slot, f"layer {li} V b={b}")
    # the per-layer entry point on the same inputs (caches restored) gives the same answer
    for spec, w, kc, vc, kc0, vc0 in layers:
        kc.copy_(kc0)
        vc.copy_(vc0)
    cur_t = h.clone()
    for spec, w, kc, vc, _, _ in layers:
        nxt = torch.empty_like(cur_t)
        B.spark_attn_decode(geom, cur_t, B.LayerWeights(**w), B.KvLayer(kc, vc, spec.ring_capacity),
                            B.SPARK_FULL if spec.is_full else B.SPARK_SLIDING, wl.positions, nxt, ws)
        cur_t = nxt
    torch.cuda.synchronize()
    ma, rel = err_stats(got - synth.to_numpy(h).astype(np.float64),
                        cur_t.cpu().numpy().astype(np.float64) - synth.to_numpy(h).astype(np.float64))
    assert ma < 2e-3 and rel < 1e-3, f"stack vs per-layer: max_abs {ma:.3e} rel {rel:.3e}"


def test_stack_full_sliding_bf16_b1_pos700(B):
    run_stack_parity(B, WORKLOADS["full+sliding_bf16_b1_pos700"])


def test_stack36_bf16_b1_ctx8192(B):
    run_stack_parity(B, WORKLOADS["stack36_bf16_b1_ctx8192"])


def test_stack_batch_edges(B):
    wl = synth.Workload("edges", "", "bf16", [0, 1, 513, 700],
                        [synth.LayerSpec(True, 0), synth.LayerSpec(False, 512), synth.LayerSpec(False, 512)],
                        seed=620)
    run_stack_parity(B, wl)


def test_stack_two_sequences_and_fallbacks(B):
    run_stack_parity(B, synth.Workload("b2", "", "bf16", [40, 3000],
                                       [synth.LayerSpec(False, 512), synth.LayerSpec(True, 0)], seed=621))
    # fp32 weights and batch 8 take the per-layer path
    run_stack_parity(B, WORKLOADS["sliding_f32_b1_pos40"])
    run_stack_parity(B, synth.Workload("b8", "", "bf16", [5, 9, 700, 1, 40, 513, 88, 300],
                                       [synth.LayerSpec(True, 0), synth.LayerSpec(False, 512)], seed=622))


def test_stack_more_layers_than_one_launch(B):
    wl = synth.Workload("stack45", "", "bf16", [600],
                        [synth.LayerSpec(i % 4 == 3, 0 if i % 4 == 3 else 512) for i in range(45)], seed=623)
    run_stack_parity(B, wl)


# ---------------------------------------------------------------------------
# a chunk of consecutive tokens of one sequence (prefill / verify)
# ---------------------------------------------------------------------------

PREFILL_CASES = [
    # id, is_full, ring, capacity, p0, m, dtype
    ("full_p0_m1", True, 0, 64, 0, 1, "bf16"),
    ("full_p0_m7", True, 0, 64, 0, 7, "bf16"),
    ("full_p700_m3", True, 0, 800, 700, 3, "bf16"),
    ("full_p700_m37", True, 0, 800, 700, 37, "bf16"),
    ("full_p100_m130", True, 0, 300, 100, 130, "bf16"),
    ("sliding_ring_fills_inside", False, 512, 512, 490, 45, "bf16"),
    ("sliding_ring_wraps_inside", False, 512, 512, 1000, 100, "bf16"),
    ("sliding_ring_outgrown", False, 512, 512, 300, 600, "bf16"),
    ("sliding_f32", False, 512, 512, 40, 3, "f32"),
    ("sliding_linear", False, 0, 2048, 1500, 20, "bf16"),
    # chunks long enough for the query-grouped kernel (one CTA per 4 tokens and KV head)
    ("grouped_full_p700_m300", True, 0, 1024, 700, 300, "bf16"),
    ("grouped_full_p0_m161", True, 0, 200, 0, 161, "bf16"),
    ("grouped_sliding_ring_wraps", False, 512, 512, 1000, 257, "bf16"),
    ("grouped_sliding_ring_fills", False, 512, 512, 300, 400, "bf16"),
    ("grouped_sliding_linear", False, 0, 2048, 1500, 170, "bf16"),
]


def _prefill_inputs(is_full, ring, cap, p0, m, dtype, seed):
    wl = synth.Workload("t", "", dtype, [p0], [synth.LayerSpec(is_full, ring)], seed=seed)
    w = synth.make_weights(wl, 0, "cuda")
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    kc = torch.randn((1, cap, N_KV, D), generator=_gen(seed + 1), device="cuda").to(tdt)
    vc = torch.randn((1, cap, N_KV, D), generator=_gen(seed + 2), device="cuda").to(tdt)
    h = torch.randn((m, 2560), generator=_gen(seed + 3), device="cuda")
    return wl, w, kc, vc, h


@pytest.mark.parametrize("case", PREFILL_CASES, ids=[c[0] for c in PREFILL_CASES])
def test_prefill_chunk_matches_oracle(B, case):
    _, is_full, ring, cap, p0, m, dtype = case
    wl, w, kc, vc, h = _prefill_inputs(is_full, ring, cap, p0, m, dtype, 900 + m)
    kc0, vc0 = kc.clone(), vc.clone()
    geom = B.spark_geom_default()
    ws = B.make_workspace(geom, m)
    out = torch.empty_like(h)
    B.spark_attn_prefill(geom, h, B.LayerWeights(**w), B.KvLayer(kc, vc, ring),
                         B.SPARK_FULL if is_full else B.SPARK_SLIDING, p0, out, ws)
    torch.cuda.synchronize()
    assert B.spark_attn_error_word(ws) == 0
    res = oracle.prefill_chunk(oracle_geom(wl), synth.to_numpy(h).astype(np.float64), np_weights(w),
                               synth.to_numpy(kc0[0]), synth.to_numpy(vc0[0]), is_full, p0, ring)
    got_o = out.cpu().numpy().astype(np.float64) - h.cpu().numpy().astype(np.float64)
    for t in range(m):
        assert_close(got_o[t], res["o"][t], f"token {t} (position {p0 + t}) o")
    # the cache afterwards: exactly the oracle's rows changed, to the same values
    want_k, want_v = res["k_cache"], res["v_cache"]
    changed = np.any((want_k != synth.to_numpy(kc0[0])).reshape(cap, -1), axis=1) | \
        np.any((want_v != synth.to_numpy(vc0[0])).reshape(cap, -1), axis=1)
    got_k, got_v = synth.to_numpy(kc[0]), synth.to_numpy(vc[0])
    for slot in range(cap):
        if changed[slot]:
            assert_close(f64(got_k[slot]), f64(want_k[slot]), f"k slot {slot}")
            assert_close(f64(got_v[slot]), f64(want_v[slot]), f"v slot {slot}")
        else:
            assert np.array_equal(got_k[slot], want_k[slot]), f"k slot {slot} changed"
            assert np.array_equal(got_v[slot], want_v[slot]), f"v slot {slot} changed"
    assert int(changed.sum()) == (min(m, ring) if ring > 0 else m)


def test_prefill_grouped_ignores_non_finite_unused_rows(B):
    # cache rows the chunk does not read (positions >= p0 of a linear cache)
    # hold NaN: the short tiles' stale rows must not reach any token
    is_full, ring, cap, p0, m = True, 0, 1024, 700, 200
    wl, w, kc, vc, h = _prefill_inputs(is_full, ring, cap, p0, m, "bf16", 4242)
    kc[0, p0:] = float("nan")
    vc[0, p0:] = float("nan")
    kc0, vc0 = kc.clone(), vc.clone()
    geom = B.spark_geom_default()
    ws = B.make_workspace(geom, m)
    out = torch.empty_like(h)
    B.spark_attn_prefill(geom, h, B.LayerWeights(**w), B.KvLayer(kc, vc, ring), B.SPARK_FULL, p0, out, ws)
    torch.cuda.synchronize()
    assert B.spark_attn_error_word(ws) == 0
    res = oracle.prefill_chunk(oracle_geom(wl), synth.to_numpy(h).astype(np.float64), np_weights(w),
                               synth.to_numpy(kc0[0]), synth.to_numpy(vc0[0]), is_full, p0, ring)
    got_o = out.cpu().numpy().astype(np.float64) - h.cpu().numpy().astype(np.float64)
    for t in range(m):
        assert_close(got_o[t], res["o"][t], f"token {t} o")


def test_prefill_one_token_agrees_with_decode(B):
    """A chunk of one token is a decode step."""
    wl, w, kc, vc, h = _prefill_inputs(False, 512, 512, 700, 1, "bf16", 950)
    kc2, vc2 = kc.clone(), vc.clone()
    geom = B.spark_geom_default()
    ws = B.make_workspace(geom, 1)
    out1, out2 = torch.empty_like(h), torch.empty_like(h)
    B.spark_attn_prefill(geom, h, B.LayerWeights(**w), B.KvLayer(kc, vc, 512), B.SPARK_SLIDING, 700, out1, ws)
    B.spark_attn_decode(geom, h, B.LayerWeights(**w), B.KvLayer(kc2, vc2, 512), B.SPARK_SLIDING, [700], out2, ws)
    torch.cuda.synchronize()
    ma, rel = err_stats(out1.cpu().numpy() - h.cpu().numpy(), out2.cpu().numpy() - h.cpu().numpy())
    assert ma < 1e-4 and rel < 1e-5, (ma, rel)
    assert torch.equal(kc, kc2) and torch.equal(vc, vc2)


# ---------------------------------------------------------------------------
# error reporting of the bounded waits
# ---------------------------------------------------------------------------

def test_a_wait_that_runs_out_reports_and_leaves_the_gpu_usable(B):
    """A wait on a phase nothing completes gives up after its limit, raises
    the wait-timeout bit of the error word, and the next call works."""
    geom = B.spark_geom_default()
    ws = B.make_workspace(geom, 1)
    assert B.spark_attn_error_word(ws) == 0
    B.spark_dbg_wait_timeout(ws, 2_000_000)          # 2 ms
    torch.cuda.synchronize()
    assert B.spark_attn_error_word(ws) == 1          # bit 1: a wait ran out; reading clears it
    assert B.spark_attn_error_word(ws) == 0
    # the context is intact: an attention call right after is correct
    positions = [40]
    wl = synth.Workload("t", "", "bf16", positions, [synth.LayerSpec(True)], seed=960)
    kc, vc = synth.make_cache(wl, 0, "cuda")
    q = torch.randn((1, Q_DIM), generator=_gen(961), device="cuda")
    a = torch.empty((1, Q_DIM), device="cuda")
    B.spark_dbg_attention(geom, q, B.KvLayer(kc, vc, 0), B.SPARK_FULL, positions, a, ws)
    torch.cuda.synchronize()
    assert B.spark_attn_error_word(ws) == 0
    want = _attention_oracle(q.cpu().numpy().astype(np.float64), synth.to_numpy(kc), synth.to_numpy(vc),
                             positions, True, 0)
    assert_close(a.cpu().numpy(), want, "attention after a timed-out wait")
