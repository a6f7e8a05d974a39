"""Parity of the rest of the decoder layer (post-attention RMSNorm, GELU-gated
MLP, residual) and of the head (final RMSNorm, tied embedding) with the CPU
oracle, through the C ABI, on the GEMV and the tensor-core paths: tiny
geometries with ragged tiles, batches across the path switch and across the
tensor-core chunk of 128 sequences, and the stand-in spark2_5 sizes (hidden
2560, intermediate 10240, vocabulary 2^17, the head on sampled rows).
"""

import numpy as np
import pytest
import torch

import oracle
from decode_attention_block_gb300 import build_lib, synth
from helpers import assert_close, np_weights

pytestmark = pytest.mark.gpu

PATHS = {"auto": 0, "gemv": 1, "mma": 2}


@pytest.fixture(scope="module")
def B():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    build_lib.build()
    from decode_attention_block_gb300 import binding
    binding.load()
    return binding


def _geom(B, hidden):
    g = B.spark_geom_default()
    g.hidden = hidden
    return g


def _f64(x):
    x = np.asarray(x)
    return oracle.cache_rows_to_f64(x) if x.dtype == np.uint16 else x.astype(np.float64)


def _run_mlp(B, hidden, inter, batch, dtype, path, seed, in_place=False):
    w = synth.make_mlp_weights(seed, hidden, inter, dtype, "cuda")
    h = synth.make_hidden(seed, batch, hidden, "cuda")
    h0 = h.clone()
    out = h if in_place else torch.full_like(h, float("nan"))
    g = _geom(B, hidden)
    ws = B.make_mlp_workspace(g, inter, batch)
    B.spark_mlp_decode(g, h, B.MlpWeights(**w), out, ws, PATHS[path])
    torch.cuda.synchronize()
    assert B.spark_attn_error_word(ws) == 0
    return w, h0, out


def _mlp_oracle(hidden, w, h0):
    geom = oracle.OracleGeometry(hidden=hidden)
    return oracle.mlp_block(geom, synth.to_numpy(h0).astype(np.float64), np_weights(w))["out"]


def _check_mlp(hidden, w, h0, out, what):
    want = _mlp_oracle(hidden, w, h0)
    h64 = synth.to_numpy(h0).astype(np.float64)
    got = out.cpu().numpy().astype(np.float64)
    for b in range(h64.shape[0]):
        assert_close(got[b] - h64[b], want[b] - h64[b], f"{what} b={b}")


MLP_SMALL = [
    # (hidden, inter, batch, dtype, path)
    (256, 40, 1, torch.bfloat16, "gemv"),
    (256, 352, 2, torch.bfloat16, "gemv"),
    (256, 352, 3, torch.float32, "gemv"),
    (512, 200, 4, torch.bfloat16, "auto"),
    (256, 40, 5, torch.bfloat16, "auto"),
    (256, 352, 13, torch.bfloat16, "mma"),
    (512, 200, 40, torch.bfloat16, "mma"),
    (256, 1000, 64, torch.bfloat16, "mma"),
    (256, 352, 130, torch.bfloat16, "mma"),
    (256, 352, 9, torch.float32, "auto"),      # fp32 weights: the GEMV path at any batch
    # more up tiles than SMs (two CTAs per SM, or a second wave), ragged last tile
    (256, 12296, 8, torch.bfloat16, "mma"),
    (512, 10248, 64, torch.bfloat16, "mma"),
    (256, 16384, 130, torch.bfloat16, "mma"),
    # five chunks of 128 sequences in one launch, the last one partial
    (256, 352, 520, torch.bfloat16, "mma"),
]


@pytest.mark.parametrize("case", MLP_SMALL, ids=[f"H{c[0]}_I{c[1]}_b{c[2]}_{str(c[3])[6:]}_{c[4]}"
                                                 for c in MLP_SMALL])
def test_mlp_matches_oracle(B, case):
    hidden, inter, batch, dtype, path = case
    w, h0, out = _run_mlp(B, hidden, inter, batch, dtype, path, seed=hidden + inter + batch)
    _check_mlp(hidden, w, h0, out, f"mlp {case}")


@pytest.mark.parametrize("batch,path", [(1, "auto"), (2, "gemv"), (64, "auto"), (8, "mma")])
def test_mlp_full_size_matches_oracle(B, batch, path):
    w, h0, out = _run_mlp(B, synth.HIDDEN, synth.INTERMEDIATE, batch, torch.bfloat16, path, seed=2000 + batch)
    _check_mlp(synth.HIDDEN, w, h0, out, f"mlp full b={batch} {path}")


@pytest.mark.parametrize("path,batch", [("gemv", 3), ("mma", 24), ("mma", 40)])
def test_mlp_in_place_and_zero_down(B, path, batch):
    hidden, inter = 256, 352
    w, h0, out = _run_mlp(B, hidden, inter, batch, torch.bfloat16, path, seed=77, in_place=True)
    _check_mlp(hidden, w, h0, out, f"mlp in place {path}")
    # down_proj = 0: the layer returns h bit for bit
    w["down_w"].zero_()
    h = h0.clone()
    out = torch.full_like(h, float("nan"))
    g = _geom(B, hidden)
    ws = B.make_mlp_workspace(g, inter, batch)
    B.spark_mlp_decode(g, h, B.MlpWeights(**w), out, ws, PATHS[path])
    torch.cuda.synchronize()
    assert torch.equal(out, h0)


def test_mlp_paths_agree_and_repeat(B):
    hidden, inter, batch = 512, 352, 8
    w = synth.make_mlp_weights(5, hidden, inter, torch.bfloat16, "cuda")
    h = synth.make_hidden(5, batch, hidden, "cuda")
    g = _geom(B, hidden)
    ws = B.make_mlp_workspace(g, inter, batch)
    outs = []
    for path in ("gemv", "mma", "mma"):
        o = torch.empty_like(h)
        B.spark_mlp_decode(g, h, B.MlpWeights(**w), o, ws, PATHS[path])
        outs.append(o)
    torch.cuda.synchronize()
    assert torch.equal(outs[1], outs[2]), "the tensor-core path is not deterministic"
    d = (outs[0] - h).double().cpu().numpy()
    assert_close((outs[1] - h).double().cpu().numpy(), d, "gemv vs mma", max_abs=2e-3, rel_l2=1e-3)


# ---------------------------------------------------------------------------
# the head
# ---------------------------------------------------------------------------

def _run_head(B, hidden, vocab, batch, dtype, path, seed):
    p = synth.make_head(seed, hidden, vocab, dtype, "cuda")
    h = synth.make_hidden(seed + 1, batch, hidden, "cuda")
    logits = torch.full((batch, vocab), float("nan"), device="cuda")
    g = _geom(B, hidden)
    ws = B.make_mlp_workspace(g, 0, batch)
    B.spark_head_logits(g, h, p["norm_w"], p["embed"], logits, ws, PATHS[path])
    torch.cuda.synchronize()
    assert B.spark_attn_error_word(ws) == 0
    return p, h, logits


HEAD_SMALL = [
    (256, 8, 1, torch.bfloat16, "gemv"),
    (256, 136, 3, torch.float32, "gemv"),
    (512, 1000, 4, torch.bfloat16, "auto"),
    (256, 136, 5, torch.bfloat16, "auto"),
    (256, 1000, 64, torch.bfloat16, "mma"),
    (256, 4104, 130, torch.bfloat16, "mma"),
    (256, 8, 16, torch.bfloat16, "mma"),
    # more tiles than SMs (several waves), ragged last tile
    (256, 40008, 16, torch.bfloat16, "mma"),
    (512, 20488, 77, torch.bfloat16, "mma"),
    (256, 1000, 300, torch.bfloat16, "mma"),
]


@pytest.mark.parametrize("case", HEAD_SMALL, ids=[f"H{c[0]}_V{c[1]}_b{c[2]}_{str(c[3])[6:]}_{c[4]}"
                                                  for c in HEAD_SMALL])
def test_head_matches_oracle(B, case):
    hidden, vocab, batch, dtype, path = case
    p, h, logits = _run_head(B, hidden, vocab, batch, dtype, path, seed=hidden + vocab + batch)
    want = oracle.head_logits(oracle.OracleGeometry(hidden=hidden), synth.to_numpy(h).astype(np.float64),
                              synth.to_numpy(p["norm_w"]), synth.to_numpy(p["embed"]))
    got = logits.cpu().numpy()
    for b in range(batch):
        assert_close(got[b], want[b], f"head {case} b={b}")


@pytest.mark.parametrize("batch,path", [(1, "auto"), (64, "auto")])
def test_head_full_size_on_sampled_rows(B, batch, path):
    vocab = synth.VOCAB
    p, h, logits = _run_head(B, synth.HIDDEN, vocab, batch, torch.bfloat16, path, seed=3000 + batch)
    rng = np.random.default_rng(batch)
    rows = np.unique(np.concatenate([rng.integers(0, vocab, 3000), np.arange(vocab - 200, vocab),
                                     np.arange(0, 200)]))
    emb = synth.to_numpy(p["embed"][torch.from_numpy(rows).cuda()])
    want = oracle.head_logits(oracle.OracleGeometry(hidden=synth.HIDDEN), synth.to_numpy(h).astype(np.float64),
                              synth.to_numpy(p["norm_w"]), emb)
    got = logits.cpu().numpy()[:, rows]
    assert np.all(np.isfinite(logits.cpu().numpy())), "a logit was never written"
    for b in range(batch):
        assert_close(got[b], want[b], f"head full b={b} {path}")


def test_many_tile_results_repeat_bit_for_bit(B):
    # launches with more tiles than SMs give the same bits call after call on
    # one workspace (split-K tickets reset, partials added in split order)
    hidden, inter, batch = 256, 12296, 8
    w = synth.make_mlp_weights(9, hidden, inter, torch.bfloat16, "cuda")
    h = synth.make_hidden(9, batch, hidden, "cuda")
    g = _geom(B, hidden)
    ws = B.make_mlp_workspace(g, inter, batch)
    outs = []
    for _ in range(3):
        o = torch.empty_like(h)
        B.spark_mlp_decode(g, h, B.MlpWeights(**w), o, ws, PATHS["mma"])
        outs.append(o)
    p = synth.make_head(9, hidden, 40008, torch.bfloat16, "cuda")
    lg = [torch.empty((batch, 40008), device="cuda") for _ in range(2)]
    for t in lg:
        B.spark_head_logits(g, h, p["norm_w"], p["embed"], t, ws, PATHS["mma"])
    torch.cuda.synchronize()
    assert B.spark_attn_error_word(ws) == 0
    assert torch.equal(outs[0], outs[1]) and torch.equal(outs[0], outs[2])
    assert torch.equal(lg[0], lg[1])
