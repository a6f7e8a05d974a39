"""Seeded synthetic inputs for the decode attention block.

The one module both the CUDA path's callers and the CPU oracle's callers use:
it draws random numbers and casts them, and holds none of the block's
arithmetic.  Value distributions: h ~ N(0, 1); input_layernorm = 1 + 0.1 N(0, 1);
q_k_v_proj and g_proj ~ N(0, 1/hidden); o_proj ~ N(0, 1/(n_q*d)); every
cache row ~ N(0, 1).  The rest of the decoder layer and the head:
post_attention_layernorm and model.norm = 1 + 0.1 N(0, 1); gate_proj and
up_proj ~ N(0, 1/hidden); down_proj ~ N(0, 1/intermediate); the tied
embedding ~ N(0, 1/hidden) (logits of order 1).  The pages print neither the
intermediate size nor the vocabulary: INTERMEDIATE and VOCAB are stand-ins
(a 4x MLP and 2^17 tokens, which with 36 layers put the model near the 4B
parameters its name states).  Values are drawn in fp32 and rounded to bf16 with
round-to-nearest-even where the workload is bf16.  No trained checkpoint and
no dataset is involved: the workloads are defined by their shapes, lengths and
distributions alone.
"""

from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np
import torch

HIDDEN = 2560
N_Q = 16
N_KV = 4
HEAD_DIM = 256
WINDOW = 512
RING = 512
INTERMEDIATE = 4 * HIDDEN
VOCAB = 1 << 17


@dataclass(frozen=True)
class LayerSpec:
    is_full: bool
    ring_capacity: int = 0    # 0: linear addressing


@dataclass
class Workload:
    name: str
    description: str
    dtype: str                 # "f32" or "bf16": weights and caches
    positions: list
    layers: list
    seed: int
    hidden: int = HIDDEN
    n_q: int = N_Q
    n_kv: int = N_KV
    head_dim: int = HEAD_DIM
    window: int = WINDOW
    extra: dict = field(default_factory=dict)

    @property
    def batch(self) -> int:
        return len(self.positions)

    @property
    def torch_dtype(self):
        return torch.float32 if self.dtype == "f32" else torch.bfloat16

    @property
    def elem_bytes(self) -> int:
        return 4 if self.dtype == "f32" else 2

    def capacity(self, li: int) -> int:
        spec = self.layers[li]
        return spec.ring_capacity if spec.ring_capacity > 0 else max(self.positions) + 1

    def rows_read(self, li: int, b: int) -> int:
        """Cache rows (positions) a sequence's token reads on layer li."""
        p = self.positions[b]
        seq_len = p + 1
        if self.layers[li].is_full:
            return seq_len
        return min(seq_len, self.window)

    def weight_bytes_per_layer(self) -> int:
        q_dim = self.n_q * self.head_dim
        kv_dim = self.n_kv * self.head_dim
        elems = (q_dim + 2 * kv_dim) * self.hidden + self.n_q * self.hidden \
            + self.hidden * q_dim + self.hidden
        return elems * self.elem_bytes

    def kv_row_bytes(self) -> int:
        """Bytes of one cache row of K plus V."""
        return 2 * self.n_kv * self.head_dim * self.elem_bytes


def _ragged_positions(seed: int, n: int, lo: int, hi: int) -> list:
    rng = np.random.default_rng(seed)
    return [int(x) for x in rng.integers(lo, hi + 1, size=n)]


def workloads() -> dict:
    """The block's workloads, by name."""
    wl = [
        Workload("sliding_f32_b1_pos40",
                 "one sliding layer (ring 512), fp32 weights and cache, batch 1, decode at "
                 "position 40 over 40 prefilled rows",
                 "f32", [40], [LayerSpec(False, RING)], seed=1000),
        Workload("full+sliding_bf16_b1_pos700",
                 "one full layer (rotary 64 @ 5e6, causal) and one sliding layer (window 512, "
                 "ring 512, wrapped), bf16, batch 1, decode at position 700",
                 "bf16", [700], [LayerSpec(True, 0), LayerSpec(False, RING)], seed=1001),
        Workload("stack36_bf16_b1_ctx8192",
                 "36-layer stack, layer i full iff i % 4 == 3, bf16, batch 1, decode at context 8192",
                 "bf16", [8192], [LayerSpec(i % 4 == 3, 0 if i % 4 == 3 else RING) for i in range(36)],
                 seed=1002),
        Workload("full+sliding_bf16_b64_ctx512-32768",
                 "64 independent sequences, context uniform in [512, 32768], one full and one "
                 "sliding layer, bf16",
                 "bf16", _ragged_positions(1003, 64, 512, 32768),
                 [LayerSpec(True, 0), LayerSpec(False, RING)], seed=1003),
        Workload("full+sliding_bf16_b8_ctx131072",
                 "8 sequences at context 131072, one full layer (rotary 64 @ 5e6) and one sliding "
                 "layer (ring 512 wrapped many times), bf16",
                 "bf16", [131072] * 8, [LayerSpec(True, 0), LayerSpec(False, RING)], seed=1004),
        Workload("full+sliding_bf16_b64_ctx512-1023",
                 "64 sequences, context uniform in [512, 1023], one full and one sliding layer, "
                 "bf16: the batched projections with caches small enough to profile",
                 "bf16", _ragged_positions(1006, 64, 512, 1023),
                 [LayerSpec(True, 0), LayerSpec(False, RING)], seed=1006),
        Workload("full_bf16_b16_ctx512-32768",
                 "the full layer of the first 16 sequences of the 64-sequence ragged batch "
                 "(contexts in [512, 32768], the same rows): its attention at a size a profiler "
                 "can capture",
                 "bf16", _ragged_positions(1003, 64, 512, 32768)[:16], [LayerSpec(True, 0)], seed=1003),
        Workload("full_bf16_b1_ctx131072",
                 "one full layer (rotary 64 @ 5e6), bf16, one sequence at context 131072 "
                 "(a single long-context attention)",
                 "bf16", [131072], [LayerSpec(True, 0)], seed=1005),
    ]
    return {w.name: w for w in wl}


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def _randn(shape, gen, device, scale=1.0, shift=0.0, dtype=torch.float32):
    x = torch.randn(shape, generator=gen, device=device, dtype=torch.float32)
    if scale != 1.0:
        x.mul_(scale)
    if shift != 0.0:
        x.add_(shift)
    return x.to(dtype)


def make_h(wl: Workload, device="cpu", gen_device=None) -> torch.Tensor:
    gd = gen_device or device
    g = _gen(wl.seed * 7919 + 1, gd)
    return _randn((wl.batch, wl.hidden), g, gd).to(device)


def make_weights(wl: Workload, li: int, device="cpu", gen_device=None) -> dict:
    """One layer's weights: norm_w [H], qkv_w [q+2kv, H], g_w [n_q, H], o_w [H, q]."""
    gd = gen_device or device
    g = _gen(wl.seed * 1000003 + 17 * li + 3, gd)
    H, q_dim, kv_dim = wl.hidden, wl.n_q * wl.head_dim, wl.n_kv * wl.head_dim
    dt = wl.torch_dtype
    out = {
        "norm_w": _randn((H,), g, gd, 0.1, 1.0, dt),
        "qkv_w": _randn((q_dim + 2 * kv_dim, H), g, gd, H ** -0.5, 0.0, dt),
        "g_w": _randn((wl.n_q, H), g, gd, H ** -0.5, 0.0, dt),
        "o_w": _randn((H, q_dim), g, gd, q_dim ** -0.5, 0.0, dt),
    }
    return {k: v.to(device) for k, v in out.items()}


def _draw_sequence_rows(wl: Workload, li: int, b: int, k_out, v_out, gd) -> None:
    """Sequence b's K and V rows of layer li into k_out, v_out [capacity, n_kv, d]:
    the generator is seeded per (layer, sequence), so a sequence's rows do not
    depend on which other sequences are drawn."""
    g = _gen(wl.seed * 1000003 + 17 * li + 7 + 104729 * (b + 1), gd)
    k_out.copy_(_randn(tuple(k_out.shape), g, gd, dtype=wl.torch_dtype))
    v_out.copy_(_randn(tuple(v_out.shape), g, gd, dtype=wl.torch_dtype))


def make_cache(wl: Workload, li: int, device="cpu", gen_device=None, sequences=None):
    """One layer's K and V caches [batch, capacity, n_kv, d], every row ~ N(0, 1).
    With ``sequences``, only those batch entries are drawn (the others are
    zero)."""
    gd = gen_device or device
    cap = wl.capacity(li)
    shape = (wl.batch, cap, wl.n_kv, wl.head_dim)
    k = torch.zeros(shape, dtype=wl.torch_dtype, device=device)
    v = torch.zeros(shape, dtype=wl.torch_dtype, device=device)
    seqs = range(wl.batch) if sequences is None else sequences
    for b in seqs:
        _draw_sequence_rows(wl, li, b, k[b], v[b], gd)
    return k, v


def make_sequence_cache(wl: Workload, li: int, b: int, device="cpu", gen_device=None):
    """Sequence b's entry of make_cache alone, as [1, capacity, n_kv, d]
    tensors (the same rows, without the other sequences' memory)."""
    gd = gen_device or device
    shape = (1, wl.capacity(li), wl.n_kv, wl.head_dim)
    k = torch.empty(shape, dtype=wl.torch_dtype, device=device)
    v = torch.empty(shape, dtype=wl.torch_dtype, device=device)
    _draw_sequence_rows(wl, li, b, k[0], v[0], gd)
    return k, v


def to_numpy(t: torch.Tensor) -> np.ndarray:
    """A CPU copy as numpy: float32 stays float32, bf16 becomes its uint16 bits."""
    t = t.detach().to("cpu").contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def make_mlp_weights(seed: int, hidden: int, inter: int, dtype=torch.bfloat16, device="cpu",
                     gen_device=None) -> dict:
    """The MLP half of one layer: norm_w [H] (post_attention_layernorm),
    gate_w, up_w [I, H], down_w [H, I]."""
    gd = gen_device or device
    g = _gen(seed * 1000033 + 11, gd)
    out = {
        "norm_w": _randn((hidden,), g, gd, 0.1, 1.0, dtype),
        "gate_w": _randn((inter, hidden), g, gd, hidden ** -0.5, 0.0, dtype),
        "up_w": _randn((inter, hidden), g, gd, hidden ** -0.5, 0.0, dtype),
        "down_w": _randn((hidden, inter), g, gd, inter ** -0.5, 0.0, dtype),
    }
    return {k: v.to(device) for k, v in out.items()}


def make_head(seed: int, hidden: int, vocab: int, dtype=torch.bfloat16, device="cpu", gen_device=None) -> dict:
    """The head: norm_w [H] (model.norm) and the tied embedding [V, H]."""
    gd = gen_device or device
    g = _gen(seed * 1000037 + 13, gd)
    out = {
        "norm_w": _randn((hidden,), g, gd, 0.1, 1.0, dtype),
        "embed": _randn((vocab, hidden), g, gd, hidden ** -0.5, 0.0, dtype),
    }
    return {k: v.to(device) for k, v in out.items()}


def make_hidden(seed: int, batch: int, hidden: int, device="cpu", gen_device=None) -> torch.Tensor:
    """A residual stream [batch, hidden] ~ N(0, 1) (fp32)."""
    gd = gen_device or device
    return _randn((batch, hidden), _gen(seed * 7919 + 5, gd), gd).to(device)
