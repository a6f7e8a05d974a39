"""float64 CPU oracle of the spark2_5 single-token decode attention block.

TEST INFRASTRUCTURE ONLY (see the package docstring): nothing on the product
path may import this module.

What it computes, step by step, in the order the source pages give.  The pages
are three files of the Rust crate ``turbospark-runtime 0.3.0``:

* ``src/families/spark/mod.rs``, module doc, "One decoder layer, transcribed"
  -- the layer's formulas (rms pre-norm with plain ``w`` and eps 1e-6, fused
  ``q_k_v_proj``, one sigmoid gate scalar per head from ``g_proj``, per-class
  rope, attention with scale ``256^-0.5``, gate before ``o_proj``, raw
  residual add);
* ``src/families/spark/attn.rs``, ``encode_attention_block`` -- the order of
  operations (split with k and v landing in their cache slots, rope of q and
  of k in the slot, window / ring set-up, attention, head gate, ``o_proj``),
  its module doc items 1-3, and ``rope_params_for`` with its unit test;
* ``src/kv_write.rs``, ``kv_write_target`` / ``encode_attention_any`` -- the
  cache slot is the write target and attention reads the layer's buffer from
  row 0.

Everything is float64.  bf16 tensors travel as ``uint16`` bit patterns and are
widened exactly; fp32 tensors are widened exactly.  The only rounding to a
narrower type is the one the method itself performs: the new k and v rows are
rounded once (round-to-nearest-even) to the cache's element type when they are
written into the cache slot, and attention then reads them back from the cache.

Parity pins (``tests/test_oracle_pins.py``) -- every function here is pinned:

* ``f64_to_bf16_bits`` / ``bf16_bits_to_f64``: torch's RNE cast on fp32 values,
  exhaustive round trip of all finite bf16 patterns, hand-made ties.
* ``rms_norm``: closed form for a constant input, scale invariance, a
  pure-Python loop.
* ``project``: one-hot weights, pure-Python loop.
* ``rope_params_for``: the values of the pages' own unit test.
* ``rope_neox``: identity at position 0, pair norms kept, dims past the rotary
  width untouched, relative-position property, closed-form angles at pair 0
  (frequency 1) and pair r/4 (frequency theta^-1/2), NeoX half-split pairing.
* ``window_params`` / ``write_slot`` / ``read_slot``: brute-force set semantics
  of the window and the ring on small integers; hand-derived values.
* ``attention_decode``: a single row returns v, equal keys give the window
  mean, GQA head map, sliding-window exclusion, pure-Python softmax.
* ``head_gate`` / ``sigmoid``: g = 0 halves the attention output.
* ``decode_step``: ``o_proj = 0`` returns ``h`` exactly, and a pure-Python
  loop implementation of the whole block at a tiny geometry.
* ``prefill_chunk``: one token equals ``decode_step``; a dense formulation
  (every token of the chunk projected at once, one causal / sliding mask over
  logical positions, softmax by rows) on a full layer with and without
  history and on a ring that wraps inside the chunk, chunks longer than the
  ring included; the final ring contents against a brute-force ring.
"""

from __future__ import annotations

import math
from dataclasses import dataclass

import numpy as np


# ----------------------------------------------------------------------------
# geometry
# ----------------------------------------------------------------------------

@dataclass(frozen=True)
class OracleGeometry:
    """Block geometry.  Defaults are spark2_5's, as ``mod.rs``'s module doc and
    ``attn.rs``'s module doc give them: hidden 2560, 16 query heads over 4 KV
    heads at head_dim 256, full layers rotate 64 dims at theta 5e6, sliding
    layers the whole head at theta 1e4, window 512, eps 1e-6, scale 256^-0.5."""

    hidden: int = 2560
    n_q: int = 16
    n_kv: int = 4
    head_dim: int = 256
    full_rotary_dim: int = 64
    window: int = 512
    full_theta: float = 5.0e6
    sliding_theta: float = 1.0e4
    eps: float = 1.0e-6
    scale: float = 256.0 ** -0.5

    @property
    def q_dim(self) -> int:
        return self.n_q * self.head_dim

    @property
    def kv_dim(self) -> int:
        return self.n_kv * self.head_dim


# ----------------------------------------------------------------------------
# element types
# ----------------------------------------------------------------------------

def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns (uint16) exactly: a bf16 value is the fp32 value
    whose upper 16 bits are the pattern and whose lower 16 bits are zero."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    with np.errstate(invalid="ignore"):       # NaN patterns stay NaN
        return b.view(np.float32).astype(np.float64)


def f64_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float64 values to bf16 with round-to-nearest-even, from the
    format's definition (8 significant bits, fp32's exponent range), and return
    the bit patterns as uint16.  Values beyond the largest finite bf16 round to
    infinity as IEEE RNE prescribes."""
    x = np.asarray(x, dtype=np.float64)
    _, e = np.frexp(x)                      # x = m * 2**e, 0.5 <= |m| < 1
    # the spacing of bf16 values around x: 2**(e-8) for normals; the subnormal
    # range shares the spacing of the smallest normal binade (e = -125)
    e = np.maximum(e, -125)
    quantum = np.ldexp(1.0, e - 8)
    with np.errstate(over="ignore", invalid="ignore"):
        r = np.round(x / quantum) * quantum   # np.round: half to even; exact scaling
        r = np.where(np.isfinite(x), r, x)
        big = np.abs(r) >= 2.0 ** 128          # past the largest finite value
        r = np.where(big, np.copysign(np.inf, r), r)
    f32 = r.astype(np.float32)                # exact: r has <= 8 significant bits
    return (f32.view(np.uint32) >> np.uint32(16)).astype(np.uint16)


def cache_rows_to_f64(rows: np.ndarray) -> np.ndarray:
    """Cache rows as float64: uint16 arrays are bf16 bit patterns, float32
    arrays are fp32 values."""
    if rows.dtype == np.uint16:
        return bf16_bits_to_f64(rows)
    if rows.dtype == np.float32:
        return rows.astype(np.float64)
    raise TypeError(f"unsupported cache element type {rows.dtype}")


def _weights_to_f64(w: np.ndarray) -> np.ndarray:
    return cache_rows_to_f64(w)


def _round_to_cache(x: np.ndarray, cache_dtype) -> np.ndarray:
    """Round float64 values once to the cache's element type (RNE)."""
    if cache_dtype == np.uint16:
        return f64_to_bf16_bits(x)
    if cache_dtype == np.float32:
        return np.asarray(x, dtype=np.float64).astype(np.float32)
    raise TypeError(f"unsupported cache element type {cache_dtype}")


# ----------------------------------------------------------------------------
# the steps
# ----------------------------------------------------------------------------

def rms_norm(h: np.ndarray, w: np.ndarray, eps: float) -> np.ndarray:
    """Input RMSNorm with a plain weight (``x = h / sqrt(mean(h^2) + eps) * w``,
    not ``1 + w``), as ``mod.rs``'s transcription of one layer writes it
    (``x = rms(h, input_layernorm, 1e-6)``, "plain w, pre-norm")."""
    h = np.asarray(h, dtype=np.float64)
    return h / np.sqrt(np.mean(h * h) + eps) * np.asarray(w, dtype=np.float64)


def project(weight: np.ndarray, x: np.ndarray) -> np.ndarray:
    """A GEMV with a row-major ``[rows x cols]`` weight: ``out[r] = sum_c
    W[r, c] * x[c]`` -- ``encode_gemv_any(name, rows, cols, in, out)`` in
    ``attn.rs``'s ``encode_attention_block``."""
    return np.asarray(weight, dtype=np.float64) @ np.asarray(x, dtype=np.float64)


def rope_params_for(is_full: bool, full_rotary_dim: int, head_dim: int,
                    full_theta: float, sliding_theta: float) -> tuple[int, float]:
    """Per-layer-class rope choice (``attn.rs``, ``rope_params_for``): a full
    layer rotates its leading ``full_rotary_dim`` dims at the full theta; a
    sliding layer rotates the whole head at the sliding theta."""
    if is_full:
        return full_rotary_dim, full_theta
    return head_dim, sliding_theta


def rope_inv_freq(rotary_dim: int, theta: float) -> np.ndarray:
    """Frequencies of the rotated pairs: ``theta^(-2i/r)`` for ``i < r/2``.
    The divisor is the rotary dim, not the head dim (``attn.rs`` module doc,
    item 2: HF partial-rotary semantics)."""
    i = np.arange(rotary_dim // 2, dtype=np.float64)
    return np.power(float(theta), -2.0 * i / float(rotary_dim))


def rope_neox(u: np.ndarray, position: int, rotary_dim: int, theta: float) -> np.ndarray:
    """NeoX-style rope over the leading ``rotary_dim`` dims of each head
    (``encode_rope_neox_subdim`` in ``attn.rs``): pair ``(i, i + r/2)`` of a
    head vector is rotated by the angle ``position * theta^(-2i/r)``; dims at
    or past ``r`` pass through.  ``u`` is ``[heads, head_dim]``."""
    u = np.asarray(u, dtype=np.float64)
    half = rotary_dim // 2
    ang = float(position) * rope_inv_freq(rotary_dim, theta)
    c, s = np.cos(ang), np.sin(ang)
    out = u.copy()
    x1 = u[:, :half]
    x2 = u[:, half:rotary_dim]
    out[:, :half] = x1 * c - x2 * s
    out[:, half:rotary_dim] = x2 * c + x1 * s
    return out


def window_params(position: int, is_full: bool, window: int,
                  ring_capacity: int) -> tuple[int, int, int]:
    """``(seq_len, kv_start, active_ring)`` as ``encode_attention_block`` sets
    them up: ``seq_len = position + 1``; a full layer reads ``[0, seq_len)``
    with identity addressing; a sliding layer reads
    ``[seq_len - window, seq_len)`` (saturating at 0), and its ring is active
    only once ``seq_len`` exceeds the ring's capacity."""
    seq_len = position + 1
    if is_full:
        return seq_len, 0, 0
    kv_start = max(0, seq_len - window)
    active_ring = ring_capacity if (ring_capacity > 0 and seq_len > ring_capacity) else 0
    return seq_len, kv_start, active_ring


def write_slot(position: int, ring_capacity: int) -> int:
    """Cache row that receives the token at ``position`` (``kv_write_target``
    hands back the layer's slot for ``position``).  A ring layer keeps
    position ``p`` in row ``p mod capacity`` -- the same addressing its
    attention uses once the ring is active; other layers keep it in row ``p``."""
    return position % ring_capacity if ring_capacity > 0 else position


def read_slot(j: int, active_ring: int) -> int:
    """Cache row that holds logical position ``j`` for attention: identity
    addressing when the ring is inactive (``active_ring == 0``), ``j mod ring``
    otherwise."""
    return j % active_ring if active_ring > 0 else j


def attention_decode(q: np.ndarray, k_rows: np.ndarray, v_rows: np.ndarray,
                     scale: float, n_kv: int) -> np.ndarray:
    """GQA decode attention of one token over the rows of its window.

    ``q`` is ``[n_q, d]``; ``k_rows`` / ``v_rows`` are ``[n, n_kv, d]``, the
    window's rows in logical order (already read through the slot mapping).
    Query head ``h`` reads KV head ``h // (n_q / n_kv)``; scores are
    ``scale * q_h . k_j``; the softmax is the plain max-subtracted one over the
    whole window; the output is the probability-weighted sum of v rows."""
    q = np.asarray(q, dtype=np.float64)
    n_q, d = q.shape
    group = n_q // n_kv
    out = np.empty((n_q, d), dtype=np.float64)
    for h in range(n_q):
        kvh = h // group
        s = scale * (k_rows[:, kvh, :] @ q[h])
        s = s - s.max()
        p = np.exp(s)
        p = p / p.sum()
        out[h] = p @ v_rows[:, kvh, :]
    return out


def sigmoid(z: np.ndarray) -> np.ndarray:
    """``1 / (1 + exp(-z))``."""
    z = np.asarray(z, dtype=np.float64)
    return 1.0 / (1.0 + np.exp(-z))


def head_gate(a: np.ndarray, g_logit: np.ndarray) -> np.ndarray:
    """Headwise output gate (``attn.rs`` module doc item 3,
    ``encode_sigmoid_head_gate_mul``): one sigmoid scalar per query head,
    broadcast over head_dim, applied to the attention output before
    ``o_proj``.  ``a`` is ``[n_q, d]``, ``g_logit`` is ``[n_q]``."""
    return np.asarray(a, dtype=np.float64) * sigmoid(g_logit)[:, None]


# ----------------------------------------------------------------------------
# the whole block
# ----------------------------------------------------------------------------

def decode_step(geom: OracleGeometry, h: np.ndarray, weights: dict,
                k_cache: np.ndarray, v_cache: np.ndarray, is_full: bool,
                positions, ring_capacity: int, sequences=None) -> dict:
    """One decode step of the attention block for a batch of independent
    sequences, following ``encode_attention_block``'s order.

    Arguments:
      h         ``[B, hidden]`` fp32/fp64 residual stream.
      weights   dict with ``norm_w [hidden]``, ``qkv_w [q_dim + 2 kv_dim,
                hidden]``, ``g_w [n_q, hidden]``, ``o_w [hidden, q_dim]``;
                float32 arrays or uint16 bf16 bit patterns.
      k_cache, v_cache  ``[B, capacity, n_kv, head_dim]``, float32 or uint16
                (bf16 bits).  They are not modified; the updated caches'
                written rows are returned.
      is_full   layer class (``True``: full attention, ``False``: sliding).
      positions ``[B]`` decode positions (token ``p`` attends to ``p+1`` rows
                of history including itself).
      ring_capacity  the layer's ring capacity (0 = linear addressing).
      sequences optional iterable of batch indices to compute (default: all).

    Returns a dict of float64 arrays keyed by batch index lists: ``x``,
    ``qkv``, ``g``, ``q``, ``k``, ``v`` (rope'd, before rounding), ``k_row``,
    ``v_row`` (the rows written, in the cache's element type), ``slot``,
    ``a`` (attention output), ``a_gated``, ``o``, ``out`` (``h + o``), and
    ``window`` (``(seq_len, kv_start, active_ring)`` per sequence)."""
    g_ = geom
    B = h.shape[0]
    seqs = list(range(B)) if sequences is None else list(sequences)
    norm_w = _weights_to_f64(weights["norm_w"])
    qkv_w = _weights_to_f64(weights["qkv_w"])
    g_w = _weights_to_f64(weights["g_w"])
    o_w = _weights_to_f64(weights["o_w"])
    rotary_dim, theta = rope_params_for(is_full, g_.full_rotary_dim, g_.head_dim,
                                        g_.full_theta, g_.sliding_theta)
    res = {key: [] for key in ("x", "qkv", "g", "q", "k", "v", "k_row", "v_row",
                               "slot", "a", "a_gated", "o", "out", "window")}
    for b in seqs:
        p = int(positions[b])
        hb = np.asarray(h[b], dtype=np.float64)
        # input_layernorm (mod.rs, one decoder layer: x = rms(h, w, 1e-6))
        x = rms_norm(hb, norm_w, g_.eps)
        # the fused q_k_v_proj GEMV; rows are q, then k, then v (attn.rs doc item 1)
        qkv = project(qkv_w, x)
        # g_proj reads the same normed x (attn.rs, the gate's projection)
        g_logit = project(g_w, x)
        # the split
        q = qkv[: g_.q_dim].reshape(g_.n_q, g_.head_dim)
        k = qkv[g_.q_dim: g_.q_dim + g_.kv_dim].reshape(g_.n_kv, g_.head_dim)
        v = qkv[g_.q_dim + g_.kv_dim:].reshape(g_.n_kv, g_.head_dim)
        # rope, per layer class, on q and on k (v untouched)
        q = rope_neox(q, p, rotary_dim, theta)
        k = rope_neox(k, p, rotary_dim, theta)
        # k and v land in their cache slot, in the cache's element type
        slot = write_slot(p, ring_capacity)
        k_row = _round_to_cache(k, k_cache.dtype)
        v_row = _round_to_cache(v, v_cache.dtype)
        # window / ring set-up
        seq_len, kv_start, active_ring = window_params(p, is_full, g_.window, ring_capacity)
        slots = np.array([read_slot(j, active_ring) for j in range(kv_start, seq_len)],
                         dtype=np.int64)
        k_rows = k_cache[b][slots].copy()
        v_rows = v_cache[b][slots].copy()
        # attention reads the new row back from its slot
        hit = slots == slot
        k_rows[hit] = k_row
        v_rows[hit] = v_row
        a = attention_decode(q, cache_rows_to_f64(k_rows), cache_rows_to_f64(v_rows),
                             g_.scale, g_.n_kv)
        # the headwise gate before o_proj, then o_proj and the raw residual add
        a_gated = head_gate(a, g_logit)
        o = project(o_w, a_gated.reshape(-1))
        out = hb + o
        for key, val in (("x", x), ("qkv", qkv), ("g", g_logit), ("q", q), ("k", k),
                         ("v", v), ("k_row", k_row), ("v_row", v_row), ("slot", slot),
                         ("a", a), ("a_gated", a_gated), ("o", o), ("out", out),
                         ("window", (seq_len, kv_start, active_ring))):
            res[key].append(val)
    res["sequences"] = seqs
    return res


def prefill_chunk(geom: OracleGeometry, h: np.ndarray, weights: dict,
                  k_cache: np.ndarray, v_cache: np.ndarray, is_full: bool,
                  p0: int, ring_capacity: int) -> dict:
    """M consecutive tokens of one sequence through the block, at positions
    ``p0 .. p0 + M - 1``: the per-token attention block run token after token
    (kv_write.rs, module doc: chunked prefill reuses the per-token attention
    block, only the K/V projections being batched), so token ``t`` sees the
    rows tokens ``< t`` of the chunk wrote, and on a ring a later token's
    row replaces the row of the position ``ring_capacity`` before it.

    Arguments as ``decode_step`` for one sequence: ``h [M, hidden]``,
    ``k_cache, v_cache [capacity, n_kv, head_dim]`` (not modified).

    Returns ``out [M, hidden]``, ``o [M, hidden]``, the caches after the
    chunk (``k_cache``, ``v_cache``) and per token ``slot``, ``k_row``,
    ``v_row``, ``q``, ``a``."""
    kc = np.array(k_cache, copy=True)
    vc = np.array(v_cache, copy=True)
    M = h.shape[0]
    res = {key: [] for key in ("out", "o", "slot", "k_row", "v_row", "q", "a")}
    for t in range(M):
        step = decode_step(geom, h[t:t + 1], weights, kc[None], vc[None], is_full, [p0 + t],
                           ring_capacity)
        slot = step["slot"][0]
        kc[slot] = step["k_row"][0]
        vc[slot] = step["v_row"][0]
        for key in ("out", "o", "slot", "k_row", "v_row", "q", "a"):
            res[key].append(step[key][0])
    res["out"] = np.stack(res["out"])
    res["o"] = np.stack(res["o"])
    res["k_cache"] = kc
    res["v_cache"] = vc
    return res
