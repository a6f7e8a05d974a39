"""float64 CPU oracle of the rest of a spark2_5 decoder layer and of the head.

TEST INFRASTRUCTURE ONLY (see the package docstring): nothing on the product
path may import this module.

What it computes follows ``src/families/spark/mod.rs`` of turbospark-runtime
0.3.0: the module doc's transcription of one decoder layer (after the
attention block's raw residual add, a second pre-norm with a plain weight and
eps 1e-6, then ``h = h + down(gelu_erf(x @ gate_proj) * (x @ up_proj))``),
the same transcription's last two lines (the final ``model.norm`` RMSNorm and
the tied head ``logits = h @ embed_tokens``), and the layer loop of
``produce_real_spark`` (the RMSNorm with ``post_attention_layernorm`` feeding
``mlp::encode_mlp_block``, whose FFN residual add ends the layer; the final
norm and one ``encode_gemv_any`` over the embedding rows with ``vocab`` rows
and ``hidden`` columns).  The body of ``mlp.rs`` is not on the pages; what
the transcription fixes is used, read plainly:

* ``gelu_erf(z) = z * Phi(z) = z / 2 * (1 + erf(z / sqrt 2))`` -- the exact
  (erf) GELU, not the tanh approximation;
* ``gate_proj`` and ``up_proj`` are ``[intermediate x hidden]``,
  ``down_proj`` is ``[hidden x intermediate]``, row-major, with
  ``out[r] = sum_c W[r, c] in[c]`` as every GEMV of the pages;
* the head's weight is the embedding matrix itself, ``[vocab x hidden]``, one
  row per token (``TIED``; no softcap, no output multiplier).

Everything is float64; bf16 weights travel as ``uint16`` bit patterns and are
widened exactly.

Parity pins (``tests/test_oracle_pins.py``):

* ``gelu_erf``: ``gelu(x) / x`` against the standard normal CDF's printed
  table values at -2, -1, 1 and 2, ``gelu(0) = 0``, the limits (identity for
  large positive inputs, zero for large negative ones); the tanh
  approximation is rejected at the table's precision.
* ``mlp_block``: a pure-Python loop at a tiny geometry; ``down_proj = 0``
  returns ``h`` exactly; gate and up are not interchangeable (a gate row that
  drives its output far negative zeroes the product whatever up gives).
* ``head_logits``: a pure-Python loop; one-hot embedding rows pick the normed
  hidden state's components.
"""

from __future__ import annotations

import math

import numpy as np

from .spark_block import OracleGeometry, _weights_to_f64, project, rms_norm


def gelu_erf(z: np.ndarray) -> np.ndarray:
    """The exact GELU of ``mod.rs``'s transcription (``gelu_erf``):
    ``z * Phi(z)`` with ``Phi`` the standard normal CDF written through erf,
    ``Phi(z) = (1 + erf(z / sqrt 2)) / 2``."""
    z = np.asarray(z, dtype=np.float64)
    erf = np.vectorize(math.erf, otypes=[np.float64])
    return 0.5 * z * (1.0 + erf(z / math.sqrt(2.0)))


def mlp_block(geom: OracleGeometry, h: np.ndarray, weights: dict) -> dict:
    """The MLP half of one decoder layer for a batch of sequences
    (``mod.rs``: ``x = rms(h, post_attention_layernorm, 1e-6)``, then
    ``h = h + down(gelu_erf(x @ gate_proj) * (x @ up_proj))``).

    ``h`` is ``[B, hidden]`` -- the residual stream after the attention
    block.  ``weights`` holds ``norm_w [hidden]``, ``gate_w``, ``up_w``
    ``[intermediate, hidden]`` and ``down_w [hidden, intermediate]`` (float32
    arrays or bf16 bit patterns).  Returns ``out [B, hidden]`` and the
    intermediates ``x``, ``gate``, ``up`` and ``m`` (the GELU product)."""
    h = np.asarray(h, dtype=np.float64)
    norm_w = _weights_to_f64(weights["norm_w"])
    gate_w = _weights_to_f64(weights["gate_w"])
    up_w = _weights_to_f64(weights["up_w"])
    down_w = _weights_to_f64(weights["down_w"])
    B = h.shape[0]
    out = np.empty_like(h)
    xs, gates, ups, ms = [], [], [], []
    for b in range(B):
        x = rms_norm(h[b], norm_w, geom.eps)
        gate = project(gate_w, x)
        up = project(up_w, x)
        m = gelu_erf(gate) * up
        out[b] = h[b] + project(down_w, m)
        xs.append(x)
        gates.append(gate)
        ups.append(up)
        ms.append(m)
    return {"out": out, "x": np.array(xs), "gate": np.array(gates), "up": np.array(ups),
            "m": np.array(ms)}


def head_logits(geom: OracleGeometry, h: np.ndarray, norm_w: np.ndarray,
                embed: np.ndarray) -> np.ndarray:
    """The head after the last layer (``mod.rs``: ``h = rms(h, model.norm,
    1e-6)``, ``logits = h @ embed_tokens`` with the embedding tied as the
    head): ``logits[b, v] = sum_c embed[v, c] * rms(h_b)[c]``.  ``h`` is
    ``[B, hidden]``, ``embed`` ``[vocab, hidden]``; returns ``[B, vocab]``."""
    h = np.asarray(h, dtype=np.float64)
    w = _weights_to_f64(norm_w)
    e = _weights_to_f64(embed)
    return np.array([project(e, rms_norm(h[b], w, geom.eps)) for b in range(h.shape[0])])
