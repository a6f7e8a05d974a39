"""Test helpers: tolerances, oracle calls on synthetic inputs, device set-up.

Tolerances are those the block's acceptance states for bf16 weights and
cache with fp32 accumulation: max-abs 2e-2 and relative L2 1e-2.  The block's
output is compared as ``o = out - h`` (the block's own contribution), because
the pass-through ``h`` would otherwise dominate the relative error.
"""

from __future__ import annotations

import numpy as np
import torch

import oracle
from decode_attention_block_gb300 import synth

MAX_ABS = 2e-2
REL_L2 = 1e-2


def err_stats(got, want):
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    d = got - want
    max_abs = float(np.max(np.abs(d))) if d.size else 0.0
    rel = float(np.linalg.norm(d) / max(np.linalg.norm(want), 1e-30))
    return max_abs, rel


def assert_close(got, want, what="", max_abs=MAX_ABS, rel_l2=REL_L2):
    assert np.all(np.isfinite(np.asarray(got, dtype=np.float64))), f"{what}: non-finite output"
    ma, rel = err_stats(got, want)
    assert ma <= max_abs and rel <= rel_l2, f"{what}: max_abs {ma:.3e} rel_l2 {rel:.3e}"
    return ma, rel


def oracle_geom(wl: synth.Workload) -> oracle.OracleGeometry:
    return oracle.OracleGeometry(hidden=wl.hidden, n_q=wl.n_q, n_kv=wl.n_kv, head_dim=wl.head_dim,
                                 window=wl.window)


def cache_as_f64(rows: np.ndarray) -> np.ndarray:
    return oracle.cache_rows_to_f64(rows)


def np_weights(w: dict) -> dict:
    return {k: synth.to_numpy(v) for k, v in w.items()}
