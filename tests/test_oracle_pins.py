"""Pins of the CPU oracle against facts other than the oracle itself.

Every function of ``oracle.spark_block`` is checked here against something
fixed independently of its own code: values printed on the source pages
(``tests/golden``), closed forms, invariants of the mathematics, library
routines for special cases, and brute force on tiny inputs written as plain
Python loops.  Each pin is chosen so that a plausible slip in the oracle (a
dropped term, a wrong sign or index, a swapped class, a wrong divisor, a
transposed operand) fails at least one test.
"""

import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from oracle import OracleGeometry

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ---------------------------------------------------------------------------
# element types
# ---------------------------------------------------------------------------

def test_bf16_round_matches_torch_rne_cast():
    rng = np.random.default_rng(0)
    x = np.concatenate([
        rng.standard_normal(20000).astype(np.float32),
        (rng.standard_normal(2000) * 1e30).astype(np.float32),
        (rng.standard_normal(2000) * 1e-30).astype(np.float32),
        (rng.standard_normal(2000) * 1e-39).astype(np.float32),   # fp32 subnormals
        np.array([0.0, -0.0, 3.3895314e38, -3.3895314e38, np.inf, -np.inf], dtype=np.float32),
    ])
    want = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = oracle.f64_to_bf16_bits(x.astype(np.float64))
    np.testing.assert_array_equal(got, want)


def test_bf16_round_trip_every_finite_pattern():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    vals = oracle.bf16_bits_to_f64(bits)
    finite = np.isfinite(vals)
    np.testing.assert_array_equal(oracle.f64_to_bf16_bits(vals[finite]), bits[finite])


def test_bf16_ties_go_to_even():
    # 1 + 2^-8 lies halfway between 1 and 1 + 2^-7: even mantissa is 1.0
    # 1 + 3*2^-8 lies halfway between 1 + 2^-7 and 1 + 2^-6: even is 1 + 2^-6
    x = np.array([1 + 2.0 ** -8, 1 + 3 * 2.0 ** -8, -(1 + 2.0 ** -8), 1 + 2.0 ** -8 + 2.0 ** -30])
    want = np.array([1.0, 1 + 2.0 ** -6, -1.0, 1 + 2.0 ** -7])
    np.testing.assert_array_equal(oracle.bf16_bits_to_f64(oracle.f64_to_bf16_bits(x)), want)


def test_bf16_widening_known_patterns():
    bits = np.array([0x3F80, 0xC000, 0x0000, 0x3E80, 0x4049], dtype=np.uint16)
    np.testing.assert_array_equal(oracle.bf16_bits_to_f64(bits),
                                  [1.0, -2.0, 0.0, 0.25, 3.140625])


# ---------------------------------------------------------------------------
# RMSNorm
# ---------------------------------------------------------------------------

def test_rms_norm_constant_input_closed_form():
    n, c, eps = 64, 3.0, 1e-6
    w = np.linspace(0.5, 1.5, n)
    x = oracle.rms_norm(np.full(n, c), w, eps)
    np.testing.assert_allclose(x, w * c / math.sqrt(c * c + eps), rtol=1e-15)


def test_rms_norm_plain_weight_and_scale_invariance():
    rng = np.random.default_rng(1)
    h = rng.standard_normal(2560)
    w = 1 + 0.1 * rng.standard_normal(2560)
    x = oracle.rms_norm(h, w, 0.0)
    np.testing.assert_allclose(oracle.rms_norm(7.5 * h, w, 0.0), x, rtol=1e-13)
    # with w = 1 the result has unit root-mean-square (plain w, not 1 + w)
    x1 = oracle.rms_norm(h, np.ones_like(h), 0.0)
    assert abs(math.sqrt(np.mean(x1 ** 2)) - 1.0) < 1e-13


def test_rms_norm_matches_python_loop():
    rng = np.random.default_rng(2)
    h = rng.standard_normal(37)
    w = rng.standard_normal(37)
    ss = 0.0
    for v in h:
        ss += v * v
    inv = 1.0 / math.sqrt(ss / len(h) + 1e-6)
    want = [h[i] * inv * w[i] for i in range(len(h))]
    np.testing.assert_allclose(oracle.rms_norm(h, w, 1e-6), want, rtol=1e-13)


# ---------------------------------------------------------------------------
# projections
# ---------------------------------------------------------------------------

def test_project_one_hot_selects_column():
    rng = np.random.default_rng(3)
    x = rng.standard_normal(11)
    W = np.zeros((5, 11))
    W[3, 7] = 1.0
    W[0, 2] = -2.0
    out = oracle.project(W, x)
    np.testing.assert_array_equal(out, [-2.0 * x[2], 0, 0, x[7], 0])


def test_project_matches_python_loop():
    rng = np.random.default_rng(4)
    W = rng.standard_normal((6, 9))
    x = rng.standard_normal(9)
    want = [sum(W[r, c] * x[c] for c in range(9)) for r in range(6)]
    np.testing.assert_allclose(oracle.project(W, x), want, rtol=1e-13)


# ---------------------------------------------------------------------------
# rope
# ---------------------------------------------------------------------------

def test_rope_selection_matches_pages_unit_test():
    with open(os.path.join(GOLDEN, "rope_selection.json")) as f:
        gold = json.load(f)
    for case in gold["cases"]:
        got = oracle.rope_params_for(case["is_full"], case["full_rotary_dim"], case["head_dim"],
                                     case["full_theta"], case["sliding_theta"])
        assert got == (case["rotary_dim"], case["theta"])


def test_rope_identity_at_position_zero():
    rng = np.random.default_rng(5)
    u = rng.standard_normal((4, 256))
    for r, theta in ((64, 5e6), (256, 1e4)):
        np.testing.assert_array_equal(oracle.rope_neox(u, 0, r, theta), u)


def test_rope_keeps_pair_norms_and_passes_tail_through():
    rng = np.random.default_rng(6)
    u = rng.standard_normal((3, 256))
    for r, theta, p in ((64, 5e6, 131072), (256, 1e4, 700), (64, 5e6, 1)):
        out = oracle.rope_neox(u, p, r, theta)
        half = r // 2
        n_in = u[:, :half] ** 2 + u[:, half:r] ** 2
        n_out = out[:, :half] ** 2 + out[:, half:r] ** 2
        np.testing.assert_allclose(n_out, n_in, rtol=1e-12)
        np.testing.assert_array_equal(out[:, r:], u[:, r:])


def test_rope_scores_depend_only_on_relative_position():
    rng = np.random.default_rng(7)
    q = rng.standard_normal((1, 256))
    k = rng.standard_normal((1, 256))
    for r, theta in ((64, 5e6), (256, 1e4)):
        base = float(oracle.rope_neox(q, 900, r, theta)[0] @ oracle.rope_neox(k, 700, r, theta)[0])
        moved = float(oracle.rope_neox(q, 1900, r, theta)[0] @ oracle.rope_neox(k, 1700, r, theta)[0])
        assert abs(base - moved) < 1e-9 * max(1.0, abs(base))


def _unit(d, i):
    u = np.zeros((1, d))
    u[0, i] = 1.0
    return u


def test_rope_neox_half_split_pairing_and_first_pair_angle():
    # pair 0 has frequency theta^0 = 1, so its angle is the position itself,
    # and NeoX pairs dim i with dim i + r/2 (not with i + 1)
    for r, theta in ((64, 5e6), (256, 1e4)):
        for p in (1, 3, 700):
            out = oracle.rope_neox(_unit(256, 0), p, r, theta)[0]
            assert abs(out[0] - math.cos(p)) < 1e-12
            assert abs(out[r // 2] - math.sin(p)) < 1e-12
            assert np.count_nonzero(np.abs(out) > 1e-15) == 2


def test_rope_frequency_divisor_is_rotary_dim():
    # at pair i = r/4 the frequency theta^(-2i/r) is theta^(-1/2); with the
    # head dim as divisor it would be theta^(-1/8) for the full class
    for r, theta, p in ((64, 5e6, 131072), (256, 1e4, 100), (256, 1e4, 40)):
        i = r // 4
        out = oracle.rope_neox(_unit(256, i), p, r, theta)[0]
        ang = math.atan2(out[i + r // 2], out[i])
        want = math.remainder(p / math.sqrt(theta), 2 * math.pi)
        assert abs(ang - want) < 1e-9
    # theta 1e4: pair 64 of 256 turns by exactly 0.01 rad per position
    out = oracle.rope_neox(_unit(256, 64), 100, 256, 1e4)[0]
    assert abs(out[64] - math.cos(1.0)) < 1e-12 and abs(out[192] - math.sin(1.0)) < 1e-12


def test_rope_class_swap_changes_result():
    rng = np.random.default_rng(8)
    u = rng.standard_normal((1, 256))
    full = oracle.rope_neox(u, 700, *oracle.rope_params_for(True, 64, 256, 5e6, 1e4))
    sliding = oracle.rope_neox(u, 700, *oracle.rope_params_for(False, 64, 256, 5e6, 1e4))
    assert np.max(np.abs(full - sliding)) > 0.1
    np.testing.assert_array_equal(full[:, 64:], u[:, 64:])


# ---------------------------------------------------------------------------
# window and ring addressing
# ---------------------------------------------------------------------------

def _simulate(positions_written, ring_capacity, capacity):
    """Write positions 0..P into a ring buffer (or a linear array) one by one
    and return the storage: row -> position it now holds."""
    store = [None] * capacity
    for pos in range(positions_written + 1):
        row = pos % ring_capacity if ring_capacity > 0 else pos
        store[row] = pos
    return store


@pytest.mark.parametrize("window,ring", [(4, 4), (4, 6), (3, 0), (5, 5), (1, 1), (7, 9)])
def test_window_and_ring_by_simulation(window, ring):
    cap = ring if ring > 0 else 64
    for p in range(0, 40 if ring > 0 else 60):
        store = _simulate(p, ring, cap)
        # write slot: where the simulation put position p
        assert store[oracle.write_slot(p, ring)] == p
        for is_full in (False, True):
            if is_full and ring > 0:
                continue  # a full layer keeps every row (no ring)
            seq_len, kv_start, active = oracle.window_params(p, is_full, window, ring)
            assert seq_len == p + 1
            want = list(range(0, p + 1)) if is_full else list(range(max(0, p + 1 - window), p + 1))
            got = [store[oracle.read_slot(j, active)] for j in range(kv_start, seq_len)]
            assert got == want


def test_window_hand_values():
    # decode at 700 on a sliding layer with window 512 and ring 512: the ring
    # has wrapped, 512 rows from position 189, the token lands in row 188
    assert oracle.window_params(700, False, 512, 512) == (701, 189, 512)
    assert oracle.write_slot(700, 512) == 188
    assert oracle.window_params(40, False, 512, 512) == (41, 0, 0)
    assert oracle.window_params(511, False, 512, 512) == (512, 0, 0)
    assert oracle.window_params(512, False, 512, 512) == (513, 1, 512)
    assert oracle.window_params(131072, True, 512, 0) == (131073, 0, 0)
    assert oracle.window_params(131072, False, 512, 512) == (131073, 130561, 512)
    assert oracle.write_slot(131072, 512) == 0


# ---------------------------------------------------------------------------
# attention
# ---------------------------------------------------------------------------

def test_attention_single_row_returns_v():
    rng = np.random.default_rng(9)
    q = rng.standard_normal((16, 256))
    k = rng.standard_normal((1, 4, 256))
    v = rng.standard_normal((1, 4, 256))
    a = oracle.attention_decode(q, k, v, 1 / 16, 4)
    for h in range(16):
        np.testing.assert_array_equal(a[h], v[0, h // 4])


def test_attention_equal_keys_give_window_mean():
    rng = np.random.default_rng(10)
    q = rng.standard_normal((16, 256))
    k = np.repeat(rng.standard_normal((1, 4, 256)), 50, axis=0)
    v = rng.standard_normal((50, 4, 256))
    a = oracle.attention_decode(q, k, v, 1 / 16, 4)
    for h in range(16):
        np.testing.assert_allclose(a[h], v[:, h // 4].mean(axis=0), rtol=1e-12, atol=1e-14)


def test_attention_gqa_head_map():
    rng = np.random.default_rng(11)
    q = rng.standard_normal((16, 256))
    k = rng.standard_normal((30, 4, 256))
    v = rng.standard_normal((30, 4, 256))
    a = oracle.attention_decode(q, k, v, 1 / 16, 4)
    for j in range(4):
        k2, v2 = k.copy(), v.copy()
        k2[:, j] += rng.standard_normal((30, 256))
        v2[:, j] += 1.0
        a2 = oracle.attention_decode(q, k2, v2, 1 / 16, 4)
        changed = [h for h in range(16) if np.max(np.abs(a2[h] - a[h])) > 1e-12]
        assert changed == [4 * j, 4 * j + 1, 4 * j + 2, 4 * j + 3]


def test_attention_matches_python_softmax():
    rng = np.random.default_rng(12)
    n_q, n_kv, d, n = 4, 2, 3, 5
    q = rng.standard_normal((n_q, d))
    k = rng.standard_normal((n, n_kv, d))
    v = rng.standard_normal((n, n_kv, d))
    scale = 0.7
    got = oracle.attention_decode(q, k, v, scale, n_kv)
    for h in range(n_q):
        kvh = h // (n_q // n_kv)
        s = [scale * sum(q[h][i] * k[j][kvh][i] for i in range(d)) for j in range(n)]
        e = [math.exp(x) for x in s]
        z = sum(e)
        want = [sum(e[j] / z * v[j][kvh][i] for j in range(n)) for i in range(d)]
        np.testing.assert_allclose(got[h], want, rtol=1e-12)


# ---------------------------------------------------------------------------
# gate and residual
# ---------------------------------------------------------------------------

def test_sigmoid_known_values_and_gate_halves():
    np.testing.assert_array_equal(oracle.sigmoid(np.array([0.0])), [0.5])
    assert abs(oracle.sigmoid(np.array([math.log(3.0)]))[0] - 0.75) < 1e-15
    rng = np.random.default_rng(13)
    a = rng.standard_normal((16, 256))
    np.testing.assert_array_equal(oracle.head_gate(a, np.zeros(16)), a * 0.5)
    # one scalar per head, broadcast over head_dim, head 5 alone is switched on
    g = np.full(16, -np.inf)
    g[5] = np.inf
    gated = oracle.head_gate(a, g)
    assert np.all(gated[np.arange(16) != 5] == 0)
    np.testing.assert_array_equal(gated[5], a[5])


# ---------------------------------------------------------------------------
# the whole block
# ---------------------------------------------------------------------------

def _tiny_inputs(rng, geom, B, cap, bf16):
    H = geom.hidden
    rows = geom.q_dim + 2 * geom.kv_dim

    def w(shape, scale):
        x = (rng.standard_normal(shape) * scale).astype(np.float32)
        return oracle.f64_to_bf16_bits(x.astype(np.float64)) if bf16 else x

    weights = {
        "norm_w": w((H,), 1.0),
        "qkv_w": w((rows, H), H ** -0.5),
        "g_w": w((geom.n_q, H), H ** -0.5),
        "o_w": w((H, geom.q_dim), geom.q_dim ** -0.5),
    }
    kc = w((B, cap, geom.n_kv, geom.head_dim), 1.0)
    vc = w((B, cap, geom.n_kv, geom.head_dim), 1.0)
    h = rng.standard_normal((B, H)).astype(np.float32)
    return h, weights, kc, vc


def test_decode_step_zero_o_proj_returns_h_exactly():
    geom = OracleGeometry(hidden=32, n_q=8, n_kv=2, head_dim=8, full_rotary_dim=4, window=6,
                          scale=8 ** -0.5)
    rng = np.random.default_rng(14)
    h, weights, kc, vc = _tiny_inputs(rng, geom, 2, 12, False)
    weights["o_w"] = np.zeros_like(weights["o_w"])
    res = oracle.decode_step(geom, h, weights, kc, vc, True, [5, 11], 0)
    for b in range(2):
        np.testing.assert_array_equal(res["out"][b], h[b].astype(np.float64))


def test_decode_step_zero_gate_halves_attention():
    geom = OracleGeometry(hidden=32, n_q=8, n_kv=2, head_dim=8, full_rotary_dim=4, window=6,
                          scale=8 ** -0.5)
    rng = np.random.default_rng(15)
    h, weights, kc, vc = _tiny_inputs(rng, geom, 1, 12, False)
    weights["g_w"] = np.zeros_like(weights["g_w"])
    res = oracle.decode_step(geom, h, weights, kc, vc, False, [9], 0)
    np.testing.assert_array_equal(res["a_gated"][0], 0.5 * res["a"][0])


def test_decode_step_sliding_window_excludes_old_rows_full_does_not():
    geom = OracleGeometry(hidden=32, n_q=8, n_kv=2, head_dim=8, full_rotary_dim=4, window=6,
                          scale=8 ** -0.5)
    rng = np.random.default_rng(16)
    h, weights, kc, vc = _tiny_inputs(rng, geom, 1, 40, True)
    p = 30
    kc2, vc2 = kc.copy(), vc.copy()
    old = slice(0, p + 1 - geom.window)        # rows older than seq_len - window
    kc2[0, old] = oracle.f64_to_bf16_bits(rng.standard_normal(kc2[0, old].shape))
    vc2[0, old] = oracle.f64_to_bf16_bits(rng.standard_normal(vc2[0, old].shape))
    s1 = oracle.decode_step(geom, h, weights, kc, vc, False, [p], 0)
    s2 = oracle.decode_step(geom, h, weights, kc2, vc2, False, [p], 0)
    np.testing.assert_array_equal(s1["out"][0], s2["out"][0])
    f1 = oracle.decode_step(geom, h, weights, kc, vc, True, [p], 0)
    f2 = oracle.decode_step(geom, h, weights, kc2, vc2, True, [p], 0)
    assert np.max(np.abs(f1["out"][0] - f2["out"][0])) > 1e-6


def _python_block(geom, h, weights, kc, vc, is_full, p, ring, bf16):
    """The whole block as plain Python loops on one sequence."""
    def f(x):
        return float(oracle.bf16_bits_to_f64(np.array([x]))[0]) if bf16 else float(x)

    H, nq, nkv, d = geom.hidden, geom.n_q, geom.n_kv, geom.head_dim
    hv = [float(x) for x in h]
    ss = sum(x * x for x in hv)
    inv = 1.0 / math.sqrt(ss / H + geom.eps)
    x = [hv[i] * inv * f(weights["norm_w"][i]) for i in range(H)]
    rows = nq * d + 2 * nkv * d
    qkv = [sum(f(weights["qkv_w"][r][c]) * x[c] for c in range(H)) for r in range(rows)]
    gl = [sum(f(weights["g_w"][r][c]) * x[c] for c in range(H)) for r in range(nq)]
    if is_full:
        rdim, theta = geom.full_rotary_dim, geom.full_theta
    else:
        rdim, theta = d, geom.sliding_theta

    def rope(vec):
        out = list(vec)
        for i in range(rdim // 2):
            ang = p * theta ** (-2.0 * i / rdim)
            a, b = vec[i], vec[i + rdim // 2]
            out[i] = a * math.cos(ang) - b * math.sin(ang)
            out[i + rdim // 2] = b * math.cos(ang) + a * math.sin(ang)
        return out

    q = [rope(qkv[hh * d:(hh + 1) * d]) for hh in range(nq)]
    k = [rope(qkv[nq * d + j * d: nq * d + (j + 1) * d]) for j in range(nkv)]
    v = [qkv[nq * d + nkv * d + j * d: nq * d + nkv * d + (j + 1) * d] for j in range(nkv)]
    # the cache as Python lists of floats; the new rows stored at cache precision
    cap = kc.shape[0]
    K = [[[f(kc[s][j][i]) for i in range(d)] for j in range(nkv)] for s in range(cap)]
    V = [[[f(vc[s][j][i]) for i in range(d)] for j in range(nkv)] for s in range(cap)]
    slot = p % ring if ring > 0 else p

    def to_cache(val):
        if bf16:
            return float(oracle.bf16_bits_to_f64(oracle.f64_to_bf16_bits(np.array([val])))[0])
        return float(np.float32(val))

    K[slot] = [[to_cache(val) for val in k[j]] for j in range(nkv)]
    V[slot] = [[to_cache(val) for val in v[j]] for j in range(nkv)]
    # visible positions: the whole history (full) or the last `window` (sliding)
    first = 0 if is_full else max(0, p + 1 - geom.window)
    positions = list(range(first, p + 1))
    grp = nq // nkv
    a = []
    for hh in range(nq):
        j = hh // grp
        rows_k = [K[pos % ring if ring > 0 else pos][j] for pos in positions]
        rows_v = [V[pos % ring if ring > 0 else pos][j] for pos in positions]
        s = [geom.scale * sum(q[hh][i] * rk[i] for i in range(d)) for rk in rows_k]
        m = max(s)
        e = [math.exp(val - m) for val in s]
        z = sum(e)
        gate = 1.0 / (1.0 + math.exp(-gl[hh]))
        a.append([gate * sum(e[t] / z * rows_v[t][i] for t in range(len(e))) for i in range(d)])
    flat = [val for head in a for val in head]
    o = [sum(f(weights["o_w"][r][c]) * flat[c] for c in range(nq * d)) for r in range(H)]
    return [hv[r] + o[r] for r in range(H)]


@pytest.mark.parametrize("is_full,ring,bf16,p", [
    (True, 0, True, 9), (False, 6, True, 13), (False, 6, False, 4), (False, 0, True, 11),
    (True, 0, False, 0)])
def test_decode_step_matches_python_block(is_full, ring, bf16, p):
    geom = OracleGeometry(hidden=16, n_q=8, n_kv=2, head_dim=8, full_rotary_dim=4, window=6,
                          full_theta=500.0, sliding_theta=10.0, scale=8 ** -0.5)
    rng = np.random.default_rng(100 + p)
    cap = ring if ring > 0 else 16
    h, weights, kc, vc = _tiny_inputs(rng, geom, 1, cap, bf16)
    res = oracle.decode_step(geom, h, weights, kc, vc, is_full, [p], ring)
    want = _python_block(geom, h[0], weights, kc[0], vc[0], is_full, p, ring, bf16)
    np.testing.assert_allclose(res["out"][0], want, rtol=1e-11, atol=1e-12)


# ---------------------------------------------------------------------------
# a chunk of consecutive tokens (prefill / verify)
# ---------------------------------------------------------------------------

def _dense_chunk(geom, h, weights, history_k, history_v, hist_pos, is_full, p0, bf16):
    """The chunk in one dense pass, written independently of decode_step:
    every token projected at once as a matrix product, the history and the
    chunk's own rows laid out by logical position, one mask (causal, and for
    a sliding layer the window) over positions, a row-wise softmax.
    history_k/v: rows of the positions in hist_pos (already in the cache)."""
    def wf(x):
        return oracle.bf16_bits_to_f64(x) if bf16 else np.asarray(x, dtype=np.float64)

    def to_cache(x):
        return oracle.bf16_bits_to_f64(oracle.f64_to_bf16_bits(x)) if bf16 else x.astype(np.float32).astype(np.float64)

    M, H = h.shape
    nq, nkv, d = geom.n_q, geom.n_kv, geom.head_dim
    hh = h.astype(np.float64)
    X = hh / np.sqrt(np.mean(hh * hh, axis=1, keepdims=True) + geom.eps) * wf(weights["norm_w"])[None]
    QKV = X @ wf(weights["qkv_w"]).T
    G = X @ wf(weights["g_w"]).T
    Q = QKV[:, :nq * d].reshape(M, nq, d)
    K = QKV[:, nq * d:(nq + nkv) * d].reshape(M, nkv, d)
    V = QKV[:, (nq + nkv) * d:].reshape(M, nkv, d)
    r, theta = (geom.full_rotary_dim, geom.full_theta) if is_full else (d, geom.sliding_theta)
    half = r // 2
    pos = p0 + np.arange(M)
    ang = pos[:, None] * theta ** (-2.0 * np.arange(half) / r)[None]      # [M, half]
    c, s = np.cos(ang)[:, None], np.sin(ang)[:, None]

    def rot(u):
        out = u.copy()
        a, b = u[..., :half], u[..., half:r]
        out[..., :half] = a * c - b * s
        out[..., half:r] = b * c + a * s
        return out

    Q, K = rot(Q), rot(K)
    Kc, Vc = to_cache(K), to_cache(V)
    keys_pos = np.concatenate([np.asarray(hist_pos, dtype=np.int64), pos])
    Kall = np.concatenate([history_k, Kc], axis=0)                          # [P, nkv, d]
    Vall = np.concatenate([history_v, Vc], axis=0)
    mask = keys_pos[None, :] <= pos[:, None]
    if not is_full:
        mask &= keys_pos[None, :] > pos[:, None] - geom.window
    grp = nq // nkv
    A = np.zeros((M, nq, d))
    for hq in range(nq):
        S = geom.scale * np.einsum("md,pd->mp", Q[:, hq], Kall[:, hq // grp])
        S = np.where(mask, S, -np.inf)
        P = np.exp(S - S.max(axis=1, keepdims=True))
        P /= P.sum(axis=1, keepdims=True)
        A[:, hq] = P @ Vall[:, hq // grp]
    A *= (1.0 / (1.0 + np.exp(-G)))[:, :, None]
    O = A.reshape(M, nq * d) @ wf(weights["o_w"]).T
    return hh + O


def _chunk_geom():
    return OracleGeometry(hidden=16, n_q=8, n_kv=2, head_dim=8, full_rotary_dim=4, window=6,
                          full_theta=500.0, sliding_theta=10.0, scale=8 ** -0.5)


def test_prefill_chunk_one_token_is_a_decode_step():
    geom = _chunk_geom()
    rng = np.random.default_rng(200)
    h, weights, kc, vc = _tiny_inputs(rng, geom, 1, 6, True)
    res = oracle.prefill_chunk(geom, h, weights, kc[0], vc[0], False, 9, 6)
    step = oracle.decode_step(geom, h, weights, kc, vc, False, [9], 6)
    np.testing.assert_array_equal(res["out"][0], step["out"][0])
    np.testing.assert_array_equal(res["k_cache"][step["slot"][0]], step["k_row"][0])


@pytest.mark.parametrize("p0,M,bf16", [(0, 7, True), (5, 9, False), (3, 1, True)])
def test_prefill_chunk_full_layer_matches_dense_causal(p0, M, bf16):
    geom = _chunk_geom()
    rng = np.random.default_rng(210 + p0 + M)
    cap = p0 + M + 3
    _, weights, kc, vc = _tiny_inputs(rng, geom, 1, cap, bf16)
    h = rng.standard_normal((M, geom.hidden)).astype(np.float32)
    res = oracle.prefill_chunk(geom, h, weights, kc[0], vc[0], True, p0, 0)
    hist = list(range(p0))
    want = _dense_chunk(geom, h, weights, oracle.cache_rows_to_f64(kc[0][:p0]),
                        oracle.cache_rows_to_f64(vc[0][:p0]), hist, True, p0, bf16)
    np.testing.assert_allclose(res["out"], want, rtol=1e-10, atol=1e-11)
    # rows past the chunk are untouched, the chunk's slots hold its rows
    np.testing.assert_array_equal(res["k_cache"][p0 + M:], kc[0][p0 + M:])
    assert res["slot"] == list(range(p0, p0 + M))


@pytest.mark.parametrize("p0,M", [(4, 5), (9, 8), (2, 15), (13, 2)])
def test_prefill_chunk_ring_wrapping_inside_the_chunk(p0, M):
    """Sliding layer, ring capacity == window: tokens late in the chunk
    overwrite ring rows that earlier tokens of the same chunk still read;
    each token must see the row of the position it needs."""
    geom = _chunk_geom()
    R = geom.window
    rng = np.random.default_rng(230 + p0 + M)
    _, weights, kc, vc = _tiny_inputs(rng, geom, 1, R, True)
    h = rng.standard_normal((M, geom.hidden)).astype(np.float32)
    res = oracle.prefill_chunk(geom, h, weights, kc[0], vc[0], False, p0, R)
    # history: the positions the ring holds before the chunk, by logical position
    hist = list(range(max(0, p0 - R), p0))
    hk = oracle.cache_rows_to_f64(kc[0][[x % R for x in hist]]) if hist else np.zeros((0, geom.n_kv, geom.head_dim))
    hv = oracle.cache_rows_to_f64(vc[0][[x % R for x in hist]]) if hist else np.zeros((0, geom.n_kv, geom.head_dim))
    want = _dense_chunk(geom, h, weights, hk, hv, hist, False, p0, True)
    np.testing.assert_allclose(res["out"], want, rtol=1e-10, atol=1e-11)
    # brute-force ring: replay the writes in order into a dict slot -> position
    holder = {x % R: x for x in range(max(0, p0 - R), p0)}
    for t in range(M):
        holder[(p0 + t) % R] = p0 + t
    for slot in range(R):
        x = holder.get(slot)
        if x is not None and x >= p0:
            np.testing.assert_array_equal(res["k_cache"][slot], res["k_row"][x - p0])
        else:
            np.testing.assert_array_equal(res["k_cache"][slot], kc[0][slot])
