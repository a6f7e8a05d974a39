"""Host-side checks of the C ABI that need no GPU.

The library loads and exports every entry point ``include/spark_attn.h``
declares; invalid arguments are rejected with the documented status before
anything touches a device (so these calls are safe without a GPU).
"""

import ctypes
import os
import re

import pytest

from decode_attention_block_gb300 import build_lib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def B():
    build_lib.build()
    from decode_attention_block_gb300 import binding
    binding.load()
    return binding


def _declared_functions():
    names = []
    inc = os.path.join(ROOT, "include")
    for f in sorted(os.listdir(inc)):
        if not f.endswith(".h"):
            continue
        text = re.sub(r"/\*.*?\*/", "", open(os.path.join(inc, f)).read(), flags=re.S)
        names += re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\**\s*(spark_[a-z0-9_]+)\s*\(",
                            text, flags=re.M)
    return sorted(set(names))


def test_every_declared_symbol_is_exported_and_bound(B):
    declared = _declared_functions()
    assert len(declared) >= 10
    lib = ctypes.CDLL(build_lib.LIB_PATH)
    for name in declared:
        assert hasattr(lib, name), f"{name} declared in include/ but not exported"
    assert sorted(B.declared_symbols()) == declared


def test_abi_version_and_status_strings(B):
    assert B.spark_attn_abi_version() == 4
    for code in range(-7, 1):
        s = B.spark_attn_status_string(code)
        assert s and s != "unknown status"
    assert B.spark_attn_status_string(-99) == "unknown status"


def test_geometry_default_is_spark2_5(B):
    g = B.spark_geom_default()
    assert (g.hidden, g.n_q, g.n_kv, g.head_dim, g.full_rotary_dim, g.window) == (2560, 16, 4, 256, 64, 512)
    assert g.full_theta == 5e6 and g.sliding_theta == 1e4
    assert abs(g.eps - 1e-6) < 1e-12 and g.scale == 0.0625


def test_workspace_bytes(B):
    g = B.spark_geom_default()
    sizes = [B.spark_attn_workspace_bytes(g, b) for b in (1, 2, 64, 1024)]
    assert all(s > 0 and s % 256 == 0 for s in sizes)
    assert sizes == sorted(sizes)
    assert B.spark_attn_workspace_bytes(g, 0) == 0
    assert B.spark_attn_workspace_bytes(g, 1025) == 0
    bad = B.spark_geom_default()
    bad.head_dim = 128
    assert B.spark_attn_workspace_bytes(bad, 1) == 0


# -- argument validation, all rejected on the host ---------------------------

FAKE = 1 << 40          # 16-byte aligned, never dereferenced: validation fails first


def _call(B, geom=None, weights=None, kv=None, cls=1, positions=(5,), batch=None, h=FAKE,
          out=FAKE, ws=FAKE, ws_bytes=None):
    lib = B.load()
    g = geom or B.spark_geom_default()
    w = weights or B.SparkLayerWeights(FAKE, FAKE, FAKE, FAKE, B.SPARK_BF16)
    k = kv or B.SparkKvLayer(FAKE, FAKE, 1024, 0, B.SPARK_BF16)
    n = len(positions) if batch is None else batch
    pos = (ctypes.c_int32 * max(1, len(positions)))(*positions)
    if ws_bytes is None:
        ws_bytes = B.spark_attn_workspace_bytes(g, max(1, min(n, 1024))) or (1 << 30)
    return lib.spark_attn_decode(ctypes.byref(g), h, ctypes.byref(w), ctypes.byref(k), cls, pos, n,
                                 out, ws, ws_bytes, None)


def test_rejects_null_and_misaligned_pointers(B):
    assert _call(B, h=0) == -1
    assert _call(B, out=0) == -1
    assert _call(B, h=FAKE + 4) == -1
    assert _call(B, weights=B.SparkLayerWeights(FAKE, 0, FAKE, FAKE, B.SPARK_BF16)) == -1
    assert _call(B, weights=B.SparkLayerWeights(FAKE, FAKE + 8, FAKE, FAKE, B.SPARK_BF16)) == -1
    assert _call(B, kv=B.SparkKvLayer(0, FAKE, 1024, 0, B.SPARK_BF16)) == -1


def test_rejects_bad_enums_and_batch(B):
    assert _call(B, cls=2) == -1
    assert _call(B, weights=B.SparkLayerWeights(FAKE, FAKE, FAKE, FAKE, 7)) == -1
    assert _call(B, kv=B.SparkKvLayer(FAKE, FAKE, 1024, 0, 5)) == -1
    assert _call(B, positions=(1,), batch=0) == -1
    assert _call(B, positions=tuple([1] * 1025)) == -1


def test_rejects_positions_outside_the_cache(B):
    assert _call(B, positions=(1024,)) == -2            # linear cache of 1024 rows: 0..1023
    assert _call(B, positions=(-1,)) == -2
    assert _call(B, positions=(3, 2000, 4)) == -2
    # a ring layer keeps any position (row p mod ring)
    ring = B.SparkKvLayer(FAKE, FAKE, 512, 512, B.SPARK_BF16)
    assert _call(B, kv=ring, cls=0, positions=(131072,), ws=FAKE + 16) == -4  # passes kv checks, fails ws


def test_rejects_bad_rings(B):
    g = B.spark_geom_default()
    # a full layer has no ring
    assert _call(B, kv=B.SparkKvLayer(FAKE, FAKE, 512, 512, B.SPARK_BF16), cls=1) == -3
    # a ring shorter than the window would evict rows the window still reads
    assert _call(B, kv=B.SparkKvLayer(FAKE, FAKE, 512, 256, B.SPARK_BF16), cls=0) == -3
    # a ring larger than the buffer
    assert _call(B, kv=B.SparkKvLayer(FAKE, FAKE, 512, 1024, B.SPARK_BF16), cls=0) == -1
    assert g.window == 512


def test_rejects_small_or_misaligned_workspace(B):
    g = B.spark_geom_default()
    need = B.spark_attn_workspace_bytes(g, 1)
    assert _call(B, ws_bytes=need - 1) == -4
    assert _call(B, ws=FAKE + 16) == -4
    assert _call(B, ws=0) == -4


def test_rejects_unsupported_geometry(B):
    for field, val in (("head_dim", 128), ("n_q", 8), ("n_kv", 16), ("hidden", 2564),
                       ("full_rotary_dim", 63), ("full_rotary_dim", 512)):
        g = B.spark_geom_default()
        setattr(g, field, val)
        if field == "n_kv":
            g.n_q = 4 * val
        assert _call(B, geom=g) == -5, field
    g = B.spark_geom_default()
    g.window = 0
    assert _call(B, geom=g) == -1
    g = B.spark_geom_default()
    g.scale = float("nan")
    assert _call(B, geom=g) == -1


def _dbg_qkv(B, path, dtype=None, batch=2):
    lib = B.load()
    g = B.spark_geom_default()
    w = B.SparkLayerWeights(FAKE, FAKE, FAKE, FAKE, B.SPARK_BF16 if dtype is None else dtype)
    k = B.SparkKvLayer(FAKE, FAKE, 1024, 0, B.SPARK_BF16)
    pos = (ctypes.c_int32 * batch)(*([5] * batch))
    need = B.spark_attn_workspace_bytes(g, batch)
    return lib.spark_dbg_qkv_rope(ctypes.byref(g), FAKE, ctypes.byref(w), ctypes.byref(k), 1, pos, batch,
                                  FAKE, FAKE, path, FAKE, need, None)


def _dbg_oproj(B, path, dtype=None, batch=2, ws_bytes=None):
    lib = B.load()
    g = B.spark_geom_default()
    w = B.SparkLayerWeights(FAKE, FAKE, FAKE, FAKE, B.SPARK_BF16 if dtype is None else dtype)
    need = B.spark_attn_workspace_bytes(g, batch) if ws_bytes is None else ws_bytes
    return lib.spark_dbg_gate_oproj(ctypes.byref(g), FAKE, FAKE, FAKE, ctypes.byref(w), batch, FAKE, path,
                                    FAKE, need, None)


def test_projection_path_argument_is_validated(B):
    # an unknown path, and the tensor-core path forced on fp32 weights, are
    # refused before anything is enqueued
    assert _dbg_qkv(B, 3) == -1
    assert _dbg_qkv(B, -1) == -1
    assert _dbg_oproj(B, 9) == -1
    assert _dbg_qkv(B, B.SPARK_PATH_MMA, dtype=B.SPARK_F32) == -5
    assert _dbg_oproj(B, B.SPARK_PATH_MMA, dtype=B.SPARK_F32) == -5
    # the stage entry points need a workspace now
    assert _dbg_oproj(B, 0, ws_bytes=16) == -4


def test_workspace_grows_with_the_tensor_core_batch(B):
    g = B.spark_geom_default()
    small, b8, b64, b128, b1024 = (B.spark_attn_workspace_bytes(g, b) for b in (1, 8, 64, 128, 1024))
    assert small < b8 < b64 < b128 < b1024


def _prefill(B, p0=5, m=3, cls=1, kv=None, ws_bytes=None):
    lib = B.load()
    g = B.spark_geom_default()
    w = B.SparkLayerWeights(FAKE, FAKE, FAKE, FAKE, B.SPARK_BF16)
    k = kv or B.SparkKvLayer(FAKE, FAKE, 1024, 0, B.SPARK_BF16)
    need = B.spark_attn_workspace_bytes(g, max(1, min(m, 1024))) if ws_bytes is None else ws_bytes
    return lib.spark_attn_prefill(ctypes.byref(g), FAKE, ctypes.byref(w), ctypes.byref(k), cls, p0, m, FAKE,
                                  FAKE, need or (1 << 30), None)


def test_prefill_arguments_are_validated(B):
    assert _prefill(B, m=0) == -1
    assert _prefill(B, m=1025) == -1
    assert _prefill(B, p0=-1) == -2
    assert _prefill(B, p0=1020, m=5) == -2                # a linear cache of 1024 rows ends at 1023
    ring = B.SparkKvLayer(FAKE, FAKE, 512, 512, B.SPARK_BF16)
    assert _prefill(B, p0=1 << 20, m=600, cls=0, kv=ring, ws_bytes=16) == -4   # any position on a ring
    assert _prefill(B, cls=1, kv=ring) == -3              # a full layer has no ring
    assert _prefill(B, ws_bytes=64) == -4


def test_wait_timeout_arguments_are_validated(B):
    lib = B.load()
    assert lib.spark_dbg_wait_timeout(FAKE, 4096, 0, None) == -1
    assert lib.spark_dbg_wait_timeout(FAKE, 4096, 3_000_000_000, None) == -1
    assert lib.spark_dbg_wait_timeout(FAKE + 16, 4096, 1000, None) == -4
    assert lib.spark_dbg_wait_timeout(0, 4096, 1000, None) == -4


# -- the rest of the decoder layer and the head ------------------------------

def _mlp(B, inter=10240, batch=1, dtype=None, path=0, ptrs=None, h=FAKE, out=FAKE, ws=FAKE, ws_bytes=None,
         geom=None):
    lib = B.load()
    g = geom or B.spark_geom_default()
    dt = B.SPARK_BF16 if dtype is None else dtype
    p = ptrs or (FAKE, FAKE, FAKE, FAKE)
    w = B.SparkMlpWeights(p[0], p[1], p[2], p[3], inter, dt)
    if ws_bytes is None:
        ws_bytes = B.spark_mlp_workspace_bytes(g, inter, max(1, min(batch, 1024))) or (1 << 30)
    return lib.spark_mlp_decode(ctypes.byref(g), h, ctypes.byref(w), batch, out, path, ws, ws_bytes, None)


def _head(B, vocab=131072, batch=1, dtype=None, path=0, norm=FAKE, embed=FAKE, ws=FAKE, ws_bytes=None):
    lib = B.load()
    g = B.spark_geom_default()
    dt = B.SPARK_BF16 if dtype is None else dtype
    if ws_bytes is None:
        ws_bytes = B.spark_mlp_workspace_bytes(g, 0, max(1, min(batch, 1024))) or (1 << 30)
    return lib.spark_head_logits(ctypes.byref(g), FAKE, norm, embed, vocab, dt, batch, FAKE, path, ws, ws_bytes,
                                 None)


def test_mlp_workspace_bytes(B):
    g = B.spark_geom_default()
    sizes = [B.spark_mlp_workspace_bytes(g, 10240, b) for b in (1, 8, 64, 1024)]
    assert all(s > 0 and s % 256 == 0 for s in sizes) and sizes == sorted(sizes)
    assert B.spark_mlp_workspace_bytes(g, 0, 1) < B.spark_mlp_workspace_bytes(g, 8, 1)
    for inter in (-8, 4, 12, 16392):
        assert B.spark_mlp_workspace_bytes(g, inter, 1) == 0
    assert B.spark_mlp_workspace_bytes(g, 10240, 0) == 0


def test_mlp_arguments_are_validated(B):
    assert _mlp(B, h=0) == -1
    assert _mlp(B, out=FAKE + 4) == -1
    assert _mlp(B, ptrs=(FAKE, FAKE, 0, FAKE)) == -1
    assert _mlp(B, ptrs=(FAKE, FAKE + 8, FAKE, FAKE)) == -1
    assert _mlp(B, dtype=3) == -1
    assert _mlp(B, batch=0) == -1
    assert _mlp(B, batch=1025) == -1
    assert _mlp(B, inter=-8) == -1
    assert _mlp(B, inter=12, ws_bytes=1 << 30) == -5      # not a multiple of 8
    assert _mlp(B, inter=16392, ws_bytes=1 << 30) == -5
    assert _mlp(B, path=5) == -1
    assert _mlp(B, batch=8, path=B.SPARK_PATH_MMA, dtype=B.SPARK_F32) == -5
    need = B.spark_mlp_workspace_bytes(B.spark_geom_default(), 10240, 1)
    assert _mlp(B, ws_bytes=need - 1) == -4
    assert _mlp(B, ws=FAKE + 16) == -4
    bad = B.spark_geom_default()
    bad.hidden = 2564
    assert _mlp(B, geom=bad, ws_bytes=1 << 30) == -5


def test_head_arguments_are_validated(B):
    assert _head(B, norm=0) == -1
    assert _head(B, embed=FAKE + 8) == -1
    assert _head(B, vocab=0) == -1
    assert _head(B, vocab=1001) == -5
    assert _head(B, vocab=(1 << 22) + 8) == -5
    assert _head(B, dtype=2) == -1
    assert _head(B, batch=0) == -1
    assert _head(B, path=7) == -1
    assert _head(B, batch=8, path=B.SPARK_PATH_MMA, dtype=B.SPARK_F32) == -5
    assert _head(B, ws_bytes=64) == -4
    assert _head(B, ws=0) == -4


def test_descriptors_cache_their_c_struct_until_a_field_changes(B, monkeypatch):
    # the struct is built (and its tensors checked) once; reassigning a field
    # drops it, so the next call builds it again from the new tensors
    built = []

    def fake_build(self):
        built.append(self)
        return object()

    monkeypatch.setattr(B.LayerWeights, "_build_c", fake_build)
    w = B.LayerWeights(None, None, None, None)
    first = w.to_c()
    assert w.to_c() is first and len(built) == 1
    w.o_w = None                      # a field reassigned: the cache is dropped
    second = w.to_c()
    assert second is not first and len(built) == 2
    assert w.to_c() is second
