"""ctypes binding of ``libspark_attn.so`` (the C ABI in ``include/spark_attn.h``
and ``include/spark_layer.h``).

Argument marshalling only: every step of the block runs in the library's CUDA
kernels.  Tensors are PyTorch CUDA tensors (PyTorch provides device memory and
streams); the functions carry the C entry points' names and check only what
the C side cannot see (tensor devices, dtypes, contiguity and shapes).  The
library must have been built (``decode_attention_block_gb300.build_lib.build``);
importing the binding without it raises instead of falling back to anything.
"""

from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass, field

import torch

from .build_lib import LIB_PATH

SPARK_OK = 0
SPARK_PATH_AUTO, SPARK_PATH_GEMV, SPARK_PATH_MMA = 0, 1, 2
SPARK_F32 = 0
SPARK_BF16 = 1
SPARK_SLIDING = 0
SPARK_FULL = 1
SPARK_MAX_BATCH = 1024

_DTYPE_CODE = {torch.float32: SPARK_F32, torch.bfloat16: SPARK_BF16}


class SparkError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {spark_attn_status_string(status)} (status {status})")


class SparkGeom(ctypes.Structure):
    _fields_ = [
        ("hidden", ctypes.c_int32),
        ("n_q", ctypes.c_int32),
        ("n_kv", ctypes.c_int32),
        ("head_dim", ctypes.c_int32),
        ("full_rotary_dim", ctypes.c_int32),
        ("window", ctypes.c_int32),
        ("full_theta", ctypes.c_float),
        ("sliding_theta", ctypes.c_float),
        ("eps", ctypes.c_float),
        ("scale", ctypes.c_float),
    ]


class SparkLayerWeights(ctypes.Structure):
    _fields_ = [
        ("norm_w", ctypes.c_void_p),
        ("qkv_w", ctypes.c_void_p),
        ("g_w", ctypes.c_void_p),
        ("o_w", ctypes.c_void_p),
        ("dtype", ctypes.c_int32),
    ]


class SparkKvLayer(ctypes.Structure):
    _fields_ = [
        ("k", ctypes.c_void_p),
        ("v", ctypes.c_void_p),
        ("capacity", ctypes.c_int64),
        ("ring_capacity", ctypes.c_int32),
        ("dtype", ctypes.c_int32),
    ]


class SparkMlpWeights(ctypes.Structure):
    _fields_ = [
        ("norm_w", ctypes.c_void_p),
        ("gate_w", ctypes.c_void_p),
        ("up_w", ctypes.c_void_p),
        ("down_w", ctypes.c_void_p),
        ("intermediate", ctypes.c_int32),
        ("dtype", ctypes.c_int32),
    ]


# every symbol include/*.h declares, with its ctypes signature
_P = ctypes.c_void_p
_SIGNATURES = {
    "spark_geom_default": (None, [ctypes.POINTER(SparkGeom)]),
    "spark_attn_workspace_bytes": (ctypes.c_size_t, [ctypes.POINTER(SparkGeom), ctypes.c_int32]),
    "spark_attn_workspace_init": (ctypes.c_int, [_P, ctypes.c_size_t, _P]),
    "spark_attn_error_word": (ctypes.c_int, [_P, ctypes.c_size_t, ctypes.POINTER(ctypes.c_uint32), _P]),
    "spark_attn_decode": (ctypes.c_int, [ctypes.POINTER(SparkGeom), _P, ctypes.POINTER(SparkLayerWeights),
                                         ctypes.POINTER(SparkKvLayer), ctypes.c_int32,
                                         ctypes.POINTER(ctypes.c_int32), ctypes.c_int32, _P, _P,
                                         ctypes.c_size_t, _P]),
    "spark_attn_prefill": (ctypes.c_int, [ctypes.POINTER(SparkGeom), _P, ctypes.POINTER(SparkLayerWeights),
                                          ctypes.POINTER(SparkKvLayer), ctypes.c_int32, ctypes.c_int32,
                                          ctypes.c_int32, _P, _P, ctypes.c_size_t, _P]),
    "spark_attn_decode_stack": (ctypes.c_int, [ctypes.POINTER(SparkGeom), _P, ctypes.c_int32,
                                               ctypes.POINTER(SparkLayerWeights), ctypes.POINTER(SparkKvLayer),
                                               ctypes.POINTER(ctypes.c_int32), ctypes.POINTER(ctypes.c_int32),
                                               ctypes.c_int32, _P, _P, ctypes.c_size_t, _P]),
    "spark_dbg_qkv_rope": (ctypes.c_int, [ctypes.POINTER(SparkGeom), _P, ctypes.POINTER(SparkLayerWeights),
                                          ctypes.POINTER(SparkKvLayer), ctypes.c_int32,
                                          ctypes.POINTER(ctypes.c_int32), ctypes.c_int32, _P, _P,
                                          ctypes.c_int32, _P, ctypes.c_size_t, _P]),
    "spark_dbg_attention": (ctypes.c_int, [ctypes.POINTER(SparkGeom), _P, ctypes.POINTER(SparkKvLayer),
                                           ctypes.c_int32, ctypes.POINTER(ctypes.c_int32), ctypes.c_int32,
                                           _P, ctypes.c_int32, _P, ctypes.c_size_t, _P]),
    "spark_dbg_attention_noalloc": (ctypes.c_int, [ctypes.POINTER(SparkGeom), _P, ctypes.POINTER(SparkKvLayer),
                                                   ctypes.c_int32, ctypes.POINTER(ctypes.c_int32), ctypes.c_int32,
                                                   _P, _P]),
    "spark_dbg_attention_noalloc_error_word": (ctypes.c_int, [ctypes.POINTER(ctypes.c_uint32), _P]),
    "spark_dbg_gate_oproj": (ctypes.c_int, [ctypes.POINTER(SparkGeom), _P, _P, _P,
                                            ctypes.POINTER(SparkLayerWeights), ctypes.c_int32, _P,
                                            ctypes.c_int32, _P, ctypes.c_size_t, _P]),
    "spark_dbg_wait_timeout": (ctypes.c_int, [_P, ctypes.c_size_t, ctypes.c_uint64, _P]),
    "spark_mlp_workspace_bytes": (ctypes.c_size_t, [ctypes.POINTER(SparkGeom), ctypes.c_int32, ctypes.c_int32]),
    "spark_mlp_decode": (ctypes.c_int, [ctypes.POINTER(SparkGeom), _P, ctypes.POINTER(SparkMlpWeights),
                                        ctypes.c_int32, _P, ctypes.c_int32, _P, ctypes.c_size_t, _P]),
    "spark_head_logits": (ctypes.c_int, [ctypes.POINTER(SparkGeom), _P, _P, _P, ctypes.c_int32, ctypes.c_int32,
                                         ctypes.c_int32, _P, ctypes.c_int32, _P, ctypes.c_size_t, _P]),
    "spark_attn_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "spark_attn_abi_version": (ctypes.c_int32, []),
}

_lib = None


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load the library once and bind every declared entry point."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it with "
                           "decode_attention_block_gb300.build_lib.build() (needs nvcc)")
    lib = ctypes.CDLL(path)
    for name, (res, args) in _SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def declared_symbols() -> list[str]:
    return list(_SIGNATURES)


# ---------------------------------------------------------------------------
# marshalling helpers
# ---------------------------------------------------------------------------

def _stream(stream) -> int | None:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _dev_ptr(t: torch.Tensor, name: str, dtype=None) -> int:
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    return t.data_ptr()


def _check(status: int, where: str) -> None:
    if status != SPARK_OK:
        raise SparkError(status, where)


class _CachedC:
    """Mixin of the weight and cache descriptors: the C struct is built and
    checked once and reused while no field is reassigned (the tensors' device
    addresses do not change in place), which keeps the per-call marshalling
    of a decode step short."""

    def __setattr__(self, name, value):
        if name != "_c":
            object.__setattr__(self, "_c", None)
        object.__setattr__(self, name, value)

    def to_c(self):
        if self._c is None:
            object.__setattr__(self, "_c", self._build_c())
        return self._c


def _positions(positions) -> ctypes.Array:
    vals = [int(p) for p in positions]
    return (ctypes.c_int32 * max(1, len(vals)))(*vals)


@dataclass
class LayerWeights(_CachedC):
    """One layer's weights as CUDA tensors (all float32 or all bfloat16):
    ``norm_w [hidden]``, ``qkv_w [n_q*d + 2*n_kv*d, hidden]``,
    ``g_w [n_q, hidden]``, ``o_w [hidden, n_q*d]``."""

    norm_w: torch.Tensor
    qkv_w: torch.Tensor
    g_w: torch.Tensor
    o_w: torch.Tensor
    _c: object = field(default=None, init=False, repr=False, compare=False)

    def _build_c(self) -> SparkLayerWeights:
        dt = self.qkv_w.dtype
        if dt not in _DTYPE_CODE:
            raise TypeError(f"weights must be float32 or bfloat16, got {dt}")
        return SparkLayerWeights(_dev_ptr(self.norm_w, "norm_w", dt), _dev_ptr(self.qkv_w, "qkv_w", dt),
                                 _dev_ptr(self.g_w, "g_w", dt), _dev_ptr(self.o_w, "o_w", dt),
                                 _DTYPE_CODE[dt])


@dataclass
class KvLayer(_CachedC):
    """One layer's cache as CUDA tensors ``k``, ``v`` of shape
    ``[batch, capacity, n_kv, head_dim]`` (float32 or bfloat16) and the ring
    capacity (0 = linear addressing)."""

    k: torch.Tensor
    v: torch.Tensor
    ring_capacity: int = 0
    _c: object = field(default=None, init=False, repr=False, compare=False)

    def _build_c(self) -> SparkKvLayer:
        dt = self.k.dtype
        if dt not in _DTYPE_CODE:
            raise TypeError(f"cache must be float32 or bfloat16, got {dt}")
        if self.k.dim() != 4 or self.k.shape != self.v.shape:
            raise ValueError("k and v must both be [batch, capacity, n_kv, head_dim]")
        return SparkKvLayer(_dev_ptr(self.k, "k", dt), _dev_ptr(self.v, "v", dt),
                            int(self.k.shape[1]), int(self.ring_capacity), _DTYPE_CODE[dt])


@dataclass
class MlpWeights(_CachedC):
    """The MLP half of one layer as CUDA tensors (all float32 or all
    bfloat16): ``norm_w [hidden]`` (post_attention_layernorm), ``gate_w`` and
    ``up_w [intermediate, hidden]``, ``down_w [hidden, intermediate]``."""

    norm_w: torch.Tensor
    gate_w: torch.Tensor
    up_w: torch.Tensor
    down_w: torch.Tensor
    _c: object = field(default=None, init=False, repr=False, compare=False)

    def _build_c(self) -> SparkMlpWeights:
        dt = self.gate_w.dtype
        if dt not in _DTYPE_CODE:
            raise TypeError(f"weights must be float32 or bfloat16, got {dt}")
        if self.gate_w.dim() != 2 or self.up_w.shape != self.gate_w.shape or \
                self.down_w.shape != (self.gate_w.shape[1], self.gate_w.shape[0]):
            raise ValueError("gate_w, up_w must be [intermediate, hidden] and down_w [hidden, intermediate]")
        return SparkMlpWeights(_dev_ptr(self.norm_w, "norm_w", dt), _dev_ptr(self.gate_w, "gate_w", dt),
                               _dev_ptr(self.up_w, "up_w", dt), _dev_ptr(self.down_w, "down_w", dt),
                               int(self.gate_w.shape[0]), _DTYPE_CODE[dt])


# ---------------------------------------------------------------------------
# the entry points
# ---------------------------------------------------------------------------

def spark_geom_default() -> SparkGeom:
    g = SparkGeom()
    load().spark_geom_default(ctypes.byref(g))
    return g


def spark_attn_workspace_bytes(geom: SparkGeom, batch: int) -> int:
    return int(load().spark_attn_workspace_bytes(ctypes.byref(geom), int(batch)))


def spark_attn_workspace_init(ws: torch.Tensor, stream=None) -> None:
    _check(load().spark_attn_workspace_init(_dev_ptr(ws, "workspace"), ws.numel() * ws.element_size(),
                                            _stream(stream)), "spark_attn_workspace_init")


def spark_attn_error_word(ws: torch.Tensor, stream=None) -> int:
    word = ctypes.c_uint32(0)
    _check(load().spark_attn_error_word(_dev_ptr(ws, "workspace"), ws.numel() * ws.element_size(),
                                        ctypes.byref(word), _stream(stream)), "spark_attn_error_word")
    return int(word.value)


def make_workspace(geom: SparkGeom, batch: int, device=None, stream=None) -> torch.Tensor:
    """Allocate (through PyTorch) and initialise a workspace for ``batch``."""
    nbytes = spark_attn_workspace_bytes(geom, batch)
    if nbytes == 0:
        raise ValueError("invalid geometry or batch for a workspace")
    ws = torch.empty(nbytes, dtype=torch.uint8, device=device or "cuda")
    spark_attn_workspace_init(ws, stream)
    return ws


def spark_attn_decode(geom: SparkGeom, h: torch.Tensor, weights: LayerWeights, kv: KvLayer,
                      layer_class: int, positions, out: torch.Tensor, ws: torch.Tensor,
                      stream=None) -> None:
    batch = len(positions)
    wc, kc, pos = weights.to_c(), kv.to_c(), _positions(positions)
    _check(load().spark_attn_decode(ctypes.byref(geom), _dev_ptr(h, "h", torch.float32),
                                    ctypes.byref(wc), ctypes.byref(kc), int(layer_class), pos,
                                    batch, _dev_ptr(out, "out", torch.float32),
                                    _dev_ptr(ws, "workspace"), ws.numel() * ws.element_size(),
                                    _stream(stream)), "spark_attn_decode")


def spark_attn_prefill(geom: SparkGeom, h: torch.Tensor, weights: LayerWeights, kv: KvLayer,
                       layer_class: int, p0: int, out: torch.Tensor, ws: torch.Tensor, stream=None) -> None:
    """h.shape[0] consecutive tokens of one sequence (positions p0, p0+1, ...)
    through one layer; kv is that sequence's cache ([1, capacity, n_kv, 256])."""
    wc, kc = weights.to_c(), kv.to_c()
    _check(load().spark_attn_prefill(ctypes.byref(geom), _dev_ptr(h, "h", torch.float32), ctypes.byref(wc),
                                     ctypes.byref(kc), int(layer_class), int(p0), int(h.shape[0]),
                                     _dev_ptr(out, "out", torch.float32), _dev_ptr(ws, "workspace"),
                                     ws.numel() * ws.element_size(), _stream(stream)),
           "spark_attn_prefill")


def spark_attn_decode_stack(geom: SparkGeom, h: torch.Tensor, weights: list, kvs: list, layer_classes,
                            positions, out: torch.Tensor, ws: torch.Tensor, stream=None) -> None:
    """One decode step through len(weights) layers (each layer's output is the
    next one's input); ``out`` receives the last layer's output."""
    n = len(weights)
    if len(kvs) != n or len(layer_classes) != n:
        raise ValueError("weights, kvs and layer_classes must have one entry per layer")
    wc = (SparkLayerWeights * n)(*[w.to_c() for w in weights])
    kc = (SparkKvLayer * n)(*[k.to_c() for k in kvs])
    cls = (ctypes.c_int32 * n)(*[int(c) for c in layer_classes])
    pos = _positions(positions)
    _check(load().spark_attn_decode_stack(ctypes.byref(geom), _dev_ptr(h, "h", torch.float32), n, wc, kc, cls,
                                          pos, len(positions), _dev_ptr(out, "out", torch.float32),
                                          _dev_ptr(ws, "workspace"), ws.numel() * ws.element_size(),
                                          _stream(stream)), "spark_attn_decode_stack")


def spark_dbg_qkv_rope(geom: SparkGeom, h: torch.Tensor, weights: LayerWeights, kv: KvLayer,
                       layer_class: int, positions, q_rot: torch.Tensor, g_logits: torch.Tensor,
                       ws: torch.Tensor, path: int = 0, stream=None) -> None:
    wc, kc, pos = weights.to_c(), kv.to_c(), _positions(positions)
    _check(load().spark_dbg_qkv_rope(ctypes.byref(geom), _dev_ptr(h, "h", torch.float32), ctypes.byref(wc),
                                     ctypes.byref(kc), int(layer_class), pos, len(positions),
                                     _dev_ptr(q_rot, "q_rot", torch.float32),
                                     _dev_ptr(g_logits, "g_logits", torch.float32), int(path),
                                     _dev_ptr(ws, "workspace"), ws.numel() * ws.element_size(),
                                     _stream(stream)),
           "spark_dbg_qkv_rope")


def spark_dbg_attention(geom: SparkGeom, q_rot: torch.Tensor, kv: KvLayer, layer_class: int, positions,
                        a: torch.Tensor, ws: torch.Tensor, n_ctas: int = 0, stream=None) -> None:
    kc, pos = kv.to_c(), _positions(positions)
    _check(load().spark_dbg_attention(ctypes.byref(geom), _dev_ptr(q_rot, "q_rot", torch.float32),
                                      ctypes.byref(kc), int(layer_class), pos, len(positions),
                                      _dev_ptr(a, "a", torch.float32), int(n_ctas),
                                      _dev_ptr(ws, "workspace"), ws.numel() * ws.element_size(),
                                      _stream(stream)), "spark_dbg_attention")


def spark_dbg_attention_noalloc(geom: SparkGeom, q_rot: torch.Tensor, kv: KvLayer, layer_class: int,
                                positions, a: torch.Tensor, stream=None) -> None:
    """spark_dbg_attention without a workspace: the library's fixed scratch
    array is used instead (for callers that cannot allocate device memory)."""
    kc, pos = kv.to_c(), _positions(positions)
    _check(load().spark_dbg_attention_noalloc(ctypes.byref(geom), _dev_ptr(q_rot, "q_rot", torch.float32),
                                              ctypes.byref(kc), int(layer_class), pos, len(positions),
                                              _dev_ptr(a, "a", torch.float32), _stream(stream)),
           "spark_dbg_attention_noalloc")


def spark_dbg_attention_noalloc_error_word(stream=None) -> int:
    """Read and clear the error word of the no-workspace attention's fixed
    array on the current device (synchronises the stream)."""
    word = ctypes.c_uint32(0)
    _check(load().spark_dbg_attention_noalloc_error_word(ctypes.byref(word), _stream(stream)),
           "spark_dbg_attention_noalloc_error_word")
    return int(word.value)


def spark_dbg_gate_oproj(geom: SparkGeom, a: torch.Tensor, g_logits: torch.Tensor, h: torch.Tensor,
                         weights: LayerWeights, out: torch.Tensor, ws: torch.Tensor, path: int = 0,
                         stream=None) -> None:
    wc = weights.to_c()
    _check(load().spark_dbg_gate_oproj(ctypes.byref(geom), _dev_ptr(a, "a", torch.float32),
                                       _dev_ptr(g_logits, "g_logits", torch.float32),
                                       _dev_ptr(h, "h", torch.float32), ctypes.byref(wc), int(h.shape[0]),
                                       _dev_ptr(out, "out", torch.float32), int(path),
                                       _dev_ptr(ws, "workspace"), ws.numel() * ws.element_size(),
                                       _stream(stream)),
           "spark_dbg_gate_oproj")


def spark_dbg_wait_timeout(ws: torch.Tensor, limit_ns: int, stream=None) -> None:
    """Run a bounded wait that nothing satisfies (see the header)."""
    _check(load().spark_dbg_wait_timeout(_dev_ptr(ws, "workspace"), ws.numel() * ws.element_size(),
                                         int(limit_ns), _stream(stream)), "spark_dbg_wait_timeout")


def spark_mlp_workspace_bytes(geom: SparkGeom, intermediate: int, batch: int) -> int:
    return int(load().spark_mlp_workspace_bytes(ctypes.byref(geom), int(intermediate), int(batch)))


def make_mlp_workspace(geom: SparkGeom, intermediate: int, batch: int, device=None, stream=None) -> torch.Tensor:
    """Allocate (through PyTorch) and initialise a workspace for
    spark_mlp_decode at this intermediate size (0: spark_head_logits only)."""
    nbytes = spark_mlp_workspace_bytes(geom, intermediate, batch)
    if nbytes == 0:
        raise ValueError("invalid geometry, intermediate size or batch for a workspace")
    ws = torch.empty(nbytes, dtype=torch.uint8, device=device or "cuda")
    spark_attn_workspace_init(ws, stream)
    return ws


def spark_mlp_decode(geom: SparkGeom, h: torch.Tensor, weights: MlpWeights, out: torch.Tensor,
                     ws: torch.Tensor, path: int = 0, stream=None) -> None:
    wc = weights.to_c()
    _check(load().spark_mlp_decode(ctypes.byref(geom), _dev_ptr(h, "h", torch.float32), ctypes.byref(wc),
                                   int(h.shape[0]), _dev_ptr(out, "out", torch.float32), int(path),
                                   _dev_ptr(ws, "workspace"), ws.numel() * ws.element_size(), _stream(stream)),
           "spark_mlp_decode")


def spark_head_logits(geom: SparkGeom, h: torch.Tensor, norm_w: torch.Tensor, embed: torch.Tensor,
                      logits: torch.Tensor, ws: torch.Tensor, path: int = 0, stream=None) -> None:
    """logits [batch, vocab] = embed [vocab, hidden] @ rms(h) * norm_w."""
    dt = embed.dtype
    if dt not in _DTYPE_CODE:
        raise TypeError(f"embed must be float32 or bfloat16, got {dt}")
    if embed.dim() != 2 or logits.dim() != 2 or logits.shape != (h.shape[0], embed.shape[0]):
        raise ValueError("embed must be [vocab, hidden] and logits [batch, vocab]")
    _check(load().spark_head_logits(ctypes.byref(geom), _dev_ptr(h, "h", torch.float32),
                                    _dev_ptr(norm_w, "norm_w", dt), _dev_ptr(embed, "embed", dt),
                                    int(embed.shape[0]), _DTYPE_CODE[dt], int(h.shape[0]),
                                    _dev_ptr(logits, "logits", torch.float32), int(path),
                                    _dev_ptr(ws, "workspace"), ws.numel() * ws.element_size(), _stream(stream)),
           "spark_head_logits")


def spark_attn_status_string(status: int) -> str:
    return load().spark_attn_status_string(int(status)).decode()


def spark_attn_abi_version() -> int:
    return int(load().spark_attn_abi_version())
