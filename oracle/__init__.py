"""Plain float64 CPU oracle for the spark2_5 decode attention block and the
rest of its decoder layer.

TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only the test-suite (``tests/``), the
``smoke()`` check in ``__graft_entry__`` and the ``cpu_baseline`` / reference
leg of ``bench.py`` may import anything from this package.  The CUDA library
and its Python binding never import, call or link it, and it imports nothing
from them: the two sides share no code beyond the seeded input generators.

Parity status of each function is stated in the headers of
``oracle.spark_block`` (the attention block) and ``oracle.spark_layer`` (the
MLP half of a decoder layer and the head).
"""

from .spark_block import (  # noqa: F401
    OracleGeometry,
    bf16_bits_to_f64,
    f64_to_bf16_bits,
    rms_norm,
    project,
    rope_params_for,
    rope_neox,
    rope_inv_freq,
    window_params,
    write_slot,
    read_slot,
    attention_decode,
    sigmoid,
    head_gate,
    decode_step,
    prefill_chunk,
    cache_rows_to_f64,
)
from .spark_layer import (  # noqa: F401
    gelu_erf,
    mlp_block,
    head_logits,
)
