"""CPU oracle for the quantized KV cache — TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` may import this package. The product
library never does, and the two share no code.

The arithmetic lives in ``kvq_oracle.cpp`` (plain single-threaded C++17, built
with ``-ffp-contract=off -fno-fast-math``); this module builds it with g++ and
wraps it with ctypes and numpy.
"""

from .oracle import (  # noqa: F401
    build,
    lib,
    f32_from_f16,
    f16_from_f32_rne,
    f16_from_f32_ru,
    qmin,
    qmax,
    quant_params,
    quantize_values,
    dequantize_value,
    kv_bytes,
    v_pos,
    pack_k_row,
    unpack_k_row,
    pack_v_token,
    unpack_v_token,
    cache_state,
    value_meta,
    dequantize_state,
    sym_params,
    sym_quantize,
    sym_dequantize_value,
    split_outliers,
    cache_state_sym,
    dequantize_state_sym,
    attention,
    OracleState,
)
