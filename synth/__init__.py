"""Seeded synthetic inputs for the quantized matvec workloads.

This module only draws random bytes and numbers and lays them out in the GGML
block byte formats. It holds none of the method's arithmetic (no decode, no
dot product, no activation quantization), so both the CPU oracle's tests and
the CUDA path's tests and benchmark can take their inputs from it without
sharing any code of the method.

Random source: splitmix64 (Steele, Lea and Flood, "Fast splittable
pseudorandom number generators", OOPSLA 2014; the output mix of Vigna's
public-domain reference). It is counter-based: draw ``i`` of a stream with seed
``s`` is ``mix(s + (i + 1) * 0x9E3779B97F4A7C15)``, so whole arrays of draws are
produced at once with numpy.
"""

from .gen import (  # noqa: F401
    Stream,
    CONFIGS,
    Q4K_BLOCK_BYTES,
    Q6K_BLOCK_BYTES,
    Q8_0_BLOCK_BYTES,
    Q4_0_BLOCK_BYTES,
    Q5K_BLOCK_BYTES,
    GEN_ROWS,
    gen_q4k_rows,
    gen_q6k_rows,
    gen_q8_0_rows,
    gen_q4_0_rows,
    gen_q5k_rows,
    gen_normal,
    gen_moe_ids,
    make_config,
    row_bytes,
)
