"""Plain CPU oracle for the int4 group-quantized matvec family.

TEST INFRASTRUCTURE ONLY.  The C sources in this folder restate, in double
precision and without any blocking or reordering, what the int4 weight-only
group-quantized matrix-vector product and its fused variants compute.  Only the
test suite, ``__graft_entry__.smoke()`` and the CPU-baseline / reference leg of
``bench.py`` may import this package.  It shares no code with the CUDA library.
"""

from .oracle import (  # noqa: F401
    build,
    dequant_f32,
    dequant_f64,
    dot_cols,
    embedding,
    from_mlx,
    gated_input_matvec,
    gated_matvec,
    load,
    matvec,
    mlx_dequant_f64,
    nibble,
    norm,
    norm_matvec,
    pack,
    quad_matvec,
    quantize,
    unpack,
)
