"""CPU oracle for the FP8 linear + normalization layer.

TEST INFRASTRUCTURE ONLY.  This package is the plain, slow, obviously correct
statement of what the GPU library computes.  Only ``tests/``, the smoke check
in ``__graft_entry__`` and the CPU-baseline leg of ``bench.py`` may import it;
the library itself never calls it and has no CPU fallback.

It shares no code with the CUDA path.  It is written in numpy, in float64
wherever the method leaves the precision open, and in float32 exactly where a
float32 operation decides an 8-bit code (the scaling multiply before the E4M3
cast), so that the decision is taken in the same precision as the kernel.

Sources (by page and section):
  * "LoKA: Low-precision Kernel Applications for Recommendation Models at
    Scale": section II-C (MERE, the FP8 linear y = Wx + b against a
    high-precision reference, Fig. 5), section III-B (normalization after the
    GEMM, fused into the epilogue; RMSNorm vs LayerNorm), section III-C
    (Dispatch: error and speedup filters, then the fastest candidate),
    section III-A 1 (the probe's online input statistics and sampler, and
    its matrix-normal weight model and weight sampler).
  * "GEM Training: How Meta Doubled the Efficiency ..." section "Low Precision
    Flash Attention" (MXFP8 block-scaled MMA, scale factors along K).
  * The pages name FP8 and MX formats without defining their bits; the E4M3
    ("fn": no infinities, max 448) and E8M0 definitions used here are the
    public OCP 8-bit floating point and Microscaling v1.0 formats that the MX
    reference on the LoKA page points to.

Parity status: every function here is pinned by tests in
``tests/test_oracle_pins.py`` (exhaustive code tables, brute force on tiny
inputs, library special cases and invariants).
"""
from . import formats, quantize, linear, probe, probe_stats, probe_weights, dispatch  # noqa: F401
