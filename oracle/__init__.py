"""CPU oracle for the quantized KV-cache hot path.  TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product path (the C-ABI library
and its Python binding) never imports, links or executes it, and this
package imports nothing from the product path.

It is a plain, slow, obviously-correct restatement of what the method
computes, in float64 NumPy (plus float32/float16 where a decision is taken in
the kernel's precision, see ``quantizer``):

* ``hadamard``   -- explicit Sylvester Hadamard matrices, block-diagonal
                    rotation by matrix multiply.
* ``fp16``       -- directed rounding to IEEE binary16.
* ``quantizer``  -- token-wise asymmetric INT-b quantization with one fp16
                    scale and one fp16 zero per vector; the symmetric
                    per-channel key quantizer of the key-per-channel mode.
* ``layout``     -- the paged-cache byte layout (pack / unpack).
* ``cache``      -- quantize-on-append into the paged cache plus the bf16
                    recent-token window (and the key-per-channel mode's
                    page-at-a-time rule).
* ``attention``  -- decode attention over the dequantized cache.
* ``logquant``   -- LogQuant's log-spaced full-precision set B (token-by-token
                    halving) and decode attention with B's positions in bf16.
* ``allocator``  -- RateQuant greedy marginal-gain bit allocation, the
                    closed-form reverse-waterfilling optimum, brute force.
* ``distortion`` -- fitting D(b) = alpha * beta^-b to measured MSE.

Pins (tests that tie each function to something other than itself) live in
``tests/test_oracle_*.py``.  Parity unpinned: the byte layout of a page, the
rounding directions of the fp16 scale and zero, the Sylvester ordering of the
Hadamard rows and the window flush rule are conventions of this library; the
pages do not fix them, so they are checked for self-consistency only.
"""
from . import allocator, attention, cache, distortion, fp16, hadamard, layout, quantizer
from . import logquant

__all__ = ["allocator", "attention", "cache", "distortion", "fp16", "hadamard", "layout",
           "logquant", "quantizer"]
