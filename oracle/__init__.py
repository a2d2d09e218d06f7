"""Float64 CPU oracle for the Mamba-2 SSD forward pass.

TEST INFRASTRUCTURE ONLY: the tests, the package smoke check and the
benchmark's CPU-baseline leg may import this package; the product path
(the CUDA library and its Python binding) never does, and shares no code
with it.

Two independent float64 implementations live here, both written from
"Accelerating Mamba-2 with High-Performance Forward Pass Kernels in NVIDIA
CUDA Tile", section "Mamba-2 architecture":

* ``recurrence`` -- the token-by-token recurrence in plain C (ssd_oracle.c),
  driven through ctypes; the reference every GPU result is compared with.
  ``recurrence_np`` is the same definition in numpy for tiny inputs.
* ``chunked`` -- the chunked log-space formulas of the same section (the
  decayed state jump and the chunked output equation), in numpy, used only
  to cross-check the recurrence and to pin the chunking semantics.
* ``decode_step`` -- one token of the recurrence for a batch of states, in
  numpy: the reference for the single-token decode step.
* ``backward`` -- the gradients of a loss through the recurrence (the
  adjoint recurrence token by token, numpy float64): the reference a
  backward pass will be checked against; no CUDA path computes it yet.
  ``backward_chunked`` restates it by the chunked formulas a chunk-parallel
  kernel would use (reverse pass over chunks, per-chunk masked products,
  the decay gradient as a reverse cumsum of dL/dG), pinned against it.

Parity status: every function here is pinned by the ``-m "not gpu"`` tests
(hand-worked example, brute-force unrolled sum, linear-attention, B = 0 and
dt = 0 special cases, chunk invariance, padding, resume, linearity in h0;
for decode_step: the hand-worked example token by token, agreement with the
C recurrence over whole sequences, dt = 0, and planted mistakes; for
backward: central finite differences of the C recurrence, closed forms of
special cases, and planted mistakes).
"""
from .ssd_oracle import (  # noqa: F401
    backward,
    backward_chunked,
    build,
    chunked,
    decode_step,
    max_threads,
    recurrence,
    recurrence_np,
    set_threads,
)
