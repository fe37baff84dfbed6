"""CPU oracle for the NVFP4 W4A4 MoE expert block.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import this package.
The CUDA library never calls it, and it shares no code, table or helper with the CUDA
path: both sides are written independently from the pages' definitions.

The oracle is plain, slow and meant to be checked by eye against the pages:

* numpy, vectorised over elements; float32 only where the method's contract fixes a
  float32 step (the scale arithmetic that decides the quantised codes), float64 for
  every sum, product and transcendental that is a plain mathematical definition;
* a library primitive (``numpy.matmul`` in float64, a stable ``argsort``) may serve as a
  step, with no blocking, fusion or reordering beyond the definition.

Pages cited (by title and section):

* [4BL] "The 4-bitter Lesson: Balancing Stability and Performance in NVFP4 RL" --
  §Baseline (the NVFP4 format), §"Why is the NVFP4 pretraining recipe not sufficient
  for RL?" (weights: per-block E4M3 + one FP32 global scale; activations: per-token FP32
  scale; stochastic rounding; MoE-experts-only scope; fused per-token quantiser),
  §"Improving Gradient Stability" and its footnote 6 (Q = clip(round(w/s), qmin, qmax);
  dequantisation DQ).
* [LBP] "Low-Bit Precision Training Is Ready for Production: What Engineering Leaders
  Need to Know Before Adopting NVFP4" -- §"What W4A4 GEMM Actually Changes" (both GEMM
  operands in FP4; expert GEMMs), §"The Cross-Engine Alignment Problem" (execution-level
  alignment: composition and accumulation order decide the result).
* [4BL] §"Improving Gradient Stability", "Results Validation with MXFP8" -- the MXFP8
  recipe the fix is first validated with (``mx.py``; the format itself is read from the
  OCP Microscaling Formats v1.0 definition, which the pages name but do not restate).
* [miniTE] "miniTE identifies and closes the execution gap in native NVFP4 reinforcement
  learning" -- §Development (NVFP4 kernels, scaling, grouped GEMMs).

Where the pages leave a bit-level step open, the reading taken is stated in the
docstring of the function that implements it.

Parity status: every function here is pinned by a ``-m "not gpu"`` test against values
fixed by the format definitions, closed forms, brute force or an independent
high-precision library (see tests/test_oracle_*.py); none is "parity unpinned".
"""

from . import formats, philox, quant, moe, mx, backward  # noqa: F401
