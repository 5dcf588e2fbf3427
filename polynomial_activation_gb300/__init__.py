"""polynomial_activation_gb300 -- packed-polynomial activations for GB300.

Short range-reduced polynomial programs replace the special-function-unit
evaluation of sigmoid, tanh, SiLU and exact GELU (and of the derivatives used
in backward), evaluated with packed FP16 / BF16 FMAs by hand-written CUDA
kernels for sm_103a, standalone or fused into a SwiGLU gate ("Fast
Polynomial Transcendentals for LLMs", arXiv 2610.00049).

``binding`` mirrors the C ABI of ``libpolyact.so`` (include/polyact.h) name
for name; ``ops`` adds allocate-and-call conveniences on torch tensors.
"""
from . import binding  # noqa: F401
from .binding import PolyError, PolyProgram  # noqa: F401
