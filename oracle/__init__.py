"""CPU oracle for the FP4 quantized linear layer -- test infrastructure only.

Only tests/, __graft_entry__.smoke() and bench.py's cpu_baseline / reference
arm may import anything under oracle/.  The CUDA library and its Python binding
never do; they share no code with it.
"""
from . import fp4_linear  # noqa: F401
