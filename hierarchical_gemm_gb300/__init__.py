"""hierarchical_gemm_gb300: the tile-level GEMM C = A * B for one GB300 GPU.

The compute path is libtsgemm.so (hand-written CUDA for sm_103a: TMA operand
loads, an mbarrier shared-memory ring, tcgen05.mma into tensor memory, a
persistent warp-specialised schedule, split-K).  This package only builds
that library (hierarchical_gemm_gb300.build) and marshals arguments to its C
ABI (include/tsgemm.h) through hierarchical_gemm_gb300.tsgemm.

The binding is loaded on first use of any of its names; if the library has
not been built that raises ImportError (there is no fallback).
"""
_EXPORTED = ("BF16", "F16", "F32", "Config", "Plan", "TsgemmError", "choose_config",
             "gemm", "status_string")


def __getattr__(name):
    if name in _EXPORTED:
        from . import tsgemm
        return getattr(tsgemm, name)
    raise AttributeError(name)
