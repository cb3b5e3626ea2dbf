"""Single-GPU MoE layer hot path for GB300 (sm_103a): softmax top-k routing (optionally from x and
router weights), per-expert token counting and index generation, token permutation, grouped SwiGLU
GEMM on tcgen05 tensor cores, and the weighted combine, forward and backward, behind the C ABI in
include/moe.h. MoELayer holds one layer's buffers and call order (and can record a pass as a CUDA
graph); HostPipeline runs passes from pinned host memory with the copies overlapped."""
from . import _lib
from ._lib import MoeError
from .layer import MoELayer
from .pipeline import HostPipeline

__all__ = ["MoELayer", "HostPipeline", "MoeError", "_lib"]
