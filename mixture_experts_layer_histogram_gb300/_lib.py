"""ctypes binding of libmoe (include/moe.h): the same entry points, argument marshalling only.

Tensors are torch CUDA tensors (PyTorch supplies device memory and streams); every step runs in
the library's kernels. There is no CPU path: calling with a CPU tensor, or without the built
library, raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

# MOE_LIBRARY selects another build of the same library (the debug build, libmoe_checks.so)
LIB_PATH = os.environ.get("MOE_LIBRARY") or os.path.join(os.path.dirname(os.path.abspath(__file__)), "libmoe.so")

MOE_F32, MOE_BF16 = 0, 1
GROUP_ROWS = 128
MAX_EXPERTS = 256
MAX_TOPK = 16
STATUS = {0: "MOE_OK", -1: "MOE_ERR_INVALID_ARG", -2: "MOE_ERR_UNSUPPORTED", -3: "MOE_ERR_CUDA",
          -4: "MOE_ERR_DEVICE_TIMEOUT", -5: "MOE_ERR_BAD_INDEX", -6: "MOE_ERR_CHECK_FAILED"}

_lock = threading.Lock()
_lib = None

_P, _I, _I64, _SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t
_SIGS = {
    "moe_route_topk": (_I, [_P, _I, _I, _I, _P, _P, _P]),
    "moe_grouped_rows_max": (_I64, [_I, _I, _I]),
    "moe_count_index_workspace_size": (_SZ, [_I, _I, _I]),
    "moe_count_index_hook_offset": (_SZ, [_I]),
    "moe_count_index": (_I, [_P, _I, _I, _I, _P, _P, _P, _P, _P, _P, _SZ, _P]),
    "moe_count_index_static": (_I, [_P, _I, _I, _I, _P, _P, _P, _P, _P, _P]),
    "moe_route_count_index": (_I, [_P, _I, _I, _I, _P, _P, _P, _P, _P, _P, _P, _P, _SZ, _P]),
    "moe_permute": (_I, [_P, _I, _I, _I, _I, _I, _P, _P, _P, _I64, _P, _P]),
    "moe_grouped_ffn_workspace_size": (_SZ, [_I, _I, _I, _I64, _I, _I]),
    "moe_grouped_ffn_fwd": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I64, _I, _P, _P, _P, _P, _SZ, _P]),
    "moe_grouped_ffn_bwd": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I64, _I, _P, _P, _P, _P, _P, _SZ, _P]),
    "moe_grouped_ffn_bwd_recompute": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I64, _I, _P, _P, _P, _P, _P,
                                           _SZ, _P]),
    "moe_grouped_ffn_fwd_gather": (_I, [_P, _P, _I, _P, _P, _P, _P, _I, _I, _I, _I64, _I, _P, _P, _P, _P, _SZ, _P]),
    "moe_grouped_ffn_bwd_gather": (_I, [_P, _P, _P, _I, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I64, _I, _P, _P, _P, _P, _P,
                                        _SZ, _P]),
    "moe_grouped_ffn_bwd_recompute_gather": (_I, [_P, _P, _P, _I, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I64, _I, _P, _P,
                                                  _P, _P, _P, _SZ, _P]),
    "moe_combine_fwd": (_I, [_P, _P, _P, _I, _I, _I, _I64, _I, _P, _P]),
    "moe_combine_bwd": (_I, [_P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I64, _I, _P, _P, _P, _P]),
    "moe_router_workspace_size": (_SZ, [_I, _I, _I, _I]),
    "moe_router_fwd": (_I, [_P, _P, _I, _I, _I, _I, _I, _P, _P, _P, _P, _SZ, _P]),
    "moe_router_bwd": (_I, [_P, _P, _P, _I, _I, _I, _I, _I, _P, _P, _P, _SZ, _P]),
    "moe_read_status": (_I, [_P, _P]),
    "moe_status_string": (ctypes.c_char_p, [_I]),
    "moe_version": (_I, []),
}


class MoeError(RuntimeError):
    def __init__(self, fn, code):
        super().__init__(f"{fn} returned {STATUS.get(code, code)}")
        self.code = code


def lib():
    """Load libmoe.so (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(f"{LIB_PATH} is missing: build it first (python -c 'import __graft_entry__ as g; g.build()')")
            L = ctypes.CDLL(LIB_PATH)
            for name, (res, args) in _SIGS.items():
                fn = getattr(L, name)
                fn.restype = res
                fn.argtypes = args
            _lib = L
    return _lib


def exported_symbols():
    return list(_SIGS)


def dtype_code(t: torch.dtype) -> int:
    if t == torch.float32:
        return MOE_F32
    if t == torch.bfloat16:
        return MOE_BF16
    raise TypeError(f"unsupported dtype {t}")


def _p(t):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("libmoe takes CUDA tensors only")
    return ctypes.c_void_p(t.data_ptr())


def _s(stream):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _ok(fn, rc):
    if rc != 0:
        raise MoeError(fn, rc)


def moe_route_topk(logits, k, topk_idx, topk_w, stream=None):
    T, E = logits.shape
    _ok("moe_route_topk", lib().moe_route_topk(_p(logits), T, E, k, _p(topk_idx), _p(topk_w), _s(stream)))


def moe_grouped_rows_max(T, k, E):
    return int(lib().moe_grouped_rows_max(T, k, E))


def moe_count_index_workspace_size(T, k, E):
    return int(lib().moe_count_index_workspace_size(T, k, E))


def moe_count_index_hook_offset(E):
    return int(lib().moe_count_index_hook_offset(E))


def moe_count_index(topk_idx, E, counts, offsets, tile_offsets, row_of_slot, token_of_row, ws, stream=None):
    T, k = topk_idx.shape
    _ok("moe_count_index", lib().moe_count_index(_p(topk_idx), T, k, E, _p(counts), _p(offsets), _p(tile_offsets),
                                                 _p(row_of_slot), _p(token_of_row), _p(ws), ws.numel() * ws.element_size(),
                                                 _s(stream)))


def moe_route_count_index(logits, k, topk_idx, topk_w, counts, offsets, tile_offsets, row_of_slot, token_of_row, ws,
                          stream=None):
    """moe_route_topk then moe_count_index, in one launch when all its blocks fit on the GPU."""
    T, E = logits.shape
    _ok("moe_route_count_index", lib().moe_route_count_index(
        _p(logits), T, E, k, _p(topk_idx), _p(topk_w), _p(counts), _p(offsets), _p(tile_offsets), _p(row_of_slot),
        _p(token_of_row), _p(ws), ws.numel() * ws.element_size(), _s(stream)))


def moe_count_index_static(topk_idx, E, counts, offsets, tile_offsets, row_of_slot, token_of_row, stream=None):
    """moe_count_index for callers that cannot allocate: the scratch is a fixed array inside libmoe."""
    T, k = topk_idx.shape
    _ok("moe_count_index_static", lib().moe_count_index_static(
        _p(topk_idx), T, k, E, _p(counts), _p(offsets), _p(tile_offsets), _p(row_of_slot), _p(token_of_row),
        _s(stream)))


def moe_permute(x, k, E, row_of_slot, counts, tile_offsets, x_perm, stream=None):
    T, d = x.shape
    _ok("moe_permute", lib().moe_permute(_p(x), dtype_code(x.dtype), T, d, k, E, _p(row_of_slot), _p(counts),
                                         _p(tile_offsets), x_perm.shape[0], _p(x_perm), _s(stream)))


def moe_grouped_ffn_workspace_size(E, d, f, rows_max, dtype, backward):
    return int(lib().moe_grouped_ffn_workspace_size(E, d, f, rows_max, dtype, int(backward)))


def moe_grouped_ffn_fwd(x_perm, w_gate_up, w_down, tile_offsets, offsets, ab, h, y_perm, ws, stream=None):
    E, twof, d = w_gate_up.shape
    _ok("moe_grouped_ffn_fwd", lib().moe_grouped_ffn_fwd(
        _p(x_perm), _p(w_gate_up), _p(w_down), _p(tile_offsets), _p(offsets), E, d, twof // 2, x_perm.shape[0],
        dtype_code(x_perm.dtype), _p(ab), _p(h), _p(y_perm), _p(ws), ws.numel() * ws.element_size(), _s(stream)))


def moe_grouped_ffn_bwd(dy_perm, x_perm, ab, h, w_gate_up, w_down, tile_offsets, offsets, dab, dx_perm, dw_gate_up,
                        dw_down, ws, stream=None):
    E, twof, d = w_gate_up.shape
    _ok("moe_grouped_ffn_bwd", lib().moe_grouped_ffn_bwd(
        _p(dy_perm), _p(x_perm), _p(ab), _p(h), _p(w_gate_up), _p(w_down), _p(tile_offsets), _p(offsets), E, d,
        twof // 2,
        x_perm.shape[0], dtype_code(x_perm.dtype), _p(dab), _p(dx_perm), _p(dw_gate_up), _p(dw_down), _p(ws),
        ws.numel() * ws.element_size(), _s(stream)))


def moe_grouped_ffn_bwd_recompute(dy_perm, x_perm, ab, h, w_gate_up, w_down, tile_offsets, offsets, dab, dx_perm,
                                  dw_gate_up, dw_down, ws, stream=None):
    E, twof, d = w_gate_up.shape
    _ok("moe_grouped_ffn_bwd_recompute", lib().moe_grouped_ffn_bwd_recompute(
        _p(dy_perm), _p(x_perm), _p(ab), _p(h), _p(w_gate_up), _p(w_down), _p(tile_offsets), _p(offsets), E, d,
        twof // 2,
        x_perm.shape[0], dtype_code(x_perm.dtype), _p(dab), _p(dx_perm), _p(dw_gate_up), _p(dw_down), _p(ws),
        ws.numel() * ws.element_size(), _s(stream)))


def moe_grouped_ffn_fwd_gather(x, token_of_row, w_gate_up, w_down, tile_offsets, offsets, ab, h, y_perm, ws,
                               stream=None):
    """moe_grouped_ffn_fwd with GEMM1 gathering its token rows from x [T, d] through token_of_row."""
    E, twof, d = w_gate_up.shape
    _ok("moe_grouped_ffn_fwd_gather", lib().moe_grouped_ffn_fwd_gather(
        _p(x), _p(token_of_row), x.shape[0], _p(w_gate_up), _p(w_down), _p(tile_offsets), _p(offsets), E, d,
        twof // 2, h.shape[0], dtype_code(x.dtype), _p(ab), _p(h), _p(y_perm), _p(ws), ws.numel() * ws.element_size(),
        _s(stream)))


def moe_grouped_ffn_bwd_gather(dy_perm, x, token_of_row, ab, h, w_gate_up, w_down, tile_offsets, offsets, dab, dx_perm,
                               dw_gate_up, dw_down, ws, stream=None):
    """moe_grouped_ffn_bwd with the gate/up weight gradient gathering its token rows from x [T, d]."""
    E, twof, d = w_gate_up.shape
    _ok("moe_grouped_ffn_bwd_gather", lib().moe_grouped_ffn_bwd_gather(
        _p(dy_perm), _p(x), _p(token_of_row), x.shape[0], _p(ab), _p(h), _p(w_gate_up), _p(w_down), _p(tile_offsets),
        _p(offsets), E, d, twof // 2, dy_perm.shape[0], dtype_code(x.dtype), _p(dab), _p(dx_perm), _p(dw_gate_up),
        _p(dw_down), _p(ws), ws.numel() * ws.element_size(), _s(stream)))


def moe_grouped_ffn_bwd_recompute_gather(dy_perm, x, token_of_row, ab, h, w_gate_up, w_down, tile_offsets, offsets,
                                         dab, dx_perm, dw_gate_up, dw_down, ws, stream=None):
    """moe_grouped_ffn_bwd_recompute with GEMM1 and the gate/up weight gradient gathering from x [T, d]."""
    E, twof, d = w_gate_up.shape
    _ok("moe_grouped_ffn_bwd_recompute_gather", lib().moe_grouped_ffn_bwd_recompute_gather(
        _p(dy_perm), _p(x), _p(token_of_row), x.shape[0], _p(ab), _p(h), _p(w_gate_up), _p(w_down), _p(tile_offsets),
        _p(offsets), E, d, twof // 2, dy_perm.shape[0], dtype_code(x.dtype), _p(dab), _p(dx_perm), _p(dw_gate_up),
        _p(dw_down), _p(ws), ws.numel() * ws.element_size(), _s(stream)))


def moe_combine_fwd(y_perm, topk_w, row_of_slot, T, k, out, stream=None):
    d = y_perm.shape[1]
    _ok("moe_combine_fwd", lib().moe_combine_fwd(_p(y_perm), _p(topk_w), _p(row_of_slot), T, d, k, y_perm.shape[0],
                                                 dtype_code(y_perm.dtype), _p(out), _s(stream)))


def moe_combine_bwd(grad_out, y_perm, topk_w, topk_idx, row_of_slot, counts, tile_offsets, E, dy_perm, d_topk_w,
                    d_logits, stream=None):
    T, d = grad_out.shape
    k = topk_idx.shape[1]
    _ok("moe_combine_bwd", lib().moe_combine_bwd(
        _p(grad_out), _p(y_perm), _p(topk_w), _p(topk_idx), _p(row_of_slot), _p(counts), _p(tile_offsets), T, d, k, E,
        y_perm.shape[0], dtype_code(y_perm.dtype), _p(dy_perm), _p(d_topk_w), _p(d_logits), _s(stream)))


def moe_router_workspace_size(T, d, E, dtype):
    return int(lib().moe_router_workspace_size(T, d, E, dtype))


def moe_router_fwd(x, w_router, k, logits, topk_idx, topk_w, ws, stream=None):
    """logits may be None (not written)."""
    T, d = x.shape
    E = w_router.shape[0]
    _ok("moe_router_fwd", lib().moe_router_fwd(
        _p(x), _p(w_router), T, d, E, k, dtype_code(x.dtype), _p(logits), _p(topk_idx), _p(topk_w), _p(ws),
        ws.numel() * ws.element_size(), _s(stream)))


def moe_router_bwd(x, w_router, d_logits, dx, dw_router, ws, accumulate_dx=False, stream=None):
    T, d = x.shape
    E = w_router.shape[0]
    _ok("moe_router_bwd", lib().moe_router_bwd(
        _p(x), _p(w_router), _p(d_logits), T, d, E, dtype_code(x.dtype), int(bool(accumulate_dx)), _p(dx),
        _p(dw_router), _p(ws), ws.numel() * ws.element_size(), _s(stream)))


def moe_read_status(ws, stream=None):
    return int(lib().moe_read_status(_p(ws), _s(stream)))


def moe_status_string(code):
    return lib().moe_status_string(code).decode()


def moe_version():
    return int(lib().moe_version())
