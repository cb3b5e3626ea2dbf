"""The C-ABI library loads, exports every symbol include/moe.h declares, and rejects bad arguments on
the host before touching the device (no GPU needed: nothing here launches a kernel)."""
import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    from mixture_experts_layer_histogram_gb300 import _lib, build
    if not os.path.exists(_lib.LIB_PATH):
        build.build()
    return _lib.lib()


def _declared():
    src = open(os.path.join(ROOT, "include", "moe.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z_0-9]+)\s*\(", src)))


def test_header_declares_the_boundary():
    names = _declared()
    for required in ("moe_route_topk", "moe_count_index", "moe_permute", "moe_grouped_ffn_fwd", "moe_grouped_ffn_bwd",
                     "moe_combine_fwd", "moe_combine_bwd", "moe_read_status"):
        assert required in names


def test_every_declared_symbol_is_exported(L):
    from mixture_experts_layer_histogram_gb300 import _lib
    out = subprocess.run(["nm", "-D", "--defined-only", _lib.LIB_PATH], capture_output=True, text=True).stdout
    exported = set(re.findall(r" T (moe_\w+)", out))
    for name in _declared():
        assert name in exported, name
        assert name in _lib.exported_symbols(), name
        getattr(L, name)


def test_version_and_status_strings(L):
    from mixture_experts_layer_histogram_gb300 import _lib
    assert _lib.moe_version() == 100
    assert _lib.moe_status_string(0) == "ok"
    assert "timed out" in _lib.moe_status_string(-4)
    assert _lib.moe_status_string(-5) == "expert index out of range"


def test_rows_max_and_workspace_sizes(L):
    from mixture_experts_layer_histogram_gb300 import _lib
    assert _lib.moe_grouped_rows_max(16384, 8, 64) == 131072 + 64 * 128
    assert _lib.moe_grouped_rows_max(1, 1, 1) == 128
    assert _lib.moe_grouped_rows_max(256, 2, 8) % 128 == 0
    assert _lib.moe_count_index_workspace_size(16384, 8, 64) >= 64 + 256 + 256 + 128 * 64 * 8
    assert _lib.moe_count_index_hook_offset(64) % 16 == 0
    assert _lib.moe_grouped_ffn_workspace_size(64, 2048, 1024, 139264, 1, 1) >= 4
    # router: header + bf16 copy of d_logits (8192 x 64) + fp32 partials of at least one token range
    assert _lib.moe_router_workspace_size(8192, 2048, 64, 1) >= 256 + 8192 * 64 * 2 + 64 * 2048 * 4
    assert _lib.moe_router_workspace_size(256, 64, 8, 0) >= 256 + 256 * 8 * 4
    assert _lib.moe_router_workspace_size(0, 64, 8, 1) >= 256


FAKE = ctypes.c_void_p(1 << 20)   # never dereferenced: every call below fails validation first
NULL = None


def test_invalid_arguments_are_rejected_on_the_host(L):
    # route: k > E, E too large, null pointers
    assert L.moe_route_topk(FAKE, 8, 4, 5, FAKE, FAKE, NULL) == -1
    assert L.moe_route_topk(FAKE, 8, 300, 2, FAKE, FAKE, NULL) == -1
    assert L.moe_route_topk(NULL, 8, 8, 2, FAKE, FAKE, NULL) == -1
    assert L.moe_route_topk(FAKE, 8, 8, 17, FAKE, FAKE, NULL) == -1
    # count_index: workspace too small, misaligned workspace
    need = L.moe_count_index_workspace_size(64, 2, 8)
    assert L.moe_count_index(FAKE, 64, 2, 8, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, need - 1, NULL) == -1
    assert L.moe_count_index(FAKE, 64, 2, 8, FAKE, FAKE, FAKE, FAKE, FAKE, ctypes.c_void_p((1 << 20) + 8), need,
                             NULL) == -1
    # permute: row size not a multiple of 16 bytes
    rm = L.moe_grouped_rows_max(64, 2, 8)
    assert L.moe_permute(FAKE, 1, 64, 12, 2, 8, FAKE, FAKE, FAKE, rm, FAKE, NULL) == -2
    assert L.moe_permute(FAKE, 1, 64, 64, 2, 8, FAKE, FAKE, FAKE, rm - 128, FAKE, NULL) == -1
    assert L.moe_permute(FAKE, 7, 64, 64, 2, 8, FAKE, FAKE, FAKE, rm, FAKE, NULL) == -1
    # grouped FFN: bf16 needs d, f multiples of 256; rows_max multiple of 128; workspace present
    ws = L.moe_grouped_ffn_workspace_size(8, 128, 256, rm, 1, 1)
    assert L.moe_grouped_ffn_fwd(FAKE, FAKE, FAKE, FAKE, FAKE, 8, 128, 256, rm, 1, FAKE, FAKE, FAKE, FAKE, ws,
                                 NULL) == -2
    assert L.moe_grouped_ffn_fwd(FAKE, FAKE, FAKE, FAKE, FAKE, 8, 256, 256, rm + 1, 1, FAKE, FAKE, FAKE, FAKE, ws,
                                 NULL) == -1
    assert L.moe_grouped_ffn_fwd(FAKE, FAKE, FAKE, FAKE, FAKE, 8, 256, 256, rm, 1, FAKE, FAKE, FAKE, NULL, ws,
                                 NULL) == -1
    assert L.moe_grouped_ffn_fwd(FAKE, FAKE, FAKE, FAKE, NULL, 8, 256, 256, rm, 1, FAKE, FAKE, FAKE, FAKE, ws,
                                 NULL) == -1                                   # offsets missing
    assert L.moe_grouped_ffn_bwd(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 8, 256, 100, rm, 1, FAKE, FAKE, FAKE,
                                 FAKE, FAKE, ws, NULL) == -2
    # combine: misaligned output, k out of range
    assert L.moe_combine_fwd(FAKE, FAKE, FAKE, 64, 64, 2, rm, 1, ctypes.c_void_p((1 << 20) + 2), NULL) == -1
    assert L.moe_combine_fwd(FAKE, FAKE, FAKE, 64, 64, 0, rm, 1, FAKE, NULL) == -1
    assert L.moe_combine_bwd(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 64, 64, 9, 8, rm, 1, FAKE, FAKE, FAKE, NULL) == -1
    # router: k > E, E too large, bf16 d not a multiple of 8, workspace too small or misaligned, nulls
    rws = L.moe_router_workspace_size(64, 256, 8, 1)
    assert L.moe_router_fwd(FAKE, FAKE, 64, 256, 8, 9, 1, FAKE, FAKE, FAKE, FAKE, rws, NULL) == -1
    assert L.moe_router_fwd(FAKE, FAKE, 64, 256, 300, 2, 1, FAKE, FAKE, FAKE, FAKE, rws, NULL) == -1
    assert L.moe_router_fwd(FAKE, FAKE, 64, 252, 8, 2, 1, FAKE, FAKE, FAKE, FAKE, rws, NULL) == -2
    assert L.moe_router_fwd(FAKE, FAKE, 64, 256, 8, 2, 1, FAKE, FAKE, FAKE, FAKE, rws - 1, NULL) == -1
    assert L.moe_router_fwd(FAKE, FAKE, 64, 256, 8, 2, 1, FAKE, FAKE, FAKE, ctypes.c_void_p((1 << 20) + 16), rws,
                            NULL) == -1
    assert L.moe_router_fwd(FAKE, NULL, 64, 256, 8, 2, 1, FAKE, FAKE, FAKE, FAKE, rws, NULL) == -1
    assert L.moe_router_fwd(FAKE, FAKE, 64, 256, 8, 2, 1, ctypes.c_void_p((1 << 20) + 4), FAKE, FAKE, FAKE, rws,
                            NULL) == -1
    assert L.moe_router_bwd(FAKE, FAKE, FAKE, 64, 256, 8, 1, 0, FAKE, NULL, FAKE, rws, NULL) == -1
    assert L.moe_router_bwd(FAKE, FAKE, FAKE, 64, 256, 8, 2, 0, FAKE, FAKE, FAKE, rws, NULL) == -1
    assert L.moe_read_status(NULL, NULL) == -1
    # allocation-free count/index: the stated limits are exactly where the 1 MiB scratch runs out
    for E, slots in ((64, 2095104), (256, 523264)):
        assert L.moe_count_index_workspace_size(slots, 1, E) <= 1 << 20 < L.moe_count_index_workspace_size(slots + 1, 1, E)
        assert L.moe_count_index_static(FAKE, slots + 1, 1, E, FAKE, FAKE, FAKE, FAKE, FAKE, NULL) == -2


def test_empty_inputs_enqueue_nothing(L):
    assert L.moe_route_topk(NULL, 0, 8, 2, NULL, NULL, NULL) == 0
    assert L.moe_combine_fwd(NULL, NULL, NULL, 0, 64, 2, 0, 1, NULL, NULL) == 0


def test_product_path_fails_loudly_without_cuda_tensors():
    import torch
    from mixture_experts_layer_histogram_gb300 import _lib
    x = torch.zeros((4, 8))
    with pytest.raises(ValueError):
        _lib.moe_route_topk(x, 2, torch.zeros((4, 2), dtype=torch.int32), torch.zeros((4, 2)))
