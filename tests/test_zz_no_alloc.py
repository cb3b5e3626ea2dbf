"""moe_count_index_static: the counting / index-generation call for callers that cannot allocate
device memory (a plugin that only receives its input and output buffers from a host framework, or
a service that forbids allocation after start-up). Its scratch is a fixed array inside libmoe
instead of a caller-provided workspace; its results must equal moe_count_index's exactly (they are
integers), call after call, even though every call reuses the same array.

This file is collected last on purpose and depends on no earlier test.
"""
import pytest
import torch

import moe_inputs

pytestmark = pytest.mark.gpu


def _outputs(T, k, E, dev):
    from mixture_experts_layer_histogram_gb300 import _lib as L
    R = L.moe_grouped_rows_max(T, k, E)
    return dict(counts=torch.full((E,), -9, dtype=torch.int32, device=dev),
                offsets=torch.full((E + 1,), -9, dtype=torch.int32, device=dev),
                tile_offsets=torch.full((E + 1,), -9, dtype=torch.int32, device=dev),
                row_of_slot=torch.full((T * k,), -9, dtype=torch.int32, device=dev),
                token_of_row=torch.full((R,), -9, dtype=torch.int32, device=dev))


def _with_workspace(idx, E):
    from mixture_experts_layer_histogram_gb300 import _lib as L
    T, k = idx.shape
    o = _outputs(T, k, E, idx.device)
    ws = torch.zeros(L.moe_count_index_workspace_size(T, k, E), dtype=torch.uint8, device=idx.device)
    L.moe_count_index(idx, E, o["counts"], o["offsets"], o["tile_offsets"], o["row_of_slot"], o["token_of_row"], ws)
    torch.cuda.synchronize()
    assert L.moe_read_status(ws) == 0
    return o


def _static(idx, E):
    from mixture_experts_layer_histogram_gb300 import _lib as L
    T, k = idx.shape
    o = _outputs(T, k, E, idx.device)
    L.moe_count_index_static(idx, E, o["counts"], o["offsets"], o["tile_offsets"], o["row_of_slot"],
                             o["token_of_row"])
    torch.cuda.synchronize()
    return o


def _routed(T, E, k, routing, alpha, seed):
    from mixture_experts_layer_histogram_gb300 import _lib as L
    w = moe_inputs.small("noalloc", T=T, d=16, E=E, k=k, f=16, routing=routing, alpha=alpha, dtype="f32", seed=seed)
    logits = moe_inputs.make_logits(w, "cuda")
    idx = torch.empty((T, k), dtype=torch.int32, device="cuda")
    wt = torch.empty((T, k), dtype=torch.float32, device="cuda")
    L.moe_route_topk(logits, k, idx, wt)
    return idx


CASES = [(3000, 32, 4, "normal", 0.0, 1), (16384, 64, 8, "zipf", 1.2, 2), (8192, 256, 16, "zipf", 0.5, 3),
         (1, 1, 1, "normal", 0.0, 4)]


def test_static_scratch_matches_workspace_version_on_consecutive_calls():
    inputs = [(_routed(T, E, k, r, a, s), E) for T, E, k, r, a, s in CASES]
    expected = [_with_workspace(idx, E) for idx, E in inputs]
    # two passes over all cases: every call reuses the array the previous call left behind
    for _ in range(2):
        for (idx, E), exp in zip(inputs, expected):
            got = _static(idx, E)
            for key in exp:
                assert torch.equal(got[key], exp[key]), (idx.shape, E, key)


def test_static_scratch_rejects_sizes_beyond_its_limit():
    from mixture_experts_layer_histogram_gb300 import _lib as L
    T, k, E = 600_000, 16, 256           # its workspace would exceed MOE_STATIC_SCRATCH_BYTES (1 MiB)
    assert L.moe_count_index_workspace_size(T, k, E) > (1 << 20)
    idx = torch.zeros((1, 1), dtype=torch.int32, device="cuda")
    fake = torch.zeros(1, dtype=torch.int32, device="cuda")
    rc = L.lib().moe_count_index_static(L._p(idx), T, k, E, L._p(fake), L._p(fake), L._p(fake), L._p(fake),
                                         L._p(fake), L._s(None))
    assert rc == -2      # MOE_ERR_UNSUPPORTED, rejected on the host before anything is enqueued
