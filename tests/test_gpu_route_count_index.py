"""moe_route_count_index (routing, counting and index generation in one launch) must give, bit for
bit, what moe_route_topk followed by moe_count_index gives: the same kernels' selection and
weights, and the same stable counting sort. Shapes cover tokens whose slots straddle two blocks
(k = 3, 5), E = 256 with k = 16, the largest problems of the kernel's two block sizes (512 slots
while that is at most one block per SM, then 1024 while every block fits on the GPU at once), one
above both (the call then makes the two calls itself), exact ties, and calls back to back on one
workspace."""
import pytest
import torch

import moe_inputs

pytestmark = pytest.mark.gpu

SHAPES = [(1, 8, 2, "normal"), (5, 256, 16, "normal"), (1023, 7, 3, "normal"), (1025, 1, 1, "normal"),
          (333, 40, 5, "zipf"), (8192, 64, 8, "router"), (16384, 64, 8, "uniform"), (16384, 128, 8, "zipf"),
          (25000, 64, 3, "normal"),       # 75,000 slots: 147 blocks of 512 slots
          (100000, 64, 3, "normal"),      # 300,000 slots: 293 blocks of 1024 slots (2 per SM)
          (40000, 256, 16, "zipf"),       # 640,000 slots: above both, the call falls back to two launches
          (777, 16, 4, "ties")]


def _logits(T, E, routing):
    if routing == "ties":   # few distinct values, signed zeros included: many exact ties
        g = torch.Generator().manual_seed(T)
        vals = torch.tensor([-1.5, -0.0, 0.0, 0.25, 2.0])
        return vals[torch.randint(0, len(vals), (T, E), generator=g)].cuda()
    w = moe_inputs.small("rci", T=T, d=256 if routing == "router" else 16, E=E, k=1, f=16, routing=routing,
                         alpha=1.0)
    return moe_inputs.make_logits(w).cuda()


def _outputs(T, E, k):
    from mixture_experts_layer_histogram_gb300 import _lib as L
    R = L.moe_grouped_rows_max(T, k, E)
    i32 = dict(dtype=torch.int32, device="cuda")
    return dict(topk_idx=torch.full((T, k), -9, **i32), topk_w=torch.full((T, k), float("nan"), device="cuda"),
                counts=torch.full((E,), -9, **i32), offsets=torch.full((E + 1,), -9, **i32),
                tile_offsets=torch.full((E + 1,), -9, **i32), row_of_slot=torch.full((T * k,), -9, **i32),
                token_of_row=torch.full((R,), -9, **i32))


@pytest.mark.parametrize("T,E,k,routing", SHAPES, ids=lambda v: str(v))
def test_fused_equals_separate_calls(T, E, k, routing):
    from mixture_experts_layer_histogram_gb300 import _lib as L
    logits = _logits(T, E, routing)
    ws = torch.full((L.moe_count_index_workspace_size(T, k, E),), 0x5A, dtype=torch.uint8, device="cuda")
    ref = _outputs(T, E, k)
    L.moe_route_topk(logits, k, ref["topk_idx"], ref["topk_w"])
    L.moe_count_index(ref["topk_idx"], E, ref["counts"], ref["offsets"], ref["tile_offsets"], ref["row_of_slot"],
                      ref["token_of_row"], ws)
    torch.cuda.synchronize()
    assert L.moe_read_status(ws) == 0
    used = int(ref["tile_offsets"][-1]) * 128
    for rep in range(2):   # the same workspace twice in a row, any content left by the previous call
        got = _outputs(T, E, k)
        L.moe_route_count_index(logits, k, got["topk_idx"], got["topk_w"], got["counts"], got["offsets"],
                                got["tile_offsets"], got["row_of_slot"], got["token_of_row"], ws)
        torch.cuda.synchronize()
        assert L.moe_read_status(ws) == 0
        for key in ("topk_idx", "topk_w", "counts", "offsets", "tile_offsets", "row_of_slot"):
            assert torch.equal(got[key], ref[key]), (rep, key)
        assert torch.equal(got["token_of_row"][:used], ref["token_of_row"][:used]), rep


def test_fused_with_no_tokens():
    from mixture_experts_layer_histogram_gb300 import _lib as L
    E, k = 8, 2
    ws = torch.zeros(L.moe_count_index_workspace_size(0, k, E), dtype=torch.uint8, device="cuda")
    got = _outputs(0, E, k)
    L.moe_route_count_index(torch.empty((0, E), device="cuda"), k, got["topk_idx"], got["topk_w"], got["counts"],
                            got["offsets"], got["tile_offsets"], got["row_of_slot"], got["token_of_row"], ws)
    torch.cuda.synchronize()
    assert (got["counts"] == 0).all() and (got["offsets"] == 0).all() and (got["tile_offsets"] == 0).all()
