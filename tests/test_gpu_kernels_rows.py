"""Row-copy kernels (permute, combine, combine backward) through the C ABI on odd row sizes:
rows of 1..40 sixteen-byte vectors (fewer than, and not a multiple of, the 32 lanes of a warp),
k up to 16, both dtypes. Expected values come from plain torch indexing of the same inputs,
with the grouped rows taken from the fp64 oracle's index definition."""
import pytest
import torch

import oracle
from helpers import rel_err, rows_max

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("dtype,d", [(torch.bfloat16, 8), (torch.bfloat16, 24), (torch.bfloat16, 320),
                                     (torch.float32, 4), (torch.float32, 36), (torch.float32, 160)])
@pytest.mark.parametrize("T,E,k", [(37, 5, 3), (64, 32, 16), (1, 1, 1)])
def test_row_kernels_small_rows(dtype, d, T, E, k):
    from mixture_experts_layer_histogram_gb300 import _lib as L
    g = torch.Generator().manual_seed(T * 131 + d)
    idx = torch.stack([torch.randperm(E, generator=g)[:k] for _ in range(T)]).to(torch.int32)
    ref = oracle.index(idx, E, 128)
    R = rows_max(T, k, E)
    x = torch.randn((T, d), generator=g).to(dtype)
    w = torch.rand((T, k), generator=g, dtype=torch.float32)
    y = torch.randn((R, d), generator=g).to(dtype)
    go = torch.randn((T, d), generator=g).to(dtype)
    dev = "cuda"
    gi = {k_: v.to(dev) for k_, v in ref.items()}
    xp = torch.full((R, d), float("nan"), dtype=dtype, device=dev)
    L.moe_permute(x.to(dev), k, E, gi["row_of_slot"], gi["counts"], gi["tile_offsets"], xp)
    out = torch.empty((T, d), dtype=dtype, device=dev)
    L.moe_combine_fwd(y.to(dev), w.to(dev), gi["row_of_slot"], T, k, out)
    dx = torch.empty((T, d), dtype=dtype, device=dev)
    L.moe_combine_fwd(y.to(dev), None, gi["row_of_slot"], T, k, dx)
    dy = torch.full((R, d), float("nan"), dtype=dtype, device=dev)
    dtw = torch.empty((T, k), dtype=torch.float32, device=dev)
    dl = torch.empty((T, E), dtype=torch.float32, device=dev)
    L.moe_combine_bwd(go.to(dev), y.to(dev), w.to(dev), idx.to(dev), gi["row_of_slot"], gi["counts"],
                      gi["tile_offsets"], E, dy, dtw, dl)
    torch.cuda.synchronize()
    ros = ref["row_of_slot"].long().view(T, k)
    used = int(ref["tile_offsets"][-1]) * 128
    real = ref["token_of_row"][:used] >= 0
    pad = (~real).nonzero().view(-1)
    # permute: exact copies, zero padding
    xp = xp.cpu()
    assert torch.equal(xp[ros.view(-1)], x.repeat_interleave(k, 0))
    assert torch.all(xp[pad] == 0)
    # combine (weighted and unweighted sum)
    yd = y.double()
    exp_out = (w.double().unsqueeze(-1) * yd[ros]).sum(1)
    tol = 1e-2 if dtype == torch.bfloat16 else 1e-6
    assert rel_err(out, exp_out) <= tol
    assert rel_err(dx, yd[ros].sum(1)) <= tol
    # combine backward
    dy = dy.cpu()
    exp_dy = w.double().unsqueeze(-1) * go.double().unsqueeze(1)
    assert rel_err(dy[ros.view(-1)].view(T, k, d), exp_dy) <= tol
    assert torch.all(dy[pad] == 0)
    exp_dtw = (go.double().unsqueeze(1) * yd[ros]).sum(-1)
    assert rel_err(dtw, exp_dtw) <= 1e-5
    sw = (w.double() * exp_dtw).sum(1, keepdim=True)
    exp_dl = torch.zeros((T, E), dtype=torch.float64)
    exp_dl.scatter_(1, idx.long(), w.double() * (exp_dtw - sw))
    assert rel_err(dl, exp_dl) <= 1e-5
