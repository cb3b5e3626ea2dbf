"""Each grouped-GEMM kind in isolation, through the C ABI, against plain fp64 matmuls of the same
stored inputs (torch on the CPU). Inputs are laid out directly in the padded grouped layout with
ragged and empty experts, so every kind's tile decoding, tails and epilogue are exercised.

Each reference uses the library's own previous-stage output as its input (e.g. y is checked
against h_gpu Wd^T), so a failure names the kind that is wrong.
"""
import itertools

import pytest
import torch

from helpers import grouped_rows, rel_err, tile_offsets_from_counts, tol_for

pytestmark = pytest.mark.gpu

CASES = [
    # E, d, f, counts: ragged, empty, single-row and tile-multiple experts. The row-grouped kinds
    # split an expert's c rows into full 256-token tiles and a last tile of the rest rounded up to a
    # multiple of 32 (700 rows -> 256 + 256 + 192, 257 -> 256 + 32, 2049 -> 8 x 256 + 32), so these
    # counts cover one- and many-tile experts, 32-token last tiles, and tails of 1..31 rows past a
    # multiple of 32.
    (4, 512, 512, [300, 0, 129, 1]),
    (3, 256, 256, [128, 256, 5]),
    (2, 256, 768, [1, 383]),
    (2, 512, 512, [700, 1000]),
    (3, 256, 512, [1100, 0, 513]),
    (4, 512, 256, [1024, 1, 640, 897]),
    (5, 256, 256, [257, 31, 32, 33, 2049]),
    (1, 768, 256, [4095]),
    # The schedulers walk each cluster's tiles by stepping forward over the experts: long runs of
    # empty experts between tiles, and many one-tile experts (each cluster steps over several).
    (64, 256, 256, [0] * 20 + [300] + [0] * 10 + [1] + [0] * 5 + [700] + [0] * 26),
    (256, 256, 256, [1 + (e * 7) % 5 for e in range(256)]),
]


def _setup(E, d, f, counts, dtype, seed=0):
    from mixture_experts_layer_histogram_gb300 import _lib as L
    g = torch.Generator().manual_seed(seed)
    toff = tile_offsets_from_counts(counts)
    R = toff[-1] * 128 + 256          # a few unused rows after the last group
    rows = grouped_rows(counts)
    real = torch.zeros(R, dtype=torch.bool)
    for rr in rows:
        real[rr] = True
    x = (torch.randn((R, d), generator=g) * real[:, None]).to(dtype)
    dy = (torch.randn((R, d), generator=g) * real[:, None]).to(dtype)
    wgu = (torch.randn((E, 2 * f, d), generator=g) * 0.05).to(dtype)
    wd = (torch.randn((E, d, f), generator=g) * 0.05).to(dtype)
    dev = "cuda"
    t = dict(x=x, dy=dy, wgu=wgu, wd=wd)
    gt = {k: v.to(dev) for k, v in t.items()}
    gt["toff"] = torch.tensor(toff, dtype=torch.int32, device=dev)
    gt["off"] = torch.tensor([0] + list(itertools.accumulate(counts)), dtype=torch.int32, device=dev)
    ws = torch.zeros(L.moe_grouped_ffn_workspace_size(E, d, f, R, L.dtype_code(dtype), 1), dtype=torch.uint8,
                     device=dev)
    act = dict(dtype=dtype, device=dev)
    out = dict(ab=torch.full((R, 2 * f), float("nan"), **act), h=torch.full((R, f), float("nan"), **act),
               y=torch.full((R, d), float("nan"), **act), dab=torch.full((R, 2 * f), float("nan"), **act),
               dx=torch.full((R, d), float("nan"), **act), dwgu=torch.full((E, 2 * f, d), float("nan"), **act),
               dwd=torch.full((E, d, f), float("nan"), **act))
    return L, t, gt, rows, ws, out


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("E,d,f,counts", CASES)
def test_grouped_gemm_kinds(E, d, f, counts, dtype):
    L, t, gt, rows, ws, o = _setup(E, d, f, counts, dtype)
    L.moe_grouped_ffn_fwd(gt["x"], gt["wgu"], gt["wd"], gt["toff"], gt["off"], o["ab"], o["h"], o["y"], ws)
    L.moe_grouped_ffn_bwd(gt["dy"], gt["x"], o["ab"], o["h"], gt["wgu"], gt["wd"], gt["toff"], gt["off"], o["dab"],
                          o["dx"], o["dwgu"], o["dwd"], ws)
    torch.cuda.synchronize()
    assert L.moe_read_status(ws) == 0
    c = {k: v.double().cpu() for k, v in o.items()}
    x, dy = t["x"].double(), t["dy"].double()
    wgu, wd = t["wgu"].double(), t["wd"].double()
    tol = tol_for(dtype)
    all_rows = [r for rr in rows for r in rr]
    errs = {}
    ref = {k: torch.zeros_like(v) for k, v in c.items()}
    for e, rr in enumerate(rows):
        if not rr:
            continue
        ab = x[rr] @ wgu[e].T                                         # GATEUP
        ref["ab"][rr] = ab
        a, b = c["ab"][rr][:, :f], c["ab"][rr][:, f:]
        ref["h"][rr] = ab[:, :f] * torch.sigmoid(ab[:, :f]) * ab[:, f:]
        ref["y"][rr] = c["h"][rr] @ wd[e].T                           # DOWN (on the library's h)
        dh = dy[rr] @ wd[e]                                           # DH (on the library's ab)
        s = torch.sigmoid(a)
        ref["dab"][rr] = torch.cat([dh * b * s * (1 + a * (1 - s)), dh * a * s], 1)
        ref["dx"][rr] = c["dab"][rr] @ wgu[e]                         # DGRAD (on the library's dab)
        ref["dwd"][e] = dy[rr].T @ c["h"][rr]                         # WGRAD down
        ref["dwgu"][e] = c["dab"][rr].T @ x[rr]                       # WGRAD gate/up
    for key in ("ab", "h", "y", "dab", "dx"):
        errs[key] = rel_err(c[key][all_rows], ref[key][all_rows])
    for key in ("dwd", "dwgu"):
        errs[key] = rel_err(c[key], ref[key])
    bad = {k: v for k, v in errs.items() if not v <= tol}
    assert not bad, f"relative errors above {tol}: {bad} (all: {errs})"
    # experts without rows get exactly zero weight gradients
    for e, rr in enumerate(rows):
        if not rr:
            assert torch.all(c["dwd"][e] == 0) and torch.all(c["dwgu"][e] == 0)
    # padding rows of every grouped output are exactly zero
    toff = tile_offsets_from_counts(counts)
    pad = [r for e, rr in enumerate(rows) for r in range(toff[e] * 128 + len(rr), toff[e + 1] * 128)]
    if pad:
        for key in ("ab", "h", "y", "dab", "dx"):
            assert torch.all(c[key][pad] == 0), key
