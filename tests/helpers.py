"""Shared test utilities (no method arithmetic: metrics, device handling, grouped-layout fixtures)."""
import math

import torch

GROUP_ROWS = 128


def rel_err(got, exp):
    """max|got - exp| / max|exp| in fp64 (the parity metric of the float outputs)."""
    got = got.detach().double().cpu()
    exp = exp.detach().double().cpu()
    den = exp.abs().max().item()
    num = (got - exp).abs().max().item()
    return num / den if den > 0 else num


def tile_offsets_from_counts(counts, BM=GROUP_ROWS):
    toff = [0]
    for c in counts:
        toff.append(toff[-1] + math.ceil(c / BM))
    return toff


def rows_max(T, k, E, BM=GROUP_ROWS):
    return ((T * k + E * (BM - 1) + BM - 1) // BM) * BM


def grouped_rows(counts, BM=GROUP_ROWS):
    """For each expert, the list of its real grouped rows."""
    toff = tile_offsets_from_counts(counts, BM)
    return [list(range(toff[e] * BM, toff[e] * BM + c)) for e, c in enumerate(counts)]


def tol_for(dtype):
    return 1e-5 if dtype == torch.float32 else 1e-2
