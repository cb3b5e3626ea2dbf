"""Routing, counting and index generation on seeded random shapes, up to 640,000 slots: every launch
form of the one-launch call (512-slot blocks while they fit one per SM, 1024-slot blocks while all
fit at once, the two separate calls above that) and the separate calls themselves, against the
fp64 oracle. Indices and counts bit for bit, routing weights within 1e-6; a few cases draw logits
from a handful of values, so that exact ties decide the selection (lower expert id first)."""
import random

import pytest
import torch

import moe_inputs
import oracle
from helpers import rel_err

pytestmark = pytest.mark.gpu


def _cases(n=12, seed=77):
    r = random.Random(seed)
    # one case per launch form, then random ones
    out = [("fzi_512blocks_T9000_E64_k8", 9000, 64, 8, False, 1),           # 72,000 slots: 141 blocks of 512
           ("fzi_1024blocks_T16384_E101_k8", 16384, 101, 8, False, 2),     # 131,072 slots, E % 4 != 0
           ("fzi_1024blocks_T25000_E128_k12_ties", 25000, 128, 12, True, 3),  # 300,000 slots
           ("fzi_twocalls_T40000_E256_k16", 40000, 256, 16, False, 4)]     # 640,000 slots: separate calls
    for i in range(n):
        E = r.choice([1, 3, 7, 8, 40, 64, 100, 128, 255, 256])
        k = r.randint(1, min(E, 16))
        T = r.choice([1, 97, 1000, 4096, 9000, 16384, 25000, 40000])
        ties = i % 5 == 0
        out.append((f"fzi{i}_T{T}_E{E}_k{k}{'_ties' if ties else ''}", T, E, k, ties, 1000 + i))
    return out


CASES = _cases()


def _logits(T, E, ties, seed):
    g = torch.Generator().manual_seed(seed)
    if ties:
        vals = torch.tensor([-2.0, -0.0, 0.0, 0.5, 1.25])
        return vals[torch.randint(0, len(vals), (T, E), generator=g)]
    return torch.randn((T, E), generator=g) * 1.5


@pytest.mark.parametrize("name,T,E,k,ties,seed", CASES, ids=[c[0] for c in CASES])
def test_random_index_shapes_match_oracle(name, T, E, k, ties, seed):
    from mixture_experts_layer_histogram_gb300 import _lib as L
    logits = _logits(T, E, ties, seed)
    idx_ref, w_ref = oracle.route_topk(logits, k)
    R = L.moe_grouped_rows_max(T, k, E)
    ref = oracle.index(idx_ref, E, 128, R)
    used = int(ref["tile_offsets"][-1]) * 128
    lg = logits.cuda()
    i32 = dict(dtype=torch.int32, device="cuda")
    ws = torch.full((L.moe_count_index_workspace_size(T, k, E),), 0x5A, dtype=torch.uint8, device="cuda")

    def outputs():
        return dict(topk_idx=torch.full((T, k), -9, **i32), topk_w=torch.full((T, k), float("nan"), device="cuda"),
                    counts=torch.full((E,), -9, **i32), offsets=torch.full((E + 1,), -9, **i32),
                    tile_offsets=torch.full((E + 1,), -9, **i32), row_of_slot=torch.full((T * k,), -9, **i32),
                    token_of_row=torch.full((R,), -9, **i32))

    fused, sep = outputs(), outputs()
    L.moe_route_count_index(lg, k, fused["topk_idx"], fused["topk_w"], fused["counts"], fused["offsets"],
                            fused["tile_offsets"], fused["row_of_slot"], fused["token_of_row"], ws)
    torch.cuda.synchronize()
    assert L.moe_read_status(ws) == 0
    L.moe_route_topk(lg, k, sep["topk_idx"], sep["topk_w"])
    L.moe_count_index(sep["topk_idx"], E, sep["counts"], sep["offsets"], sep["tile_offsets"], sep["row_of_slot"],
                      sep["token_of_row"], ws)
    torch.cuda.synchronize()
    assert L.moe_read_status(ws) == 0
    for got in (fused, sep):
        assert torch.equal(got["topk_idx"].cpu(), idx_ref)
        assert rel_err(got["topk_w"].cpu(), w_ref) <= 1e-6
        for key in ("counts", "offsets", "tile_offsets", "row_of_slot"):
            assert torch.equal(got[key].cpu(), ref[key]), key
        assert torch.equal(got["token_of_row"][:used].cpu(), ref["token_of_row"][:used])
