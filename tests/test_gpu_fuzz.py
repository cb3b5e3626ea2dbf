"""Whole-layer parity on seeded random shapes: T from 1 to 700, E from 1 to 40, k from 1 to
min(E, 16), bf16 (d, f multiples of 256) and fp32 (any d multiple of 4, any f), normal or skewed
routing, with and without the router. Every case runs the full forward and backward through the
C ABI and compares indices bit for bit and every float output with the fp64 oracle."""
import random

import pytest
import torch

import moe_inputs
import oracle
from helpers import rel_err, tol_for

pytestmark = pytest.mark.gpu


def _cases(n=24, seed=2024):
    r = random.Random(seed)
    out = []
    for i in range(n):
        dtype = "bf16" if i % 3 else "f32"
        E = r.choice([1, 2, 3, 5, 8, 13, 16, 24, 33, 40])
        k = r.randint(1, min(E, 16))
        T = r.choice([1, 2, 31, 127, 128, 129, 255, 300, 513, 700])
        if dtype == "bf16":
            d, f = r.choice([256, 512]), r.choice([256, 512])
        else:
            d, f = 4 * r.randint(1, 40), r.randint(1, 70)
        routing = r.choice(["normal", "normal", "zipf"])
        router = dtype == "bf16" and i % 4 == 1
        out.append((f"fz{i}_{dtype}_T{T}_d{d}_E{E}_k{k}_f{f}_{routing}{'_router' if router else ''}",
                    moe_inputs.small(f"fz{i}", T=T, d=d, E=E, k=k, f=f, dtype=dtype, routing=routing, alpha=1.0,
                                     seed=i + 1), router))
    return out


CASES = _cases()


@pytest.mark.parametrize("name,w,router", CASES, ids=[c[0] for c in CASES])
def test_random_shape_layer_matches_oracle(name, w, router):
    from mixture_experts_layer_histogram_gb300 import MoELayer
    inp = moe_inputs.make_all(w)
    wr = None
    if router:
        wr = (moe_inputs.make_router_weight(w).float() * (2048.0 / w.d) ** 0.5).to(w.torch_dtype)
    g = {key: v.cuda() for key, v in inp.items()}
    layer = MoELayer(w.T, w.d, w.E, w.k, w.f, w.torch_dtype, "cuda", router=router)
    out = layer.forward(g["x"], None if router else g["logits"], g["w_gate_up"], g["w_down"],
                        w_router=wr.cuda() if router else None)
    res = layer.backward(g["g"], g["w_gate_up"], g["w_down"])
    torch.cuda.synchronize()
    assert not any(layer.status())
    logits = layer.logits.cpu() if router else inp["logits"]
    if router:
        assert rel_err(logits, oracle.router_logits(inp["x"], wr)) <= 1e-4
    idx, wt = oracle.route_topk(logits, w.k)
    assert torch.equal(layer.topk_idx.cpu(), idx)
    ref_i = oracle.index(idx, w.E, 128, layer.rows_max)
    for key in ("counts", "offsets", "tile_offsets", "row_of_slot"):
        assert torch.equal(getattr(layer, key).cpu(), ref_i[key]), key
    tol = tol_for(w.torch_dtype)
    assert rel_err(layer.topk_w, wt) <= 1e-5
    ref = oracle.moe_tokens(inp["x"], idx, wt, inp["w_gate_up"], inp["w_down"], inp["g"])
    assert rel_err(out, ref["out"]) <= tol
    assert rel_err(res["d_logits"], ref["d_logits"]) <= tol
    assert rel_err(res["d_topk_w"], ref["d_topk_w"]) <= tol
    ref_dx = ref["dx"] + (oracle.router_dx(ref["d_logits"], wr) if router else 0.0)
    assert rel_err(res["dx"], ref_dx) <= tol
    dwgu, dwd = oracle.moe_dweights(inp["x"], idx, wt, inp["w_gate_up"], inp["w_down"], inp["g"])
    assert rel_err(res["dw_gate_up"], dwgu) <= tol
    assert rel_err(res["dw_down"], dwd) <= tol
    if router:
        assert rel_err(res["dw_router"], oracle.router_dw(inp["x"], ref["d_logits"])) <= tol
