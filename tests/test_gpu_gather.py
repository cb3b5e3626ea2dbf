"""The permutation fused into the grouped GEMMs' token loads (moe_grouped_ffn_*_gather): GEMM1 and the
gate/up weight gradient read token rows of x through token_of_row instead of rows of x_perm.

The same bytes reach the tensor cores either way, so every output of a layer pass in gather mode
must equal, bit for bit, the output of the pass that runs moe_permute first; the gather path is also
compared with the fp64 oracle directly, on small shapes element by element and at the benchmark size
on sampled tokens.

A forward-only layer (and the recomputing one) passes no ab buffer: GEMM1 then stores h but not a and
b. Its output must equal the training layer's, bit for bit, and the ab buffer must stay untouched."""
import numpy as np
import pytest
import torch

import moe_inputs
import oracle
from helpers import rel_err, tol_for

pytestmark = pytest.mark.gpu

KEYS = ("dx", "d_logits", "d_topk_w", "dw_gate_up", "dw_down")

CASES = [
    moe_inputs.small("g_ragged", T=1000, d=512, E=8, k=2, f=512),                              # several tiles, ragged
    moe_inputs.small("g_zipf_empty", T=700, d=256, E=64, k=4, f=256, routing="zipf", alpha=1.5),  # empty experts
    moe_inputs.small("g_one_expert", T=300, d=256, E=1, k=1, f=256),
    moe_inputs.small("g_big_tiles", T=4096, d=256, E=4, k=2, f=256),                            # 8 full tiles per expert
    moe_inputs.small("g_f32", T=333, d=96, E=5, k=3, f=40, dtype="f32"),                        # SIMT fp32 path
]


def _pass(w, inp, gather, recompute=False):
    from mixture_experts_layer_histogram_gb300 import MoELayer
    layer = MoELayer(w.T, w.d, w.E, w.k, w.f, w.torch_dtype, "cuda", recompute=recompute, gather=gather)
    layer.forward(inp["x"], inp["logits"], inp["w_gate_up"], inp["w_down"])
    out = layer.out.clone()
    res = {k: v.clone() for k, v in layer.backward(inp["g"], inp["w_gate_up"], inp["w_down"]).items()}
    torch.cuda.synchronize()
    assert layer.status() == (0, 0)
    return layer, out, res


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_gather_pass_is_bit_identical_to_permute_pass(w):
    inp = moe_inputs.make_all(w, "cuda")
    _, out0, r0 = _pass(w, inp, gather=False)
    layer, out1, r1 = _pass(w, inp, gather=True)
    assert layer.x_perm is None
    assert torch.equal(out0, out1)
    for k in KEYS:
        assert torch.equal(r0[k], r1[k]), k


@pytest.mark.parametrize("gather", [False, True])
@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_forward_only_layer_stores_no_ab(w, gather):
    from mixture_experts_layer_histogram_gb300 import MoELayer
    inp = moe_inputs.make_all(w, "cuda")
    _, out0, _ = _pass(w, inp, gather=False)
    layer = MoELayer(w.T, w.d, w.E, w.k, w.f, w.torch_dtype, "cuda", backward=False, gather=gather)
    layer.ab.fill_(float("nan"))
    layer.forward(inp["x"], inp["logits"], inp["w_gate_up"], inp["w_down"])
    torch.cuda.synchronize()
    assert layer.status() == (0, 0)
    assert torch.equal(layer.out, out0)
    assert torch.isnan(layer.ab).all()


@pytest.mark.parametrize("w", CASES[:2] + CASES[-1:], ids=lambda w: w.name)
def test_gather_recompute_is_bit_identical(w):
    inp = moe_inputs.make_all(w, "cuda")
    _, out0, r0 = _pass(w, inp, gather=False)
    _, out1, r1 = _pass(w, inp, gather=True, recompute=True)
    assert torch.equal(out0, out1)
    for k in KEYS:
        assert torch.equal(r0[k], r1[k]), k


@pytest.mark.parametrize("w", [CASES[0], CASES[1], CASES[-1]], ids=lambda w: w.name)
def test_gather_pass_matches_oracle(w):
    inp = moe_inputs.make_all(w, "cuda")
    layer, out, res = _pass(w, inp, gather=True)
    cpu = {k: v.cpu() for k, v in inp.items()}
    idx, wt = oracle.route_topk(cpu["logits"], w.k)
    assert torch.equal(layer.topk_idx.cpu(), idx)
    ref = oracle.moe_tokens(cpu["x"], idx, wt, cpu["w_gate_up"], cpu["w_down"], cpu["g"])
    dwgu, dwd = oracle.moe_dweights(cpu["x"], idx, wt, cpu["w_gate_up"], cpu["w_down"], cpu["g"])
    errs = {"out": rel_err(out, ref["out"]), "dx": rel_err(res["dx"], ref["dx"]),
            "d_logits": rel_err(res["d_logits"], ref["d_logits"]),
            "d_topk_w": rel_err(res["d_topk_w"], ref["d_topk_w"]),
            "dw_gate_up": rel_err(res["dw_gate_up"], dwgu), "dw_down": rel_err(res["dw_down"], dwd)}
    tol = tol_for(w.torch_dtype)
    bad = {k: v for k, v in errs.items() if not v <= tol}
    assert not bad, (bad, errs)


@pytest.mark.parametrize("name", ["fwd_t4096", "fwdbwd_t8192"])
def test_gather_full_size(name):
    """At the benchmark sizes: bit-identical to the permute pass, and sampled tokens against the oracle."""
    w = moe_inputs.WORKLOADS[name]
    inp = moe_inputs.make_all(w, "cuda")
    if not w.backward:   # a forward-only workload: give the backward a seeded gradient all the same
        inp["g"] = torch.randn((w.T, w.d), device="cuda", generator=torch.Generator(device="cuda").manual_seed(9)).to(
            w.torch_dtype)
    _, out0, r0 = _pass(w, inp, gather=False)
    _, out1, r1 = _pass(w, inp, gather=True)
    assert torch.equal(out0, out1)
    for k in KEYS:
        assert torch.equal(r0[k], r1[k]), k
    cpu = {k: v.cpu() for k, v in inp.items()}
    idx, wt = oracle.route_topk(cpu["logits"], w.k)
    tokens = np.sort(np.random.default_rng(77).choice(w.T, size=48, replace=False))
    ref = oracle.moe_tokens(cpu["x"], idx, wt, cpu["w_gate_up"], cpu["w_down"], cpu["g"], tokens=tokens)
    tok = torch.from_numpy(tokens)
    errs = {"out": rel_err(out1.cpu()[tok], ref["out"]), "dx": rel_err(r1["dx"].cpu()[tok], ref["dx"]),
            "d_logits": rel_err(r1["d_logits"].cpu()[tok], ref["d_logits"])}
    bad = {k: v for k, v in errs.items() if not v <= 1e-2}
    assert not bad, (bad, errs)
