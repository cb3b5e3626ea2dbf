"""Backward with recomputation (moe_grouped_ffn_bwd_recompute): ab and h are rebuilt from x_perm,
so the forward may keep them in scratch that other layers overwrite.

Two checks. The recomputing backward is compared with the fp64 oracle directly (every element on
small shapes; sampled tokens and weight-gradient entries at the full benchmark size), with the
scratch poisoned between forward and backward, so that a backward that read stale activations
instead of recomputing them fails. And it must be bit-identical to the backward that reads the
saved activations (the kernels are deterministic)."""
import numpy as np
import pytest
import torch

import moe_inputs
import oracle
from helpers import rel_err, tol_for

pytestmark = pytest.mark.gpu

CASES = [
    moe_inputs.small("sac_many_tiles", T=2048, d=256, E=8, k=2, f=256),    # several token tiles per expert
    moe_inputs.small("sac_one_tile", T=300, d=256, E=8, k=2, f=512),       # one short token tile per expert
    moe_inputs.small("sac_f32", T=333, d=96, E=5, k=3, f=40, dtype="f32"),  # SIMT fp32 path
]


def _sac_layer(w, inp):
    """Forward into shared scratch, poison the scratch (another layer used it), then backward."""
    from mixture_experts_layer_histogram_gb300 import MoELayer, _lib as L
    R = L.moe_grouped_rows_max(w.T, w.k, w.E)
    scratch = {"ab": torch.empty((R, 2 * w.f), dtype=w.torch_dtype, device="cuda"),
               "h": torch.empty((R, w.f), dtype=w.torch_dtype, device="cuda")}
    sac = MoELayer(w.T, w.d, w.E, w.k, w.f, w.torch_dtype, "cuda", recompute=True, scratch=scratch)
    sac.forward(inp["x"], inp["logits"], inp["w_gate_up"], inp["w_down"])
    out = sac.out.clone()
    scratch["ab"].fill_(float("nan"))
    scratch["h"].fill_(float("nan"))
    res = sac.backward(inp["g"], inp["w_gate_up"], inp["w_down"])
    torch.cuda.synchronize()
    assert sac.status() == (0, 0)
    return sac, out, res


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_recompute_backward_matches_oracle(w):
    inp = moe_inputs.make_all(w, "cuda")
    sac, out, res = _sac_layer(w, inp)
    cpu = {k: v.cpu() for k, v in inp.items()}
    idx, wt = oracle.route_topk(cpu["logits"], w.k)
    assert torch.equal(sac.topk_idx.cpu(), idx)
    ref = oracle.moe_tokens(cpu["x"], idx, wt, cpu["w_gate_up"], cpu["w_down"], cpu["g"])
    dwgu, dwd = oracle.moe_dweights(cpu["x"], idx, wt, cpu["w_gate_up"], cpu["w_down"], cpu["g"])
    errs = {"out": rel_err(out, ref["out"]), "dx": rel_err(res["dx"], ref["dx"]),
            "d_logits": rel_err(res["d_logits"], ref["d_logits"]),
            "d_topk_w": rel_err(res["d_topk_w"], ref["d_topk_w"]),
            "dw_gate_up": rel_err(res["dw_gate_up"], dwgu), "dw_down": rel_err(res["dw_down"], dwd)}
    tol = tol_for(w.torch_dtype)
    bad = {k: v for k, v in errs.items() if not v <= tol}
    assert not bad, (bad, errs)


def test_recompute_backward_matches_oracle_full_size_sampled():
    """The benchmark workload (T=8192, d=2048, E=64, k=8, f=1024, bf16): sampled tokens for dx,
    d_logits, d_topk_w, and sampled dW entries of the most, least and randomly loaded experts."""
    w = moe_inputs.WORKLOADS["fwdbwd_t8192"]
    inp = moe_inputs.make_all(w, "cuda")
    sac, out, res = _sac_layer(w, inp)
    cpu = {k: v.cpu() for k, v in inp.items()}
    idx, wt = oracle.route_topk(cpu["logits"], w.k)
    assert torch.equal(sac.topk_idx.cpu(), idx)
    gen = np.random.default_rng(4321)
    tokens = np.sort(gen.choice(w.T, size=64, replace=False))
    ref = oracle.moe_tokens(cpu["x"], idx, wt, cpu["w_gate_up"], cpu["w_down"], cpu["g"], tokens=tokens)
    tok = torch.from_numpy(tokens)
    errs = {"out": rel_err(out.cpu()[tok], ref["out"]), "dx": rel_err(res["dx"].cpu()[tok], ref["dx"]),
            "d_logits": rel_err(res["d_logits"].cpu()[tok], ref["d_logits"]),
            "d_topk_w": rel_err(res["d_topk_w"].cpu()[tok], ref["d_topk_w"])}
    counts = sac.counts.cpu().numpy()
    experts = sorted(set([int(counts.argmax()), int(counts.argmin())] + gen.choice(w.E, 3, replace=False).tolist()))
    mats, es, rs, cs = [], [], [], []
    for e in experts:
        for _ in range(6):
            mats.append(0); es.append(e); rs.append(int(gen.integers(0, 2 * w.f))); cs.append(int(gen.integers(0, w.d)))
            mats.append(1); es.append(e); rs.append(int(gen.integers(0, w.d))); cs.append(int(gen.integers(0, w.f)))
    val = oracle.dweight_entries(cpu["x"], idx, wt, cpu["w_gate_up"], cpu["w_down"], cpu["g"], mats, es, rs, cs)
    dwgu, dwd = res["dw_gate_up"].cpu(), res["dw_down"].cpu()
    got = torch.tensor([float(dwgu[e, r, c]) if m == 0 else float(dwd[e, r, c])
                        for m, e, r, c in zip(mats, es, rs, cs)], dtype=torch.float64)
    m = torch.tensor(mats)
    errs["dw_gate_up"] = rel_err(got[m == 0], val[m == 0])
    errs["dw_down"] = rel_err(got[m == 1], val[m == 1])
    bad = {k: v for k, v in errs.items() if not v <= 1e-2}
    assert not bad, (bad, errs)


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_recompute_backward_is_bit_identical(w):
    from mixture_experts_layer_histogram_gb300 import MoELayer
    inp = moe_inputs.make_all(w, "cuda")
    ref = MoELayer(w.T, w.d, w.E, w.k, w.f, w.torch_dtype, "cuda")
    ref.forward(inp["x"], inp["logits"], inp["w_gate_up"], inp["w_down"])
    r1 = {k: v.clone() for k, v in ref.backward(inp["g"], inp["w_gate_up"], inp["w_down"]).items()}
    sac, out, r2 = _sac_layer(w, inp)
    assert torch.equal(out, ref.out)
    for k in r1:
        assert torch.equal(r1[k], r2[k]), k
