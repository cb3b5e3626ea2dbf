"""Backward with recomputation (moe_grouped_ffn_bwd_recompute): ab and h are rebuilt from x_perm,
so the forward may keep them in scratch that other layers overwrite. The results must be
bit-identical to the backward that reads the saved activations (the kernels are deterministic),
and that backward is itself checked against the oracle in test_gpu_parity.py."""
import pytest
import torch

import moe_inputs

pytestmark = pytest.mark.gpu

CASES = [
    moe_inputs.small("sac_pair", T=2048, d=256, E=8, k=2, f=256),          # row-grouped kinds on the CTA-pair kernel
    moe_inputs.small("sac_single", T=300, d=256, E=8, k=2, f=512),         # single-CTA kernel
    moe_inputs.small("sac_f32", T=333, d=96, E=5, k=3, f=40, dtype="f32"),  # SIMT fp32 path
]


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_recompute_backward_is_bit_identical(w):
    from mixture_experts_layer_histogram_gb300 import MoELayer
    inp = {k: v.cuda() for k, v in moe_inputs.make_all(w, "cuda").items()}
    ref = MoELayer(w.T, w.d, w.E, w.k, w.f, w.torch_dtype, "cuda")
    ref.forward(inp["x"], inp["logits"], inp["w_gate_up"], inp["w_down"])
    r1 = {k: v.clone() for k, v in ref.backward(inp["g"], inp["w_gate_up"], inp["w_down"]).items()}
    R = ref.rows_max
    scratch = {"ab": torch.empty((R, 2 * w.f), dtype=w.torch_dtype, device="cuda"),
               "h": torch.empty((R, w.f), dtype=w.torch_dtype, device="cuda")}
    sac = MoELayer(w.T, w.d, w.E, w.k, w.f, w.torch_dtype, "cuda", recompute=True, scratch=scratch)
    out = sac.forward(inp["x"], inp["logits"], inp["w_gate_up"], inp["w_down"])
    assert torch.equal(out, ref.out)
    scratch["ab"].fill_(float("nan"))      # another layer used the scratch in between
    scratch["h"].fill_(float("nan"))
    r2 = sac.backward(inp["g"], inp["w_gate_up"], inp["w_down"])
    torch.cuda.synchronize()
    assert sac.status() == (0, 0)
    for k in r1:
        assert torch.equal(r1[k], r2[k]), k
