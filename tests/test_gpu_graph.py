"""A layer pass captured into a CUDA graph (MoELayer.capture) and replayed must give, bit for bit,
what the same pass gives launched call by call (the kernels are deterministic), on new inputs
copied into the captured tensors, for bf16, fp32 and router layers."""
import pytest
import torch

import moe_inputs

pytestmark = pytest.mark.gpu

CASES = [
    (moe_inputs.small("graph_bf16", T=700, d=256, E=16, k=4, f=256), False),
    (moe_inputs.small("graph_f32", T=256, d=64, E=8, k=2, f=128, dtype="f32"), False),
    (moe_inputs.small("graph_router", T=500, d=256, E=16, k=4, f=256, routing="router"), True),
]


@pytest.mark.parametrize("w,router", CASES, ids=lambda c: c.name if hasattr(c, "name") else str(c))
def test_graph_replay_matches_eager(w, router):
    from mixture_experts_layer_histogram_gb300 import MoELayer
    inp = {k: v.cuda() for k, v in moe_inputs.make_all(w).items()}
    wr = (moe_inputs.make_router_weight(w).float() * 3.0).to(w.torch_dtype).cuda() if router else None
    lg = None if router else inp["logits"]
    eager = MoELayer(w.T, w.d, w.E, w.k, w.f, w.torch_dtype, "cuda", router=router)
    graphed = MoELayer(w.T, w.d, w.E, w.k, w.f, w.torch_dtype, "cuda", router=router)
    x = inp["x"].clone()
    g = inp["g"].clone()
    graph = graphed.capture(x, None if router else lg, inp["w_gate_up"], inp["w_down"], grad_out=g, w_router=wr)
    gen = torch.Generator(device="cuda").manual_seed(3)
    for _ in range(3):   # new inputs in the captured tensors, then one replay
        x.copy_(torch.randn(x.shape, generator=gen, device="cuda").to(x.dtype))
        g.copy_(torch.randn(g.shape, generator=gen, device="cuda").to(g.dtype))
        graph.replay()
        eager.forward(x, lg, inp["w_gate_up"], inp["w_down"], w_router=wr)
        ref = eager.backward(g, inp["w_gate_up"], inp["w_down"])
        torch.cuda.synchronize()
        assert torch.equal(graphed.out, eager.out)
        for k in ("dx", "d_logits", "dw_gate_up", "dw_down") + (("dw_router",) if router else ()):
            assert torch.equal(getattr(graphed, k), ref[k]), k
    assert not any(graphed.status()) and not any(eager.status())
