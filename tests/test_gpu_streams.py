"""Two layers run at the same time on two CUDA streams, with every call of one issued between calls
of the other and no ordering between the streams, must each give, bit for bit, what it gives run
alone. The library keeps no state shared between calls beyond each call's own workspace.

The large case has two fused routing + counting + indexing calls of 256 blocks each. Each fits on
the GPU by itself, but not both at once. The fused kernel's blocks wait for one another. Its
cooperative launch guarantees that a grid starts only when all of it can be resident; without it,
that rests on the order in which the hardware places the two grids' blocks. A grid that started
partly resident would run its blocks' bounded waits out, and the status word would say so."""
import pytest
import torch

import moe_inputs

pytestmark = pytest.mark.gpu

CASES = [
    # (name, [workload of layer 1, workload of layer 2])
    ("fused_grids_exceed_gpu", [moe_inputs.small("streams_a", T=32768, d=256, E=64, k=8, f=256, seed=11),
                                moe_inputs.small("streams_b", T=32768, d=256, E=64, k=8, f=256, routing="zipf",
                                                 alpha=1.0, seed=12)]),
    ("two_gemm_grids", [moe_inputs.small("streams_c", T=3000, d=256, E=16, k=4, f=512, seed=13),
                        moe_inputs.small("streams_d", T=2000, d=512, E=32, k=8, f=256, routing="zipf",
                                         alpha=1.0, seed=14)]),
]
KEYS = ("dx", "d_logits", "d_topk_w", "dw_gate_up", "dw_down")


def _run(layer, inp, stream=None):
    layer.forward(inp["x"], inp["logits"], inp["w_gate_up"], inp["w_down"], stream=stream)
    return layer.backward(inp["g"], inp["w_gate_up"], inp["w_down"], stream=stream)


@pytest.mark.parametrize("name,ws", CASES, ids=[c[0] for c in CASES])
def test_layers_on_two_streams_match_each_alone(name, ws):
    from mixture_experts_layer_histogram_gb300 import MoELayer
    inps = [{k: v.cuda() for k, v in moe_inputs.make_all(w).items()} for w in ws]
    refs = []
    for w, inp in zip(ws, inps):   # each layer alone, on the current stream
        layer = MoELayer(w.T, w.d, w.E, w.k, w.f, w.torch_dtype, "cuda")
        res = _run(layer, inp)
        torch.cuda.synchronize()
        assert not any(layer.status())
        refs.append({"out": layer.out.clone()} | {k: res[k].clone() for k in KEYS})
        del layer
    layers = [MoELayer(w.T, w.d, w.E, w.k, w.f, w.torch_dtype, "cuda") for w in ws]
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    for s in streams:   # the inputs and buffers were written on the current stream
        s.wait_stream(torch.cuda.current_stream())
    for _ in range(3):
        for layer, inp, s in zip(layers, inps, streams):
            layer.forward(inp["x"], inp["logits"], inp["w_gate_up"], inp["w_down"], stream=s)
        outs = [layer.backward(inp["g"], inp["w_gate_up"], inp["w_down"], stream=s)
                for layer, inp, s in zip(layers, inps, streams)]
        torch.cuda.synchronize()
        for layer, res, ref in zip(layers, outs, refs):
            assert not any(layer.status()), layer.status()
            assert torch.equal(layer.out, ref["out"])
            for k in KEYS:
                assert torch.equal(res[k], ref[k]), k
