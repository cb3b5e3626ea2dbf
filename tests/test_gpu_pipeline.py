"""Host-buffer pipeline (HostPipeline): uploads, compute and downloads of consecutive steps overlap
on three streams. Every step's host results must equal those of the plain layer run on the same
device inputs (the kernels are deterministic), for more steps than there are slots, with each
slot's pass replayed from a CUDA graph and launched kernel by kernel, and when the weights change
between steps (the graphs are recorded again)."""
import pytest
import torch

import moe_inputs

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("graphs", [True, False], ids=["graphs", "eager"])
@pytest.mark.parametrize("backward,router", [(True, False), (False, False), (True, True)],
                         ids=["fwdbwd", "fwd", "fwdbwd_router"])
def test_pipeline_matches_layer(backward, router, graphs):
    from mixture_experts_layer_histogram_gb300 import HostPipeline, MoELayer
    w = moe_inputs.small("pipe", T=1000, d=256, E=8, k=2, f=256)
    wts = moe_inputs.make_all(w, "cuda")
    # steps 0-2 use one set of weights, steps 3-4 another (new tensors: the graphs are recorded again)
    wgu1, wd1 = wts["w_gate_up"], wts["w_down"]
    wgu2, wd2 = (wgu1.float() * 0.5).to(w.torch_dtype), (wd1.float() * 1.5).to(w.torch_dtype)
    wts_of = lambda i: (wgu1, wd1) if i < 3 else (wgu2, wd2)
    wr = (moe_inputs.make_router_weight(w).float() * 3.0).to(w.torch_dtype).cuda() if router else None
    batches = []
    for i in range(5):
        gen = torch.Generator().manual_seed(100 + i)
        b = dict(x=torch.randn(w.T, w.d, generator=gen).to(w.torch_dtype))
        if not router:
            b["logits"] = torch.randn(w.T, w.E, generator=gen)
        if backward:
            b["g"] = torch.randn(w.T, w.d, generator=gen).to(w.torch_dtype)
        batches.append({k: v.pin_memory() for k, v in b.items()})
    ref = MoELayer(w.T, w.d, w.E, w.k, w.f, w.torch_dtype, "cuda", backward=backward, router=router)
    expect = []
    for i, b in enumerate(batches):
        d = {k: v.cuda() for k, v in b.items()}
        wgu, wd = wts_of(i)
        ref.forward(d["x"], d.get("logits"), wgu, wd, w_router=wr)
        r = dict(out=ref.out.cpu())
        if backward:
            ref.backward(d["g"], wgu, wd)
            r.update(dx=ref.dx.cpu(), d_logits=ref.d_logits.cpu())   # dx includes the router's share
        expect.append(r)
    lay = MoELayer(w.T, w.d, w.E, w.k, w.f, w.torch_dtype, "cuda", backward=backward, router=router)
    pipe = HostPipeline(lay, graphs=graphs)
    assert pipe.h2d_bytes() == sum(v.numel() * v.element_size() for v in batches[0].values())
    got, prev = [], None
    for i, b in enumerate(batches):
        wgu, wd = wts_of(i)
        step = pipe.submit(b, wgu, wd, next_batch=batches[i + 1] if i + 1 < len(batches) else None, w_router=wr)
        if prev is not None:                        # step i-1's download overlaps step i's compute
            got.append({k: v.clone() for k, v in prev.wait().items()})
        prev = step
    got.append({k: v.clone() for k, v in prev.wait().items()})
    pipe.join()
    torch.cuda.synchronize()
    assert not any(lay.status())
    for i, (e, g) in enumerate(zip(expect, got)):
        assert set(e) == set(g)
        for k in e:
            assert torch.equal(e[k], g[k]), (i, k)
