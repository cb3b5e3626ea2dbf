"""Parity of the router (moe_router_fwd / moe_router_bwd, through the C ABI) with the fp64 oracle.

Logits: max|gpu - oracle| / max|oracle| <= 1e-4 (fp32 accumulation of exact bf16 products; the
float bar of the layer is 1e-2 for bf16 and 1e-5 for fp32). The selection is a decision taken on
the kernel's fp32 logits, so topk_idx must equal, bit for bit, the oracle's selection on the
kernel's own logits, and topk_w its weights within 1e-5. Backward: dx and dw_router within the
dtype's bar (bf16 rounds d_logits once; fp32 not at all).
"""
import pytest
import torch

import moe_inputs
import oracle
from helpers import rel_err, tol_for

pytestmark = pytest.mark.gpu

# (name, T, d, E, k, dtype)
SHAPES = [
    ("bench_like", 1000, 256, 64, 8, "bf16"),
    ("ragged_E40_d264", 333, 264, 40, 5, "bf16"),     # E not a multiple of 16, d not of 64
    ("max_E256_k16", 257, 512, 256, 16, "bf16"),
    ("tiny_E8", 130, 64, 8, 2, "bf16"),
    ("E5_k_eq_E", 200, 128, 5, 5, "bf16"),            # E not a multiple of 4: scalar logit stores
    ("single_expert", 64, 128, 1, 1, "bf16"),
    ("many_tiles", 40000, 128, 16, 4, "bf16"),        # 313 token tiles: the persistent loop reuses TMEM
    ("f32_tiny", 256, 64, 8, 2, "f32"),
    ("f32_ragged", 333, 96, 5, 3, "f32"),
]


def _inputs(T, d, E, dtype, seed=0):
    w = moe_inputs.small("router", T=T, d=d, E=E, k=1, f=8, dtype=dtype, routing="router", seed=seed)
    x = moe_inputs.make_x(w)
    wr = moe_inputs.make_router_weight(w)
    if dtype == "bf16":   # N(0, 0.02) router weights give logits of std ~0.9 at d = 2048: scale up for small d
        wr = (wr.float() * (2048.0 / d) ** 0.5).to(torch.bfloat16)
    return x, wr


def _fwd(x, wr, k, with_logits=True):
    from mixture_experts_layer_histogram_gb300 import _lib as L
    T, d = x.shape
    E = wr.shape[0]
    ws = torch.zeros(L.moe_router_workspace_size(T, d, E, L.dtype_code(x.dtype)), dtype=torch.uint8, device="cuda")
    logits = torch.full((T, E), float("nan"), device="cuda") if with_logits else None
    idx = torch.full((T, k), -7, dtype=torch.int32, device="cuda")
    w = torch.full((T, k), float("nan"), device="cuda")
    L.moe_router_fwd(x.cuda(), wr.cuda(), k, logits, idx, w, ws)
    torch.cuda.synchronize()
    assert L.moe_read_status(ws) == 0
    return logits, idx, w


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: s[0])
def test_router_fwd_matches_oracle(shape):
    from mixture_experts_layer_histogram_gb300 import _lib as L
    _, T, d, E, k, dt = shape
    x, wr = _inputs(T, d, E, dt)
    logits, idx, w = _fwd(x, wr, k)
    ref_L = oracle.router_logits(x, wr)
    assert rel_err(logits, ref_L) <= 1e-4
    lg = logits.cpu()
    ref_idx, ref_w = oracle.route_topk(lg, k)           # the decision in the kernel's precision
    assert torch.equal(idx.cpu(), ref_idx)
    assert rel_err(w, ref_w) <= 1e-5
    # the same selection as the stand-alone routing kernel on those logits
    idx2 = torch.empty_like(idx)
    w2 = torch.empty_like(w)
    L.moe_route_topk(logits, k, idx2, w2)
    assert torch.equal(idx, idx2)
    assert rel_err(w, w2) <= 1e-6
    # without the logits output the kernel decides the same
    _, idx3, w3 = _fwd(x, wr, k, with_logits=False)
    assert torch.equal(idx, idx3) and torch.equal(w, w3)


def test_router_ties_pick_lower_ids():
    """Identical router rows give bit-identical logits; the lower expert id wins each tie."""
    T, d, E, k = 300, 256, 16, 4
    x, wr = _inputs(T, d, E, "bf16", seed=1)
    wr[7] = wr[3]
    wr[11] = wr[10]
    wr[12] = wr[10]
    logits, idx, w = _fwd(x, wr, k)
    lg = logits.cpu()
    assert torch.equal(lg[:, 3], lg[:, 7]) and torch.equal(lg[:, 10], lg[:, 12])
    ref_idx, ref_w = oracle.route_topk(lg, k)
    assert torch.equal(idx.cpu(), ref_idx)
    assert rel_err(w, ref_w) <= 1e-5
    # every router row equal: the first k experts, each with weight exactly 1/k
    wr_all = wr[:1].expand(E, d).contiguous()
    _, idx, w = _fwd(x, wr_all, k)
    assert (idx.cpu() == torch.arange(k, dtype=torch.int32)).all()
    assert (w.cpu() == 1.0 / k).all()


def _bwd(x, wr, dl, dx_in, accumulate):
    from mixture_experts_layer_histogram_gb300 import _lib as L
    T, d = x.shape
    E = wr.shape[0]
    ws = torch.full((L.moe_router_workspace_size(T, d, E, L.dtype_code(x.dtype)),), 0xAB, dtype=torch.uint8,
                    device="cuda")   # any content
    dx = dx_in.clone().cuda()
    dw = torch.full((E, d), float("nan"), dtype=x.dtype, device="cuda")
    L.moe_router_bwd(x.cuda(), wr.cuda(), dl.cuda(), dx, dw, ws, accumulate_dx=accumulate)
    torch.cuda.synchronize()
    assert L.moe_read_status(ws) == 0
    return dx, dw


@pytest.mark.parametrize("accumulate", [False, True], ids=["dx_set", "dx_add"])
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: s[0])
def test_router_bwd_matches_oracle(shape, accumulate):
    _, T, d, E, k, dt = shape
    x, wr = _inputs(T, d, E, dt)
    gen = torch.Generator().manual_seed(5)
    dl = torch.randn(T, E, generator=gen)
    dx_in = torch.randn(T, d, generator=gen).to(x.dtype)
    dx, dw = _bwd(x, wr, dl, dx_in, accumulate)
    tol = tol_for(x.dtype)
    ref_dx = oracle.router_dx(dl, wr) + (dx_in.double() if accumulate else 0.0)
    assert rel_err(dx, ref_dx) <= tol
    assert rel_err(dw, oracle.router_dw(x, dl)) <= tol


def test_router_bwd_deterministic():
    T, d, E = 4096, 512, 64
    x, wr = _inputs(T, d, E, "bf16")
    dl = torch.randn(T, E, generator=torch.Generator().manual_seed(6))
    z = torch.zeros(T, d, dtype=torch.bfloat16)
    a = _bwd(x, wr, dl, z, False)
    b = _bwd(x, wr, dl, z, False)
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


def test_router_empty_tokens():
    from mixture_experts_layer_histogram_gb300 import _lib as L
    d, E = 256, 8
    for dt in (torch.bfloat16, torch.float32):
        x = torch.empty((0, d), dtype=dt, device="cuda")
        wr = torch.ones((E, d), dtype=dt, device="cuda")
        ws = torch.zeros(L.moe_router_workspace_size(0, d, E, L.dtype_code(dt)), dtype=torch.uint8, device="cuda")
        L.moe_router_fwd(x, wr, 2, torch.empty((0, E), device="cuda"), torch.empty((0, 2), dtype=torch.int32,
                         device="cuda"), torch.empty((0, 2), device="cuda"), ws)
        dw = torch.full((E, d), 3.0, dtype=dt, device="cuda")
        L.moe_router_bwd(x, wr, torch.empty((0, E), device="cuda"), torch.empty((0, d), dtype=dt, device="cuda"), dw,
                         ws)
        torch.cuda.synchronize()
        assert L.moe_read_status(ws) == 0
        assert (dw == 0).all()


# ----------------------------------------------------------------------------- full size ---------
FULL = [("fwdbwd_t8192", 8192, 2048, 64, 8), ("large_a0.8", 16384, 4096, 128, 8)]


@pytest.mark.parametrize("shape", FULL, ids=lambda s: s[0])
def test_router_full_size(shape):
    """Full-size router: every logit (T=8192) or sampled tokens' logits, the whole selection on the
    kernel's logits, sampled dx rows and dw_router columns (all columns at T=8192)."""
    name, T, d, E, k = shape
    w = moe_inputs.small(name, T=T, d=d, E=E, k=k, f=8, dtype="bf16", routing="router")
    x, wr = moe_inputs.make_x(w), moe_inputs.make_router_weight(w)
    logits, idx, tw = _fwd(x, wr, k)
    lg = logits.cpu()
    gen = torch.Generator().manual_seed(7)
    tok = torch.randperm(T, generator=gen)[:256].sort().values
    if T <= 8192:
        assert rel_err(lg, oracle.router_logits(x, wr)) <= 1e-4
    else:
        assert rel_err(lg[tok], oracle.router_logits(x, wr, tokens=tok)) <= 1e-4
    ref_idx, ref_w = oracle.route_topk(lg, k)
    assert torch.equal(idx.cpu(), ref_idx)
    assert rel_err(tw, ref_w) <= 1e-5
    dl = torch.randn(T, E, generator=gen) * 0.01
    dx_in = torch.randn(T, d, generator=gen).to(torch.bfloat16) * 0.01
    dx, dw = _bwd(x, wr, dl, dx_in, True)
    assert rel_err(dx.cpu()[tok], oracle.router_dx(dl, wr, tokens=tok) + dx_in[tok].double()) <= 1e-2
    if T <= 8192:
        assert rel_err(dw, oracle.router_dw(x, dl)) <= 1e-2
    else:
        cols = torch.randperm(d, generator=gen)[:96].sort().values
        assert rel_err(dw.cpu()[:, cols], oracle.router_dw(x, dl, cols=cols)) <= 1e-2


# ----------------------------------------------------------------------------- layer -------------
LAYERS = [
    moe_inputs.small("router_layer_bf16", T=1000, d=256, E=16, k=4, f=256, routing="router"),
    moe_inputs.small("router_layer_f32", T=333, d=96, E=5, k=3, f=40, dtype="f32", routing="router"),
]


@pytest.mark.parametrize("w", LAYERS, ids=lambda w: w.name)
def test_layer_with_router_matches_oracle(w):
    """The whole layer fed by the router: out, dx (experts + router), d_logits, dw_router, dW."""
    from mixture_experts_layer_histogram_gb300 import MoELayer
    inp = moe_inputs.make_all(w)
    wr = moe_inputs.make_router_weight(w)
    if w.dtype == "bf16":
        wr = (wr.float() * (2048.0 / w.d) ** 0.5).to(torch.bfloat16)
    g = {kk: v.cuda() for kk, v in inp.items()}
    layer = MoELayer(w.T, w.d, w.E, w.k, w.f, w.torch_dtype, "cuda", router=True)
    out = layer.forward(g["x"], None, g["w_gate_up"], g["w_down"], w_router=wr.cuda())
    res = layer.backward(g["g"], g["w_gate_up"], g["w_down"])
    torch.cuda.synchronize()
    assert layer.status() == (0, 0, 0)
    tol = tol_for(w.torch_dtype)
    lg = layer.logits.cpu()
    assert rel_err(lg, oracle.router_logits(inp["x"], wr)) <= 1e-4
    idx, wt = oracle.route_topk(lg, w.k)
    assert torch.equal(layer.topk_idx.cpu(), idx)
    ref = oracle.moe_tokens(inp["x"], idx, wt, inp["w_gate_up"], inp["w_down"], inp["g"])
    assert rel_err(out, ref["out"]) <= tol
    assert rel_err(res["d_logits"], ref["d_logits"]) <= tol
    ref_dx = ref["dx"] + oracle.router_dx(ref["d_logits"], wr)
    assert rel_err(res["dx"], ref_dx) <= tol
    assert rel_err(res["dw_router"], oracle.router_dw(inp["x"], ref["d_logits"])) <= tol
    dwgu, dwd = oracle.moe_dweights(inp["x"], idx, wt, inp["w_gate_up"], inp["w_down"], inp["g"])
    assert rel_err(res["dw_gate_up"], dwgu) <= tol
    assert rel_err(res["dw_down"], dwd) <= tol
