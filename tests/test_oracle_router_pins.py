"""Pins of the router part of the fp64 oracle (L = x Wr^T and its backward) against things other
than itself: central finite differences of the whole layer's loss through the router (which fixes
every transpose and index of router_dx / router_dw and of their composition with the experts'
dx), a library matrix product, exact bf16 widening, and subset / full agreement."""
import numpy as np
import torch

import moe_inputs
import oracle


def _rng(seed):
    return np.random.default_rng(seed)


def _problem(seed, T=5, d=6, E=4, k=2, f=4, gap=0.3):
    """Tiny fp64 layer with a router whose top-k margin is at least `gap` for every token, so that
    perturbations of size 1e-5 keep the selection."""
    r = _rng(seed)
    while True:
        x = r.standard_normal((T, d))
        wr = r.standard_normal((E, d))
        L = x @ wr.T
        s = -np.sort(-L, axis=1)
        if np.all(s[:, k - 1] - s[:, k] > gap):
            break
    return dict(x=x, wr=wr, wgu=r.standard_normal((E, 2 * f, d)) * 0.5, wd=r.standard_normal((E, d, f)) * 0.5,
                g=r.standard_normal((T, d)), k=k)


def _loss(p, idx_fixed=None):
    X = torch.from_numpy(p["x"])
    L = oracle.router_logits(X, torch.from_numpy(p["wr"]))
    idx, w = oracle.route_topk(L, p["k"])
    if idx_fixed is not None:
        assert torch.equal(idx, idx_fixed), "selection changed under the perturbation"
    out = oracle.moe_tokens(X, idx, w, torch.from_numpy(p["wgu"]), torch.from_numpy(p["wd"]))["out"].numpy()
    return float((out * p["g"]).sum())


def _fd(p, key, idx, h=1e-5):
    base = p[key]
    grad = np.zeros_like(base)
    for i in np.ndindex(base.shape):
        q = dict(p)
        q[key] = base.copy()
        q[key][i] += h
        lp = _loss(q, idx)
        q[key][i] -= 2 * h
        lm = _loss(q, idx)
        grad[i] = (lp - lm) / (2 * h)
    return grad


def test_layer_gradients_through_router_match_finite_differences():
    """d loss / d x = experts' dx + dL Wr, d loss / d Wr = dL^T x (selection held fixed).
    d != E, so a transposed Wr or a swapped operand cannot pass."""
    p = _problem(0)
    X, Wr = torch.from_numpy(p["x"]), torch.from_numpy(p["wr"])
    L = oracle.router_logits(X, Wr)
    idx, w = oracle.route_topk(L, p["k"])
    tok = oracle.moe_tokens(X, idx, w, torch.from_numpy(p["wgu"]), torch.from_numpy(p["wd"]), torch.from_numpy(p["g"]))
    dL = tok["d_logits"]
    dx = tok["dx"].numpy() + oracle.router_dx(dL, Wr).numpy()
    dwr = oracle.router_dw(X, dL).numpy()
    for key, got in (("x", dx), ("wr", dwr)):
        fd = _fd(p, key, idx)
        err = np.abs(got - fd).max() / np.abs(fd).max()
        assert err < 1e-7, (key, err)
    # without the router term dx is wrong: the pin sees the router path
    fd_x = _fd(p, "x", idx)
    assert np.abs(tok["dx"].numpy() - fd_x).max() > 1e-3


def test_router_matches_library_matrix_products():
    r = _rng(1)
    T, d, E = 9, 13, 6
    x, wr, dL = r.standard_normal((T, d)), r.standard_normal((E, d)), r.standard_normal((T, E))
    X, Wr, DL = (torch.from_numpy(v) for v in (x, wr, dL))
    np.testing.assert_allclose(oracle.router_logits(X, Wr).numpy(), x @ wr.T, rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(oracle.router_dx(DL, Wr).numpy(), dL @ wr, rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(oracle.router_dw(X, DL).numpy(), dL.T @ x, rtol=1e-13, atol=1e-13)


def test_router_subsets_agree_with_full():
    r = _rng(2)
    T, d, E = 11, 8, 5
    X, Wr, DL = (torch.from_numpy(r.standard_normal(s)) for s in ((T, d), (E, d), (T, E)))
    tok = [10, 0, 4]
    assert torch.equal(oracle.router_logits(X, Wr, tokens=tok), oracle.router_logits(X, Wr)[tok])
    assert torch.equal(oracle.router_dx(DL, Wr, tokens=tok), oracle.router_dx(DL, Wr)[tok])
    cols = [7, 2]
    assert torch.equal(oracle.router_dw(X, DL, cols=cols), oracle.router_dw(X, DL)[:, cols])


def test_router_reads_bf16_and_f32_exactly():
    gen = torch.Generator().manual_seed(3)
    x = torch.randn(6, 16, generator=gen).to(torch.bfloat16)
    wr = (torch.randn(4, 16, generator=gen) * 0.02).to(torch.bfloat16)
    dL = torch.randn(6, 4, generator=gen)
    assert torch.equal(oracle.router_logits(x, wr), oracle.router_logits(x.double(), wr.double()))
    assert torch.equal(oracle.router_dx(dL, wr), oracle.router_dx(dL.double(), wr.double()))
    assert torch.equal(oracle.router_dw(x, dL), oracle.router_dw(x.double(), dL.double()))


def test_router_logits_of_generator_match_router_workload_logits():
    """The 'router' input recipe rounds fp64 x Wr^T to fp32: the oracle's logits round to the same
    values (within one fp32 ulp: the two fp64 sums may differ in their last bits)."""
    w = moe_inputs.small(T=64, d=32, E=8, k=2, f=32, routing="router", dtype="bf16")
    x = moe_inputs.make_x(w)
    wr = moe_inputs.make_router_weight(w)
    L = moe_inputs.make_logits(w)
    torch.testing.assert_close(oracle.router_logits(x, wr).float(), L, rtol=2.0 ** -23, atol=0)
