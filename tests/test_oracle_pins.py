"""Pins of the fp64 oracle against things other than itself (no GPU needed).

Each test states what fixes the expected value: brute force on tiny inputs, a closed form, an
invariant, a special case that reduces to a textbook routine, or central finite differences.
"""
import itertools
import json
import math
import os

import numpy as np
import pytest
import torch
from scipy.special import expit, softmax

import moe_inputs
import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rng(seed):
    return np.random.default_rng(seed)


# ----------------------------------------------------------------------------- routing ----------

def _topk_bruteforce(L, k):
    """Python sort with the key (-logit, id): highest logit first, lower id on ties (-0 == +0)."""
    out = []
    for row in L.tolist():
        order = sorted(range(len(row)), key=lambda e: (-row[e], e))
        out.append(order[:k])
    return np.array(out, dtype=np.int32)


@pytest.mark.parametrize("seed,T,E,k", [(0, 64, 8, 2), (1, 33, 16, 5), (2, 50, 7, 7), (3, 40, 64, 8)])
def test_topk_matches_bruteforce_with_ties(seed, T, E, k):
    r = _rng(seed)
    # few distinct values (including -0.0 and +0.0) so that ties are common
    vals = np.array([-1.5, -0.0, 0.0, 0.25, 2.0, 3.0], dtype=np.float32)
    L = vals[r.integers(0, len(vals), size=(T, E))]
    idx, w = oracle.route_topk(torch.from_numpy(L), k)
    assert np.array_equal(idx.numpy(), _topk_bruteforce(L, k))
    np.testing.assert_allclose(w.sum(1).numpy(), 1.0, rtol=0, atol=1e-15)


def test_equal_logits_pick_lowest_ids_with_equal_weights():
    L = torch.zeros((5, 12), dtype=torch.float32)
    L[1] = -0.0
    L[2] = 7.25
    idx, w = oracle.route_topk(L, 4)
    assert (idx == torch.arange(4, dtype=torch.int32)).all()
    assert torch.all(w == 0.25)


def test_dense_routing_weights_are_softmax():
    """k = E: renormalised top-k over all experts is the plain softmax (scipy)."""
    L = _rng(4).standard_normal((20, 6)).astype(np.float32)
    idx, w = oracle.route_topk(torch.from_numpy(L), 6)
    dense = np.zeros((20, 6))
    for t in range(20):
        dense[t, idx[t].numpy()] = w[t].numpy()
    np.testing.assert_allclose(dense, softmax(L.astype(np.float64), axis=1), rtol=1e-14, atol=0)


def test_topk_weights_relative_to_full_softmax():
    """w equals softmax over all E restricted to S_t and renormalised (scipy softmax, then renorm)."""
    L = _rng(5).standard_normal((30, 16)).astype(np.float32)
    idx, w = oracle.route_topk(torch.from_numpy(L), 3)
    p = softmax(L.astype(np.float64), axis=1)
    sel = np.take_along_axis(p, idx.numpy().astype(np.int64), axis=1)
    np.testing.assert_allclose(w.numpy(), sel / sel.sum(1, keepdims=True), rtol=1e-14)


# ----------------------------------------------------------------------------- indexing ---------

def _index_bruteforce(idx, E, BM):
    T, k = idx.shape
    slots = [(int(idx[t, j]), t * k + j) for t in range(T) for j in range(k)]
    counts = [sum(1 for e, _ in slots if e == ee) for ee in range(E)]
    tiles = [math.ceil(c / BM) for c in counts]
    start = [BM * sum(tiles[:e]) for e in range(E)]
    row = [None] * (T * k)
    for ee in range(E):
        mine = sorted(s for e, s in slots if e == ee)
        for rank, s in enumerate(mine):
            row[s] = start[ee] + rank
    return counts, tiles, row


@pytest.mark.parametrize("seed,T,E,k,BM", [(0, 37, 8, 2, 4), (1, 64, 5, 3, 16), (2, 20, 16, 4, 1),
                                          (3, 50, 6, 6, 128), (4, 1, 3, 1, 8)])
def test_index_matches_bruteforce(seed, T, E, k, BM):
    r = _rng(seed)
    idx = np.stack([r.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    got = oracle.index(torch.from_numpy(idx), E, BM)
    counts, tiles, row = _index_bruteforce(idx, E, BM)
    assert got["counts"].tolist() == counts
    assert got["offsets"].tolist() == list(itertools.accumulate([0] + counts))
    assert got["tile_offsets"].tolist() == list(itertools.accumulate([0] + tiles))
    assert got["row_of_slot"].tolist() == row
    tor = got["token_of_row"].tolist()
    for s, rr in enumerate(row):
        assert tor[rr] == s // k
    assert sum(1 for v in tor if v >= 0) == T * k


def test_index_bm1_is_compact_exclusive_scan():
    """With BM = 1 the grouped layout is the unpadded counting sort: row = offsets[e] + rank."""
    r = _rng(7)
    idx = np.stack([r.permutation(9)[:3] for _ in range(40)]).astype(np.int32)
    got = oracle.index(torch.from_numpy(idx), 9, 1)
    assert got["tile_offsets"].tolist() == got["offsets"].tolist()
    assert sorted(got["row_of_slot"].tolist()) == list(range(120))


def test_index_invariants_random():
    r = _rng(8)
    T, E, k, BM = 3000, 64, 8, 128
    L = r.standard_normal((T, E)).astype(np.float32)
    idx, _ = oracle.route_topk(torch.from_numpy(L), k)
    got = oracle.index(idx, E, BM)
    c = got["counts"].numpy()
    assert c.sum() == T * k and c.min() >= 0 and c.max() <= T
    assert np.array_equal(got["offsets"].numpy(), np.concatenate([[0], np.cumsum(c)]))
    ros = got["row_of_slot"].numpy()
    assert len(set(ros.tolist())) == T * k                   # injective
    tor = got["token_of_row"].numpy()
    assert np.array_equal(tor[ros], np.repeat(np.arange(T), k))
    tile = got["tile_offsets"].numpy()
    ids = idx.numpy()
    for e in range(E):
        rows = tor[tile[e] * BM: tile[e] * BM + c[e]]
        assert np.all(np.diff(rows) > 0)                      # stable: strictly increasing tokens
        assert np.all(tor[tile[e] * BM + c[e]: tile[e + 1] * BM] == -1)
        assert np.all((ids[rows] == e).any(1))
    assert np.all([len(set(row)) == k for row in ids.tolist()])


def test_forced_uniform_routing_counts_exact():
    w = moe_inputs.small(T=512, d=16, E=16, k=4, f=16, routing="uniform", dtype="f32")
    L = moe_inputs.make_logits(w)
    idx, _ = oracle.route_topk(L, w.k)
    got = oracle.index(idx, w.E, 128)
    assert got["counts"].tolist() == [w.T * w.k // w.E] * w.E


def test_zipf_routing_is_skewed_toward_low_ids():
    w = moe_inputs.small(T=4096, d=16, E=16, k=2, f=16, routing="zipf", alpha=1.2, dtype="f32")
    idx, _ = oracle.route_topk(moe_inputs.make_logits(w), w.k)
    c = oracle.index(idx, w.E, 1)["counts"].numpy()
    assert c[0] > 3 * c[-1]


# ----------------------------------------------------------------------------- expert FFN -------

def _swiglu_ffn_numpy(x, wg, wu, wd):
    """Textbook SwiGLU FFN: (silu(x Wg^T) * (x Wu^T)) Wd^T, with scipy's logistic function."""
    a = x @ wg.T
    b = x @ wu.T
    return (a * expit(a) * b) @ wd.T


def test_single_expert_is_plain_swiglu_ffn():
    r = _rng(9)
    T, d, f = 12, 10, 6
    x = r.standard_normal((T, d))
    wgu = r.standard_normal((1, 2 * f, d)) * 0.3
    wd = r.standard_normal((1, d, f)) * 0.3
    idx, w = oracle.route_topk(torch.zeros((T, 1), dtype=torch.float32), 1)
    got = oracle.moe_tokens(torch.from_numpy(x), idx, w, torch.from_numpy(wgu), torch.from_numpy(wd))["out"].numpy()
    ref = _swiglu_ffn_numpy(x, wgu[0, :f], wgu[0, f:], wd[0])
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-14)
    swapped = _swiglu_ffn_numpy(x, wgu[0, f:], wgu[0, :f], wd[0])  # gate/up swapped must differ
    assert np.abs(swapped - ref).max() > 1e-3


def test_dense_routing_is_softmax_mixture():
    r = _rng(10)
    T, d, f, E = 9, 8, 5, 4
    x = r.standard_normal((T, d))
    L = r.standard_normal((T, E)).astype(np.float32)
    wgu = r.standard_normal((E, 2 * f, d)) * 0.3
    wd = r.standard_normal((E, d, f)) * 0.3
    idx, w = oracle.route_topk(torch.from_numpy(L), E)
    got = oracle.moe_tokens(torch.from_numpy(x), idx, w, torch.from_numpy(wgu), torch.from_numpy(wd))["out"].numpy()
    p = softmax(L.astype(np.float64), axis=1)
    ref = sum(p[:, [e]] * _swiglu_ffn_numpy(x, wgu[e, :f], wgu[e, f:], wd[e]) for e in range(E))
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-14)


def _tiny_f64(seed=11, T=4, d=8, E=4, k=2, f=8, gap=0.5):
    """Tiny fp64 problem whose top-k margin is at least `gap` (so small perturbations keep S_t)."""
    r = _rng(seed)
    while True:
        L = r.standard_normal((T, E)) * 2
        s = -np.sort(-L, axis=1)
        if np.all(s[:, k - 1] - s[:, k] > gap):
            break
    return dict(x=r.standard_normal((T, d)), L=L, wgu=r.standard_normal((E, 2 * f, d)) * 0.5,
                wd=r.standard_normal((E, d, f)) * 0.5, g=r.standard_normal((T, d)), k=k)


def _fwd(p):
    idx, w = oracle.route_topk(torch.from_numpy(p["L"]), p["k"])
    return oracle.moe_tokens(torch.from_numpy(p["x"]), idx, w, torch.from_numpy(p["wgu"]),
                             torch.from_numpy(p["wd"]))["out"].numpy()


def _loss(p):
    return float((_fwd(p) * p["g"]).sum())


def _fd(p, key, h=1e-5):
    base = p[key]
    grad = np.zeros_like(base)
    for i in np.ndindex(base.shape):
        q = dict(p)
        q[key] = base.copy()
        q[key][i] += h
        lp = _loss(q)
        q[key][i] -= 2 * h
        lm = _loss(q)
        grad[i] = (lp - lm) / (2 * h)
    return grad


def test_gradients_match_central_finite_differences():
    p = _tiny_f64()
    idx, w = oracle.route_topk(torch.from_numpy(p["L"]), p["k"])
    X, G = torch.from_numpy(p["x"]), torch.from_numpy(p["g"])
    Wgu, Wd = torch.from_numpy(p["wgu"]), torch.from_numpy(p["wd"])
    tok = oracle.moe_tokens(X, idx, w, Wgu, Wd, G)
    dwgu, dwd = oracle.moe_dweights(X, idx, w, Wgu, Wd, G)
    for key, got in (("x", tok["dx"].numpy()), ("L", tok["d_logits"].numpy()),
                     ("wgu", dwgu.numpy()), ("wd", dwd.numpy())):
        fd = _fd(p, key)
        err = np.abs(got - fd).max() / np.abs(fd).max()
        assert err < 1e-7, (key, err)


def test_d_topk_w_is_directional_derivative():
    """d_topk_w[t,j] = d loss / d w[t,j] = <g_t, y_{t,e_j}> (check by perturbing w directly)."""
    p = _tiny_f64(seed=12)
    idx, w = oracle.route_topk(torch.from_numpy(p["L"]), p["k"])
    args = (torch.from_numpy(p["x"]), idx)
    W = (torch.from_numpy(p["wgu"]), torch.from_numpy(p["wd"]))
    got = oracle.moe_tokens(*args, w, *W, torch.from_numpy(p["g"]))["d_topk_w"].numpy()
    h = 1e-6
    for t, j in itertools.product(range(w.shape[0]), range(w.shape[1])):
        wp, wm = w.clone(), w.clone()
        wp[t, j] += h
        wm[t, j] -= h
        lp = (oracle.moe_tokens(*args, wp, *W)["out"].numpy() * p["g"]).sum()
        lm = (oracle.moe_tokens(*args, wm, *W)["out"].numpy() * p["g"]).sum()
        assert abs((lp - lm) / (2 * h) - got[t, j]) < 1e-6 * max(1.0, abs(got[t, j]))


def test_zero_down_projection_gives_zero_output_and_logit_grad():
    p = _tiny_f64(seed=13)
    p["wd"][:] = 0.0
    idx, w = oracle.route_topk(torch.from_numpy(p["L"]), p["k"])
    X, G = torch.from_numpy(p["x"]), torch.from_numpy(p["g"])
    tok = oracle.moe_tokens(X, idx, w, torch.from_numpy(p["wgu"]), torch.from_numpy(p["wd"]), G)
    assert np.all(tok["out"].numpy() == 0) and np.all(tok["d_logits"].numpy() == 0)
    assert np.all(tok["dx"].numpy() == 0)
    dwgu, dwd = oracle.moe_dweights(X, idx, w, torch.from_numpy(p["wgu"]), torch.from_numpy(p["wd"]), G)
    assert np.all(dwgu.numpy() == 0) and np.abs(dwd.numpy()).max() > 0


def test_output_is_linear_in_down_projection():
    p = _tiny_f64(seed=14)
    o1 = _fwd(p)
    p2 = dict(p, wd=p["wd"] * 2.0)
    assert np.array_equal(_fwd(p2), 2.0 * o1)


def test_logit_gradient_sums_to_zero_per_token():
    """Softmax is shift invariant, so sum_e dL[t,e] = 0 (a dropped term in the closed form breaks it)."""
    p = _tiny_f64(seed=15, T=6, E=6, k=3)
    idx, w = oracle.route_topk(torch.from_numpy(p["L"]), p["k"])
    tok = oracle.moe_tokens(torch.from_numpy(p["x"]), idx, w, torch.from_numpy(p["wgu"]), torch.from_numpy(p["wd"]),
                            torch.from_numpy(p["g"]))
    np.testing.assert_allclose(tok["d_logits"].numpy().sum(1), 0.0, atol=1e-13)


def test_token_subset_and_entries_agree_with_full():
    p = _tiny_f64(seed=16, T=7, d=6, E=5, k=2, f=4)
    idx, w = oracle.route_topk(torch.from_numpy(p["L"]), p["k"])
    X, G = torch.from_numpy(p["x"]), torch.from_numpy(p["g"])
    Wgu, Wd = torch.from_numpy(p["wgu"]), torch.from_numpy(p["wd"])
    full = oracle.moe_tokens(X, idx, w, Wgu, Wd, G)
    sub = oracle.moe_tokens(X, idx, w, Wgu, Wd, G, tokens=[5, 0, 3])
    for key in ("out", "dx", "d_logits", "d_topk_w"):
        assert torch.equal(sub[key], full[key][[5, 0, 3]])
    dwgu, dwd = oracle.moe_dweights(X, idx, w, Wgu, Wd, G)
    mats, es, rs, cs, ref = [], [], [], [], []
    for e in range(5):
        for r, c in ((0, 1), (3, 5), (7, 0)):
            mats.append(0), es.append(e), rs.append(r), cs.append(c), ref.append(float(dwgu[e, r, c]))
        for r, c in ((0, 0), (5, 3)):
            mats.append(1), es.append(e), rs.append(r), cs.append(c), ref.append(float(dwd[e, r, c]))
    val = oracle.dweight_entries(X, idx, w, Wgu, Wd, G, mats, es, rs, cs).numpy()
    np.testing.assert_allclose(val, ref, rtol=1e-12, atol=1e-15)


def test_worked_example_closed_form():
    with open(os.path.join(GOLDEN, "worked_example.json")) as fh:
        ex = json.load(fh)
    env = {"ln3": math.log(3.0), "__builtins__": {}}
    inp = {k: np.array(eval(v, env), dtype=np.float64) for k, v in ex["inputs"].items() if k != "k"}
    exp = {k: np.array(eval(v, env), dtype=np.float64) for k, v in ex["expected"].items()}
    k = int(ex["inputs"]["k"])
    idx, w = oracle.route_topk(torch.from_numpy(inp["logits"]), k)
    assert idx.tolist() == exp["topk_idx"].astype(int).tolist()
    np.testing.assert_allclose(w.numpy(), exp["topk_w"], rtol=1e-15)
    X, G = torch.from_numpy(inp["x"]), torch.from_numpy(inp["g"])
    Wgu, Wd = torch.from_numpy(inp["w_gate_up"]), torch.from_numpy(inp["w_down"])
    tok = oracle.moe_tokens(X, idx, w, Wgu, Wd, G)
    dwgu, dwd = oracle.moe_dweights(X, idx, w, Wgu, Wd, G)
    for key, got in (("out", tok["out"]), ("d_topk_w", tok["d_topk_w"]), ("d_logits", tok["d_logits"]),
                     ("dx", tok["dx"]), ("dw_gate_up", dwgu), ("dw_down", dwd)):
        np.testing.assert_allclose(got.numpy(), exp[key], rtol=1e-13, atol=1e-15, err_msg=key)


def test_bf16_inputs_are_read_exactly():
    """The oracle widens stored bf16 exactly: feeding bf16 or its fp64 widening gives identical results."""
    w = moe_inputs.small(T=16, d=16, E=4, k=2, f=16, dtype="bf16")
    inp = moe_inputs.make_all(w)
    idx, wt = oracle.route_topk(inp["logits"], w.k)
    a = oracle.moe_tokens(inp["x"], idx, wt, inp["w_gate_up"], inp["w_down"], inp["g"])
    b = oracle.moe_tokens(inp["x"].double(), idx, wt, inp["w_gate_up"].double(), inp["w_down"].double(),
                          inp["g"].double())
    for key in a:
        assert torch.equal(a[key], b[key])
