"""Parity of the CUDA path (through the C ABI) with the fp64 oracle, on seeded synthetic inputs.

Index tensors (topk_idx, counts, offsets, tile_offsets, row_of_slot, token_of_row) are compared
bit-exactly. Float outputs use max|gpu - oracle| / max|oracle| <= 1e-2 for bf16 layers and <= 1e-5
for fp32 layers. Small cases compare every element; the full-size workloads compare the complete
index path and a seeded sample of tokens (out, dx, d_logits, d_topk_w) and of weight-gradient
entries, each of which the oracle computes one by one.
"""
import numpy as np
import pytest
import torch

import moe_inputs
import oracle
from helpers import rel_err, tol_for

pytestmark = pytest.mark.gpu


def _run(w, inp=None, device="cuda"):
    from mixture_experts_layer_histogram_gb300 import MoELayer
    if inp is None:
        inp = moe_inputs.make_all(w, device)
    g = {k: v.to(device) for k, v in inp.items()}
    layer = MoELayer(w.T, w.d, w.E, w.k, w.f, w.torch_dtype, device, backward=w.backward)
    layer.forward(g["x"], g["logits"], g["w_gate_up"], g["w_down"])
    res = layer.backward(g["g"], g["w_gate_up"], g["w_down"]) if w.backward else None
    torch.cuda.synchronize()
    assert layer.status() == (0, 0)
    return layer, res, inp


def _check_index(layer, w, logits_cpu):
    idx, wt = oracle.route_topk(logits_cpu, w.k)
    assert torch.equal(layer.topk_idx.cpu(), idx), "topk_idx"
    ref = oracle.index(idx, w.E, 128, layer.rows_max)
    for key in ("counts", "offsets", "tile_offsets", "row_of_slot"):
        assert torch.equal(getattr(layer, key).cpu(), ref[key]), key
    used = int(ref["tile_offsets"][-1]) * 128
    assert torch.equal(layer.token_of_row.cpu()[:used], ref["token_of_row"][:used]), "token_of_row"
    return idx, wt, ref


SMALL = [
    moe_inputs.WORKLOADS["tiny_f32"],
    moe_inputs.small("bf16_ragged", T=1000, d=512, E=8, k=2, f=512),
    moe_inputs.small("bf16_many_experts", T=512, d=256, E=64, k=8, f=256, routing="zipf", alpha=1.2),
    moe_inputs.small("bf16_uniform", T=512, d=256, E=16, k=4, f=512, routing="uniform"),
    moe_inputs.small("bf16_single_expert", T=300, d=256, E=1, k=1, f=256),
    moe_inputs.small("f32_ragged", T=333, d=96, E=5, k=3, f=40, dtype="f32"),
    moe_inputs.small("bf16_max_experts_topk", T=512, d=256, E=256, k=16, f=256),    # E and k at the ABI maximum
    moe_inputs.small("f32_topk16", T=100, d=32, E=32, k=16, f=24, dtype="f32"),
]


@pytest.mark.parametrize("w", SMALL, ids=lambda w: w.name)
def test_layer_matches_oracle_small(w):
    layer, res, inp = _run(w)
    idx, wt, _ = _check_index(layer, w, inp["logits"])
    tol = tol_for(w.torch_dtype)
    assert rel_err(layer.topk_w, wt) <= 1e-6
    ref = oracle.moe_tokens(inp["x"], idx, wt, inp["w_gate_up"], inp["w_down"], inp["g"])
    dwgu, dwd = oracle.moe_dweights(inp["x"], idx, wt, inp["w_gate_up"], inp["w_down"], inp["g"])
    errs = {"out": rel_err(layer.out, ref["out"]), "dx": rel_err(res["dx"], ref["dx"]),
            "d_logits": rel_err(res["d_logits"], ref["d_logits"]),
            "d_topk_w": rel_err(res["d_topk_w"], ref["d_topk_w"]),
            "dw_gate_up": rel_err(res["dw_gate_up"], dwgu), "dw_down": rel_err(res["dw_down"], dwd)}
    bad = {k: v for k, v in errs.items() if not v <= tol}
    assert not bad, (bad, errs)


def test_expert_outputs_per_row_match_oracle():
    """y_perm row of (token t, slot j) equals the oracle's y_{t, e_j} (checks the grouping end to end)."""
    w = moe_inputs.small("rows", T=400, d=256, E=8, k=2, f=256)
    layer, _, inp = _run(w)
    idx, wt = oracle.route_topk(inp["logits"], w.k)
    ref = oracle.moe_tokens(inp["x"], idx, wt, inp["w_gate_up"], inp["w_down"], want_y=True)
    rows = layer.row_of_slot.cpu().long().view(w.T, w.k)
    y = layer.y_perm.cpu()[rows.view(-1)].view(w.T, w.k, w.d)
    assert rel_err(y, ref["y"]) <= 1e-2


def test_permute_is_exact_copy_and_padding_is_zero():
    w = moe_inputs.small("perm", T=777, d=256, E=16, k=4, f=256, routing="zipf", alpha=0.8, backward=False)
    layer, _, inp = _run(w)
    xp = layer.x_perm.cpu()
    ros = layer.row_of_slot.cpu().long()
    assert torch.equal(xp[ros], inp["x"].cpu().repeat_interleave(w.k, 0))
    tor = layer.token_of_row.cpu()
    used = int(layer.tile_offsets[-1]) * 128
    pad = (tor[:used] < 0).nonzero().view(-1)
    assert torch.all(xp[pad] == 0)


def test_repeat_runs_are_bitwise_identical():
    w = moe_inputs.small("det", T=2048, d=256, E=32, k=4, f=256, routing="zipf", alpha=0.8)
    l1, r1, inp = _run(w)
    used = int(l1.tile_offsets[-1]) * 128          # rows past the groups are never written
    snap = {k: getattr(l1, k).clone() for k in ("row_of_slot", "out", "counts", "tile_offsets")}
    snap["token_of_row"] = l1.token_of_row[:used].clone()
    snap.update({k: v.clone() for k, v in r1.items()})
    l2, r2, _ = _run(w, inp)
    for k in ("row_of_slot", "out", "counts", "tile_offsets"):
        assert torch.equal(getattr(l2, k), snap[k]), k
    assert torch.equal(l2.token_of_row[:used], snap["token_of_row"])
    for k, v in r2.items():
        assert torch.equal(v, snap[k]), k


@pytest.mark.parametrize("T,E,k,routing,alpha", [
    (1, 8, 2, "normal", 0.0), (5, 256, 16, "normal", 0.0), (1023, 7, 3, "normal", 0.0), (1025, 1, 1, "normal", 0.0),
    (16384, 64, 8, "uniform", 0.0), (16384, 64, 8, "zipf", 1.2), (16384, 128, 8, "zipf", 0.8),
    (40000, 256, 16, "zipf", 0.5)])
def test_index_path_bit_exact(T, E, k, routing, alpha):
    from mixture_experts_layer_histogram_gb300 import _lib as L
    w = moe_inputs.small("idx", T=T, d=16, E=E, k=k, f=16, routing=routing, alpha=alpha, dtype="f32")
    logits = moe_inputs.make_logits(w)
    dev = "cuda"
    R = L.moe_grouped_rows_max(T, k, E)
    idx = torch.empty((T, k), dtype=torch.int32, device=dev)
    wt = torch.empty((T, k), dtype=torch.float32, device=dev)
    L.moe_route_topk(logits.to(dev), k, idx, wt)
    outs = dict(counts=torch.empty(E, dtype=torch.int32, device=dev),
                offsets=torch.empty(E + 1, dtype=torch.int32, device=dev),
                tile_offsets=torch.empty(E + 1, dtype=torch.int32, device=dev),
                row_of_slot=torch.empty(T * k, dtype=torch.int32, device=dev),
                token_of_row=torch.full((R,), -7, dtype=torch.int32, device=dev))
    ws = torch.full((L.moe_count_index_workspace_size(T, k, E),), 0, dtype=torch.uint8, device=dev)
    L.moe_count_index(idx, E, outs["counts"], outs["offsets"], outs["tile_offsets"], outs["row_of_slot"],
                      outs["token_of_row"], ws)
    torch.cuda.synchronize()
    assert L.moe_read_status(ws) == 0
    ridx, rw = oracle.route_topk(logits, k)
    assert torch.equal(idx.cpu(), ridx)
    assert rel_err(wt, rw) <= 1e-6
    ref = oracle.index(ridx, E, 128, R)
    for key in ("counts", "offsets", "tile_offsets", "row_of_slot"):
        assert torch.equal(outs[key].cpu(), ref[key]), key
    used = int(ref["tile_offsets"][-1]) * 128
    assert torch.equal(outs["token_of_row"].cpu()[:used], ref["token_of_row"][:used])
    assert torch.all(outs["token_of_row"].cpu()[used:] == -7)      # rows past the groups are untouched
    if routing == "uniform":
        assert torch.all(outs["counts"].cpu() == T * k // E)


def test_route_topk_ties_and_signed_zero():
    from mixture_experts_layer_histogram_gb300 import _lib as L
    r = np.random.default_rng(3)
    vals = np.array([-1.0, -0.0, 0.0, 0.5, 2.0], dtype=np.float32)
    for E, k in ((8, 2), (64, 8), (100, 7), (256, 16), (33, 16)):
        logits = torch.from_numpy(vals[r.integers(0, len(vals), size=(500, E))])
        idx = torch.empty((500, k), dtype=torch.int32, device="cuda")
        wt = torch.empty((500, k), dtype=torch.float32, device="cuda")
        L.moe_route_topk(logits.cuda(), k, idx, wt)
        ridx, rw = oracle.route_topk(logits, k)
        assert torch.equal(idx.cpu(), ridx), (E, k)
        assert rel_err(wt, rw) <= 1e-6


def test_bad_expert_index_reports_status_without_writing_out_of_bounds():
    from mixture_experts_layer_histogram_gb300 import _lib as L
    T, k, E = 300, 2, 8
    idx = torch.randint(0, E, (T, k), dtype=torch.int32, device="cuda")
    idx[17, 1] = E + 3
    idx[200, 0] = -1
    R = L.moe_grouped_rows_max(T, k, E)
    o = [torch.empty(E, dtype=torch.int32, device="cuda"), torch.empty(E + 1, dtype=torch.int32, device="cuda"),
         torch.empty(E + 1, dtype=torch.int32, device="cuda"), torch.empty(T * k, dtype=torch.int32, device="cuda"),
         torch.empty(R, dtype=torch.int32, device="cuda")]
    ws = torch.zeros(L.moe_count_index_workspace_size(T, k, E), dtype=torch.uint8, device="cuda")
    L.moe_count_index(idx, E, *o, ws)
    assert L.moe_read_status(ws) == -5
    ros = o[3].cpu()
    assert ros[17 * k + 1] == -1 and ros[200 * k] == -1
    assert int(o[0].sum()) == T * k - 2
    # the workspace is reusable: a clean call reports OK again
    idx[17, 1] = 0
    idx[200, 0] = 1
    L.moe_count_index(idx, E, *o, ws)
    assert L.moe_read_status(ws) == 0


def test_lookback_wait_is_bounded_and_reported():
    """A scan block that withholds its prefix (fault hook) makes its successor's bounded wait run out:
    the call returns MOE_ERR_DEVICE_TIMEOUT in well under a second and the context stays usable."""
    import time
    from mixture_experts_layer_histogram_gb300 import _lib as L
    T, k, E = 8192, 8, 64      # 64 scan blocks
    idx = torch.randint(0, E, (T, k), dtype=torch.int32, device="cuda")
    R = L.moe_grouped_rows_max(T, k, E)
    o = [torch.empty(E, dtype=torch.int32, device="cuda"), torch.empty(E + 1, dtype=torch.int32, device="cuda"),
         torch.empty(E + 1, dtype=torch.int32, device="cuda"), torch.empty(T * k, dtype=torch.int32, device="cuda"),
         torch.empty(R, dtype=torch.int32, device="cuda")]
    ws = torch.zeros(L.moe_count_index_workspace_size(T, k, E), dtype=torch.uint8, device="cuda")
    hook = L.moe_count_index_hook_offset(E)
    ws[hook:hook + 4].view(torch.int32).fill_(5 + 1)      # block 5 withholds
    torch.cuda.synchronize()
    t0 = time.time()
    L.moe_count_index(idx, E, *o, ws)
    st = L.moe_read_status(ws)
    dt = time.time() - t0
    assert st == -4 and dt < 5.0
    assert int(ws[hook:hook + 4].view(torch.int32).item()) == 0          # the hook is consumed
    L.moe_count_index(idx, E, *o, ws)                                      # and the next call is clean
    assert L.moe_read_status(ws) == 0
    ridx = idx.cpu()
    ref = oracle.index(ridx, E, 128, R)
    assert torch.equal(o[3].cpu(), ref["row_of_slot"])


# ----------------------------------------------------------------------------- full sizes -------

FULL = ["fwd_t4096", "fwdbwd_t8192", "skew_a0", "skew_a0.8", "skew_a1.2", "large_a0.8"]


@pytest.mark.parametrize("name", FULL)
def test_full_size_workloads_sampled(name):
    w = moe_inputs.WORKLOADS[name]
    inp = moe_inputs.make_all(w, "cuda")
    layer, res, _ = _run(w, inp)
    cpu = {k: v.cpu() for k, v in inp.items()}
    idx, wt, ref_idx = _check_index(layer, w, cpu["logits"])
    if w.routing == "uniform":
        assert torch.all(layer.counts.cpu() == w.T * w.k // w.E)
    assert rel_err(layer.topk_w, wt) <= 1e-6
    gen = np.random.default_rng(1234)
    tokens = np.sort(gen.choice(w.T, size=96, replace=False))
    ref = oracle.moe_tokens(cpu["x"], idx, wt, cpu["w_gate_up"], cpu["w_down"], cpu.get("g"), tokens=tokens)
    tok = torch.from_numpy(tokens)
    errs = {"out": rel_err(layer.out.cpu()[tok], ref["out"])}
    if w.backward:
        errs.update(dx=rel_err(res["dx"].cpu()[tok], ref["dx"]),
                    d_logits=rel_err(res["d_logits"].cpu()[tok], ref["d_logits"]),
                    d_topk_w=rel_err(res["d_topk_w"].cpu()[tok], ref["d_topk_w"]))
        # sampled weight-gradient entries: the most and least loaded experts plus random ones
        counts = layer.counts.cpu().numpy()
        experts = sorted(set([int(counts.argmax()), int(counts.argmin())] + gen.choice(w.E, 4, replace=False).tolist()))
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
