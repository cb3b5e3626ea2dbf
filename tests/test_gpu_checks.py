"""The debug build (libmoe_checks.so, -DMOE_CHECKS=1): the grouped-GEMM kernels check on the device
that every tile lies inside its expert's row group and inside the buffers, record
MOE_ERR_CHECK_FAILED when a check fails and skip the tile (no trap, nothing written outside the
buffers).

Each case runs in a child process with MOE_LIBRARY pointing at the debug build, so the release
library of this process is untouched. Valid layers of awkward shapes must report status 0 and give
the release build's results; offsets that contradict tile_offsets must be reported."""
import os
import subprocess
import sys
import textwrap

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run_with_checks(code):
    from mixture_experts_layer_histogram_gb300 import build
    lib = build.build(checks=True)
    env = dict(os.environ, MOE_LIBRARY=lib, PYTHONPATH=ROOT)
    r = subprocess.run([sys.executable, "-c", textwrap.dedent(code)], env=env, cwd=ROOT, capture_output=True,
                       text=True, timeout=600)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "libmoe_checks.so" in r.stdout, r.stdout
    return r.stdout


def test_debug_build_passes_awkward_valid_layers():
    out = _run_with_checks("""
        import torch, moe_inputs
        from mixture_experts_layer_histogram_gb300 import MoELayer, _lib as L
        print(L.LIB_PATH)
        cases = [moe_inputs.small("one_expert", T=300, d=256, E=1, k=1, f=256),
                 moe_inputs.small("empty_experts", T=200, d=256, E=64, k=2, f=256, routing="zipf", alpha=1.5),
                 moe_inputs.small("ragged", T=1000, d=512, E=8, k=2, f=512),
                 moe_inputs.small("f32", T=333, d=96, E=5, k=3, f=40, dtype="f32")]
        for w in cases:
            inp = moe_inputs.make_all(w, "cuda")
            counts = None
            for gather in (False, True):
                layer = MoELayer(w.T, w.d, w.E, w.k, w.f, w.torch_dtype, "cuda", gather=gather)
                layer.forward(inp["x"], inp["logits"], inp["w_gate_up"], inp["w_down"])
                layer.backward(inp["g"], inp["w_gate_up"], inp["w_down"])
                torch.cuda.synchronize()
                assert layer.status() == (0, 0), (w.name, gather, layer.status())
                counts = layer.counts.cpu()
            if w.name == "empty_experts":
                assert int((counts == 0).sum()) > 0
            print(w.name, "ok")
    """)
    assert out.count(" ok") == 4


def test_debug_build_reports_inconsistent_offsets():
    out = _run_with_checks("""
        import torch
        from mixture_experts_layer_histogram_gb300 import _lib as L
        print(L.LIB_PATH)
        E, d, f = 2, 256, 256
        R = 4 * 128
        dev = "cuda"
        x = torch.randn((R, d), device=dev).to(torch.bfloat16)
        wgu = (torch.randn((E, 2 * f, d), device=dev) * 0.05).to(torch.bfloat16)
        wd = (torch.randn((E, d, f), device=dev) * 0.05).to(torch.bfloat16)
        ab = torch.zeros((R, 2 * f), dtype=torch.bfloat16, device=dev)
        h = torch.zeros((R, f), dtype=torch.bfloat16, device=dev)
        y = torch.zeros((R, d), dtype=torch.bfloat16, device=dev)
        ws = torch.zeros(L.moe_grouped_ffn_workspace_size(E, d, f, R, 1, 1), dtype=torch.uint8, device=dev)
        # expert 0 claims 300 routed rows but owns one 128-row group: its tiles must be skipped
        toff = torch.tensor([0, 1, 2], dtype=torch.int32, device=dev)
        off = torch.tensor([0, 300, 350], dtype=torch.int32, device=dev)
        L.moe_grouped_ffn_fwd(x, wgu, wd, toff, off, ab, h, y, ws)
        assert L.moe_read_status(ws) == -6, L.moe_read_status(ws)
        assert torch.all(ab[:128] == 0) and torch.all(y[:128] == 0)        # nothing written for expert 0
        assert torch.any(y[128:178] != 0)                                  # expert 1 was computed
        # consistent offsets on a fresh status word: no report
        ws.zero_()
        off = torch.tensor([0, 100, 150], dtype=torch.int32, device=dev)
        L.moe_grouped_ffn_fwd(x, wgu, wd, toff, off, ab, h, y, ws)
        assert L.moe_read_status(ws) == 0
        # weight gradients over groups that run backwards (tile_offsets decreasing)
        ws.zero_()
        dab = torch.zeros((R, 2 * f), dtype=torch.bfloat16, device=dev)
        dx = torch.zeros((R, d), dtype=torch.bfloat16, device=dev)
        dwgu = torch.zeros((E, 2 * f, d), dtype=torch.bfloat16, device=dev)
        dwd = torch.zeros((E, d, f), dtype=torch.bfloat16, device=dev)
        bad_toff = torch.tensor([0, 2, 1], dtype=torch.int32, device=dev)
        L.moe_grouped_ffn_bwd(y, x, ab, h, wgu, wd, bad_toff, off, dab, dx, dwgu, dwd, ws)
        assert L.moe_read_status(ws) == -6
        print("reported ok")
    """)
    assert "reported ok" in out
