"""Seeded synthetic inputs for one MoE layer (routing logits, tokens, expert weights, output gradient).

This module only draws tensors. It holds none of the layer's arithmetic (no top-k, no softmax, no
expert FFN) and imports neither the CUDA package nor the oracle: both sides are fed the same bytes
from here, so a parity test compares the two implementations on identical inputs.

Workloads (the shapes of the MoE layers the source pages train; their per-layer sizes are not
printed there, so these are the synthetic stand-ins):

  tiny_f32        T=256   d=64   E=8   k=2 f=128  fp32  fwd+bwd  logits ~ N(0,1)
  fwd_t4096       T=4096  d=2048 E=64  k=8 f=1024 bf16  fwd      logits = x . W_r, W_r ~ N(0,0.02)
  fwdbwd_t8192    T=8192  d=2048 E=64  k=8 f=1024 bf16  fwd+bwd  as above
  skew_a0/.8/1.2  T=16384 d=2048 E=64  k=8 f=1024 bf16  fwd+bwd  forced-uniform / Zipf(0.8) / Zipf(1.2)
  large_a0.8      T=16384 d=4096 E=128 k=8 f=1536 bf16  fwd+bwd  Zipf(0.8)
  large_shape_e16 T=2048  d=4096 E=16  k=8 f=1536 bf16  fwd+bwd  Zipf(0.8)  (profiling stand-in for large_a0.8)

Expert weights ~ N(0, 0.02), tokens x ~ N(0, 1), grad_out ~ N(0, 1). bf16 tensors are drawn in
fp32 and rounded to nearest-even bf16; the rounded values are the inputs both sides see.

Skewed routing ("Scalable Pretraining of Large MoE LMs on Aurora", brief, section 局限与风险,
names forced uniform routing; the Zipf construction is this library's reading):
  Zipf(alpha):   L[t,e] = -alpha * ln(e+1) + G[t,e], G ~ Gumbel(0,1). By the Gumbel-top-k property
                 the top-k of a row is a draw of k experts without replacement with P(e) ~ (e+1)^-alpha.
  forced uniform: S_t = {(t*k + j) mod E : j < k}; L[t,e] = G[t,e] + 30 [e in S_t]. Each expert then
                 receives exactly T*k/E rows. Rows whose selected minimum does not clear the
                 unselected maximum are redrawn (a plain min/max comparison).
"""
from __future__ import annotations

import dataclasses
import math

import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    T: int
    d: int
    E: int
    k: int
    f: int
    dtype: str          # "f32" or "bf16": storage type of x, weights, grad_out and the layer outputs
    backward: bool
    routing: str        # "normal" | "router" | "zipf" | "uniform"
    alpha: float = 0.0
    seed: int = 0

    @property
    def torch_dtype(self):
        return torch.float32 if self.dtype == "f32" else torch.bfloat16

    def describe(self):
        return dataclasses.asdict(self)


WORKLOADS = {
    "tiny_f32": Workload("tiny_f32", 256, 64, 8, 2, 128, "f32", True, "normal"),
    "fwd_t4096": Workload("fwd_t4096", 4096, 2048, 64, 8, 1024, "bf16", False, "router"),
    "fwdbwd_t8192": Workload("fwdbwd_t8192", 8192, 2048, 64, 8, 1024, "bf16", True, "router"),
    "skew_a0": Workload("skew_a0", 16384, 2048, 64, 8, 1024, "bf16", True, "uniform"),
    "skew_a0.8": Workload("skew_a0.8", 16384, 2048, 64, 8, 1024, "bf16", True, "zipf", 0.8),
    "skew_a1.2": Workload("skew_a1.2", 16384, 2048, 64, 8, 1024, "bf16", True, "zipf", 1.2),
    "large_a0.8": Workload("large_a0.8", 16384, 4096, 128, 8, 1536, "bf16", True, "zipf", 0.8),
    # large_a0.8's per-expert shapes (d, f, k, Zipf(0.8), about 1,024 rows per expert) on 16 experts:
    # a case small enough (about 1.5 GB) for multi-pass profiler captures of the same kernels
    "large_shape_e16": Workload("large_shape_e16", 2048, 4096, 16, 8, 1536, "bf16", True, "zipf", 0.8),
}

# Each tensor has its own stream so that drawing one never shifts another.
_STREAM = {"x": 1, "logits": 2, "router": 3, "wgu": 4, "wd": 5, "g": 6, "redraw": 7}


def _gen(device, seed, name):
    g = torch.Generator(device=device)
    g.manual_seed(seed * 1000 + _STREAM[name])
    return g


def _normal(shape, std, dtype, device, seed, name):
    t = torch.randn(shape, generator=_gen(device, seed, name), device=device, dtype=torch.float32)
    if std != 1.0:
        t.mul_(std)
    return t.to(dtype)


def _gumbel(shape, device, gen):
    u = torch.rand(shape, generator=gen, device=device, dtype=torch.float64)
    u.clamp_(min=1e-300)
    return -torch.log(-torch.log(u))


def make_logits(w: Workload, device="cpu", x=None):
    """Router logits [T, E] fp32 (see the module docstring for each routing recipe)."""
    T, E, k = w.T, w.E, w.k
    if w.routing == "normal":
        return _normal((T, E), 1.0, torch.float32, device, w.seed, "logits")
    if w.routing == "router":
        if x is None:
            x = make_x(w, device)
        wr = _normal((w.d, E), 0.02, w.torch_dtype, device, w.seed, "router")
        return (x.to(torch.float64) @ wr.to(torch.float64)).to(torch.float32)
    gen = _gen(device, w.seed, "logits")
    G = _gumbel((T, E), device, gen)
    if w.routing == "zipf":
        bias = -w.alpha * torch.log(torch.arange(1, E + 1, device=device, dtype=torch.float64))
        return (G + bias).to(torch.float32)
    if w.routing == "uniform":
        t = torch.arange(T, device=device).unsqueeze(1)
        sel = (t * k + torch.arange(k, device=device).unsqueeze(0)) % E          # [T, k]
        mask = torch.zeros((T, E), dtype=torch.bool, device=device)
        mask.scatter_(1, sel, True)
        L = G + 30.0 * mask
        regen = _gen(device, w.seed, "redraw")
        for _ in range(100):
            Lf = L.to(torch.float32)
            lo = torch.where(mask, Lf, torch.full_like(Lf, math.inf)).amin(1)
            hi = torch.where(mask, torch.full_like(Lf, -math.inf), Lf).amax(1)
            bad = lo <= hi
            if not bool(bad.any()):
                return Lf
            nb = int(bad.sum())
            L[bad] = _gumbel((nb, E), device, regen) + 30.0 * mask[bad]
        raise RuntimeError("forced-uniform logits: redraw did not converge")
    raise ValueError(w.routing)


def make_router_weight(w: Workload, device="cpu"):
    """Router weight W_r [E, d] (row e scores expert e), ~ N(0, 0.02): the same draw that the
    "router" logits recipe multiplies by, stored transposed (L = x W_r^T)."""
    return _normal((w.d, w.E), 0.02, w.torch_dtype, device, w.seed, "router").t().contiguous()


def make_x(w: Workload, device="cpu"):
    return _normal((w.T, w.d), 1.0, w.torch_dtype, device, w.seed, "x")


def make_weights(w: Workload, device="cpu"):
    """w_gate_up [E, 2f, d] (rows 0..f-1 gate, f..2f-1 up) and w_down [E, d, f], ~ N(0, 0.02)."""
    wgu = _normal((w.E, 2 * w.f, w.d), 0.02, w.torch_dtype, device, w.seed, "wgu")
    wd = _normal((w.E, w.d, w.f), 0.02, w.torch_dtype, device, w.seed, "wd")
    return wgu, wd


def make_grad_out(w: Workload, device="cpu"):
    return _normal((w.T, w.d), 1.0, w.torch_dtype, device, w.seed, "g")


def make_all(w: Workload, device="cpu"):
    """Every input of one layer pass: dict with x, logits, w_gate_up, w_down and (if backward) g."""
    x = make_x(w, device)
    out = {"x": x, "logits": make_logits(w, device, x)}
    out["w_gate_up"], out["w_down"] = make_weights(w, device)
    if w.backward:
        out["g"] = make_grad_out(w, device)
    return out


def small(name="small", T=300, d=256, E=8, k=2, f=256, dtype="bf16", routing="normal", alpha=0.0,
          seed=0, backward=True):
    """A workload of arbitrary (test) size with the same recipes."""
    return Workload(name, T, d, E, k, f, dtype, backward, routing, alpha, seed)
