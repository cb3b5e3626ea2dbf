"""fp64 CPU oracle of one MoE layer (routing, counting/indexing, expert SwiGLU FFNs, combine; fwd + bwd).

TEST INFRASTRUCTURE. Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` use this package. It shares no code with the CUDA library and imports nothing from it.

The arithmetic lives in ``moe_oracle.c`` (plain loops, fp64, OpenMP over tokens or experts); this
module compiles it with gcc on first use and marshals torch/numpy buffers. Every function states
the definition it computes in the C source; the short form:

  route_topk      S_t = top-k of L[t,:] by (value desc, id asc); w = softmax over the selected logits
  index           counts, offsets (exclusive scan), tile_offsets (exclusive scan of ceil(counts/BM)),
                  row_of_slot (expert e's rows start at tile_offsets[e]*BM, stable in slot order),
                  token_of_row (-1 on padding rows)
  moe_tokens      out_t = sum_{e in S_t} w_te * Wd[e] (silu(Wg[e] x_t) * (Wu[e] x_t)), and with g:
                  dw, d_logits (softmax backward on S_t), dx_t
  moe_dweights    dW_gate_up, dW_down summed over all tokens
  dweight_entries selected dW entries, each summed over the tokens routed to its expert
  router_logits   L[t,e] = sum_c x[t,c] Wr[e,c]   (the router before the selection)
  router_dx       dx_r[t,c] = sum_e dL[t,e] Wr[e,c];  router_dw  dWr[e,c] = sum_t dL[t,e] x[t,c]

Parity pins (tests/test_oracle_*.py): brute-force index/top-k on tiny inputs, invariants, the E=1/k=1
reduction to a plain SwiGLU FFN, dense routing k=E, W_down=0, equal logits, forced-uniform counts,
central finite differences for every gradient, and a hand-derived worked example (tests/golden).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

F32, BF16, F64 = 0, 1, 2


def build(force=False):
    """Compile liboracle.so with gcc (plain C, OpenMP). Portable flags only: the same source builds on x86_64 and aarch64."""
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    subprocess.check_call(["gcc", "-O3", "-fopenmp", "-fPIC", "-shared", "-std=c11", "-o", tmp, _SRC, "-lm"])
    os.replace(tmp, _LIB)
    return _LIB


def lib():
    global _lib
    with _lock:
        if _lib is None:
            build()
            L = ctypes.CDLL(_LIB)
            P, I, I64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64
            L.oracle_num_threads.restype = I
            L.oracle_route_topk.argtypes = [P, I, I, I, I, P, P]
            L.oracle_index.argtypes = [P, I, I, I, I, P, P, P, P, P, I64]
            L.oracle_moe_tokens.argtypes = [I, I, I, I, I, P, I, P, P, P, P, I, P, I, P, I64, P, P, P, P, P]
            L.oracle_moe_dweights.argtypes = [I, I, I, I, I, P, I, P, P, P, P, I, P, I, P, P]
            L.oracle_moe_dweight_entries.argtypes = [I, I, I, I, I, P, I, P, P, P, P, I, P, I, I64, P, P, P, P, P]
            L.oracle_router_logits.argtypes = [I, I, I, P, I, P, I, P, I64, P]
            L.oracle_router_dx.argtypes = [I, I, I, P, I, P, I, P, I64, P]
            L.oracle_router_dw.argtypes = [I, I, I, P, I, P, I, P, I64, P]
            for fn in ("oracle_route_topk", "oracle_index", "oracle_moe_tokens", "oracle_moe_dweights",
                       "oracle_moe_dweight_entries", "oracle_router_logits", "oracle_router_dx", "oracle_router_dw"):
                getattr(L, fn).restype = I
            _lib = L
    return _lib


def num_threads():
    return lib().oracle_num_threads()


def _cpu(t):
    """Contiguous CPU tensor (torch) from a torch tensor or numpy array, plus its oracle dtype code."""
    if isinstance(t, np.ndarray):
        t = torch.from_numpy(np.ascontiguousarray(t))
    t = t.detach().to("cpu").contiguous()
    code = {torch.float32: F32, torch.bfloat16: BF16, torch.float64: F64}.get(t.dtype)
    return t, code


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else None


def _check(rc, what):
    if rc != 0:
        raise RuntimeError(f"oracle {what} failed with code {rc}")


def route_topk(logits, k):
    L, ldt = _cpu(logits)
    T, E = L.shape
    idx = torch.empty((T, k), dtype=torch.int32)
    w = torch.empty((T, k), dtype=torch.float64)
    _check(lib().oracle_route_topk(_ptr(L), ldt, T, E, k, _ptr(idx), _ptr(w)), "route_topk")
    return idx, w


def index(topk_idx, E, BM, rows_cap=None):
    idx, _ = _cpu(topk_idx.to(torch.int32) if isinstance(topk_idx, torch.Tensor) else topk_idx)
    T, k = idx.shape
    if rows_cap is None:
        rows_cap = rows_max(T, k, E, BM)
    counts = torch.empty(E, dtype=torch.int32)
    offsets = torch.empty(E + 1, dtype=torch.int32)
    tile_offsets = torch.empty(E + 1, dtype=torch.int32)
    row_of_slot = torch.empty(T * k, dtype=torch.int32)
    token_of_row = torch.empty(rows_cap, dtype=torch.int32)
    _check(lib().oracle_index(_ptr(idx), T, k, E, BM, _ptr(counts), _ptr(offsets), _ptr(tile_offsets),
                              _ptr(row_of_slot), _ptr(token_of_row), rows_cap), "index")
    return dict(counts=counts, offsets=offsets, tile_offsets=tile_offsets, row_of_slot=row_of_slot,
                token_of_row=token_of_row)


def rows_max(T, k, E, BM):
    """Upper bound on the padded grouped row count: sum_e ceil(c_e/BM)*BM <= T*k + E*(BM-1)."""
    return ((T * k + E * (BM - 1) + BM - 1) // BM) * BM


def moe_tokens(x, idx, w, w_gate_up, w_down, g=None, tokens=None, want_y=False):
    """Forward (+ token-side backward if g is given) for the listed tokens (all if None). fp64 outputs."""
    X, xdt = _cpu(x)
    T, d = X.shape
    Wgu, wdt = _cpu(w_gate_up)
    Wd, wdt2 = _cpu(w_down)
    assert wdt == wdt2
    E, twof, _ = Wgu.shape
    f = twof // 2
    I, _ = _cpu(idx.to(torch.int32))
    k = I.shape[1]
    W, _ = _cpu(w.to(torch.float64))
    G, gdt = (_cpu(g) if g is not None else (None, 0))
    if tokens is None:
        tok = None
        n = T
    else:
        tok = torch.as_tensor(tokens, dtype=torch.int64).contiguous()
        n = tok.numel()
    out = torch.empty((n, d), dtype=torch.float64)
    y = torch.empty((n, k, d), dtype=torch.float64) if want_y else None
    dx = torch.empty((n, d), dtype=torch.float64) if G is not None else None
    dl = torch.empty((n, E), dtype=torch.float64) if G is not None else None
    dw = torch.empty((n, k), dtype=torch.float64) if G is not None else None
    _check(lib().oracle_moe_tokens(T, d, E, k, f, _ptr(X), xdt, _ptr(I), _ptr(W), _ptr(Wgu), _ptr(Wd), wdt,
                                   _ptr(G), gdt, _ptr(tok), n, _ptr(out), _ptr(y), _ptr(dx), _ptr(dl), _ptr(dw)),
           "moe_tokens")
    res = dict(out=out)
    if want_y:
        res["y"] = y
    if G is not None:
        res.update(dx=dx, d_logits=dl, d_topk_w=dw)
    return res


def moe_dweights(x, idx, w, w_gate_up, w_down, g):
    X, xdt = _cpu(x)
    T, d = X.shape
    Wgu, wdt = _cpu(w_gate_up)
    Wd, _ = _cpu(w_down)
    E, twof, _ = Wgu.shape
    f = twof // 2
    I, _ = _cpu(idx.to(torch.int32))
    k = I.shape[1]
    W, _ = _cpu(w.to(torch.float64))
    G, gdt = _cpu(g)
    dwgu = torch.empty((E, 2 * f, d), dtype=torch.float64)
    dwd = torch.empty((E, d, f), dtype=torch.float64)
    _check(lib().oracle_moe_dweights(T, d, E, k, f, _ptr(X), xdt, _ptr(I), _ptr(W), _ptr(Wgu), _ptr(Wd), wdt,
                                     _ptr(G), gdt, _ptr(dwgu), _ptr(dwd)), "moe_dweights")
    return dwgu, dwd


def dweight_entries(x, idx, w, w_gate_up, w_down, g, mat, e, r, c):
    X, xdt = _cpu(x)
    T, d = X.shape
    Wgu, wdt = _cpu(w_gate_up)
    Wd, _ = _cpu(w_down)
    E, twof, _ = Wgu.shape
    f = twof // 2
    I, _ = _cpu(idx.to(torch.int32))
    k = I.shape[1]
    W, _ = _cpu(w.to(torch.float64))
    G, gdt = _cpu(g)
    cols = [torch.as_tensor(v, dtype=torch.int32).contiguous() for v in (mat, e, r, c)]
    n = cols[0].numel()
    val = torch.empty(n, dtype=torch.float64)
    _check(lib().oracle_moe_dweight_entries(T, d, E, k, f, _ptr(X), xdt, _ptr(I), _ptr(W), _ptr(Wgu), _ptr(Wd),
                                            wdt, _ptr(G), gdt, n, *[_ptr(v) for v in cols], _ptr(val)),
           "dweight_entries")
    return val


def _tokens(tokens, T):
    if tokens is None:
        return None, T
    tok = torch.as_tensor(tokens, dtype=torch.int64).contiguous()
    return tok, tok.numel()


def router_logits(x, w_router, tokens=None):
    """L = x Wr^T for the listed tokens (all if None); Wr is [E, d]. fp64 [n, E]."""
    X, xdt = _cpu(x)
    Wr, wdt = _cpu(w_router)
    T, d = X.shape
    E = Wr.shape[0]
    tok, n = _tokens(tokens, T)
    out = torch.empty((n, E), dtype=torch.float64)
    _check(lib().oracle_router_logits(T, d, E, _ptr(X), xdt, _ptr(Wr), wdt, _ptr(tok), n, _ptr(out)), "router_logits")
    return out


def router_dx(d_logits, w_router, tokens=None):
    """dx_r = dL Wr for the listed tokens (all if None). fp64 [n, d]."""
    DL, dldt = _cpu(d_logits)
    Wr, wdt = _cpu(w_router)
    T, E = DL.shape
    d = Wr.shape[1]
    tok, n = _tokens(tokens, T)
    out = torch.empty((n, d), dtype=torch.float64)
    _check(lib().oracle_router_dx(T, d, E, _ptr(DL), dldt, _ptr(Wr), wdt, _ptr(tok), n, _ptr(out)), "router_dx")
    return out


def router_dw(x, d_logits, cols=None):
    """dWr = dL^T x for the listed columns of Wr (all if None). fp64 [E, ncols]."""
    X, xdt = _cpu(x)
    DL, dldt = _cpu(d_logits)
    T, d = X.shape
    E = DL.shape[1]
    if cols is None:
        cl, nc = None, d
    else:
        cl = torch.as_tensor(cols, dtype=torch.int32).contiguous()
        nc = cl.numel()
    out = torch.empty((E, nc), dtype=torch.float64)
    _check(lib().oracle_router_dw(T, d, E, _ptr(X), xdt, _ptr(DL), dldt, _ptr(cl), nc, _ptr(out)), "router_dw")
    return out
