"""One MoE layer's expert computation on one GPU: resident buffers and the call sequence.

Forward (one stream, no host synchronisation):
  moe_route_count_index  logits [T,E]  -> topk_idx [T,k], topk_w [T,k], counts, offsets, tile_offsets,
                                          row_of_slot, token_of_row   (routing + counting + indexing)
   (or, given router weights: moe_router_fwd  x, w_router [E,d] -> logits, topk_idx, topk_w, then
    moe_count_index  topk_idx -> counts, offsets, tile_offsets, row_of_slot, token_of_row)
  moe_permute      x [T,d]             -> x_perm [rows_max,d]
  moe_grouped_ffn_fwd                  -> ab [rows_max,2f], h [rows_max,f], y_perm [rows_max,d]
   (gather=True: no moe_permute and no x_perm; moe_grouped_ffn_fwd_gather reads x [T,d] through
    token_of_row, and the backward's moe_grouped_ffn_bwd_gather does the same)
  moe_combine_fwd  y_perm, topk_w      -> out [T,d]
Backward:
  moe_combine_bwd  grad_out            -> dy_perm, d_topk_w [T,k], d_logits [T,E]
  moe_grouped_ffn_bwd                  -> dab, dx_perm, dw_gate_up [E,2f,d], dw_down [E,d,f]
  moe_combine_fwd  dx_perm, w = NULL   -> dx [T,d]      (backward of the permutation)
  moe_router_bwd   d_logits            -> dx += d_logits w_router, dw_router [E,d]   (router layers)

Every step runs in libmoe's kernels; this module only allocates buffers (PyTorch device memory)
and calls the C ABI in order.
"""
from __future__ import annotations

import torch

from . import _lib as L


class MoELayer:
    """Buffers of one layer pass, allocated once and reused every step (no allocation per step)."""

    def __init__(self, T, d, E, k, f, dtype=torch.bfloat16, device="cuda", backward=True, recompute=False,
                 scratch=None, router=False, gather=False):
        """recompute: the backward recomputes ab and h from x_perm instead of reading them (selective
        activation checkpointing); ab and h may then live in `scratch` (a dict with tensors "ab" [R, 2f]
        and "h" [R, f] shared with other layers).
        router: the layer computes its logits from x and router weights (forward(..., w_router=W_r)),
        and its backward adds the router's share to dx and returns dw_router.
        gather: the permutation is fused into the grouped GEMMs' token loads (x_perm is never formed;
        the backward reads the x passed to forward, which must stay unchanged until then)."""
        if not torch.cuda.is_available():
            raise RuntimeError("MoELayer needs a CUDA device")
        self.T, self.d, self.E, self.k, self.f = T, d, E, k, f
        self.dtype = dtype
        self.device = torch.device(device)
        self.rows_max = L.moe_grouped_rows_max(T, k, E)
        R = self.rows_max
        i32 = dict(dtype=torch.int32, device=self.device)
        act = dict(dtype=dtype, device=self.device)
        self.topk_idx = torch.empty((T, k), **i32)
        self.topk_w = torch.empty((T, k), dtype=torch.float32, device=self.device)
        self.counts = torch.empty(E, **i32)
        self.offsets = torch.empty(E + 1, **i32)
        self.tile_offsets = torch.empty(E + 1, **i32)
        self.row_of_slot = torch.empty(T * k, **i32)
        self.token_of_row = torch.empty(R, **i32)
        self.ws_index = torch.zeros(L.moe_count_index_workspace_size(T, k, E), dtype=torch.uint8, device=self.device)
        self.ws_ffn = torch.zeros(L.moe_grouped_ffn_workspace_size(E, d, f, R, L.dtype_code(dtype), backward),
                                  dtype=torch.uint8, device=self.device)
        self.gather = gather
        self.x_perm = None if gather else torch.empty((R, d), **act)
        self._xin = None
        self.recompute = recompute
        if scratch is not None:
            self.ab, self.h = scratch["ab"], scratch["h"]
        else:
            self.ab = torch.empty((R, 2 * f), **act)
            self.h = torch.empty((R, f), **act)
        self.y_perm = torch.empty((R, d), **act)
        self.out = torch.empty((T, d), **act)
        self.backward_enabled = backward
        self.router = router
        self._x = self._w_router = None
        if router:
            self.logits = torch.empty((T, E), dtype=torch.float32, device=self.device)
            self.ws_router = torch.zeros(L.moe_router_workspace_size(T, d, E, L.dtype_code(dtype)), dtype=torch.uint8,
                                         device=self.device)
            if backward:
                self.dw_router = torch.empty((E, d), **act)
        if backward:
            self.dy_perm = torch.empty((R, d), **act)
            self.dab = torch.empty((R, 2 * f), **act)
            self.dx_perm = torch.empty((R, d), **act)
            self.dx = torch.empty((T, d), **act)
            self.d_topk_w = torch.empty((T, k), dtype=torch.float32, device=self.device)
            self.d_logits = torch.empty((T, E), dtype=torch.float32, device=self.device)
            self.dw_gate_up = torch.empty((E, 2 * f, d), **act)
            self.dw_down = torch.empty((E, d, f), **act)

    def forward(self, x, logits, w_gate_up, w_down, stream=None, w_router=None):
        """logits [T, E] fp32, or None with w_router [E, d] on a router layer (logits = x w_router^T,
        fused with the top-k selection)."""
        if w_router is not None:
            if not self.router or logits is not None:
                raise ValueError("w_router needs a layer built with router=True and logits=None")
            L.moe_router_fwd(x, w_router, self.k, self.logits, self.topk_idx, self.topk_w, self.ws_router, stream)
            self._x, self._w_router = x, w_router
            L.moe_count_index(self.topk_idx, self.E, self.counts, self.offsets, self.tile_offsets,
                              self.row_of_slot, self.token_of_row, self.ws_index, stream)
        else:   # routing, counting and index generation in one launch
            L.moe_route_count_index(logits, self.k, self.topk_idx, self.topk_w, self.counts, self.offsets,
                                    self.tile_offsets, self.row_of_slot, self.token_of_row, self.ws_index, stream)
            self._x = self._w_router = None
        # a and b are stored only for a backward that reads them (not for a forward-only layer, nor for
        # the recomputing backward, which forms them again)
        ab = self.ab if self.backward_enabled and not self.recompute else None
        if self.gather:
            self._xin = x
            L.moe_grouped_ffn_fwd_gather(x, self.token_of_row, w_gate_up, w_down, self.tile_offsets, self.offsets,
                                         ab, self.h, self.y_perm, self.ws_ffn, stream)
        else:
            L.moe_permute(x, self.k, self.E, self.row_of_slot, self.counts, self.tile_offsets, self.x_perm, stream)
            L.moe_grouped_ffn_fwd(self.x_perm, w_gate_up, w_down, self.tile_offsets, self.offsets, ab, self.h,
                                  self.y_perm, self.ws_ffn, stream)
        L.moe_combine_fwd(self.y_perm, self.topk_w, self.row_of_slot, self.T, self.k, self.out, stream)
        return self.out

    def backward(self, grad_out, w_gate_up, w_down, stream=None):
        if not self.backward_enabled:
            raise RuntimeError("layer was built without backward buffers")
        L.moe_combine_bwd(grad_out, self.y_perm, self.topk_w, self.topk_idx, self.row_of_slot, self.counts,
                          self.tile_offsets, self.E, self.dy_perm, self.d_topk_w, self.d_logits, stream)
        if self.gather:
            bwd = L.moe_grouped_ffn_bwd_recompute_gather if self.recompute else L.moe_grouped_ffn_bwd_gather
            bwd(self.dy_perm, self._xin, self.token_of_row, self.ab, self.h, w_gate_up, w_down, self.tile_offsets,
                self.offsets, self.dab, self.dx_perm, self.dw_gate_up, self.dw_down, self.ws_ffn, stream)
        else:
            bwd = L.moe_grouped_ffn_bwd_recompute if self.recompute else L.moe_grouped_ffn_bwd
            bwd(self.dy_perm, self.x_perm, self.ab, self.h, w_gate_up, w_down, self.tile_offsets, self.offsets,
                self.dab, self.dx_perm, self.dw_gate_up, self.dw_down, self.ws_ffn, stream)
        L.moe_combine_fwd(self.dx_perm, None, self.row_of_slot, self.T, self.k, self.dx, stream)
        res = dict(dx=self.dx, d_logits=self.d_logits, d_topk_w=self.d_topk_w, dw_gate_up=self.dw_gate_up,
                   dw_down=self.dw_down)
        if self._w_router is not None:
            L.moe_router_bwd(self._x, self._w_router, self.d_logits, self.dx, self.dw_router, self.ws_router,
                             accumulate_dx=True, stream=stream)
            res["dw_router"] = self.dw_router
        return res

    def capture(self, x, logits, w_gate_up, w_down, grad_out=None, w_router=None):
        """Record one pass (forward, and backward when grad_out is given) on these tensors into a
        CUDA graph and return it; graph.replay() re-runs the whole pass on whatever the tensors hold
        then, with one launch from the host instead of one per kernel. The call runs the pass
        twice on a side stream first (the library's one-time set-up happens outside the capture)."""
        def step():
            self.forward(x, logits, w_gate_up, w_down, w_router=w_router)
            if grad_out is not None:
                self.backward(grad_out, w_gate_up, w_down)
        side = torch.cuda.Stream(self.device)
        side.wait_stream(torch.cuda.current_stream(self.device))
        with torch.cuda.stream(side):
            for _ in range(2):
                step()
        torch.cuda.current_stream(self.device).wait_stream(side)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            step()
        return graph

    def status(self, stream=None):
        """Device status words (synchronises): (count_index, grouped_ffn), plus the router's on a router layer."""
        st = (L.moe_read_status(self.ws_index, stream), L.moe_read_status(self.ws_ffn, stream))
        return st + (L.moe_read_status(self.ws_router, stream),) if self.router else st

    # kernels launched per pass, for the bench's launch count
    def launches(self, backward=True):
        if self._w_router is not None:
            index = 1 + 2                     # router GEMM with top-k, count, index
        else:                                 # one fused kernel while its blocks fit at once (2 per SM)
            sms = torch.cuda.get_device_properties(self.device).multi_processor_count
            index = 1 if -(-self.T * self.k // 1024) <= 2 * sms else 3
        fwd = index + (0 if self.gather else 1) + 2 + 1
        bwd = 1 + 4 + 1 + (1 if self.recompute else 0)
        if self._w_router is not None:
            bwd += 4   # prep, dx GEMM, dW GEMM, reduce
        return fwd + (bwd if backward else 0)
