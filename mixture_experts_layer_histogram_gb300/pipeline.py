"""Host-buffer pipeline: layer passes fed from, and returned to, pinned host memory.

Each step copies the pass's inputs (x, logits -- or none on a router layer, which computes them
from x --, and grad_out for a training pass) from host to device, runs the layer through the C ABI, and copies the per-token results (out, and dx, d_logits
for a training pass) back to host memory. The copies run on two streams of their own and overlap
the neighbouring steps' compute: step i+1's inputs are uploaded while step i computes, and step
i's results are downloaded while step i+1 computes. Device inputs and the layer's result tensors
rotate over `depth` slots, so a copy never touches memory that a running kernel reads or writes;
events order every reuse of a slot. Each slot's pass is recorded once into a CUDA graph (on its
first step, and again whenever the weight tensors change) and replayed, so a step costs the host
one launch instead of one per kernel.

    pipe = HostPipeline(layer)
    for i, batch in enumerate(batches):      # dicts of pinned host tensors: x, logits (and g)
        step = pipe.submit(batch, w_gate_up, w_down, next_batch=batches[i + 1] if i + 1 < len(batches) else None)
        ...                                  # step.wait(), then read step.tensors before depth more steps run
"""
from __future__ import annotations

import torch


class StepResult:
    """Pinned host result tensors of one step and the event that marks their arrival. The tensors
    belong to a slot that the pipeline reuses `depth` steps later."""

    def __init__(self, tensors, event):
        self.tensors = tensors
        self.event = event

    def wait(self):
        self.event.synchronize()
        return self.tensors


class HostPipeline:
    def __init__(self, layer, depth=2, graphs=True):
        """graphs: replay each slot's pass from a CUDA graph (False: launch the kernels one by one)."""
        self.layer = layer
        self.graphs = graphs
        self._graph = [None] * depth     # per slot: (weight pointers, graph)
        self.backward = layer.backward_enabled
        self.depth = depth
        dev = layer.device
        self.compute = torch.cuda.current_stream(dev)
        self.h2d = torch.cuda.Stream(dev)
        self.d2h = torch.cuda.Stream(dev)
        T, d, E = layer.T, layer.d, layer.E
        act = dict(dtype=layer.dtype, device=dev)
        f32 = dict(dtype=torch.float32, device=dev)
        self.inputs = []
        self.results = []
        for _ in range(depth):
            inp = dict(x=torch.empty((T, d), **act))
            if not layer.router:
                inp["logits"] = torch.empty((T, E), **f32)
            res = dict(out=torch.empty((T, d), **act))
            if self.backward:
                inp["g"] = torch.empty((T, d), **act)
                res["dx"] = torch.empty((T, d), **act)
                res["d_logits"] = torch.empty((T, E), **f32)
            self.inputs.append(inp)
            self.results.append(res)
        self.host_out = [{k: torch.empty(v.shape, dtype=v.dtype).pin_memory() for k, v in r.items()}
                         for r in self.results]
        self.in_free = [torch.cuda.Event() for _ in range(depth)]     # compute has finished reading the slot's inputs
        self.in_ready = [torch.cuda.Event() for _ in range(depth)]    # the slot's inputs are uploaded
        self.res_ready = [torch.cuda.Event() for _ in range(depth)]   # the slot's results are written
        self.res_free = [torch.cuda.Event() for _ in range(depth)]    # the slot's results are downloaded
        for s in range(depth):
            self.in_free[s].record(self.compute)
            self.res_free[s].record(self.compute)
        self.done = self.res_free[0]
        self.n_run = 0
        self.pending = []

    def h2d_bytes(self):
        return sum(v.numel() * v.element_size() for v in self.inputs[0].values())

    def d2h_bytes(self):
        return sum(v.numel() * v.element_size() for v in self.host_out[0].values())

    def upload(self, batch):
        """Enqueue the host->device copy of a step's inputs; call it one step ahead to overlap."""
        if len(self.pending) >= self.depth:
            raise RuntimeError("every input slot already holds an uploaded step")
        s = (self.n_run + len(self.pending)) % self.depth
        self.h2d.wait_event(self.in_free[s])
        with torch.cuda.stream(self.h2d):
            for k, dst in self.inputs[s].items():
                dst.copy_(batch[k], non_blocking=True)
        self.in_ready[s].record(self.h2d)
        self.pending.append(s)

    def run(self, w_gate_up, w_down, w_router=None):
        """Compute the oldest uploaded step and enqueue the download of its results (w_router: the
        router weights of a router layer)."""
        s = self.pending.pop(0)
        inp, res, lay = self.inputs[s], self.results[s], self.layer
        self.compute.wait_event(self.in_ready[s])
        self.compute.wait_event(self.res_free[s])
        lay.out = res["out"]
        if self.backward:
            lay.dx, lay.d_logits = res["dx"], res["d_logits"]
        if self.graphs:
            key = (w_gate_up.data_ptr(), w_down.data_ptr(), None if w_router is None else w_router.data_ptr())
            if self._graph[s] is None or self._graph[s][0] != key:
                with torch.cuda.stream(self.compute):   # the capture's warm-up passes follow the waits above
                    graph = lay.capture(inp["x"], inp.get("logits"), w_gate_up, w_down,
                                        grad_out=inp["g"] if self.backward else None, w_router=w_router)
                self._graph[s] = (key, graph)
            with torch.cuda.stream(self.compute):
                self._graph[s][1].replay()
        else:
            lay.forward(inp["x"], inp.get("logits"), w_gate_up, w_down, self.compute, w_router=w_router)
            if self.backward:
                lay.backward(inp["g"], w_gate_up, w_down, self.compute)
        self.in_free[s].record(self.compute)
        self.res_ready[s].record(self.compute)
        self.d2h.wait_event(self.res_ready[s])
        with torch.cuda.stream(self.d2h):
            for k, v in res.items():
                self.host_out[s][k].copy_(v, non_blocking=True)
        ev = torch.cuda.Event()
        ev.record(self.d2h)
        self.res_free[s] = ev
        self.done = ev
        self.n_run += 1
        return StepResult(self.host_out[s], ev)

    def submit(self, batch, w_gate_up, w_down, next_batch=None, w_router=None):
        """One step: upload `batch` unless it is already uploaded, enqueue the upload of `next_batch`
        (if given) so that it overlaps this step's compute, then run this step."""
        if not self.pending:
            self.upload(batch)
        if next_batch is not None:
            self.upload(next_batch)
        return self.run(w_gate_up, w_down, w_router)

    def join(self, stream=None):
        """Make `stream` (default: the compute stream) wait for every enqueued copy."""
        stream = stream or self.compute
        stream.wait_stream(self.h2d)
        stream.wait_stream(self.d2h)

    def wait(self):
        """Block the host until the last run step's results are in host memory."""
        self.done.synchronize()
