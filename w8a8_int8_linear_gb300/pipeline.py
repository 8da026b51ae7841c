"""Host-to-host W8A8 Linear over a sequence of batches.

A caller whose activations live in (pinned) host memory pays a host -> device
copy of every batch and a device -> host copy of every result.  `HostPipeline`
overlaps them with the Linear itself: three CUDA streams (copy in, compute,
copy out) and `depth` device buffers per side, so while batch i runs its
Linear, batch i+1 is being copied in and the result of batch i-1 copied out.
Each batch still makes its own two copies; only their order in time changes.
Every kernel is the library's (the Linear runs on the compute stream through
the C ABI); PyTorch provides the streams, events and copies.
"""
import torch


class HostPipeline:
    """Run `fn(X_dev, Y_dev)` (a W8A8 Linear writing Y_dev from X_dev on the
    current stream) over host batches xs[i] -> ys[i].

    x_shape / y_shape: the per-batch shapes; dtype bf16.  Host tensors should
    be pinned for the copies to be asynchronous.  `fn` may also take the batch
    index as a third argument (fn(X, Y, i)), e.g. to pick a weight copy."""

    def __init__(self, fn, x_shape, y_shape, device=None, depth=2, pass_index=False):
        if depth < 1:
            raise ValueError("depth must be >= 1")
        self.fn = fn
        self.pass_index = pass_index
        self.device = torch.device(device if device is not None else "cuda")
        self.depth = depth
        self.xd = [torch.empty(x_shape, dtype=torch.bfloat16, device=self.device) for _ in range(depth)]
        self.yd = [torch.empty(y_shape, dtype=torch.bfloat16, device=self.device) for _ in range(depth)]
        self.s_in = torch.cuda.Stream(device=self.device)
        self.s_comp = torch.cuda.Stream(device=self.device)
        self.s_out = torch.cuda.Stream(device=self.device)
        self.in_done = [torch.cuda.Event() for _ in range(depth)]
        self.comp_done = [torch.cuda.Event() for _ in range(depth)]
        self.out_done = [torch.cuda.Event() for _ in range(depth)]

    def run(self, xs, ys):
        """Enqueue every batch; returns without synchronizing.  The caller's
        current stream waits for all of it, so work queued there afterwards
        (an event, a synchronize) sees every result in ys."""
        if len(xs) != len(ys):
            raise ValueError("xs and ys must have the same length")
        caller = torch.cuda.current_stream(self.device)
        for s in (self.s_in, self.s_comp, self.s_out):
            s.wait_stream(caller)
        for i, (xh, yh) in enumerate(zip(xs, ys)):
            b = i % self.depth
            reuse = i >= self.depth
            with torch.cuda.stream(self.s_in):
                if reuse:  # the Linear of batch i - depth has read this input buffer
                    self.s_in.wait_event(self.comp_done[b])
                self.xd[b].copy_(xh, non_blocking=True)
                self.in_done[b].record(self.s_in)
            with torch.cuda.stream(self.s_comp):
                self.s_comp.wait_event(self.in_done[b])
                if reuse:  # the result of batch i - depth has left this output buffer
                    self.s_comp.wait_event(self.out_done[b])
                if self.pass_index:
                    self.fn(self.xd[b], self.yd[b], i)
                else:
                    self.fn(self.xd[b], self.yd[b])
                self.comp_done[b].record(self.s_comp)
            with torch.cuda.stream(self.s_out):
                self.s_out.wait_event(self.comp_done[b])
                yh.copy_(self.yd[b], non_blocking=True)
                self.out_done[b].record(self.s_out)
        for s in (self.s_in, self.s_comp, self.s_out):
            caller.wait_stream(s)
        # the device buffers are used on the side streams: keep the allocator
        # from handing them out again before that work is done
        for t in self.xd + self.yd:
            t.record_stream(self.s_in)
            t.record_stream(self.s_comp)
            t.record_stream(self.s_out)
        return ys
