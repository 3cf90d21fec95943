"""Step pipeline for a dynamic table: the lookup-or-insert of step t+1 (and
the expiry of step t) on a low-priority side stream while step t's work --
the caller's dense network and emb_backward_update -- runs on a
higher-priority main stream (RecIS §3.3, the PRE_FORWARD stage of the next
step on its own stream).  Host orchestration only: every step of the path
runs in the library's kernels; nothing here reads embedding values ahead of
time (the lookup hands out row numbers and initialises newly admitted rows).

Per step t (lag = 1 when ttl >= 1, else 0):
    main:  wait L(t) -> emb_forward(t) -> record F(t) -> [dense work] -> backward(t)
    side:  wait F(t - lag) -> expiry(t) -> lookup-or-insert(t+1) -> record L(t+1)
With lag 1 the next lookup also overlaps this step's forward; the row
numbers alternate between two buffers.

The result is the sequential one (lookup, forward, backward, expiry per
step):
  * expiry(t) removes keys with t - last_seen > ttl.  Rows the main stream
    may still use belong to keys of steps t - lag .. t (everything older
    finished before F(t - lag)); their last_seen is >= t - lag >= t - ttl,
    so none of them is freed;
  * lookup(t+1) only changes slot metadata, which the forward and backward
    never read, and initialises rows that were free after expiry(t), which
    no key in use holds; it writes the buffer forward(t - 1) read, and
    forward(t - 1) finished before F(t - lag);
  * forward(t+1) follows backward(t) on the main stream, so it reads the
    updated weights; the side stream stays at most lag + 1 steps ahead.
"""
from __future__ import annotations


class DynamicPipeline:
    """Pipelined steps over a HashTable and a training Plan whose columns are
    rows_given over the table's row pool.  Call per step:
    ``forward(t, offsets, out)``, then ``prefetch(t + 1, table_ids, keys)``
    (when there is a next step), the caller's dense work on ``main``, then
    ``backward(grad_out, lr, eps)``; ``finish()`` after the last step.
    Each call first orders its stream after the caller's current stream, so
    inputs produced there before the call are ready."""

    def __init__(self, table, plan, ttl, batch, max_keys, device="cuda"):
        import torch
        self.table, self.plan, self.ttl, self.batch = table, plan, ttl, batch
        self.main = torch.cuda.Stream(device=device, priority=-1)
        self.side = torch.cuda.Stream(device=device, priority=0)
        self.lag = 1 if ttl >= 1 else 0
        self.rows = [torch.empty(max(max_keys, 1), dtype=torch.int64, device=device) for _ in range(2)]
        self._looked = None          # (step, n, event) of the last queued lookup
        self._fwd_events = [None, None]   # completions of the last two forwards (older first)
        self._evict_step = None      # step whose expiry is still to be queued

    def prefetch(self, step, table_ids, keys):
        """Queue expiry of the previous step and lookup-or-insert of `step` on
        the side stream, after the previous step's forward."""
        import torch
        n = keys.numel()
        self.side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(self.side):
            gate = self._fwd_events[1 - self.lag]   # F(step - 1 - lag)
            if gate is not None:
                self.side.wait_event(gate)
            if self._evict_step is not None:
                self.table.evict_expired(self._evict_step, self.ttl, stream=self.side)
                self._evict_step = None
            self.table.lookup_or_insert(table_ids, keys, step, rows_out=self.rows[step % 2][:n],
                                        stream=self.side)
            ev = torch.cuda.Event()
            ev.record(self.side)
        self._looked = (step, n, ev)

    def forward(self, step, offsets, out, rows_copy=None, events=None):
        """emb_forward of `step` on the main stream, over the rows its queued
        lookup produces; rows_copy (optional) receives the step's row numbers
        (the next lookup overwrites the pipeline's own buffer); events
        (optional start, end CUDA events) are recorded around the launch."""
        import torch
        if self._looked is None or self._looked[0] != step:
            raise RuntimeError("prefetch(step, ...) must be queued before forward(step)")
        _, n, ev = self._looked
        self.main.wait_stream(torch.cuda.current_stream())
        self.main.wait_event(ev)
        rows = self.rows[step % 2][:n]
        if events is not None:
            events[0].record(self.main)
        self.plan.forward(self.batch, rows, offsets, None, None, out=out, stream=self.main)
        if events is not None:
            events[1].record(self.main)
        if rows_copy is not None:
            with torch.cuda.stream(self.main):
                rows_copy[:n].copy_(rows)
        f = torch.cuda.Event()
        f.record(self.main)
        self._fwd_events = [self._fwd_events[1], f]
        self._evict_step = step

    def backward(self, grad_out, lr, eps):
        import torch
        self.main.wait_stream(torch.cuda.current_stream())
        self.plan.backward_update(grad_out, None, lr, eps, stream=self.main)

    def finish(self):
        """Queue the last expiry and make the caller's current stream wait for
        both streams."""
        import torch
        if self._evict_step is not None:
            with torch.cuda.stream(self.side):
                if self._fwd_events[1] is not None:
                    self.side.wait_event(self._fwd_events[1])
                self.table.evict_expired(self._evict_step, self.ttl, stream=self.side)
            self._evict_step = None
        cur = torch.cuda.current_stream()
        cur.wait_stream(self.main)
        cur.wait_stream(self.side)
