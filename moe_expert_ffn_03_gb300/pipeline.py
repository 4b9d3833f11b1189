"""Steps of an ExpertFFN fed from pinned host memory, with the copies overlapped.

A step's inputs (x, logits and, for training, dout) arrive from pinned host
buffers and its results (out and, for training, dx) go back to pinned host
buffers.  The copies run on two streams of their own, one per direction (the
GPU has separate copy engines for each), while the kernels run on the compute
stream:

  input stream    H2D inputs[i+1] -> slot (i+1)%2
  output stream                                        D2H out[i]     D2H dx[i]
  compute stream  step i on slot i%2 ............ combine_out ..... combine_dx

* Two device slots hold the inputs, so the next step's inputs land while this
  step computes.  A slot is refilled only after the step that read it has run
  its backward (or its forward, without training).
* A step quantizes its weights before it waits for its inputs (the weights are
  already on the device), and its forward waits only for x and logits: dout has
  an event of its own and is awaited by the backward.  So the inputs of a step
  whose predecessor left no time to copy them (the first one) land under work.
* out and dx are single device buffers.  A step's combine waits until the
  previous step's copy of that buffer has left the device, so a result is
  never overwritten before it is read out.

All ordering is by CUDA events; the host never waits inside ``run``.
"""
from __future__ import annotations

import torch


class HostPipeline:
    def __init__(self, layer, w_gu, w_d, stream: torch.cuda.Stream | None = None):
        self.L = layer
        self.w_gu, self.w_d = w_gu, w_d
        self.train = layer.training
        dev = layer.ws.device
        self.compute = stream if stream is not None else torch.cuda.current_stream(dev)
        self.copy_in = torch.cuda.Stream(dev)
        self.copy_out = torch.cuda.Stream(dev)
        T, H, E = layer.T, layer.H, layer.E
        names = ("x", "logits", "dout") if self.train else ("x", "logits")
        shapes = {"x": ((T, H), torch.bfloat16), "logits": ((T, E), torch.float32),
                  "dout": ((T, H), torch.bfloat16)}
        self.names = names
        self.slots = [{n: torch.empty(shapes[n][0], dtype=shapes[n][1], device=dev) for n in names}
                      for _ in range(2)]
        ev = lambda: torch.cuda.Event()                                 # noqa: E731
        self.landed = [ev(), ev()]        # H2D of a slot's x and logits finished
        self.landed_dout = [ev(), ev()]   # H2D of a slot's dout finished (training)
        self.released = [ev(), ev()]      # the compute stream is done reading a slot
        self.out_done, self.dx_done = ev(), ev()        # a result is complete on the device
        self.out_copied, self.dx_copied = ev(), ev()    # a result has left the device
        self._first = True

    def _h2d(self, slot: int, host: dict, wait_release: bool):
        with torch.cuda.stream(self.copy_in):
            if wait_release:
                self.copy_in.wait_event(self.released[slot])
            for n in ("x", "logits"):
                self.slots[slot][n].copy_(host[n], non_blocking=True)
            self.landed[slot].record(self.copy_in)
            if self.train:
                self.slots[slot]["dout"].copy_(host["dout"], non_blocking=True)
                self.landed_dout[slot].record(self.copy_in)

    def run(self, host_inputs: list, host_outputs: list, after: torch.cuda.Event | None = None):
        """One step per entry of host_inputs (dicts of pinned tensors named x, logits[,
        dout]); step i's out (and dx) are copied into host_outputs[i] (dicts of pinned
        tensors named out[, dx]).  Both copy streams first wait for `after` if given.
        Returns without waiting; synchronize (or join()) before reading the results."""
        n = len(host_inputs)
        if n == 0:
            return
        L, st = self.L, self.compute
        if after is not None:
            self.copy_in.wait_event(after)
            self.copy_out.wait_event(after)
        self._h2d(0, host_inputs[0], wait_release=not self._first)
        for i in range(n):
            s = i % 2
            if i + 1 < n:
                self._h2d(1 - s, host_inputs[i + 1], wait_release=not self._first or i >= 1)
            inp = self.slots[s]
            L.quantize_weights(self.w_gu, self.w_d, st)
            st.wait_event(self.landed[s])
            L.route(inp["logits"], inp["x"], st)
            L.ffn_forward(st)
            if not self._first or i > 0:
                st.wait_event(self.out_copied)
            L.combine_out(st)
            self.out_done.record(st)
            if self.train:
                st.wait_event(self.landed_dout[s])
                L.ffn_backward(inp["dout"], st)
                self.released[s].record(st)
                if not self._first or i > 0:
                    st.wait_event(self.dx_copied)
                L.combine_dx(st)
                self.dx_done.record(st)
            else:
                self.released[s].record(st)
            with torch.cuda.stream(self.copy_out):
                self.copy_out.wait_event(self.out_done)
                host_outputs[i]["out"].copy_(L.out, non_blocking=True)
                self.out_copied.record(self.copy_out)
                if self.train:
                    self.copy_out.wait_event(self.dx_done)
                    host_outputs[i]["dx"].copy_(L.dx, non_blocking=True)
                    self.dx_copied.record(self.copy_out)
        self._first = False

    def join(self):
        """Make the compute stream wait for every copy issued so far."""
        for st in (self.copy_in, self.copy_out):
            e = torch.cuda.Event()
            e.record(st)
            self.compute.wait_event(e)
