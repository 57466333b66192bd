"""Forward + backward over logits that live in host memory.

Rows are independent and every row's bits are independent of the batch it is
computed in ("Batch-Invariance" section of the operator page), so a batch
can be cut into row chunks and streamed: while chunk i is computed, chunk i+1
is copied in and chunk i-1 is copied out, on three CUDA streams.  The result
is bit for bit the one-shot result.  Every computing step runs in the CUDA
library; the copies are asynchronous DMA from and to pinned host memory.
"""
from __future__ import annotations

import torch

from .logp import DEFAULT_TILE_V, IGNORE_INDEX, logp_bwd, logp_fwd


class HostStreamedLogp:
    """Reusable device buffers and streams for host-resident batches of one shape.

    ``run(...)`` takes pinned host tensors: logits [N, V], target_ids [N],
    grad_logp [N] (float32), and writes logp [N] (float32) and dlogits [N, V]
    back to pinned host tensors.  ``chunk_rows`` rows are in flight per stage;
    two chunks of device buffers are used in turn.
    """

    def __init__(self, n_rows: int, vocab: int, dtype: torch.dtype, dlogits_dtype: torch.dtype,
                 chunk_rows: int = 2048, device: torch.device | str = "cuda"):
        self.device = torch.device(device)
        self.n_rows, self.vocab, self.chunk = n_rows, vocab, max(1, min(chunk_rows, n_rows))
        dev = self.device
        self.x = [torch.empty(self.chunk, vocab, dtype=dtype, device=dev) for _ in range(2)]
        self.t = [torch.empty(self.chunk, dtype=torch.int64, device=dev) for _ in range(2)]
        self.g = [torch.empty(self.chunk, dtype=torch.float32, device=dev) for _ in range(2)]
        self.lp = [torch.empty(self.chunk, dtype=torch.float32, device=dev) for _ in range(2)]
        self.lse = [torch.empty(self.chunk, dtype=torch.float32, device=dev) for _ in range(2)]
        self.d = [torch.empty(self.chunk, vocab, dtype=dlogits_dtype, device=dev) for _ in range(2)]
        self.s_in = torch.cuda.Stream(dev)
        self.s_comp = torch.cuda.Stream(dev)
        self.s_out = torch.cuda.Stream(dev)
        # per chunk buffer, kept from one call to the next: its inputs have been
        # read by the kernels (computed) and its outputs copied out (drained)
        self._computed = [None, None]
        self._drained = [None, None]

    def run(self, logits_h: torch.Tensor, target_h: torch.Tensor, grad_h: torch.Tensor, logp_h: torch.Tensor,
            dlogits_h: torch.Tensor, ignore_index: int = IGNORE_INDEX, tile_v: int = DEFAULT_TILE_V,
            order_inputs: bool = True) -> int:
        """Queue the whole batch; returns the number of CUDA-library kernel launches queued.

        The caller's current stream waits for the last copy out.  With
        ``order_inputs`` (the default) the batch's copies and kernels also wait
        for the work already queued on the caller's stream, as if they ran on
        it.  ``order_inputs=False`` drops that wait, for host inputs that the
        CPU wrote (no queued work produces them): the next batch's copies in
        then overlap this batch's last copies out, and the chunk buffers are
        guarded by the pipeline's own events."""
        n, c = self.n_rows, self.chunk
        cur = torch.cuda.current_stream(self.device)
        if order_inputs:
            for s in (self.s_in, self.s_comp, self.s_out):
                s.wait_stream(cur)
        loaded = [None, None]      # event: chunk buffer b holds its inputs
        computed = self._computed  # event: chunk buffer b holds its outputs
        drained = self._drained    # event: chunk buffer b's outputs are copied out
        launches = 0
        for i, r0 in enumerate(range(0, n, c)):
            r1 = min(n, r0 + c)
            m = r1 - r0
            b = i % 2
            with torch.cuda.stream(self.s_in):
                if computed[b] is not None:
                    self.s_in.wait_event(computed[b])        # inputs of chunk i-2 no longer needed
                self.x[b][:m].copy_(logits_h[r0:r1], non_blocking=True)
                self.t[b][:m].copy_(target_h[r0:r1], non_blocking=True)
                self.g[b][:m].copy_(grad_h[r0:r1], non_blocking=True)
                loaded[b] = self.s_in.record_event()
            with torch.cuda.stream(self.s_comp):
                self.s_comp.wait_event(loaded[b])
                if drained[b] is not None:
                    self.s_comp.wait_event(drained[b])       # outputs of chunk i-2 copied out
                logp_fwd(self.x[b][:m], self.t[b][:m], ignore_index, tile_v, out=self.lp[b][:m],
                         lse=self.lse[b][:m])
                logp_bwd(self.x[b][:m], self.t[b][:m], self.lse[b][:m], self.g[b][:m], ignore_index,
                         out=self.d[b][:m])
                launches += 2
                computed[b] = self.s_comp.record_event()
            with torch.cuda.stream(self.s_out):
                self.s_out.wait_event(computed[b])
                logp_h[r0:r1].copy_(self.lp[b][:m], non_blocking=True)
                dlogits_h[r0:r1].copy_(self.d[b][:m], non_blocking=True)
                drained[b] = self.s_out.record_event()
        cur.wait_stream(self.s_out)
        return launches
