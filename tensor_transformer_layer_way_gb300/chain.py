"""Host bookkeeping of the GTP_remat prefetch chain (two gathered slots, a side stream, events).

Source: "Generalized Tensor Parallelism(GTP)是什么?" -- concept "Prefetch chain" and Fig. 1:
weights form a chain in forward order; while layer l's GEMM runs, layer l+1's all-gather is
already issued; the chain head's gather is exposed and the other L-1 are hidden; every
weight's first gather is synchronous (cold start); backward walks the chain in reverse with
layer l-1's gather beside layer l's dgrad; the wgrad reduce-scatter's finalize is deferred by
one backward layer and the last one is synchronous.

Only scheduling lives here: every gather, GEMM, reduce-scatter and finalize is a call into
the C library.  Slot k (k = layer parity) is reused every other layer, so a gather into it
first waits for the event recorded after the last GEMM that read it.
"""
from __future__ import annotations


class GtpChain:
    def __init__(self, ttl, torch, shards, slots):
        """``shards[l][j]``: layer l's GTP shard j ([K/g, N] bf16); ``slots``: two [K, N] buffers."""
        self.ttl = ttl
        self.torch = torch
        self.shards = shards
        self.slots = slots
        self.L = len(shards)
        self.side = torch.cuda.Stream()
        self.fin = torch.cuda.Stream()                         # deferred finalizes
        self.wg = torch.cuda.Stream()                          # weight gradients beside the dgrads
        self.ready = [torch.cuda.Event() for _ in range(2)]
        self.free = [torch.cuda.Event() for _ in range(2)]
        self.wgrad_done = [torch.cuda.Event() for _ in range(self.L)]

    def _gather_async(self, l, wait_free):
        k = l % 2
        with self.torch.cuda.stream(self.side):
            if wait_free:
                self.side.wait_event(self.free[k])
            self.ttl.gtp_gather(self.shards[l], self.slots[k], stream=self.side, done_event=self.ready[k])

    def forward(self, X, Y, *, cold=False, folded=False):
        """Y[l] = X W_l for every layer.  cold: each gather synchronous on the compute stream
        (first pass); folded: the gather is folded into the GEMM's operand loads."""
        ttl = self.ttl
        main = self.torch.cuda.current_stream()
        if folded:
            for l in range(self.L):
                ttl.gtp_gather_gemm(X, self.shards[l], Y[l])
            return
        if cold:
            for l in range(self.L):
                ttl.gtp_gather(self.shards[l], self.slots[l % 2], stream=main)
                ttl.gtp_gather_gemm(X, self.shards[l], Y[l], slot=self.slots[l % 2])
            return
        self.side.wait_stream(main)
        self._gather_async(0, wait_free=False)                  # chain head: exposed
        for l in range(self.L):
            if l + 1 < self.L:
                self._gather_async(l + 1, wait_free=True)       # AG(W_{l+1}) beside GEMM(W_l)
            main.wait_event(self.ready[l % 2])
            ttl.gtp_gather_gemm(X, self.shards[l], Y[l], slot=self.slots[l % 2])
            self.free[l % 2].record(main)

    def backward(self, X, dY, dX, staging, main_grad, *, folded=False, finalize_stream=True, wgrad_stream=True):
        """Reverse chain: dX = dY[l] W_l^T with the gather of layer l-1 beside it; the wgrad of
        layer l is reduce-scattered into staging[l] and finalized into main_grad[l] one backward
        layer later (layer 0 at once).  ``dX`` may be one buffer or a list per layer.

        With ``finalize_stream`` the deferred finalize of layer l+1 is issued at the start of
        backward step l on a stream of its own (after the event recorded behind layer l+1's
        weight gradient), so it runs beside step l's GEMMs instead of between them; the
        compute stream joins it before returning.  Otherwise it runs on the compute stream,
        inside the weight-gradient call of step l.

        With ``wgrad_stream`` (and ``finalize_stream``) the weight gradients run on a stream of
        their own: they depend only on X and dY, so layer l's weight gradient can fill the SMs
        that layer l-1's dgrad leaves idle in its last wave; the compute stream joins that
        stream before returning."""
        ttl = self.ttl
        main = self.torch.cuda.current_stream()
        L = self.L
        if finalize_stream:
            self.fin.wait_stream(main)
        wgs = wgrad_stream and finalize_stream
        if wgs:
            self.wg.wait_stream(main)                           # X and every dY[l] are ready
        if not folded:
            self.side.wait_stream(main)
            self._gather_async(L - 1, wait_free=False)          # head of the reverse chain
        for l in range(L - 1, -1, -1):
            prev = l + 1 if l + 1 < L else None
            if finalize_stream and prev is not None:
                self.fin.wait_event(self.wgrad_done[prev])
                ttl.gtp_finalize(staging[prev], main_grad[prev], stream=self.fin)
            out = dX[l] if isinstance(dX, (list, tuple)) else dX
            if folded:
                ttl.gtp_gather_gemm(dY[l], self.shards[l], out, transpose_w=True)
            else:
                if l - 1 >= 0:
                    self._gather_async(l - 1, wait_free=True)   # AG(W_{l-1}) beside dgrad(W_l)
                main.wait_event(self.ready[l % 2])
                ttl.gtp_gather_gemm(dY[l], self.shards[l], out, slot=self.slots[l % 2], transpose_w=True)
                self.free[l % 2].record(main)
            in_stream = prev is not None and not finalize_stream
            ws = self.wg if wgs else main
            ttl.gtp_wgrad_rs_finalize(X, dY[l], staging[l],
                                      staging_prev=staging[prev] if in_stream else None,
                                      main_grad_prev=main_grad[prev] if in_stream else None,
                                      sync=(l == 0), main_grad_cur=main_grad[0] if l == 0 else None,
                                      stream=ws)
            self.wgrad_done[l].record(ws)
        if wgs:
            main.wait_stream(self.wg)
        if finalize_stream:
            main.wait_stream(self.fin)
