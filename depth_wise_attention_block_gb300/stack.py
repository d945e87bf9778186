"""Synthetic L-layer Block AttnRes stack forward on the GPU.

Per layer l = 1..L: one fused `attnres_layer_step` (fold v_{l-1} into the
partial sum or emit b_n at a block boundary, then aggregate layer l), then
the stand-in layer body v_l = tanh(r_l * g_l) * s_l.  After layer L, the
final output aggregation (l = L+1) folds v_L into the last block and
aggregates [h_0, b_1 .. b_N] (Kimi K3 chaptered tutorial, ch. 4.3: the final
output layer aggregates all block representations).  2L+1 launches per
forward; `capture()` records them into one CUDA graph so a decode-sized
forward is not bound by launch latency.

schedule="two_phase" runs the same forward as the tutorial's two-phase
inference schedule (ch. 4.4, 4.6): at the start of block n the previous
block is closed (attnres_block_step), one inter-block pass aggregates the
cached [h_0, b_1 .. b_{n-1}] for all of the block's layer queries
(attnres_interblock), and each layer merges its partial sum in
(attnres_intrablock_step).  schedule="hybrid" runs the blocks before
`two_phase_from` (default 6) in single pass and the later ones (the most
cached sources, where one shared pass saves the most re-reads) two-phase.
A block whose pass would take more than 9 cached sources or 16 queries
(more than K3's 8 blocks of 12) runs single pass in either schedule.
The hybrid schedule is the faster one here:
on a GB300 the 93-layer T = 2048 prefill then takes 4.35 ms against
4.51 ms in single pass.
"""
from __future__ import annotations

import torch

from . import (
    AttnResState,
    attnres_aggregate,
    attnres_aggregate_backward,
    attnres_aggregate_backward_workspace_size,
    attnres_aggregate_fold,
    attnres_block_step,
    attnres_interblock,
    attnres_interblock_workspace_size,
    attnres_intrablock_step,
    attnres_layer_sources,
    attnres_layer_step,
    attnres_num_sources,
    attnres_synthetic_layer,
    attnres_synthetic_layer_backward,
)


def stack_forward_bytes(T: int, d: int, esz: int, num_layers: int, block_size: int) -> int:
    """Byte model of one single-pass stack forward (T tokens of d channels,
    esz bytes per stored element): each layer step reads its stored sources,
    the previous partial sum (if the block has one) and F_{l-1} once, and
    writes the new partial sum or block sum, r and the fp32 weights once;
    each layer body reads r and writes F (and reads its fp32 g and s)."""
    L, B = num_layers, block_size
    row = T * d * esz
    total = 0
    for l in range(1, L + 2):
        S = attnres_num_sources(l, B, L)
        if l == 1:
            total += row + row                       # read h_0, write r
        else:
            p = l - 1
            first = (p - 1) // B * B + 1
            has_prev = p > first
            total += (S - 1) * row                   # stored sources
            total += row * (2 if has_prev else 1)    # partial (if any) + F_{l-1}
            total += row                             # new partial / b_n
            total += row                             # r_l
        total += T * S * 4                           # weights
        if l <= L:
            total += 2 * row + 2 * d * 4             # F_l: read r, write F (+ g, s)
    return total


class StackForward:
    """Buffers and launch sequence of one stack forward over T tokens.

    h0: [T, d] embedding (bf16 or fp32); W: [L+1, d] fp32 pseudo-queries
    (row L is the final aggregation's); G, Sc: [L, d] fp32 gains and scales
    of the synthetic layer body.  Outputs: `r` ([T, d], the final residual
    stream after `run()`), `weights[l-1]` ([T, S_l] fp32, l = 1..L+1).
    With `early_loads` the fused steps load their stored rows before the
    body before them has finished (ATTNRES_STATE_EARLY_LOADS); the results
    are the same bits.
    """

    def __init__(self, h0, W, G, Sc, num_layers: int, block_size: int, eps: float = 1e-5,
                 keep_weights: bool = True, dev_err: torch.Tensor | None = None, schedule: str = "single",
                 two_phase_from: int = 6, early_loads: bool = True, first_layer_from_pass: bool = True):
        self.L, self.B, self.eps = num_layers, block_size, eps
        T, d = h0.shape
        self.T, self.d = T, d
        self.W, self.G, self.Sc = W, G, Sc
        # the kernel before each fused step is the layer body, which writes
        # only F and signals its dependents after its own wait: the steps may
        # load their stored rows early (ATTNRES_STATE_EARLY_LOADS).  on_layer
        # hooks must not write the state's rows then.
        self.early_loads = early_loads
        # a two-phase block's first layer written by the inter-block pass
        # itself (its merge would fold nothing and give the same bits)
        self.first_layer_from_pass = first_layer_from_pass
        self.state = AttnResState.allocate(h0, num_layers, block_size, eps, early_loads=early_loads)
        self.r = torch.empty_like(h0)
        self.F = torch.empty_like(h0)
        self.S = [attnres_num_sources(l, block_size, num_layers) for l in range(1, num_layers + 2)]
        self.weights = None
        if keep_weights:
            flat = torch.empty(T * sum(self.S), dtype=torch.float32, device=h0.device)
            self.weights, off = [], 0
            for s in self.S:
                self.weights.append(flat[off:off + T * s].view(T, s))
                off += T * s
        self.dev_err = dev_err
        self.graph = None
        if schedule not in ("single", "two_phase", "hybrid"):
            raise ValueError("schedule must be 'single', 'two_phase' or 'hybrid'")
        self.schedule = schedule
        # the first block run two-phase
        self.first_two_phase = {"single": None, "two_phase": 1, "hybrid": max(1, int(two_phase_from))}[schedule]
        self.inter_ws = None
        if any(self._runs_two_phase(n) for n in range(1, -(-num_layers // block_size) + 1)):
            q = min(block_size, num_layers)
            n_max = min(-(-num_layers // block_size), self.PASS_MAX_SOURCES)  # cached sources, at most
            self.R_inter = torch.empty((q, T, d), dtype=torch.float32, device=h0.device)
            self.lse_inter = torch.empty((q, T), dtype=torch.float32, device=h0.device)
            self.A_flat = torch.empty(q * T * n_max, dtype=torch.float32, device=h0.device)
            # the tensor-core logits' workspace, sized for the largest block
            need = max(attnres_interblock_workspace_size(n, T, d, h0.dtype, q) for n in range(1, n_max + 1))
            self.inter_ws = torch.empty(need, dtype=torch.uint8, device=h0.device) if need > 0 else None

    # what one inter-block pass takes (attnres_interblock): cached sources and queries
    PASS_MAX_SOURCES = 9
    PASS_MAX_QUERIES = 16

    def _runs_two_phase(self, n: int) -> bool:
        """Block n runs two-phase: from the schedule's first two-phase block
        on, while one pass can take its cached sources and its queries (a
        block beyond that runs single pass)."""
        if self.first_two_phase is None or n < self.first_two_phase:
            return False
        q = min(n * self.B, self.L) - (n - 1) * self.B
        return n <= self.PASS_MAX_SOURCES and q <= self.PASS_MAX_QUERIES

    def launches_per_forward(self) -> int:
        if self.schedule == "single":
            return 2 * self.L + 1
        N = -(-self.L // self.B)
        two = [n for n in range(1, N + 1) if self._runs_two_phase(n)]
        n2 = len(two)                                        # blocks run two-phase
        closes = sum(1 for n in two if n >= 2)               # block_step closing the block before
        own = n2 if self.first_layer_from_pass else 0        # first layers the pass writes itself
        per_pass = 2 if self.inter_ws is not None else 1     # tensor-core logits + weighted sums, or one kernel
        return per_pass * n2 + closes + 2 * self.L + 1 - own

    def _issue_two_phase(self, stream=None, on_layer=None) -> None:
        st, L, B = self.state, self.L, self.B
        st.reset()
        bufs = {t.data_ptr(): t for t in [st.h0] + st.block_reps}
        T = self.T
        for n in range(1, -(-L // B) + 1):
            first, last = (n - 1) * B + 1, min(n * B, L)
            if not self._runs_two_phase(n):
                # single pass: each step folds the previous layer's output
                for l in range(first, last + 1):
                    attnres_layer_step(st, self.F if l > 1 else None, self.W[l - 1], l, self.r,
                                       self.weights[l - 1] if self.weights is not None else None,
                                       dev_err=self.dev_err, stream=stream)
                    attnres_synthetic_layer(self.r, self.G[l - 1], self.Sc[l - 1], self.F, stream=stream)
                    if on_layer is not None:
                        on_layer(l, self)
                continue
            if n >= 2:
                attnres_block_step(st, self.F, first - 1, dev_err=self.dev_err, stream=stream)
            cached = [bufs[p] for p in attnres_layer_sources(st, first)]
            Q = last - first + 1
            A = self.A_flat[: Q * T * n].view(Q, T, n)
            own = self.first_layer_from_pass
            attnres_interblock(cached, self.W[first - 1:last], self.R_inter[:Q], self.lse_inter[:Q], A,
                               workspace=self.inter_ws, tensor_cores=self.inter_ws is not None,
                               dev_err=self.dev_err, stream=stream, out_r0=self.r if own else None,
                               out_weights0=self.weights[first - 1] if own and self.weights is not None else None)
            for layer in range(first, last + 1):
                q = layer - first
                if not (own and layer == first):
                    attnres_intrablock_step(st, self.F if layer > first else None, self.W[layer - 1], layer,
                                            self.R_inter[q], self.lse_inter[q], A[q], self.r,
                                            self.weights[layer - 1] if self.weights is not None else None,
                                            dev_err=self.dev_err, stream=stream)
                attnres_synthetic_layer(self.r, self.G[layer - 1], self.Sc[layer - 1], self.F, stream=stream)
                if on_layer is not None:
                    on_layer(layer, self)
        attnres_layer_step(st, self.F, self.W[L], L + 1, self.r,
                           self.weights[L] if self.weights is not None else None, dev_err=self.dev_err, stream=stream)
        if on_layer is not None:
            on_layer(L + 1, self)

    def _issue_layers(self, first: int, last: int, stream=None, on_layer=None) -> None:
        """Layers first..last from a state with v_1 .. v_{first-1} folded:
        the first layer aggregates the state's sources as they are, each
        later one folds its predecessor's output in the same launch.  If
        last == L the final aggregation follows (folding v_L); otherwise v_last
        is folded on its own, so that the state holds everything a later
        stage needs ([Tutorial] ch. 4.6, pipeline stages)."""
        for l in range(first, last + 1):
            attnres_layer_step(self.state, self.F if l > first else None, self.W[l - 1], l, self.r,
                               self.weights[l - 1] if self.weights is not None else None,
                               dev_err=self.dev_err, stream=stream)
            attnres_synthetic_layer(self.r, self.G[l - 1], self.Sc[l - 1], self.F, stream=stream)
            if on_layer is not None:
                on_layer(l, self)
        if last == self.L:
            attnres_layer_step(self.state, self.F, self.W[self.L], self.L + 1, self.r,
                               self.weights[self.L] if self.weights is not None else None,
                               dev_err=self.dev_err, stream=stream)
            if on_layer is not None:
                on_layer(self.L + 1, self)
        else:
            attnres_block_step(self.state, self.F, last, dev_err=self.dev_err, stream=stream)

    def _issue(self, stream=None, on_layer=None) -> None:
        if self.schedule != "single":
            self._issue_two_phase(stream, on_layer)
            return
        self.state.reset()
        self._issue_layers(1, self.L, stream, on_layer)

    def run(self, stream=None, on_layer=None) -> torch.Tensor:
        """One forward (replays the captured graph if there is one).
        on_layer(l, self), eager runs only, is called after layer l's step
        and body have been issued (l = L+1: after the final aggregation)."""
        if self.graph is not None:
            if on_layer is not None:
                raise ValueError("on_layer needs an eager run (this forward is a captured graph)")
            self.graph.replay()
        else:
            self._issue(stream, on_layer)
        return self.r

    def run_chunk(self, first: int, last: int, stream=None, on_layer=None) -> torch.Tensor:
        """Layers first..last only (a pipeline stage, eager).  first == 1
        starts the stack; otherwise the state must hold v_1 .. v_{first-1}
        folded (its own earlier chunk, or buffers received and
        AttnResState.resume(first - 1)).  Ends with the final aggregation
        when last == L, else with v_last folded into the state."""
        if self.schedule != "single":
            raise ValueError("run_chunk runs the single-pass schedule")
        if not (1 <= first <= last <= self.L):
            raise ValueError("need 1 <= first <= last <= L")
        if first == 1:
            self.state.reset()
        self._issue_layers(first, last, stream, on_layer)
        return self.r

    def capture(self) -> None:
        """Record the whole forward into a CUDA graph (after one eager run)."""
        self._issue()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            self._issue()
        self.graph = g

    def bytes_moved(self) -> int:
        """Minimum HBM bytes one forward must move (every source row, F row,
        partial/b_n row read once; r, F, partial/b_n and weights written once)."""
        return stack_forward_bytes(self.T, self.d, self.state.h0.element_size(), self.L, self.B)


class StackBackward:
    """Gradients of the loss sum(r_out * dr_out) of a StackForward's stack
    with respect to h_0 and every pseudo-query W[0..L], with the forward
    recomputed block by block from what the forward keeps (h_0 and the block
    representations b_1 .. b_N: activation checkpointing at block
    granularity, [Tutorial] ch. 4.6).

    Per block n, from the last block down:
      recompute: v_l = F_l(r_l) and r_{l+1} = aggregate over [h_0,
        b_1..b_{n-1}, P_{l+1}] with P_{l+1} = P_l + v_l formed in the same
        launch (attnres_aggregate_fold; the block's first layer a plain
        attnres_aggregate), keeping every r_l and partial sum P_l;
      backward, layer by layer from the block's last: dL/dv_l is the
        gradient of b_n (from later blocks and the final aggregation) plus
        that of the partial sums of the block's later layers, dL/dr_l =
        dL/dv_l F_l'(r_l) (attnres_synthetic_layer_backward), and
        attnres_aggregate_backward (accumulate) adds layer l's gradients into
        those of h_0, b_1..b_{n-1} and the block's running partial-sum
        gradient, and writes dW[l-1].
    The final aggregation's backward (over [h_0, b_1..b_N]) starts it.
    Gradients are kept in the stack's storage dtype.  Outputs: `dh0` [T, d],
    `dW` [L+1, d] fp32.
    """

    def __init__(self, fwd: StackForward):
        self.fwd = fwd
        st, T, d, B = fwd.state, fwd.T, fwd.d, fwd.B
        dt, dev = st.h0.dtype, st.h0.device
        self.N = -(-fwd.L // B)
        self.dh0 = torch.empty((T, d), dtype=dt, device=dev)
        self.gb = [torch.empty((T, d), dtype=dt, device=dev) for _ in range(self.N)]
        self.gpart = torch.empty((T, d), dtype=dt, device=dev)
        self.gr = torch.empty((T, d), dtype=dt, device=dev)
        self.v = torch.empty((T, d), dtype=dt, device=dev)
        q = min(B, fwd.L)
        self.R = torch.empty((q, T, d), dtype=dt, device=dev)       # r_l of the block being processed
        self.P = torch.empty((q, T, d), dtype=dt, device=dev)       # P[i-1]: partial sum read by position i >= 2
        self.dW = torch.empty((fwd.L + 1, d), dtype=torch.float32, device=dev)
        nbytes = attnres_aggregate_backward_workspace_size(T, d)
        self.ws = torch.empty((nbytes + 3) // 4, dtype=torch.float32, device=dev)
        self.graph = None

    def _issue(self, dr_out, stream=None, on_call=None) -> None:
        f, st = self.fwd, self.fwd.state
        L, B, eps = f.L, f.B, f.eps
        b = st.block_reps[: self.N]
        if on_call is not None:
            on_call(L + 1, [st.h0] + b, dr_out, [self.dh0] + self.gb, self.dW[L], False, "before")
        attnres_aggregate_backward([st.h0] + b, f.W[L], dr_out, [self.dh0] + self.gb, self.dW[L],
                                   workspace=self.ws, eps=eps, accumulate=False, stream=stream)
        if on_call is not None:
            on_call(L + 1, [st.h0] + b, dr_out, [self.dh0] + self.gb, self.dW[L], False, "after")
        for n in range(self.N, 0, -1):
            first, last = (n - 1) * B + 1, min(n * B, L)
            cached = [st.h0] + b[: n - 1]
            for layer in range(first, last + 1):
                i = layer - first + 1
                if i == 1:
                    attnres_aggregate(cached, f.W[layer - 1], self.R[0], eps=eps, stream=stream)
                else:
                    # P[i-1] = P[i-2] + v_{i-1} (or v_1) formed in the aggregation's launch
                    # (early loads: the body just before writes only v, and every kernel
                    # here signals its dependents after its own wait)
                    attnres_aggregate_fold(cached, self.P[i - 2] if i >= 3 else None, self.v, self.P[i - 1],
                                           f.W[layer - 1], self.R[i - 1], eps=eps, early_loads=f.early_loads,
                                           stream=stream)
                if layer < last:
                    attnres_synthetic_layer(self.R[i - 1], f.G[layer - 1], f.Sc[layer - 1], self.v, stream=stream)
            # the block's partial sums have no gradient yet (one memset)
            if stream is None:
                self.gpart.zero_()
            else:
                with torch.cuda.stream(stream):
                    self.gpart.zero_()
            for layer in range(last, first - 1, -1):
                i = layer - first + 1
                attnres_synthetic_layer_backward(self.R[i - 1], f.G[layer - 1], f.Sc[layer - 1], self.gb[n - 1],
                                                 self.gpart if layer < last else None, self.gr, stream=stream)
                srcs = cached + ([self.P[i - 1]] if i >= 2 else [])
                grads = [self.dh0] + self.gb[: n - 1] + ([self.gpart] if i >= 2 else [])
                if on_call is not None:
                    on_call(layer, srcs, self.gr, grads, self.dW[layer - 1], True, "before")
                attnres_aggregate_backward(srcs, f.W[layer - 1], self.gr, grads, self.dW[layer - 1],
                                           workspace=self.ws, eps=eps, accumulate=True, stream=stream)
                if on_call is not None:
                    on_call(layer, srcs, self.gr, grads, self.dW[layer - 1], True, "after")

    def run(self, dr_out=None, stream=None, on_call=None):
        """One backward (replays the captured graph, recorded for the dr_out
        given to capture(), if there is one); the forward must have run on
        the same inputs.  on_call(layer, sources, grad_r, grad_sources,
        grad_w, accumulate, phase), eager runs only, is called just before
        (phase "before") and after ("after") each layer's
        attnres_aggregate_backward is issued."""
        if self.graph is not None:
            if on_call is not None:
                raise ValueError("on_call needs an eager run (this backward is a captured graph)")
            self.graph.replay()
        else:
            self._issue(dr_out, stream, on_call)
        return self.dh0, self.dW

    def capture(self, dr_out) -> None:
        """Record the whole backward for dr_out into a CUDA graph (after one
        eager run)."""
        self._issue(dr_out)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            self._issue(dr_out)
        self.graph = g

    def bytes_moved(self) -> int:
        """Minimum HBM bytes one backward moves: every row each call reads or
        writes, once (the model behind its achieved bandwidth)."""
        f = self.fwd
        L, B, N = f.L, f.B, self.N
        row = f.T * f.d * f.state.h0.element_size()
        rows = (N + 2) + (N + 1)                               # final: sources + dr read, grads written
        for n in range(1, N + 1):
            q = min(n * B, L) - (n - 1) * B
            for i in range(1, q + 1):
                S = n + (1 if i >= 2 else 0)
                if i == 1:
                    rows += n + 1                              # recompute: aggregate reads h_0, b_1.., writes r
                else:
                    rows += n + (2 if i >= 3 else 1) + 2       # aggregate_fold: stored, (P +) v in; P', r out
                if i < q:
                    rows += 2                                  # body: r -> v
                rows += (3 if i < q else 2) + 1                # body backward: r, gb (+ gpart) -> gr
                rows += (2 * S + 1) + S                        # aggregation backward, accumulating
            rows += 1                                          # memset of the partial-sum gradient
        return rows * row + (L + 1) * f.d * 4

    def launches_per_backward(self) -> int:
        """Kernel launches (plus one memset per block) of one backward."""
        L, B, N = self.fwd.L, self.fwd.B, self.N
        n = 2                                                  # final aggregation backward (+ its dw reduction)
        for k in range(1, N + 1):
            q = min(k * B, L) - (k - 1) * B
            n += q + (q - 1)                                   # recompute: aggregate (fold fused), body
            n += q * (1 + 2)                                   # body backward, aggregation backward (+ dw reduction)
        return n
