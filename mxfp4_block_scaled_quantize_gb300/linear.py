"""The MXFP4 linear layer's data path, Y = X . W^T, as a sequence of C-ABI calls.

Follows the dataflow of `MXFP4LinearFunction` in primus_turbo_mxfp4_local.py:
  forward   dual-quantize X and W (row-only when no backward follows, the "row-only
            packing" of Primus PR #1107), Y = X_row . W_row^T, with the layer's bias add
            (`output + bias` of `_forward_impl`) fused into the GEMM when a bias is given
  backward  dual-quantize dY (optionally with stochastic rounding, the gradient
            quantizer's `use_sr`), dX = dY_row . (W_col)^T, dW = dY_col . (X_col)^T;
            or, with backward="fp8", the pages' hybrid backward (tensorwise E5M2 of dY,
            X, W and FP8 GEMMs)
With weight_2d, W is quantized with one scale per 32 x 32 block in both packings (the
weight recipe of `_quantize_weight_dual`, `rowwise_use_2d_block` / `colwise_use_2d_block`);
with rht_signs, the column blobs of X and dY -- the two wgrad operands -- are those of their
Hadamard-transformed columns, with the same signs (`colwise_use_rht` of
`_quantize_input_dual` / `_quantize_grad_dual`).  The shuffle flags are off.  In the
MXFP4 backward only the column blobs of X and W live from forward to backward; bf16 X
and W are not kept.  All buffers are allocated once (torch as the allocator) and reused,
so an MXFP4 step is four launches on one stream: X and W quantized together, the forward
GEMM, dY, and dgrad with wgrad in one GEMM launch.
"""
import torch

from . import abi


class MXFP4Linear:
    """backward = "mxfp4" (the default) or "fp8": the hybrid mode of the pages
    (`mxfp4_backward_precision == "fp8"`, `backward_is_fp8`), where the forward keeps the
    bf16 X and W and the backward quantizes dY, X and W tensorwise to E5M2 and runs dgrad
    and wgrad as FP8 GEMMs.  In that mode the forward quantizes X and W row-only: their
    column blobs would only feed an MXFP4 backward."""

    def __init__(self, M: int, N: int, K: int, train: bool = True, device="cuda",
                 out_dtype=torch.bfloat16, backward: str = "mxfp4", weight_2d: bool = False,
                 rht_signs=None):
        assert backward in ("mxfp4", "fp8")
        self.M, self.N, self.K, self.train = M, N, K, train
        self.weight_2d = weight_2d
        self.rht_signs = rht_signs
        assert rht_signs is None or backward == "mxfp4", "the transform belongs to the MXFP4 wgrad"
        self.fp8_backward = train and backward == "fp8"
        L = abi.MXFP4_SCALE_TC
        self.x_row = abi.alloc_blob(M, K, L, device)
        self.w_row = abi.alloc_blob(N, K, L, device)
        self.y = torch.empty((M, N), dtype=out_dtype, device=device)
        if self.fp8_backward:
            p = abi.fp8_pitch
            self.dy_f8 = torch.empty((M, p(N)), dtype=torch.uint8, device=device)
            self.dy_f8_col = torch.empty((N, p(M)), dtype=torch.uint8, device=device)
            self.x_f8_col = torch.empty((K, p(M)), dtype=torch.uint8, device=device)
            self.w_f8_col = torch.empty((K, p(N)), dtype=torch.uint8, device=device)
            self.f8_scalars = torch.zeros(6, dtype=torch.float32, device=device)   # (amax, scale_inv) x dY, X, W
            self.dx = torch.empty((M, K), dtype=out_dtype, device=device)
            self.dw = torch.empty((N, K), dtype=out_dtype, device=device)
            self._saved = None
        elif train:
            self.x_col = abi.alloc_blob(K, M, L, device)
            self.w_col = abi.alloc_blob(K, N, L, device)
            self.dy_row = abi.alloc_blob(M, N, L, device)
            self.dy_col = abi.alloc_blob(N, M, L, device)
            self.dx = torch.empty((M, K), dtype=out_dtype, device=device)
            self.dw = torch.empty((N, K), dtype=out_dtype, device=device)

    # -- steps a1..a4 of the path ---------------------------------------------------------
    def quantize_x(self, x, stream=None):
        M, K = self.M, self.K
        if self.train and self.rht_signs is not None:
            abi.mxfp4_quantize_dual_rht(x, M, K, x.stride(0), *self.x_row, *self.x_col,
                                        abi.MXFP4_SCALE_TC, self.rht_signs, stream)
        elif self.train:
            abi.mxfp4_quantize_dual(x, M, K, x.stride(0), *self.x_row, *self.x_col,
                                    abi.MXFP4_SCALE_TC, stream)
        else:
            abi.mxfp4_quantize(x, M, K, x.stride(0), *self.x_row, abi.MXFP4_SCALE_TC, stream)

    def quantize_w(self, w, stream=None):
        N, K = self.N, self.K
        if self.train and not self.fp8_backward:
            quant = abi.mxfp4_quantize_dual_2d if self.weight_2d else abi.mxfp4_quantize_dual
            quant(w, N, K, w.stride(0), *self.w_row, *self.w_col, abi.MXFP4_SCALE_TC, stream)
        else:
            flags = abi.MXFP4_QUANT_2D_BLOCKS if self.weight_2d else 0
            abi.mxfp4_quantize_batch([(w, N, K, w.stride(0), *self.w_row, None, None, flags)], False,
                                     abi.MXFP4_SCALE_TC, stream)

    def quantize_dy(self, dy, stream=None, sr_seed=None):
        """dY's two blobs; with sr_seed, stochastically rounded (the gradient quantizer's
        `use_sr`, the layer's `mxfp4_gradient_stochastic_rounding` option); with the layer's
        rht_signs, the col blob of the transformed columns (both together: the gradient
        recipe of `_quantize_grad_dual` with `use_sr`)."""
        if self.rht_signs is not None and sr_seed is not None:
            abi.mxfp4_quantize_dual_rht_sr(dy, self.M, self.N, dy.stride(0), *self.dy_row, *self.dy_col,
                                           abi.MXFP4_SCALE_TC, self.rht_signs, sr_seed, stream)
        elif self.rht_signs is not None:
            abi.mxfp4_quantize_dual_rht(dy, self.M, self.N, dy.stride(0), *self.dy_row, *self.dy_col,
                                        abi.MXFP4_SCALE_TC, self.rht_signs, stream)
        elif sr_seed is None:
            abi.mxfp4_quantize_dual(dy, self.M, self.N, dy.stride(0), *self.dy_row, *self.dy_col,
                                    abi.MXFP4_SCALE_TC, stream)
        else:
            abi.mxfp4_quantize_dual_sr(dy, self.M, self.N, dy.stride(0), *self.dy_row, *self.dy_col,
                                       abi.MXFP4_SCALE_TC, sr_seed, stream)

    # -- steps a5..a7 ---------------------------------------------------------------------
    def fwd_gemm(self, stream=None, bias=None):
        """Y = X . W^T, plus the layer's bf16 bias[N] fused into the GEMM's output when given
        (the `output + bias` that follows the GEMM in `_forward_impl`)."""
        abi.gemm(*self.x_row, *self.w_row, self.M, self.N, self.K, out=self.y, stream=stream, bias=bias)
        return self.y

    def dgrad_gemm(self, stream=None):
        abi.gemm(*self.dy_row, *self.w_col, self.M, self.K, self.N, out=self.dx, stream=stream)
        return self.dx

    def wgrad_gemm(self, stream=None):
        abi.gemm(*self.dy_col, *self.x_col, self.N, self.K, self.M, out=self.dw, stream=stream)
        return self.dw

    def bwd_gemms(self, stream=None):
        """dgrad and wgrad in one launch (they read the same dY blobs)."""
        code = abi.MXFP4_OUT_F32 if self.dx.dtype == torch.float32 else abi.MXFP4_OUT_BF16
        abi.mxfp4_gemm_batch([
            (*self.dy_row, *self.w_col, self.M, self.K, self.N, self.dx, self.dx.stride(0), code),
            (*self.dy_col, *self.x_col, self.N, self.K, self.M, self.dw, self.dw.stride(0), code),
        ], stream)
        return self.dx, self.dw

    # -- a8: the whole step ---------------------------------------------------------------
    def quantize_xw(self, x, w, stream=None):
        """X and W in one launch (steps a1-a4 for both)."""
        M, N, K = self.M, self.N, self.K
        if self.fp8_backward:
            self._saved = (x, w)   # the hybrid backward re-quantizes the bf16 tensors
        wf = abi.MXFP4_QUANT_2D_BLOCKS if self.weight_2d else 0
        if self.train and not self.fp8_backward:
            xf = abi.MXFP4_QUANT_RHT_COL if self.rht_signs is not None else 0
            tasks = [(x, M, K, x.stride(0), *self.x_row, *self.x_col, xf, self.rht_signs or 0),
                     (w, N, K, w.stride(0), *self.w_row, *self.w_col, wf)]
        elif self.fp8_backward:
            # the row-only forward quantization also gives X's and W's tensorwise amax, so the
            # hybrid backward's FP8 quantization of them skips its own amax pass
            sc = self.f8_scalars
            tasks = [(x, M, K, x.stride(0), *self.x_row, None, None, 0, 0, sc[2:3]),
                     (w, N, K, w.stride(0), *self.w_row, None, None, wf, 0, sc[4:5])]
        else:
            tasks = [(x, M, K, x.stride(0), *self.x_row, None, None),
                     (w, N, K, w.stride(0), *self.w_row, None, None, wf)]
        abi.mxfp4_quantize_batch(tasks, self.train and not self.fp8_backward, abi.MXFP4_SCALE_TC, stream)

    def forward(self, x, w, stream=None, bias=None):
        self.quantize_xw(x, w, stream)
        return self.fwd_gemm(stream, bias)

    def backward(self, dy, stream=None, sr_seed=None):
        assert self.train, "backward needs the column blobs of the dual quantizer"
        if self.fp8_backward:
            assert sr_seed is None, "stochastic rounding belongs to the MXFP4 backward"
            self.quantize_fp8_bwd(dy, stream)
            return self.fp8_bwd_gemms(stream)
        self.quantize_dy(dy, stream, sr_seed)
        return self.bwd_gemms(stream)

    # -- hybrid FP8 backward ----------------------------------------------------------------
    def quantize_fp8_bwd(self, dy, stream=None):
        """`_quantize_fp8_tw` of dY (row and column copies), X and W (column copies: the
        K-major operands of the two TN GEMMs); X's and W's amax come from the forward's
        quantization."""
        x, w = self._saved
        sc = self.f8_scalars
        abi.mxfp4_fp8_quantize_tw_batch([
            (dy, self.M, self.N, dy.stride(0), self.dy_f8, self.dy_f8_col, sc[0:1], sc[1:2]),
            (x, self.M, self.K, x.stride(0), None, self.x_f8_col, sc[2:3], sc[3:4], True),
            (w, self.N, self.K, w.stride(0), None, self.w_f8_col, sc[4:5], sc[5:6], True),
        ], stream)

    def fp8_bwd_gemms(self, stream=None):
        """dX = dY . W (A = dY codes, B = W^T codes) and dW = dY^T . X (A = dY^T codes,
        B = X^T codes) in one launch, each scaled by its operands' inverse scales."""
        code = abi.MXFP4_OUT_F32 if self.dx.dtype == torch.float32 else abi.MXFP4_OUT_BF16
        sc = self.f8_scalars
        abi.mxfp4_fp8_gemm_batch([
            (self.dy_f8, sc[1:2], self.w_f8_col, sc[5:6], self.M, self.K, self.N, self.dx,
             self.dx.stride(0), code),
            (self.dy_f8_col, sc[1:2], self.x_f8_col, sc[3:4], self.N, self.K, self.M, self.dw,
             self.dw.stride(0), code),
        ], stream)
        return self.dx, self.dw

    def step(self, x, w, dy=None, stream=None, bias=None, sr_seed=None):
        y = self.forward(x, w, stream, bias)
        if not self.train:
            return (y,)
        dx, dw = self.backward(dy, stream, sr_seed)
        return y, dx, dw

    # -- the step from pinned host buffers to pinned host buffers --------------------------
    def step_host(self, hx, hw, hdy=None, hy=None, hdx=None, hdw=None, bias=None, sr_seed=None):
        """One step with bf16 inputs in pinned host memory and results copied back to pinned
        host memory.  Host-to-device copies run on one copy stream, device-to-host copies on
        another, and the kernels on the current stream; each kernel waits only for the copy
        it reads, and each result starts back as soon as its GEMM is done (measured on
        GB300: 2.46 ms per Flux MLP step with serial copies, 1.84 ms overlapped; the link
        moves ~200 GB/s each way).  Returns when the
        work is queued; the current stream is ordered after every copy of the step."""
        if not hasattr(self, "_h2d"):
            dev = self.y.device
            self._h2d = torch.cuda.Stream(device=dev)
            self._d2h = torch.cuda.Stream(device=dev)
            self._x = torch.empty((self.M, self.K), dtype=torch.bfloat16, device=dev)
            self._w = torch.empty((self.N, self.K), dtype=torch.bfloat16, device=dev)
            self._dy = (torch.empty((self.M, self.N), dtype=torch.bfloat16, device=dev)
                        if self.train else None)
        compute = torch.cuda.current_stream(self.y.device)
        h2d, d2h = self._h2d, self._d2h
        # The previous step's kernels are done with the input buffers before they refill.
        h2d.wait_stream(compute)
        d2h.wait_stream(compute)
        ins = [(self._x, hx), (self._w, hw)] + ([(self._dy, hdy)] if self.train else [])
        ready = []
        for dst, src in ins:
            with torch.cuda.stream(h2d):
                dst.copy_(src, non_blocking=True)
                ev = torch.cuda.Event()
                ev.record(h2d)
            ready.append(ev)

        def send_back(dev_t, host_t):
            if host_t is None:
                return
            ev = torch.cuda.Event()
            ev.record(compute)
            d2h.wait_event(ev)
            with torch.cuda.stream(d2h):
                host_t.copy_(dev_t, non_blocking=True)

        compute.wait_event(ready[0])
        compute.wait_event(ready[1])
        self.quantize_xw(self._x, self._w)
        send_back(self.fwd_gemm(bias=bias), hy)
        if self.train:
            compute.wait_event(ready[2])
            self.backward(self._dy, sr_seed=sr_seed)
            send_back(self.dw, hdw)
            send_back(self.dx, hdx)
        compute.wait_stream(d2h)
        compute.wait_stream(h2d)

    # launches per step (for the benchmark's launch count)
    @property
    def launches_per_step(self) -> int:
        if self.fp8_backward:
            # X+W (amax zeroing, row-only quantization), fwd; FP8 quantization of dY, X, W
            # (zeroing, dY's amax, dY's conversion, X's and W's conversion); the FP8 GEMMs
            return 2 + 1 + 4 + 1
        return 4 if self.train else 2


class MXFP4Block:
    """The MXFP4 linears of one transformer block, stepped in the order of a training step:
    every forward in order, then every backward in reverse order (Flux-12B's single-stream
    block: linear1 and linear2 forward, linear2 and linear1 backward; the pages' Flux-12B
    campaign of Primus PR #1107 runs its MXFP4 linears this way, block after block).  In
    this data path each linear's inputs are given, so the linears share no buffer.

    shapes: sequence of (name, M, N, K).  Options as MXFP4Linear."""

    def __init__(self, shapes, train: bool = True, device="cuda", out_dtype=torch.bfloat16,
                 backward: str = "mxfp4", weight_2d: bool = False, rht_signs=None):
        self.names = [s[0] for s in shapes]
        self.train = train
        self.layers = [MXFP4Linear(M, N, K, train=train, device=device, out_dtype=out_dtype,
                                   backward=backward, weight_2d=weight_2d, rht_signs=rht_signs)
                       for _, M, N, K in shapes]
        self._ws = None
        self._pws = None   # the pipelined host step's workspace (two output sets)

    def ops(self, inputs, bias=None, sr_seed=None):
        """One step as a list of (name, callable, launches): each callable enqueues one
        stage of the step on the current stream.  inputs: per linear a dict with "X", "W"
        (and "dY" when training) CUDA bf16 tensors; bias: per linear a bf16 vector or None."""
        bias = bias or [None] * len(self.layers)
        out = []
        for name, L, t, b in zip(self.names, self.layers, inputs, bias):
            kind = "row" if (not self.train or L.fp8_backward) else "dual"
            # the hybrid forward's quantizer also zeroes and fills the X / W amax words
            out.append((f"{name}.quant_{kind}_XW", lambda L=L, t=t: L.quantize_xw(t["X"], t["W"]),
                        2 if L.fp8_backward else 1))
            out.append((f"{name}.gemm_fwd", lambda L=L, b=b: L.fwd_gemm(bias=b), 1))
        if self.train:
            for name, L, t in reversed(list(zip(self.names, self.layers, inputs))):
                if L.fp8_backward:
                    # zero, dY's amax and conversion, X's and W's conversions
                    out.append((f"{name}.quant_fp8_dY_X_W", lambda L=L, t=t: L.quantize_fp8_bwd(t["dY"]), 4))
                    out.append((f"{name}.gemm_fp8_dgrad_wgrad", lambda L=L: L.fp8_bwd_gemms(), 1))
                else:
                    out.append((f"{name}.quant_dual_dY",
                                lambda L=L, t=t: L.quantize_dy(t["dY"], sr_seed=sr_seed), 1))
                    out.append((f"{name}.gemm_dgrad_wgrad", lambda L=L: L.bwd_gemms(), 1))
        return out

    def step(self, inputs, bias=None, sr_seed=None):
        for _, fn, _ in self.ops(inputs, bias, sr_seed):
            fn()
        return [(L.y, L.dx, L.dw) if self.train else (L.y,) for L in self.layers]

    def host_tasks(self, host_inputs, host_outputs):
        code = abi.MXFP4_OUT_F32 if self.layers[0].y.dtype == torch.float32 else abi.MXFP4_OUT_BF16
        tasks = []
        for L, t, o in zip(self.layers, host_inputs, host_outputs):
            tasks.append((t["X"], t["W"], t.get("dY"), o[0], o[1] if self.train else None,
                          o[2] if self.train else None, L.M, L.N, L.K, self.train, code))
        return tasks

    def step_host(self, host_inputs, host_outputs, stream=None):
        """One step from host buffers to host buffers through the library's own host step
        (mxfp4_linear_step_host): the copies run on the library's copy streams, overlapped
        with the kernels.  host_outputs: per linear (Y, dX, dW) (or (Y,) forward-only) host
        tensors, pinned for asynchrony.  Returns when the step is enqueued; the current
        stream is ordered after every copy."""
        assert not any(L.fp8_backward or L.weight_2d or L.rht_signs is not None for L in self.layers), \
            "the host step runs the plain MXFP4 recipe"
        tasks = self.host_tasks(host_inputs, host_outputs)
        need = abi.mxfp4_linear_workspace_bytes(tasks)
        if self._ws is None or self._ws.numel() < need:
            self._ws = torch.empty(need, dtype=torch.uint8, device=self.layers[0].y.device)
        abi.mxfp4_linear_step_host(tasks, self._ws, self._ws.numel(), stream)

    def step_host_pipelined(self, host_inputs, host_outputs, stream=None):
        """step_host for a loop of steps (mxfp4_linear_step_host_pipelined): consecutive
        calls overlap one step's copies out with the next step's copies in and kernels.
        Call host_wait() and synchronize the stream before reading the host outputs."""
        assert not any(L.fp8_backward or L.weight_2d or L.rht_signs is not None for L in self.layers), \
            "the host step runs the plain MXFP4 recipe"
        tasks = self.host_tasks(host_inputs, host_outputs)
        need = abi.mxfp4_linear_pipelined_workspace_bytes(tasks)
        if self._pws is None or self._pws.numel() < need:
            self._pws = torch.empty(need, dtype=torch.uint8, device=self.layers[0].y.device)
        abi.mxfp4_linear_step_host_pipelined(tasks, self._pws, self._pws.numel(), stream)

    def host_wait(self, stream=None):
        """Orders the stream after every copy of the host steps enqueued so far."""
        abi.mxfp4_linear_host_wait(stream)

    @property
    def launches_per_step(self) -> int:
        return sum(L.launches_per_step for L in self.layers)
