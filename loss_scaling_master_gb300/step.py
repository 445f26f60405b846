"""One mixed-precision optimizer step on the device, as four C-ABI calls.

``AmpOptimizerStep`` owns the device-resident optimizer state (fp32 m, v,
the bf16 working copy, the optional FP8 copies, and the scaler state
{scale, growth_tracker, step, found_inf, amax[], inv_scale[]}) and the list
handles, and enqueues, per step:

1. ``amp_unscale_check``      scaled grads -> found_inf
2. ``amp_adamw_master_step``  skip or update master/m/v, emit bf16 (+ amax)
3. ``fp8_quant_tensorwise_list``  e4m3fn copies (+ transposed) of the FP8
   weights, skipped on inf (only when FP8 weights are configured)
4. ``amp_update_scale``       scale state machine; clears found_inf and amax

No call reads anything back to the host; ``state()`` does, for monitoring.
"""
from __future__ import annotations

import torch

from . import _lib as A


class AmpOptimizerStep:
    def __init__(self, master, grads, *, lr, beta1, beta2, eps, weight_decay,
                 init_scale=65536.0, growth_factor=2.0, backoff_factor=0.5,
                 growth_interval=2000, emit_bf16=True, fp8_shapes=None, fp8_eps=1e-12,
                 max_norm=None, stream=None):
        """master: fp32 device tensors (updated in place); grads: device
        tensors (f16/bf16/f32) the caller fills with scaled gradients before
        each step.  fp8_shapes: per tensor (rows, cols) for weights that get
        e4m3fn copies, None for the others (requires emit_bf16).  max_norm:
        clip the unscaled gradients to this global L2 norm (None: no clipping)."""
        dev = master[0].device
        self.stream = stream
        self.master = list(master)
        self.grads = list(grads)
        self.exp_avg = [torch.zeros_like(p) for p in self.master]
        self.exp_avg_sq = [torch.zeros_like(p) for p in self.master]
        self.bf16 = [torch.empty(p.shape, dtype=torch.bfloat16, device=dev) for p in self.master] \
            if emit_bf16 else None
        self.hyper = (lr, beta1, beta2, eps, weight_decay)
        self.growth, self.backoff, self.interval = growth_factor, backoff_factor, growth_interval
        self.scale = torch.tensor([init_scale], dtype=torch.float32, device=dev)
        self.growth_tracker = torch.zeros(1, dtype=torch.int32, device=dev)
        self.step_count = torch.zeros(1, dtype=torch.int32, device=dev)
        self.found_inf = torch.zeros(1, dtype=torch.int32, device=dev)
        self.max_norm = max_norm
        self.grad_sumsq = torch.zeros(1, dtype=torch.float64, device=dev)
        self.fp8_eps = fp8_eps
        mk = lambda ts, two_d=False: A.amp_tensor_list_create(ts, two_d=two_d, stream=stream)
        self.L_master, self.L_m, self.L_v = mk(self.master), mk(self.exp_avg), mk(self.exp_avg_sq)
        self.L_g = mk(self.grads)
        self.grad_lists = [self.L_g]
        self.graphs = {}
        self.L_b = mk(self.bf16) if emit_bf16 else None
        self.n_fp8 = 0
        self.fp8, self.fp8_t = [], []
        if fp8_shapes is not None:
            assert emit_bf16, "FP8 weight copies are cast from the bf16 copy"
            slots, xs = [], []
            for i, sh in enumerate(fp8_shapes):
                if sh is None:
                    slots.append(-1)
                    continue
                slots.append(self.n_fp8)
                self.n_fp8 += 1
                xs.append(self.bf16[i].view(sh[0], sh[1]))
                self.fp8.append(torch.empty(sh, dtype=torch.float8_e4m3fn, device=dev))
                self.fp8_t.append(torch.empty((sh[1], sh[0]), dtype=torch.float8_e4m3fn,
                                              device=dev))
            A.amp_tensor_list_set_amax_slots(self.L_b, slots, stream=stream)
            self.L_x8 = mk(xs, True)
            self.L_q = mk(self.fp8, True)
            self.L_qt = mk(self.fp8_t, True)
        self.amax = torch.zeros(max(self.n_fp8, 1), dtype=torch.float32, device=dev)
        self.inv_scale = torch.zeros(max(self.n_fp8, 1), dtype=torch.float32, device=dev)

    @property
    def launches_per_step(self) -> int:
        """Kernels one step enqueues (check [+ norm reduce], AdamW prologue + main,
        [quant], update)."""
        return 4 + (1 if self.n_fp8 else 0) + (1 if self.max_norm is not None else 0)

    def add_grad_buffer(self, grads) -> int:
        """Register another set of gradient buffers (same shapes and dtype) and
        return its index for step(grad_buffer=...): with two buffers the host
        can fill one while the GPU steps on the other."""
        grads = list(grads)
        if [g.numel() for g in grads] != [g.numel() for g in self.grads] or \
                any(a.dtype != b.dtype for a, b in zip(grads, self.grads)):
            raise ValueError("gradient buffers must match the first set in sizes and dtype")
        self.grad_lists.append(A.amp_tensor_list_create(grads, stream=self.stream))
        return len(self.grad_lists) - 1

    def capture_graph(self, stream=None, grad_buffer: int = 0):
        """Record one step into a CUDA graph; later step() calls on the same
        gradient buffer replay it.  Every call of the step is stream-ordered
        and allocation-free, so the graph is the same calls with the same
        device pointers; the caller keeps writing each step's gradients into
        the same buffers."""
        s = stream if stream is not None else (self.stream or torch.cuda.Stream())
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            self._enqueue(None, grad_buffer)
        self.graphs[grad_buffer] = g
        return g

    def step(self, stream=None, grad_buffer: int = 0):
        g = self.graphs.get(grad_buffer)
        if g is not None:
            if stream is not None:
                with torch.cuda.stream(stream):
                    g.replay()
            else:
                g.replay()
            return
        self._enqueue(stream if stream is not None else self.stream, grad_buffer)

    def _enqueue(self, s, grad_buffer: int = 0):
        L_g = self.grad_lists[grad_buffer]
        amax = self.amax if self.n_fp8 else None
        if self.max_norm is None:
            A.amp_unscale_check(L_g, self.scale, self.found_inf, stream=s)
            A.amp_adamw_master_step(self.L_master, self.L_m, self.L_v, L_g, self.L_b, self.scale,
                                    self.found_inf, self.step_count, *self.hyper, amax=amax,
                                    stream=s)
        else:
            A.amp_unscale_check_norm(L_g, self.scale, self.found_inf, self.grad_sumsq, stream=s)
            A.amp_adamw_master_step_clip(self.L_master, self.L_m, self.L_v, L_g, self.L_b,
                                         self.scale, self.found_inf, self.step_count, *self.hyper,
                                         self.grad_sumsq, self.max_norm, amax=amax, stream=s)
        if self.n_fp8:
            A.fp8_quant_tensorwise_list(self.L_x8, self.L_q, self.L_qt, "e4m3fn", self.amax,
                                        self.inv_scale, eps=self.fp8_eps, skip_if=self.found_inf,
                                        stream=s)
        A.amp_update_scale(self.scale, self.growth_tracker, self.found_inf, self.growth,
                           self.backoff, self.interval, amax=self.amax if self.n_fp8 else None,
                           n_amax=self.n_fp8, stream=s)

    def state(self) -> dict:
        """Host copy of the scaler/optimizer counters (synchronises)."""
        return {"scale": float(self.scale.item()), "growth_tracker": int(self.growth_tracker.item()),
                "step": int(self.step_count.item()), "found_inf": int(self.found_inf.item())}

    def close(self):
        for name in ("L_master", "L_m", "L_v", "L_b", "L_x8", "L_q", "L_qt"):
            lst = getattr(self, name, None)
            if lst is not None:
                lst.close()
        for lst in self.grad_lists:
            lst.close()
