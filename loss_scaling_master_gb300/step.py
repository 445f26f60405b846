"""One mixed-precision optimizer step on the device, as four C-ABI calls.

``AmpOptimizerStep`` owns the device-resident optimizer state (fp32 m, v,
the bf16 working copy, the optional FP8 copies, and the scaler state
{scale, growth_tracker, step, found_inf, amax[], inv_scale[]}) and the list
handles, and enqueues, per step:

1. ``amp_unscale_check``      scaled grads -> found_inf (data-parallel:
   then an all-reduce(MAX) of found_inf across the ranks)
2. ``amp_adamw_master_step``  skip or update master/m/v, emit bf16 (+ amax)
3. ``fp8_quant_tensorwise_list``  FP8 copies (+ transposed) of the FP8
   weights, skipped on inf (only when FP8 weights are configured)
4. ``amp_update_scale``       scale state machine; clears found_inf and amax

No call reads anything back to the host; ``state()`` does, for monitoring.
"""
from __future__ import annotations

import contextlib

import torch

from . import _lib as A

_nullctx = contextlib.nullcontext


class AmpOptimizerStep:
    def __init__(self, master, grads, *, lr, beta1, beta2, eps, weight_decay,
                 init_scale=65536.0, growth_factor=2.0, backoff_factor=0.5,
                 growth_interval=2000, emit_bf16=True, fp8_shapes=None, fp8_eps=1e-12,
                 max_norm=None, fp8_scaling="dynamic", amax_history_len=1, sr_seed=None,
                 min_scale=None, fp8_format="e4m3fn", data_parallel=False, dp_group=None,
                 fp8_slots=None, n_fp8_total=None, stream=None):
        """master: fp32 device tensors (updated in place); grads: device
        tensors (f16/bf16/f32) the caller fills with scaled gradients before
        each step.  fp8_shapes: per tensor (rows, cols) for weights that get
        FP8 copies, None for the others (requires emit_bf16).  max_norm:
        clip the unscaled gradients to this global L2 norm (None: no clipping).
        fp8_scaling: "dynamic" (this step's amax, a separate cast pass) or
        "delayed" (the max of the last amax_history_len steps' amax, cast in
        the update pass; the history starts from the initial bf16 copy).
        sr_seed: round the copies each step emits stochastically with this
        64-bit seed - the bf16 copy and the FP8 weight copies cast from it, in
        every form of the step (None: round to nearest-even).  The first
        working copies, made before any step, round to nearest-even.  min_scale: after every step, set the
        sticky health bits of amp_scale_health in page-locked host memory when
        the loss scale is not finite (1) or below min_scale (2); health()
        reads them without synchronising (None: no check).  fp8_format: the
        format of the FP8 weight copies, "e4m3fn" (the pages' choice for
        weights) or "e5m2".  data_parallel: this object steps one rank's shard
        of a data-parallel parameter set; after the non-finite check, found_inf
        is all-reduced (MAX) over dp_group (None: the default group of
        torch.distributed) on the step's stream, so every rank skips together,
        and with max_norm the fp64 sum of squares is all-reduced (SUM) too, so
        every rank clips by the global norm.  fp8_slots / n_fp8_total: flat
        (FSDP-style) shards, where a weight can span ranks (sharded.
        partition_flat): per tensor of this rank the weight's index among all
        n_fp8_total FP8 weights of the model (None for tensors without an FP8
        copy), fp8_shapes giving the rank's band of rows of each.  amax and
        inv_scale are then indexed by that global number, and with
        data_parallel the amax array is all-reduced (MAX) after each update,
        before the FP8 cast (dynamic scaling, round-to-nearest).  Without
        fp8_slots whole tensors belong to one rank and the amax needs no
        exchange."""
        # a data-parallel shard may hold no tensor at all (partition_flat can
        # give a rank an empty slice); it still takes part in every exchange
        dev = master[0].device if len(master) else torch.device("cuda", torch.cuda.current_device())
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
        self.min_scale = min_scale
        self.data_parallel, self.dp_group = bool(data_parallel), dp_group
        if fp8_format not in ("e4m3fn", "e5m2"):
            raise ValueError(fp8_format)
        self.fp8_format = fp8_format
        fp8_tdt = torch.float8_e4m3fn if fp8_format == "e4m3fn" else torch.float8_e5m2
        self.health_word = torch.zeros(1, dtype=torch.int32).pin_memory() \
            if min_scale is not None else None
        self._state_host = A.ScalerState()
        self.grad_sumsq = torch.zeros(1, dtype=torch.float64, device=dev)
        self.fp8_eps = fp8_eps
        mk = lambda ts, two_d=False, dt=None: A.amp_tensor_list_create(ts, two_d=two_d, dtype=dt,
                                                                        stream=stream)
        # empty lists take their dtype explicitly; others take it from their tensors
        e = lambda ts, dt: None if len(ts) else dt
        self.L_master = mk(self.master, dt=e(self.master, "f32"))
        self.L_m = mk(self.exp_avg, dt=e(self.exp_avg, "f32"))
        self.L_v = mk(self.exp_avg_sq, dt=e(self.exp_avg_sq, "f32"))
        self.L_g = mk(self.grads, dt=e(self.grads, "f16"))
        self.grad_lists = [self.L_g]
        self.graphs = {}
        self.L_b = mk(self.bf16, dt=e(self.bf16, "bf16")) if emit_bf16 else None
        self.n_fp8 = 0
        self.fp8, self.fp8_t = [], []
        self.flat = fp8_slots is not None
        if self.flat and (fp8_shapes is None or n_fp8_total is None or
                          len(fp8_slots) != len(self.master)):
            raise ValueError("flat shards need fp8_shapes, fp8_slots per tensor and n_fp8_total")
        if self.flat and (fp8_scaling != "dynamic" or sr_seed is not None):
            raise ValueError("flat shards are offered with dynamic scaling and "
                             "round-to-nearest copies")
        if fp8_shapes is not None:
            if not emit_bf16:
                raise ValueError("FP8 weight copies are cast from the bf16 copy (emit_bf16=True)")
            slots, xs = [], []
            for i, sh in enumerate(fp8_shapes):
                if sh is None:
                    slots.append(-1)
                    continue
                if self.flat:
                    if fp8_slots[i] is None or not 0 <= fp8_slots[i] < n_fp8_total:
                        raise ValueError(f"tensor {i}: FP8 slot {fp8_slots[i]} outside "
                                         f"0..{n_fp8_total - 1}")
                    slots.append(int(fp8_slots[i]))
                else:
                    slots.append(self.n_fp8)
                self.n_fp8 += 1
                xs.append(self.bf16[i].view(sh[0], sh[1]))
                self.fp8.append(torch.empty(sh, dtype=fp8_tdt, device=dev))
                self.fp8_t.append(torch.empty((sh[1], sh[0]), dtype=fp8_tdt,
                                              device=dev))
            A.amp_tensor_list_set_amax_slots(self.L_b, slots, stream=stream)
            # explicit dtypes: a flat shard may hold no FP8 weight at all, and
            # still takes part in the amax exchange through empty lists
            self.L_x8 = mk(xs, True, "bf16")
            if self.flat:
                A.amp_tensor_list_set_amax_slots(self.L_x8, [x for x in slots if x >= 0],
                                                 stream=stream)
            self.L_q = mk(self.fp8, True, fp8_format)
            self.L_qt = mk(self.fp8_t, True, fp8_format)
        # amax / inv_scale entries: one per FP8 weight of this object, or (flat
        # shards) one per FP8 weight of the whole model
        self.n_amax = int(n_fp8_total) if self.flat else self.n_fp8
        self.amax = torch.zeros(max(self.n_amax, 1), dtype=torch.float32, device=dev)
        self.inv_scale = torch.zeros(max(self.n_amax, 1), dtype=torch.float32, device=dev)
        if fp8_scaling == "delayed" and fp8_shapes is not None and not self.n_fp8:
            # no FP8 weight in this set (a data-parallel shard can own none):
            # nothing to cast and no history to keep, so the step is the plain
            # one, with the same exchanges as the other ranks
            fp8_scaling = "dynamic"
        self.fp8_scaling = fp8_scaling
        self.hist_len = amax_history_len
        self.sr_seed = sr_seed
        if sr_seed is not None and not emit_bf16:
            raise ValueError("stochastic rounding applies to the emitted copies (emit_bf16=True)")
        if fp8_scaling == "delayed":
            if not self.n_fp8 or max_norm is not None:
                raise ValueError("delayed FP8 scaling needs FP8 weights and no clipping")
            self._setup_delayed(fp8_shapes, stream)
        elif fp8_scaling != "dynamic":
            raise ValueError(fp8_scaling)
        else:
            self._emit_working_copies(stream)

    def _groups(self, grads):
        """1-D lists of the plain tensors and 2-D lists of the FP8 weights."""
        mk = lambda ts, two_d=False, dt=None: A.amp_tensor_list_create(ts, two_d=two_d, dtype=dt,
                                                                        stream=self.stream)
        plain = [i for i, sh in enumerate(self.fp8_shapes) if sh is None]
        fp8 = [i for i, sh in enumerate(self.fp8_shapes) if sh is not None]
        v2 = lambda ts: [ts[i].view(*self.fp8_shapes[i]) for i in fp8]
        gdt = A.dtype_name(grads[0])
        P = (mk([self.master[i] for i in plain], dt="f32"), mk([self.exp_avg[i] for i in plain], dt="f32"),
             mk([self.exp_avg_sq[i] for i in plain], dt="f32"), mk([grads[i] for i in plain], dt=gdt),
             mk([self.bf16[i] for i in plain], dt="bf16"))
        F = (mk(v2(self.master), True), mk(v2(self.exp_avg), True), mk(v2(self.exp_avg_sq), True),
             mk(v2(grads), True), mk(v2(self.bf16), True))
        return P, F

    def _setup_delayed(self, fp8_shapes, stream):
        self.fp8_shapes = list(fp8_shapes)
        dev = self.scale.device
        self.amax_history = torch.zeros((self.n_fp8, self.hist_len), dtype=torch.float32,
                                        device=dev)
        self.delayed_groups = [self._groups(self.grads)]
        # the first working copies; their amax opens the history
        self._emit_working_copies(stream)

    def _emit_working_copies(self, stream):
        """The working copies before the first step, for the first forward
        pass: bf16 = RNE(master) (amp_emit_bf16, which folds the FP8 weights'
        amax) and the FP8 copies cast dynamically from that amax.  With
        delayed scaling that amax is the first entry of each history.  amax is
        left zeroed for the first step's fold."""
        if self.bf16 is None:
            return
        A.amp_emit_bf16(self.L_master, self.L_b, self.amax if self.n_fp8 else None, stream=stream)
        if not self.n_fp8 and not self.flat:
            return
        self._combine_amax(stream)
        if not self.n_fp8:
            with torch.cuda.stream(stream) if stream is not None else _nullctx():
                self.amax.zero_()
            return
        A.fp8_quant_tensorwise_list(self.L_x8, self.L_q, self.L_qt, self.fp8_format, self.amax,
                                    self.inv_scale, eps=self.fp8_eps, stream=stream)
        with torch.cuda.stream(stream) if stream is not None else _nullctx():
            if self.fp8_scaling == "delayed":
                self.amax_history[:, 0].copy_(self.amax[:self.n_fp8])
            self.amax.zero_()

    @property
    def launches_per_step(self) -> int:
        """Kernels one step enqueues (check [+ norm reduce], AdamW prologue + main,
        [quant], update; delayed FP8: check, prologue, plain + FP8 mains, update)."""
        health = 1 if self.min_scale is not None else 0
        if self.fp8_scaling == "delayed":
            return 5 + health
        return 4 + (1 if self.n_fp8 else 0) + (1 if self.max_norm is not None else 0) + health

    def add_grad_buffer(self, grads) -> int:
        """Register another set of gradient buffers (same shapes and dtype) and
        return its index for step(grad_buffer=...): with two buffers the host
        can fill one while the GPU steps on the other."""
        grads = list(grads)
        if [g.numel() for g in grads] != [g.numel() for g in self.grads] or \
                any(a.dtype != b.dtype for a, b in zip(grads, self.grads)):
            raise ValueError("gradient buffers must match the first set in sizes and dtype")
        self.grad_lists.append(A.amp_tensor_list_create(
            grads, dtype=None if grads else self.L_g.dtype, stream=self.stream))
        if self.fp8_scaling == "delayed":
            self.delayed_groups.append(self._groups(grads))
        return len(self.grad_lists) - 1

    def capture_graph(self, stream=None, grad_buffer: int = 0):
        """Record one step into a CUDA graph; later step() calls on the same
        gradient buffer replay it.  Every call of the step is stream-ordered
        and allocation-free, so the graph is the same calls with the same
        device pointers; the caller keeps writing each step's gradients into
        the same buffers.  With data_parallel over more than one rank the
        exchanges are recorded too, which needs collectives that can be
        captured (NCCL's; gloo's run on the host and cannot be)."""
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
        if self.fp8_scaling == "delayed":
            P, F = self.delayed_groups[grad_buffer]
            A.amp_unscale_check(L_g, self.scale, self.found_inf, stream=s)
            self._combine(s)
            if self.sr_seed is None:
                A.amp_adamw_master_step_fp8_delayed(P, F, self.L_q, self.L_qt, self.fp8_format,
                                                    self.amax_history, self.hist_len, self.amax,
                                                    self.inv_scale, self.scale, self.found_inf,
                                                    self.step_count, *self.hyper,
                                                    fp8_eps=self.fp8_eps, stream=s)
            else:
                A.amp_adamw_master_step_fp8_delayed_sr(P, F, self.L_q, self.L_qt, self.fp8_format,
                                                       self.amax_history, self.hist_len,
                                                       self.amax, self.inv_scale, self.scale,
                                                       self.found_inf, self.step_count,
                                                       *self.hyper, self.sr_seed,
                                                       fp8_eps=self.fp8_eps, stream=s)
            A.amp_update_scale_fp8_history(self.scale, self.growth_tracker, self.found_inf,
                                           self.growth, self.backoff, self.interval, self.amax,
                                           self.amax_history, self.n_fp8, self.hist_len,
                                           stream=s)
            self._health(s)
            return
        sr = self.sr_seed is not None
        if self.max_norm is None:
            A.amp_unscale_check(L_g, self.scale, self.found_inf, stream=s)
            self._combine(s)
            if sr:
                A.amp_adamw_master_step_sr(self.L_master, self.L_m, self.L_v, L_g, self.L_b,
                                           self.scale, self.found_inf, self.step_count,
                                           *self.hyper, self.sr_seed, amax=amax, stream=s)
            else:
                A.amp_adamw_master_step(self.L_master, self.L_m, self.L_v, L_g, self.L_b,
                                        self.scale, self.found_inf, self.step_count, *self.hyper,
                                        amax=amax, stream=s)
        else:
            A.amp_unscale_check_norm(L_g, self.scale, self.found_inf, self.grad_sumsq, stream=s)
            self._combine(s, norm=True)
            if sr:
                A.amp_adamw_master_step_clip_sr(self.L_master, self.L_m, self.L_v, L_g, self.L_b,
                                                self.scale, self.found_inf, self.step_count,
                                                *self.hyper, self.grad_sumsq, self.max_norm,
                                                self.sr_seed, amax=amax, stream=s)
            else:
                A.amp_adamw_master_step_clip(self.L_master, self.L_m, self.L_v, L_g, self.L_b,
                                             self.scale, self.found_inf, self.step_count,
                                             *self.hyper, self.grad_sumsq, self.max_norm,
                                             amax=amax, stream=s)
        self._combine_amax(s)
        if self.n_fp8:
            if sr:
                A.fp8_quant_tensorwise_list_sr(self.L_x8, self.L_q, self.L_qt, self.fp8_format,
                                               self.amax, self.inv_scale, self.sr_seed,
                                               self.step_count, eps=self.fp8_eps,
                                               skip_if=self.found_inf, stream=s)
            else:
                A.fp8_quant_tensorwise_list(self.L_x8, self.L_q, self.L_qt, self.fp8_format,
                                            self.amax, self.inv_scale, eps=self.fp8_eps,
                                            skip_if=self.found_inf, stream=s)
        A.amp_update_scale(self.scale, self.growth_tracker, self.found_inf, self.growth,
                           self.backoff, self.interval, amax=self.amax if self.n_amax else None,
                           n_amax=self.n_amax, stream=s)
        self._health(s)

    def _combine(self, s, norm: bool = False):
        """All-reduce(MAX) of found_inf over the data-parallel group, and with
        norm the all-reduce(SUM) of grad_sumsq, on stream s."""
        if not self.data_parallel:
            return
        from .sharded import combine_found_inf, combine_grad_sumsq
        with torch.cuda.stream(s) if s is not None else _nullctx():
            combine_found_inf(self.found_inf, self.dp_group)
            if norm:
                combine_grad_sumsq(self.grad_sumsq, self.dp_group)

    def _combine_amax(self, s):
        """Flat data-parallel shards: all-reduce(MAX) of the amax array over the
        group, so every rank casts its band with its weight's global amax."""
        if not (self.flat and self.data_parallel):
            return
        from .sharded import combine_amax
        with torch.cuda.stream(s) if s is not None else _nullctx():
            combine_amax(self.amax, self.dp_group)

    def _health(self, s):
        if self.min_scale is not None:
            A.amp_scale_health(self.scale, self.min_scale, self.health_word, stream=s)

    def health(self) -> int:
        """Sticky health bits of the loss scale (0 when min_scale is None); no sync."""
        return 0 if self.health_word is None else int(self.health_word[0])

    def check(self, stream=None):
        """Raise AmpError(AMP_ETIMEOUT) if an AdamW kernel's bounded wait on its
        bulk copies gave up since the last check (synchronises)."""
        holder = self.L_q if self.fp8_scaling == "delayed" else self.L_master
        A.amp_tensor_list_check(holder, stream=stream if stream is not None else self.stream)

    def state(self, stream=None) -> dict:
        """Host copy of the scaler/optimizer counters (amp_read_state), read on
        `stream` (default: the object's stream, else the current one), which it
        synchronises: pass the stream the steps ran on."""
        s = stream if stream is not None else self.stream
        st = self._state_host
        A.amp_read_state(self.scale, self.growth_tracker, self.step_count, self.found_inf, st,
                         stream=s)
        if s is None:
            torch.cuda.current_stream(self.scale.device).synchronize()
        else:
            s.synchronize()
        return {"scale": float(st.scale), "growth_tracker": int(st.growth_tracker),
                "step": int(st.step), "found_inf": int(st.found_inf)}

    def state_dict(self) -> dict:
        """Host copies of everything a resumed run needs: master, m, v, the
        bf16 and FP8 copies, the scaler and step counters, FP8 scales and the
        amax history.  Synchronises."""
        cpu = lambda ts: [t.detach().cpu().clone() for t in ts]
        d = {"master": cpu(self.master), "exp_avg": cpu(self.exp_avg),
             "exp_avg_sq": cpu(self.exp_avg_sq),
             "bf16": cpu(self.bf16) if self.bf16 is not None else None,
             "fp8": cpu(self.fp8), "fp8_t": cpu(self.fp8_t),
             "scale": self.scale.cpu().clone(), "growth_tracker": self.growth_tracker.cpu().clone(),
             "step": self.step_count.cpu().clone(), "found_inf": self.found_inf.cpu().clone(),
             "amax": self.amax.cpu().clone(), "inv_scale": self.inv_scale.cpu().clone()}
        if self.fp8_scaling == "delayed":
            d["amax_history"] = self.amax_history.cpu().clone()
        return d

    def load_state_dict(self, d: dict):
        """Copy a state_dict() back into this step's device buffers (same
        parameter set and options); the list handles keep pointing at them."""
        def put(dst, src):
            for a, b in zip(dst, src):
                a.copy_(b)
        put(self.master, d["master"])
        put(self.exp_avg, d["exp_avg"])
        put(self.exp_avg_sq, d["exp_avg_sq"])
        if self.bf16 is not None and d["bf16"] is not None:
            put(self.bf16, d["bf16"])
        put(self.fp8, d["fp8"])
        put(self.fp8_t, d["fp8_t"])
        for name in ("scale", "growth_tracker", "step_count", "found_inf", "amax", "inv_scale"):
            getattr(self, name).copy_(d["step" if name == "step_count" else name])
        if self.fp8_scaling == "delayed":
            self.amax_history.copy_(d["amax_history"])
        torch.cuda.synchronize(self.scale.device)

    def state_fp8(self) -> dict:
        """Host copies of the FP8 scaling state (synchronises)."""
        d = {"amax": self.amax[:self.n_amax].cpu(), "inv_scale": self.inv_scale[:self.n_amax].cpu()}
        if self.fp8_scaling == "delayed":
            d["amax_history"] = self.amax_history.cpu()
        return d

    def close(self):
        for name in ("L_master", "L_m", "L_v", "L_b", "L_x8", "L_q", "L_qt"):
            lst = getattr(self, name, None)
            if lst is not None:
                lst.close()
        for lst in self.grad_lists:
            lst.close()
        for P, F in getattr(self, "delayed_groups", []):
            for lst in P + F:
                lst.close()
