"""One DP rank's blockwise-FP8 ZeRO-1 optimizer, sequencing the C-ABI calls.

"面向 Blockwise FP8 量化的 ZeRO 优化器设计" §总结 gives the order this class
follows on its shard [b0, b1):
  init : fold the row-major FP32 master params (and moments) into the 1-D
         block buffers of the shard (§参数布局变换, §块粒度切分);
  step : fold the (reduced) row-major grads of the shard, global grad norm
         ("DeepSpeed ZeRO 优化" §七), fused unscale + clip + AdamW + per-block
         E4M3 quantise, unfold the codes back into the row-major FP8 params;
         with ``fused=True`` (the default) that is two kernels: the norm read
         straight from the row-major grads, and the step reading the grads
         through the block table and writing the codes row-major;
         the scales need no unfold: block order (e, rb, cb) makes the scale
         buffer of a param a [E, R/128, C/128] view.
  host : read found_inf and update the loss scale / step count (§六).
Every step of the path runs in libfp8z1.so; this class only owns torch
buffers and calls the entry points in order.  One process, one GPU: with
dp_size > 1 the other ranks' norm partials come through ``norm_hook``.

The step loops (same results):
  step / launch_step + finish_step     one step at a time;
  launch_step_async + drain            each step enqueued before the previous
                                       one's found_inf is read (_AsyncSteps);
  step_from_host (+ finish_host_step)  grads from pinned host memory, FP8
                                       weights back to it, copies overlapped;
  capture -> CapturedStep              the step as a CUDA graph.
MxShardOptimizer runs the MXFP8 variant (one step at a time, or async).
"""
from __future__ import annotations

import ctypes as C
import json
from collections import OrderedDict
from typing import Callable, List, Optional, Sequence

import torch

from . import fp8z1 as F


def shard_scale_view(layout, scales: torch.Tensor, b0: int, b1: int, param: int):
    """``(e0, view)`` over the experts of ``param`` whose blocks all lie in the
    shard [b0, b1), where ``scales`` holds the shard's b1 - b0 block scales
    (block b0 first); None when there are none.  The block order is the
    layout's (fp8z1_param_blocks): the view is a slice of ``scales``."""
    g = F.fp8z1_param_blocks(layout, param, b0, b1)
    if g.e_end <= g.e_begin:
        return None
    per = g.row_blocks * g.col_blocks
    lo = g.first_block + g.e_begin * per - b0
    n = g.e_end - g.e_begin
    return g.e_begin, scales[lo:lo + n * per].view(n, g.row_blocks, g.col_blocks)


class _AsyncSteps:
    """Steps enqueued ahead of their found_inf, shared by both optimizers.

    The method reads found_inf after every step to set the next step's t
    and S ("DeepSpeed ZeRO 优化" §六).  Here the host reads it one step late:
    while step k-1 may still run, step k is enqueued with both candidate
    hyper-parameter sets (step k-1 clean: t+1 and S after growth; skipped: t
    and S/2), and its kernel picks one by step k-1's found_inf (the *_select
    entry points).  Each step's norm accumulators alternate between two slots,
    and its found_inf is copied to pinned memory right after its norm, on a
    side stream, so that the update does not wait for the copy; the host waits
    only for that copy of step k-2 before enqueuing step k (whose norm then
    reuses the slot).  Results equal the synchronous steps'."""

    def _async_launch(self, norm, step, stream, events) -> List[int]:
        """norm(sumsq, found, s) enqueues the norm; step(hp, hp_if_set,
        d_select, sumsq, found, s) the update (hp_if_set / d_select None when
        no step is unresolved)."""
        st = getattr(self, "_async", None)
        if st is None:
            st = self._async = {
                "sumsq": torch.zeros(2, dtype=torch.float64, device=self.device),
                "found": torch.zeros(2, dtype=torch.int32, device=self.device),
                "flags": [torch.zeros(1, dtype=torch.int32, pin_memory=True) for _ in range(2)],
                "done": [torch.cuda.Event() for _ in range(2)],
                "normed": [torch.cuda.Event() for _ in range(2)],
                "side": torch.cuda.Stream(self.device),  # the flag copies
                "k": 0, "inflight": [],  # slots of unresolved steps, oldest first
            }
        s = self._torch_stream(stream, self.device)
        resolved = []
        while len(st["inflight"]) >= 2:  # resolve step k-2: its flag copy ran long ago
            resolved.append(self._resolve_async())
        slot = st["k"] % 2
        st["k"] += 1
        sumsq, found = st["sumsq"][slot:slot + 1], st["found"][slot:slot + 1]
        ev = events or {}
        if "norm" in ev:
            ev["norm"][0].record(s)
        F.fp8z1_norm_reset(sumsq, found, s)
        norm(sumsq, found, s)
        if self.norm_hook is not None:
            with torch.cuda.stream(s):
                self.norm_hook(sumsq, found)
        if "norm" in ev:
            ev["norm"][1].record(s)
        st["normed"][slot].record(s)
        side = st["side"]
        side.wait_event(st["normed"][slot])
        with torch.cuda.stream(side):
            st["flags"][slot].copy_(found, non_blocking=True)
        st["done"][slot].record(side)
        if "step" in ev:
            ev["step"][0].record(s)
        if not st["inflight"]:
            step(self._hp_after(None), None, None, sumsq, found, s)
        else:
            prev = st["inflight"][0]
            step(self._hp_after(0), self._hp_after(1), st["found"][prev:prev + 1], sumsq, found, s)
        if "step" in ev:
            ev["step"][1].record(s)
        st["inflight"].append(slot)
        # the latest step's accumulators, for stats() once drained
        self.sumsq, self.found_inf = sumsq, found
        return resolved

    @staticmethod
    def _torch_stream(stream, device):
        """A torch stream for ``stream`` (None: the current one; a raw
        cudaStream_t is wrapped)."""
        if stream is None:
            return torch.cuda.current_stream(device)
        return stream if isinstance(stream, torch.cuda.Stream) else torch.cuda.ExternalStream(stream)

    def _run_norm_hook(self, stream):
        """The norm hook (the other ranks' partials), on the step's stream."""
        if self.norm_hook is not None:
            with torch.cuda.stream(self._torch_stream(stream, self.device)):
                self.norm_hook(self.sumsq, self.found_inf)

    def _async_busy(self) -> bool:
        st = getattr(self, "_async", None)
        return st is not None and bool(st["inflight"])

    def _hp_after(self, found_prev: Optional[int]):
        """The hyper-parameters of the next step, given the resolved scaler and,
        when one step is unresolved, its found_inf."""
        sc = self.scaler
        if found_prev is not None:
            sc = F.fp8z1_loss_scaler(sc.scale, sc.step, sc.good_steps, sc.growth_interval)
            F.fp8z1_scaler_update(sc, int(found_prev))
        return F.make_hp(step=sc.step + 1, loss_scale=sc.scale, **self.hp)

    def _resolve_async(self) -> int:
        st = self._async
        slot = st["inflight"].pop(0)
        st["done"][slot].synchronize()
        found = int(st["flags"][slot].item())
        F.fp8z1_scaler_update(self.scaler, found)
        return found

    def drain(self) -> List[int]:
        """Wait for every step enqueued by ``launch_step_async`` and return
        their found_inf, oldest first (the loss scaler and t then count them)."""
        out = []
        while self._async_busy():
            out.append(self._resolve_async())
        return out


class ShardOptimizer(_AsyncSteps):
    def __init__(self, shapes: Sequence[Sequence[int]], *, dp_size: int = 1, rank: int = 0,
                 lr=1e-3, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.1, max_norm=1.0,
                 loss_scale=1024.0, growth_interval=1000, device="cuda", fused: bool = True):
        self.device = torch.device(device)
        self.layout = F.fp8z1_build_layout(shapes, dp_size)
        self.shapes = self.layout.shapes
        self.b0, self.b1 = F.fp8z1_shard_range(self.layout, rank)
        self.nblk, self.n_padded, self.n_real = F.fp8z1_layout_info(self.layout)
        nb = self.b1 - self.b0
        n = nb * F.BLOCK_ELEMS
        kw = dict(device=self.device)
        self.master = torch.zeros(n, dtype=torch.float32, **kw)
        self.m = torch.zeros(n, dtype=torch.float32, **kw)
        self.v = torch.zeros(n, dtype=torch.float32, **kw)
        self.fused = fused
        # the folded grads are only materialised on the unfused path
        self.grad = None if fused else torch.zeros(n, dtype=torch.float32, **kw)
        self.codes = torch.zeros(n, dtype=torch.uint8, **kw)
        self.scales = torch.ones(nb, dtype=torch.float32, **kw)
        self.sumsq = torch.zeros(1, dtype=torch.float64, **kw)
        self.found_inf = torch.zeros(1, dtype=torch.int32, **kw)
        self.hp = dict(lr=lr, beta1=beta1, beta2=beta2, eps=eps, weight_decay=weight_decay,
                       max_norm=max_norm)
        self.scaler = F.fp8z1_loss_scaler(float(loss_scale), 0, 0, int(growth_interval))
        self.norm_hook: Optional[Callable[[torch.Tensor, torch.Tensor], None]] = None
        self._ptr_cache: "OrderedDict[tuple, torch.Tensor]" = OrderedDict()
        self._host_pending: Optional[int] = None  # step_from_host(wait=False) in flight
        self._host_slot = 0
        self._async = None  # launch_step_async state, made on first use

    # -- pointer arrays for fold/unfold ------------------------------------
    _PTR_CACHE = 16  # distinct tensor sets whose device pointer arrays are kept

    def pointers(self, tensors: Sequence[torch.Tensor]) -> torch.Tensor:
        """The device array of the params' data pointers that the step calls
        read.  A step loop over the same tensors can pass it instead of the
        tensor list, which spares the per-call check of every tensor (it
        matters with thousands of params)."""
        return self._ptrs(tensors)

    def _ptrs(self, tensors) -> torch.Tensor:
        """Device array of the tensors' data pointers (cached per tensor set);
        a device int64 array of n_params pointers passes through."""
        if isinstance(tensors, torch.Tensor):
            if tensors.dtype != torch.int64 or tensors.numel() != len(self.shapes) or tensors.device.type != "cuda":
                raise ValueError("a pointer array must be a device int64 tensor with one entry per param")
            return tensors
        if len(tensors) != len(self.shapes):
            raise ValueError(f"expected {len(self.shapes)} tensors, got {len(tensors)}")
        for t, shp in zip(tensors, self.shapes):
            if tuple(t.shape) != tuple(shp) and t.numel() != shp[0] * shp[1] * shp[2]:
                raise ValueError(f"a tensor of shape {tuple(t.shape)} for a param of shape {shp}")
            if not t.is_contiguous():
                raise ValueError("param tensors must be contiguous (row-major)")
        key = tuple(t.data_ptr() for t in tensors)
        hit = self._ptr_cache.get(key)
        if hit is None:
            hit = F.param_pointers(tensors, self.device)
            self._ptr_cache[key] = hit
            if len(self._ptr_cache) > self._PTR_CACHE:
                self._ptr_cache.popitem(last=False)
        else:
            self._ptr_cache.move_to_end(key)
        return hit

    def fold_into(self, params: Sequence[torch.Tensor], dst: torch.Tensor, stream=None):
        esz = params[0].element_size()
        F.fp8z1_fold(self.layout, self._ptrs(params), dst, esz, self.b0, self.b1, stream)

    def unfold_from(self, src: torch.Tensor, params: Sequence[torch.Tensor], stream=None):
        esz = params[0].element_size()
        F.fp8z1_unfold(self.layout, src, self._ptrs(params), esz, self.b0, self.b1, stream)

    # -- state --------------------------------------------------------------
    def init_state(self, master: Sequence[torch.Tensor], m=None, v=None, stream=None):
        """Fold row-major FP32 params (and optionally moments) into the shard."""
        self.fold_into(master, self.master, stream)
        if m is not None:
            self.fold_into(m, self.m, stream)
        if v is not None:
            self.fold_into(v, self.v, stream)

    def scale_view(self, param: int):
        """The scales of param ``param``'s experts that this shard holds whole,
        as ``(e0, view)``: ``view[e - e0, rb, cb]`` is the scale of block
        (e, rb, cb) of the param, a [n, ceil(R/128), ceil(C/128)] view of the
        scale buffer (no copy).  None when the shard holds no whole expert of
        the param.  Where the blocks sit comes from the layout
        (fp8z1_param_blocks)."""
        return shard_scale_view(self.layout, self.scales, self.b0, self.b1, param)

    def scale_views(self) -> List[Optional[torch.Tensor]]:
        """Per param, its [E, ceil(R/128), ceil(C/128)] scale tensor as a view
        of the scale buffer when this shard holds the whole param, else None
        ("面向 Blockwise FP8 量化的 ZeRO 优化器设计" §总结: the 1-D blockwise
        scales unfolded back into 2-D / 3-D scales)."""
        out = []
        for p, shp in enumerate(self.shapes):
            v = self.scale_view(p)
            out.append(v[1] if v is not None and v[0] == 0 and v[1].shape[0] == shp[0] else None)
        return out

    # -- checkpoint / resume --------------------------------------------------
    def state_dict(self) -> dict:
        """Everything a resumed run needs: the shard's folded FP32 master / m /
        v, the codes and scales, and the host scalars (t, S, clean-step count).
        The buffers are the 1-D block layout itself, so a reload is a copy."""
        self.finish_host_step()
        self.drain()
        return {
            "shapes": [tuple(s) for s in self.shapes], "b0": self.b0, "b1": self.b1,
            "master": self.master.cpu(), "m": self.m.cpu(), "v": self.v.cpu(),
            "codes": self.codes.cpu(), "scales": self.scales.cpu(), "hp": dict(self.hp),
            "scaler": {"scale": self.scaler.scale, "step": self.scaler.step,
                       "good_steps": self.scaler.good_steps,
                       "growth_interval": self.scaler.growth_interval},
        }

    def load_state_dict(self, sd: dict):
        self.finish_host_step()
        self.drain()
        if [tuple(s) for s in sd["shapes"]] != [tuple(s) for s in self.shapes] or \
                (sd["b0"], sd["b1"]) != (self.b0, self.b1):
            raise ValueError("checkpoint was taken for another layout or shard")
        for name in ("master", "m", "v", "codes", "scales"):
            getattr(self, name).copy_(sd[name])
        self.hp = dict(sd["hp"])
        sc = sd["scaler"]
        self.scaler = F.fp8z1_loss_scaler(sc["scale"], sc["step"], sc["good_steps"],
                                          sc["growth_interval"])

    # -- one step -------------------------------------------------------------
    def launch_step(self, grads: Sequence[torch.Tensor], fp8_params: Optional[Sequence[torch.Tensor]],
                    stream=None):
        """Enqueue one step (no host synchronisation)."""
        if self._host_pending is not None:
            raise RuntimeError("a step_from_host(wait=False) is in flight: call finish_host_step() first")
        if self._async_busy():
            raise RuntimeError("steps from launch_step_async are in flight: call drain() first")
        F.fp8z1_norm_reset(self.sumsq, self.found_inf, stream)
        hp = F.make_hp(step=self.scaler.step + 1, loss_scale=self.scaler.scale, **self.hp)
        if self.fused:
            gptrs = self._ptrs(grads)
            F.fp8z1_fold_norm(self.layout, gptrs, None, self.b0, self.b1, self.sumsq, self.found_inf,
                              stream)
            self._run_norm_hook(stream)
            # codes go row-major when FP8 params are given, else to the folded buffer
            F.fp8z1_step_fused(self.layout, hp, d_grad_params=gptrs, master_shard=self.master,
                               m_shard=self.m, v_shard=self.v,
                               fp8_shard=self.codes if fp8_params is None else None,
                               d_fp8_params=None if fp8_params is None else self._ptrs(fp8_params),
                               scale_shard=self.scales, b0=self.b0, b1=self.b1, d_sumsq=self.sumsq,
                               d_found_inf=self.found_inf, stream=stream)
            return
        self.fold_into(grads, self.grad, stream)
        F.fp8z1_grad_norm(self.layout, self.grad, self.b0, self.b1, self.sumsq, self.found_inf, stream)
        self._run_norm_hook(stream)
        F.fp8z1_step(self.layout, hp, self.grad, self.master, self.m, self.v, self.codes, self.scales,
                     self.b0, self.b1, self.sumsq, self.found_inf, stream)
        if fp8_params is not None:
            self.unfold_from(self.codes, fp8_params, stream)

    # -- host-resident grads and FP8 weights ----------------------------------
    def _host_chunks(self, target_blocks: int):
        """Contiguous block ranges of this shard whose grads are contiguous rows
        of one param (one expert, or a run of row blocks of a 2-D weight), read
        off the library's block table: (param, expert, row0, row1, k0, k1)."""
        lut = F.fp8z1_copy_lut(self.layout)[self.b0:self.b1]
        out = []
        k = 0
        n = len(lut)
        while k < n:
            p, e, rb = int(lut["param"][k]), int(lut["expert"][k]), int(lut["row_block"][k])
            j = k
            while (j < n and int(lut["param"][j]) == p and int(lut["expert"][j]) == e
                   and (j - k < target_blocks or int(lut["row_block"][j]) == int(lut["row_block"][j - 1]))):
                j += 1
            rb_last = int(lut["row_block"][j - 1])
            rows_last = int(lut["rows_real"][j - 1])
            out.append((p, e, 128 * rb, 128 * rb_last + rows_last, self.b0 + k, self.b0 + j))
            k = j
        return out

    def step_from_host(self, host_grads: Sequence[torch.Tensor], host_fp8: Sequence[torch.Tensor],
                       host_scales: Optional[torch.Tensor] = None, grads: Optional[Sequence[torch.Tensor]] = None,
                       fp8_params: Optional[Sequence[torch.Tensor]] = None, target_blocks: int = 1792,
                       wait: bool = True) -> Optional[int]:
        """One step whose grads arrive from (pinned) host memory and whose FP8
        weights (and scales) go back to it, with the copies overlapped: chunk
        c's grads are copied on a copy stream while chunk c-1's norm runs, and
        after the norm chunk c's update runs while chunk c-1's FP8 weights are
        copied back.  ``grads`` / ``fp8_params`` are the device tensors used
        (allocated on first use when not given).  Fused path, whole-buffer
        shards only: the copies move whole rows, and a shard that starts or
        ends inside a row of blocks would copy back rows it did not update.
        Host tensors should be pinned for the copies to overlap.

        ``wait=False`` returns None once the step is enqueued, so that the
        next call's grads go in while this step's update runs and its FP8
        weights come out.  A chunk's grads then wait only for this step's
        update of that chunk, and its update waits only for this step's copy
        of that chunk's FP8 weights.  The step's found_inf is read when the next
        call needs t and S (the norm has long finished by then), or by
        ``finish_host_step``, which also waits for the copies back: the host
        FP8 weights and scales are complete only after it."""
        assert self.fused, "step_from_host runs the fused path"
        if self._async_busy():
            raise RuntimeError("steps from launch_step_async are in flight: call drain() first")
        if (self.b0, self.b1) != (0, self.nblk):
            raise ValueError("step_from_host needs the whole buffer as the shard (dp_size 1)")
        if grads is None:
            grads = getattr(self, "_dev_grads", None) or [torch.empty(s, dtype=torch.float32, device=self.device)
                                                          for s in self.shapes]
            self._dev_grads = grads
        if fp8_params is None:
            fp8_params = getattr(self, "_dev_fp8", None) or [torch.empty(s, dtype=torch.uint8, device=self.device)
                                                             for s in self.shapes]
            self._dev_fp8 = fp8_params
        if getattr(self, "_chunks_cache", None) is None or self._chunks_cache[0] != target_blocks:
            if self._host_pending is not None:
                self.finish_host_step()
            chunks = self._host_chunks(target_blocks)
            self._chunks_cache = (target_blocks, chunks)
            self._copy_in = torch.cuda.Stream(self.device)
            self._copy_out = torch.cuda.Stream(self.device)
            self._flags = [torch.zeros(1, dtype=torch.int32, pin_memory=True) for _ in range(2)]
            self._norm_done = [torch.cuda.Event() for _ in range(2)]
            self._h2d_done = [torch.cuda.Event() for _ in chunks]
            self._upd_done = [torch.cuda.Event() for _ in chunks]
            self._d2h_done = [torch.cuda.Event() for _ in chunks]
            self._scales_done = torch.cuda.Event()
        chunks = self._chunks_cache[1]
        prev = self._host_pending  # the step still in flight, if any
        comp = torch.cuda.current_stream(self.device)
        gptrs, fptrs = self._ptrs(grads), self._ptrs(fp8_params)
        F.fp8z1_norm_reset(self.sumsq, self.found_inf, comp)  # after the previous step's update
        for c, (p, e, r0, r1, k0, k1) in enumerate(chunks):  # grads in, norm as each chunk lands
            with torch.cuda.stream(self._copy_in):
                if prev is not None:
                    self._copy_in.wait_event(self._upd_done[c])
                grads[p][e, r0:r1].copy_(host_grads[p][e, r0:r1], non_blocking=True)
                self._h2d_done[c].record(self._copy_in)
            comp.wait_event(self._h2d_done[c])
            F.fp8z1_fold_norm(self.layout, gptrs, None, k0, k1, self.sumsq, self.found_inf, comp)
        if self.norm_hook is not None:
            self.norm_hook(self.sumsq, self.found_inf)
        slot = self._host_slot
        self._host_slot ^= 1
        self._flags[slot].copy_(self.found_inf, non_blocking=True)
        self._norm_done[slot].record(comp)
        if prev is not None:  # t and S of this step follow the previous step's found_inf
            self._retire_host_step(prev)
        hp = F.make_hp(step=self.scaler.step + 1, loss_scale=self.scaler.scale, **self.hp)
        if prev is not None:
            comp.wait_event(self._scales_done)
        for c, (p, e, r0, r1, k0, k1) in enumerate(chunks):  # update, FP8 weights out as each chunk is done
            if prev is not None:
                comp.wait_event(self._d2h_done[c])
            o = (k0 - self.b0) * F.BLOCK_ELEMS
            F.fp8z1_step_fused(self.layout, hp, d_grad_params=gptrs, master_shard=self.master[o:],
                               m_shard=self.m[o:], v_shard=self.v[o:], d_fp8_params=fptrs,
                               scale_shard=self.scales[k0 - self.b0:], b0=k0, b1=k1, d_sumsq=self.sumsq,
                               d_found_inf=self.found_inf, stream=comp)
            self._upd_done[c].record(comp)
            self._copy_out.wait_event(self._upd_done[c])
            with torch.cuda.stream(self._copy_out):
                host_fp8[p][e, r0:r1].copy_(fp8_params[p][e, r0:r1], non_blocking=True)
                self._d2h_done[c].record(self._copy_out)
        with torch.cuda.stream(self._copy_out):
            if host_scales is not None:
                host_scales.copy_(self.scales, non_blocking=True)
            self._scales_done.record(self._copy_out)
        self._host_pending = slot
        return self.finish_host_step() if wait else None

    def _retire_host_step(self, slot: int) -> int:
        self._norm_done[slot].synchronize()
        found = int(self._flags[slot].item())
        F.fp8z1_scaler_update(self.scaler, found)
        return found

    def finish_host_step(self) -> Optional[int]:
        """Wait for the last ``step_from_host`` to finish, its FP8 weights and
        scales to reach the host, and return its found_inf (None when no step
        is in flight)."""
        if self._host_pending is None:
            return None
        self._copy_out.synchronize()
        found = self._retire_host_step(self._host_pending)
        self._host_pending = None
        return found

    # -- steps enqueued ahead of their found_inf --------------------------------
    def launch_step_async(self, grads, fp8_params, stream=None, events: Optional[dict] = None) -> List[int]:
        """Enqueue one fused step without waiting for the previous one
        (``_AsyncSteps``; fp8z1_step_fused_select).  ``grads`` / ``fp8_params``:
        the param tensors or their ``pointers``.  Returns the found_inf of the
        steps resolved by this call, oldest first; ``drain`` resolves the
        rest.  ``events``: optional {"norm": (start, end), "step": (start,
        end)} CUDA events to record around the two kernels on ``stream``."""
        if not self.fused:
            raise ValueError("launch_step_async runs the fused path")
        if self._host_pending is not None:
            raise RuntimeError("a step_from_host(wait=False) is in flight: call finish_host_step() first")
        gptrs = self._ptrs(grads)
        fptrs = None if fp8_params is None else self._ptrs(fp8_params)

        def norm(sumsq, found, s):
            F.fp8z1_fold_norm(self.layout, gptrs, None, self.b0, self.b1, sumsq, found, s)

        def step(hp, hp_set, select, sumsq, found, s):
            kw = dict(d_grad_params=gptrs, master_shard=self.master, m_shard=self.m, v_shard=self.v,
                      fp8_shard=self.codes if fptrs is None else None, d_fp8_params=fptrs,
                      scale_shard=self.scales, b0=self.b0, b1=self.b1, d_sumsq=sumsq, d_found_inf=found,
                      stream=s)
            if hp_set is None:
                F.fp8z1_step_fused(self.layout, hp, **kw)
            else:
                F.fp8z1_step_fused_select(self.layout, hp, hp_set, select, **kw)

        return self._async_launch(norm, step, stream, events)

    def finish_step(self) -> int:
        """Read found_inf (synchronises) and update the loss scale and t."""
        found = int(self.found_inf.item())
        F.fp8z1_scaler_update(self.scaler, found)
        return found

    def step(self, grads, fp8_params=None, stream=None) -> int:
        self.launch_step(grads, fp8_params, stream)
        return self.finish_step()

    def capture(self, grads: Sequence[torch.Tensor], fp8_params: Optional[Sequence[torch.Tensor]] = None,
                pool=None, slots: int = 2, mode: str = "auto") -> "CapturedStep":
        """Capture one fused step over these grad (and FP8 weight) tensors in a
        CUDA graph; see ``CapturedStep``."""
        return CapturedStep(self, grads, fp8_params, pool, slots, mode)

    def stats(self, loss_scale: Optional[float] = None) -> dict:
        """Numbers for logging the last step (reads two device scalars): the
        global grad norm and clip coefficient (on this shard's sum of squares,
        after any norm hook), the loss scale the step used (pass it when the
        scaler has moved since), t and S now, whether it was skipped, and how
        many of this shard's blocks have scale 1 (amax 0 -- an all-zero block
        -- or exactly 448)."""
        self.finish_host_step()
        self.drain()
        s = float(self.sumsq.item())
        found = int(self.found_inf.item())
        used = self.scaler.scale if loss_scale is None else loss_scale
        norm, coef = (float("nan"), float("nan")) if found else F.fp8z1_clip_coef(s, self.hp["max_norm"], used)
        return {"global_norm": norm, "clip_coef": coef, "clipped": bool(not found and coef < 1.0),
                "skipped": bool(found), "loss_scale": self.scaler.scale, "step": self.scaler.step,
                "unit_scale_blocks": int((self.scales == 1.0).sum().item())}

    def log_step(self, out, step_ms: Optional[float] = None, **extra) -> dict:
        """Write ``stats()`` (plus the step time, the elements per second of
        this shard, and any ``extra`` keys) as one JSON line to the text file
        ``out``; return the line's dict."""
        line = self.stats()
        if step_ms is not None:
            line["step_ms"] = step_ms
            line["elem_per_s"] = (self.b1 - self.b0) * F.BLOCK_ELEMS / (step_ms / 1e3)
        line.update(extra)
        out.write(json.dumps(line) + "\n")
        return line


class CapturedStep:
    """One fused step of a ``ShardOptimizer`` as a CUDA graph: zero the norm
    accumulators, the norm read from the row-major grads (then the norm hook,
    which is captured too, so it must be capturable: an NCCL all-reduce is),
    and the step.  A replay costs one graph launch however many entry points
    the step has.

    t and S change every step, so the graph cannot replay the scalars it was
    captured with.  Two ways of feeding it this step's:
      "patch"  the step is the by-value kernel (fp8z1_step_fused), and before
               each replay its scalars are rewritten in the instantiated graph
               (fp8z1_graph_set_step_hp): the kernel runs at full speed.
               Needs torch's raw graph handles (CUDAGraph(keep_graph=True)).
      "device" the step reads its scalars from device memory, copied in the
               graph from a pinned slot that ``replay`` rewrites
               (fp8z1_step_fused_dev); the kernel holds the scalars in
               registers and runs a few per cent slower.  The step is captured
               ``slots`` times, each graph copying from its own slot and
               replayed in turn, so the host can enqueue step k+1 before step
               k's copy of its scalars has run.
    "auto" takes "patch" when torch offers it.

    The graph holds the addresses of the tensors it was captured with: each
    step, write the new grads into those same ``grads`` tensors, and read the
    FP8 weights from those ``fp8_params`` (or ``codes`` when None).  t, S and
    the other hyper-parameters are the optimizer's when ``replay`` runs (a
    schedule may change lr); ``step`` also reads found_inf and updates the
    loss scaler, like ``ShardOptimizer.step``."""

    def __init__(self, opt: "ShardOptimizer", grads, fp8_params=None, pool=None, slots: int = 2,
                 mode: str = "auto"):
        if not opt.fused:
            raise ValueError("a captured step runs the fused path")
        if mode == "auto":
            mode = "patch" if self.patch_supported() else "device"
        if mode not in ("patch", "device"):
            raise ValueError(f"unknown mode {mode!r}")
        self.mode = mode
        self.opt = opt
        self.grads = list(grads)
        self.fp8_params = None if fp8_params is None else list(fp8_params)
        # the graph reads these pointer arrays: keep them alive with it
        self._gptrs = opt._ptrs(self.grads)
        self._fptrs = None if fp8_params is None else opt._ptrs(self.fp8_params)
        nsc = C.sizeof(F.fp8z1_step_scalars) // 4
        n_slots = slots if mode == "device" else 0
        self._h = [torch.zeros(nsc, dtype=torch.float32, pin_memory=True) for _ in range(n_slots)]
        self._d = torch.zeros(nsc, dtype=torch.float32, device=opt.device)
        self._done = [torch.cuda.Event() for _ in range(n_slots)]
        self._next = 0
        # load every kernel once outside the capture: found_inf preset makes
        # the step a no-op, and the accumulators are zeroed in the graph
        side = torch.cuda.Stream(opt.device)
        side.wait_stream(torch.cuda.current_stream(opt.device))
        with torch.cuda.stream(side):
            if mode == "device":
                self._write(self._h[0])
            opt.found_inf.fill_(1)
            self._enqueue(self._h[0] if mode == "device" else None, norm_hook=False)
            F.fp8z1_norm_reset(opt.sumsq, opt.found_inf)
        side.synchronize()
        torch.cuda.current_stream(opt.device).wait_stream(side)
        self.graphs = []
        if mode == "patch":
            g = torch.cuda.CUDAGraph(keep_graph=True)
            with torch.cuda.graph(g, pool=pool, stream=side):  # nothing is allocated inside
                F.fp8z1_norm_reset(opt.sumsq, opt.found_inf)
                self._enqueue(None, norm_hook=True)
            g.instantiate()
            self.graphs.append(g)
            self._nodes, self._n_nodes = F.fp8z1_graph_step_nodes(g.raw_cuda_graph())
            if self._n_nodes == 0:
                raise RuntimeError("no step kernel found in the captured graph")
            return
        for h in self._h:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, pool=pool, stream=side):  # nothing is allocated inside
                F.fp8z1_norm_reset(opt.sumsq, opt.found_inf)
                self._enqueue(h, norm_hook=True)
            self.graphs.append(g)

    @staticmethod
    def patch_supported() -> bool:
        """Whether torch exposes the raw graph handles the "patch" mode needs."""
        try:
            torch.cuda.CUDAGraph(keep_graph=True)
        except TypeError:
            return False
        return hasattr(torch.cuda.CUDAGraph, "raw_cuda_graph") and hasattr(torch.cuda.CUDAGraph,
                                                                          "raw_cuda_graph_exec")

    def _hp(self):
        o = self.opt
        return F.make_hp(step=o.scaler.step + 1, loss_scale=o.scaler.scale, **o.hp)

    def _write(self, h: torch.Tensor):
        """This step's scalars into pinned slot ``h``: t and S from the scaler,
        the rest from ``opt.hp`` as it is now (a schedule may change lr)."""
        F.fp8z1_step_scalars_from_hp(self._hp(), h)

    def _enqueue(self, h, norm_hook: bool):
        o = self.opt
        F.fp8z1_fold_norm(o.layout, self._gptrs, None, o.b0, o.b1, o.sumsq, o.found_inf)
        if norm_hook and o.norm_hook is not None:
            o.norm_hook(o.sumsq, o.found_inf)
        kw = dict(d_grad_params=self._gptrs, master_shard=o.master, m_shard=o.m, v_shard=o.v,
                  fp8_shard=o.codes if self._fptrs is None else None, d_fp8_params=self._fptrs,
                  scale_shard=o.scales, b0=o.b0, b1=o.b1, d_sumsq=o.sumsq, d_found_inf=o.found_inf)
        if h is None:
            F.fp8z1_step_fused(o.layout, self._hp(), **kw)
        else:
            F.fp8z1_step_fused_dev(o.layout, h, self._d, **kw)

    def replay(self):
        """Enqueue one step on the current stream (in "device" mode, no host
        synchronisation unless this slot's previous replay has not finished).
        t and S are the scaler's when the step is enqueued: ``finish_step``
        between replays advances them, as with ``ShardOptimizer.launch_step``."""
        if self.mode == "patch":
            g = self.graphs[0]
            F.fp8z1_graph_set_step_hp(g.raw_cuda_graph_exec(), self._nodes, self._n_nodes, self._hp())
            g.replay()
            return
        k = self._next
        self._next = (k + 1) % len(self.graphs)
        self._done[k].synchronize()  # its pinned scalars are about to be overwritten
        self._write(self._h[k])
        self.graphs[k].replay()
        self._done[k].record()

    def step(self) -> int:
        self.replay()
        return self.opt.finish_step()


class MxShardOptimizer(_AsyncSteps):
    """The same optimizer step with MXFP8 weights (E8M0 scale per 32
    consecutive elements) instead of 128x128 blocks.

    The blocks of MXFP8 are memory-contiguous ("面向 Blockwise FP8 量化的 ZeRO
    优化器设计" §Blockwise 量化 / §Blockwise 量化给 ZeRO-1 带来的挑战), so no
    fold or table is needed: the state is the params' row-major elements back
    to back, the shard a flat run of whole groups, and a step is two kernels
    (the grad norm, then the fused update + MX quantise).  Every C must be a
    multiple of 32."""

    def __init__(self, shapes: Sequence[Sequence[int]], *, dp_size: int = 1, rank: int = 0,
                 lr=1e-3, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.1, max_norm=1.0,
                 loss_scale=1024.0, growth_interval=1000, device="cuda"):
        self.device = torch.device(device)
        self.layout = F.fp8z1_mx_build_layout(shapes, dp_size)
        self.shapes = self.layout.shapes
        self.g0, self.g1 = F.fp8z1_mx_shard_range(self.layout, rank)
        self.n_groups, self.n_elems = F.fp8z1_mx_layout_info(self.layout)
        n = (self.g1 - self.g0) * F.MX_GROUP
        kw = dict(device=self.device)
        self.master = torch.zeros(n, dtype=torch.float32, **kw)
        self.m = torch.zeros(n, dtype=torch.float32, **kw)
        self.v = torch.zeros(n, dtype=torch.float32, **kw)
        self.codes = torch.zeros(n, dtype=torch.uint8, **kw)
        self.scales = torch.full((self.g1 - self.g0,), 127, dtype=torch.uint8, **kw)
        self.sumsq = torch.zeros(1, dtype=torch.float64, **kw)
        self.found_inf = torch.zeros(1, dtype=torch.int32, **kw)
        self.hp = dict(lr=lr, beta1=beta1, beta2=beta2, eps=eps, weight_decay=weight_decay,
                       max_norm=max_norm)
        self.scaler = F.fp8z1_loss_scaler(float(loss_scale), 0, 0, int(growth_interval))
        self.norm_hook: Optional[Callable[[torch.Tensor, torch.Tensor], None]] = None

    def shard_of(self, flat: torch.Tensor) -> torch.Tensor:
        """This rank's slice of a whole flat buffer (grads, say)."""
        return flat[self.g0 * F.MX_GROUP:self.g1 * F.MX_GROUP]

    def launch_step_async(self, grad_shard: torch.Tensor, stream=None, events: Optional[dict] = None) -> List[int]:
        """Enqueue one step without waiting for the previous one (``_AsyncSteps``;
        fp8z1_mx_step_select).  Returns the found_inf of the steps resolved by
        this call; ``drain`` resolves the rest."""
        def norm(sumsq, found, s):
            F.fp8z1_mx_grad_norm(self.layout, grad_shard, self.g0, self.g1, sumsq, found, s)

        def step(hp, hp_set, select, sumsq, found, s):
            args = (grad_shard, self.master, self.m, self.v, self.codes, self.scales, self.g0, self.g1, sumsq,
                    found, s)
            if hp_set is None:
                F.fp8z1_mx_step(self.layout, hp, *args)
            else:
                F.fp8z1_mx_step_select(self.layout, hp, hp_set, select, *args)

        return self._async_launch(norm, step, stream, events)

    def launch_step(self, grad_shard: torch.Tensor, stream=None):
        if self._async_busy():
            raise RuntimeError("steps from launch_step_async are in flight: call drain() first")
        F.fp8z1_norm_reset(self.sumsq, self.found_inf, stream)
        F.fp8z1_mx_grad_norm(self.layout, grad_shard, self.g0, self.g1, self.sumsq, self.found_inf,
                             stream)
        self._run_norm_hook(stream)
        hp = F.make_hp(step=self.scaler.step + 1, loss_scale=self.scaler.scale, **self.hp)
        F.fp8z1_mx_step(self.layout, hp, grad_shard, self.master, self.m, self.v, self.codes,
                        self.scales, self.g0, self.g1, self.sumsq, self.found_inf, stream)

    def finish_step(self) -> int:
        found = int(self.found_inf.item())
        F.fp8z1_scaler_update(self.scaler, found)
        return found

    def step(self, grad_shard: torch.Tensor, stream=None) -> int:
        self.launch_step(grad_shard, stream)
        return self.finish_step()

    # -- checkpoint / resume and logging, as ShardOptimizer's ------------------
    def state_dict(self) -> dict:
        self.drain()
        return {
            "shapes": [tuple(s) for s in self.shapes], "g0": self.g0, "g1": self.g1,
            "master": self.master.cpu(), "m": self.m.cpu(), "v": self.v.cpu(),
            "codes": self.codes.cpu(), "scales": self.scales.cpu(), "hp": dict(self.hp),
            "scaler": {"scale": self.scaler.scale, "step": self.scaler.step,
                       "good_steps": self.scaler.good_steps,
                       "growth_interval": self.scaler.growth_interval},
        }

    def load_state_dict(self, sd: dict):
        self.drain()
        if [tuple(s) for s in sd["shapes"]] != [tuple(s) for s in self.shapes] or \
                (sd["g0"], sd["g1"]) != (self.g0, self.g1):
            raise ValueError("checkpoint was taken for another layout or shard")
        for name in ("master", "m", "v", "codes", "scales"):
            getattr(self, name).copy_(sd[name])
        self.hp = dict(sd["hp"])
        sc = sd["scaler"]
        self.scaler = F.fp8z1_loss_scaler(sc["scale"], sc["step"], sc["good_steps"],
                                          sc["growth_interval"])

    def stats(self, loss_scale: Optional[float] = None) -> dict:
        """The last step's global norm, clip coefficient, skip, t and S, and how
        many of this shard's groups have scale 1 (E8M0 code 127)."""
        self.drain()
        s = float(self.sumsq.item())
        found = int(self.found_inf.item())
        used = self.scaler.scale if loss_scale is None else loss_scale
        norm, coef = (float("nan"), float("nan")) if found else F.fp8z1_clip_coef(s, self.hp["max_norm"], used)
        return {"global_norm": norm, "clip_coef": coef, "clipped": bool(not found and coef < 1.0),
                "skipped": bool(found), "loss_scale": self.scaler.scale, "step": self.scaler.step,
                "unit_scale_groups": int((self.scales == 127).sum().item())}
