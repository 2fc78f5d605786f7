"""An emulated data-parallel group on one GPU, driven through libzr's C ABI.

``DPGroup`` owns what each of the N ranks would hold under ZeRO stage 1/2
("Megatron-LM 分布式训练（四）" §"ZeRO 各档"; "DeepSpeed ZeRO 通信优化深度解析"
§二, §三.3): its fp32 master, m and v partition of S elements (views of one
flat buffer per state, partition r at offset rS), its IPG bucket
buffer (reused bucket after bucket, as stage 2 releases it once the slice is
reduced), and the full bf16 parameter buffer the all-gather refreshes. One
``step`` runs, for every bucket in order, the packing of each rank's
per-parameter gradients into its bucket and the fused reduce-scatter + AdamW
+ bf16 cast; nothing here computes, every step is a libzr kernel.
"""
from __future__ import annotations

from typing import List, Optional, Sequence

import torch

from . import zr


class DPGroup:
    def __init__(self, numel: Sequence[int], world: int,
                 reduce_bucket_size: int = zr.ZR_DEFAULT_REDUCE_BUCKET_SIZE,
                 grad_dtype: torch.dtype = torch.bfloat16, device: str = "cuda",
                 allocate_buckets: bool = True, arrival: Optional[Sequence[int]] = None):
        self.layout = zr.Layout(numel, world, reduce_bucket_size, arrival=arrival)
        self.world = world
        self.device = torch.device(device)
        self.grad_dtype = grad_dtype
        self.zr_dtype = {torch.bfloat16: zr.ZR_BF16, torch.float16: zr.ZR_FP16, torch.float32: zr.ZR_FP32}[grad_dtype]
        L = self.layout
        S = L.S
        f32 = dict(dtype=torch.float32, device=self.device)
        # Each state is one flat [P] buffer laid out like the parameters, partition
        # r its view at r*S: partition elements keep the parameters' 16-byte
        # phases, so the fused kernels store the bf16 params in aligned chunks.
        self._flat_state = [torch.zeros(max(L.P, 1), **f32) for _ in range(3)]
        self.master, self.m, self.v = ([buf[r * S:(r + 1) * S] for r in range(world)] for buf in self._flat_state)
        self.param = torch.zeros(max(L.P, 1), dtype=torch.bfloat16, device=self.device)
        self.max_bucket = max((L.bucket(b)[1] for b in range(L.n_buckets)), default=0)
        self.buckets: List[torch.Tensor] = []
        if allocate_buckets:
            self.buckets = [torch.empty(max(self.max_bucket, 1), dtype=grad_dtype, device=self.device)
                            for _ in range(world)]
        self._p_master = zr.PtrArray(self.master)
        self._p_m = zr.PtrArray(self.m)
        self._p_v = zr.PtrArray(self.v)
        self._p_buckets = zr.PtrArray(self.buckets) if self.buckets else None
        self.scale = float(torch.tensor(1.0 / world, dtype=torch.float32).item())

    # ---- state ------------------------------------------------------------------
    def load_flat(self, master: torch.Tensor, m: Optional[torch.Tensor] = None,
                  v: Optional[torch.Tensor] = None) -> None:
        """Scatter flat [T] fp32 state into the N partitions (padding zero)."""
        L = self.layout
        for dst, src in ((self.master, master), (self.m, m), (self.v, v)):
            if src is None:
                continue
            for r in range(self.world):
                lo, hi = r * L.S, min((r + 1) * L.S, L.T)
                dst[r].zero_()
                if hi > lo:
                    dst[r][: hi - lo].copy_(src[lo:hi])

    def flat(self, shards: Sequence[torch.Tensor]) -> torch.Tensor:
        return torch.cat(list(shards))[: self.layout.T]

    def flat_state(self) -> List[torch.Tensor]:
        """master, m and v as the flat [P] buffers whose views are the partitions."""
        return [buf[: self.layout.P] for buf in self._flat_state]

    def grad_table(self, grads: Sequence[Sequence[torch.Tensor]]) -> zr.PtrArray:
        """Host array [world * n_params] of device pointers, built once per set of grads."""
        return zr.PtrArray([t for row in grads for t in row])

    # ---- the step -------------------------------------------------------------------
    def pack(self, b: int, grad_table: zr.PtrArray, stream=None) -> None:
        zr.zr_bucket_pack(self.layout, b, grad_table, self._p_buckets, dtype=self.zr_dtype, stream=stream)

    def pack_plan(self, grad_table: zr.PtrArray) -> zr.PackPlan:
        """Device-resident packing descriptors for these gradient tensors (build once)."""
        return zr.PackPlan(self.layout, grad_table, self._p_buckets, dtype=self.zr_dtype)

    def pack_planned(self, b: int, plan: zr.PackPlan, stream=None) -> None:
        zr.zr_bucket_pack_planned(plan, b, stream=stream)

    def fused(self, b: int, hp, bucket_in: Optional[zr.PtrArray] = None, shard_grad_out=None,
              write_param: bool = True, stream=None) -> None:
        zr.zr_rs_adam_fused(self.layout, b, bucket_in or self._p_buckets, self.scale, self._p_master,
                            self._p_m, self._p_v, hp, self.param if write_param else None,
                            shard_grad_out, dtype=self.zr_dtype, stream=stream)

    def step(self, grad_table: zr.PtrArray, hp, stream=None, plan: Optional[zr.PackPlan] = None) -> None:
        """Every bucket in order: pack each rank's grads, then the fused step."""
        for b in range(self.layout.n_buckets):
            if plan is not None:
                self.pack_planned(b, plan, stream)
            else:
                self.pack(b, grad_table, stream)
            self.fused(b, hp, stream=stream)

    def bucket_plan(self, buffer_set: int = 0) -> zr.DirectPlan:
        """A direct-step plan whose gradients are bucket buffers (set 0: the
        group's own, set 1: step_overlapped's second set): replica k's gradient
        of param i is its slice of bucket buffer k, at the param's offset inside
        its bucket. Once bucket b is packed, zr_step_direct with this plan
        reduces it in flat order, whatever order the params arrived in. Built
        on first use; the bucket buffers stay."""
        plans = self.__dict__.setdefault("_bucket_plans", {})
        if buffer_set not in plans:
            bufs = self.buckets if buffer_set == 0 else getattr(self, "_buckets2", None)
            if not bufs:
                raise ValueError(f"the group has no bucket buffer set {buffer_set}")
            L = self.layout
            boff = L.bucket_positions()
            es = bufs[0].element_size()
            addrs = [int(buf.data_ptr()) + int(o) * es for buf in bufs for o in boff]
            plans[buffer_set] = zr.DirectPlan(L, zr.PtrArray(addrs), dtype=self.zr_dtype)
        return plans[buffer_set]

    def reduce_packed(self, b: int, hp, write_param: bool = True, stream=None, buffer_set: int = 0) -> None:
        """Steps 2-4 of packed bucket b, read from a bucket buffer set in flat
        order (zr_step_direct over bucket_plan): the same result as fused()."""
        self.direct(b, self.bucket_plan(buffer_set), hp, write_param=write_param, stream=stream)

    def step_packed(self, plan: zr.PackPlan, hp, stream=None) -> None:
        """The two-kernel step with the reduction in flat order: every bucket
        packed by its plan, then reduced by reduce_packed."""
        for b in range(self.layout.n_buckets):
            self.pack_planned(b, plan, stream)
            self.reduce_packed(b, hp, stream=stream)

    def overlap_plans(self, grad_table: zr.PtrArray):
        """Two pack plans over two sets of bucket buffers, for step_overlapped:
        bucket b+1 is packed into one set while bucket b is reduced from the
        other (allocated on first use)."""
        if not getattr(self, "_buckets2", None):
            self._buckets2 = [torch.empty(max(self.max_bucket, 1), dtype=self.grad_dtype, device=self.device)
                              for _ in range(self.world)]
            self._p_buckets2 = zr.PtrArray(self._buckets2)
        return (zr.PackPlan(self.layout, grad_table, self._p_buckets, dtype=self.zr_dtype),
                zr.PackPlan(self.layout, grad_table, self._p_buckets2, dtype=self.zr_dtype))

    def step_overlapped(self, plans, hp, stream=None, side_stream=None, flat_order: bool = False) -> None:
        """The two-kernel step with packing and reduction overlapped
        ("DeepSpeed ZeRO 通信优化深度解析" §四, §五 overlap_comm: the copy into the
        IPG bucket and the reduction of the previous bucket run on different
        streams): bucket b+1 is packed on side_stream into one buffer set while
        the fused step reduces bucket b from the other. Events order each
        buffer's reuse; nothing waits on the device. `stream` waits for all
        of it at the end. flat_order: each bucket reduced by reduce_packed
        instead of the fused kernel."""
        cur = stream or torch.cuda.current_stream(self.device)
        side = side_stream or torch.cuda.Stream(self.device)
        nb = self.layout.n_buckets
        if nb == 0:
            return
        sets = (self._p_buckets, self._p_buckets2)
        packed = [torch.cuda.Event() for _ in range(nb)]
        used = [torch.cuda.Event() for _ in range(nb)]
        side.wait_stream(cur)
        with torch.cuda.stream(side):
            zr.zr_bucket_pack_planned(plans[0], 0, stream=side)
            packed[0].record(side)
        for b in range(nb):
            if b + 1 < nb:
                with torch.cuda.stream(side):
                    if b >= 1:
                        side.wait_event(used[b - 1])  # buffer set (b+1) % 2 was read by bucket b-1
                    zr.zr_bucket_pack_planned(plans[(b + 1) % 2], b + 1, stream=side)
                    packed[b + 1].record(side)
            cur.wait_event(packed[b])
            if flat_order:
                self.reduce_packed(b, hp, stream=cur, buffer_set=b % 2)
            else:
                self.fused(b, hp, bucket_in=sets[b % 2], stream=cur)
            used[b].record(cur)
        cur.wait_stream(side)

    def direct_plan(self, grad_table: zr.PtrArray) -> zr.DirectPlan:
        """Device-resident map of these gradient tensors for the direct step (build once)."""
        return zr.DirectPlan(self.layout, grad_table, dtype=self.zr_dtype)

    def direct(self, b: int, plan: zr.DirectPlan, hp, shard_grad_out=None, write_param: bool = True,
               stream=None) -> None:
        zr.zr_step_direct(plan, b, self.scale, self._p_master, self._p_m, self._p_v, hp,
                          self.param if write_param else None, shard_grad_out, stream=stream)

    def step_direct(self, plan: zr.DirectPlan, hp, stream=None, per_bucket: bool = False,
                    param_out: Optional[torch.Tensor] = None) -> None:
        """Steps 1-4 for every bucket in one pass each, no bucket buffer: one
        zr_step_direct_range call, which groups consecutive buckets into as few
        launches as it can (per_bucket: one zr_step_direct call per bucket, as a
        step that reduces buckets while backward fills them runs).

        The plan's gradient tensors may be pinned host tensors, and param_out
        (bf16, at least P elements; default: self.param) a pinned host tensor:
        the kernels then read the gradients and write the params in place over
        the host link, with no copy and no staging buffer."""
        param = self.param if param_out is None else param_out
        if param_out is not None and (param_out.dtype != torch.bfloat16 or param_out.numel() < self.layout.P):
            raise ValueError("param_out must be bf16 with at least P elements")
        if per_bucket:
            for b in range(self.layout.n_buckets):
                zr.zr_step_direct(plan, b, self.scale, self._p_master, self._p_m, self._p_v, hp, param,
                                  None, stream=stream)
            return
        zr.zr_step_direct_range(plan, 0, self.layout.n_buckets, self.scale, self._p_master, self._p_m, self._p_v,
                                hp, param, stream=stream)

    # ---- the step with a global gradient check ---------------------------------------
    def grad_shards(self) -> List[torch.Tensor]:
        """Each rank's fp32 averaged-gradient partition (S elements), allocated on
        first use: the two-pass step keeps the whole averaged gradient until
        the check has seen all of it (the partition gradient of stage 2)."""
        if getattr(self, "_grad", None) is None:
            S = self.layout.S  # views of one flat buffer, like master, m and v
            buf = torch.zeros(max(self.layout.P, 1), dtype=torch.float32, device=self.device)
            self._grad_flat = buf[: self.layout.P]
            self._grad = [buf[r * S:(r + 1) * S] for r in range(self.world)]
            self._p_grad = zr.PtrArray(self._grad)
            self.check = zr.GradCheck()
        return self._grad

    def step_direct_clipped(self, plan: zr.DirectPlan, hp, max_norm: float, stream=None) -> None:
        """The step with the global gradient check before the update ("Megatron-LM
        分布式训练（四）" §"跨 model-parallel 的梯度收尾": DP sync, then the gradient
        fix-ups, then optimizer.step()): every bucket averaged into the
        gradient partitions while the norm is summed, the check (norm,
        overflow, clip coefficient for max_norm; <= 0 disables clipping), then
        the clipped AdamW + bf16 cast over every partition, or nothing when
        the check found an overflow. The outcome stays on the device
        (``zr.zr_gradcheck_read(self.check)`` reads it)."""
        self.grad_shards()
        zr.zr_rs_direct_norm_range(plan, 0, self.layout.n_buckets, self.scale, self._p_grad, self.check, stream=stream)
        self.finish_clipped(hp, max_norm, stream)

    def step_clipped(self, grad_table: zr.PtrArray, hp, max_norm: float, stream=None,
                     plan: Optional[zr.PackPlan] = None) -> None:
        """The same from packed buckets: pack, then the averaging with the norm."""
        self.grad_shards()
        for b in range(self.layout.n_buckets):
            if plan is not None:
                self.pack_planned(b, plan, stream)
            else:
                self.pack(b, grad_table, stream)
            zr.zr_reduce_scatter_avg_norm(self.layout, b, self._p_buckets, self.scale, self._p_grad, self.check,
                                          dtype=self.zr_dtype, stream=stream)
        self.finish_clipped(hp, max_norm, stream)

    def finish_clipped(self, hp, max_norm: float, stream=None) -> None:
        zr.zr_grad_check_finalize(self.check, max_norm, stream=stream)
        zr.zr_adam_clip_step(self.layout, self._p_master, self._p_m, self._p_v, self._p_grad, hp, self.check,
                             self.param, stream=stream)

    def step_direct_from_host(self, plan: zr.DirectPlan, hp, h2d: Sequence[Sequence[tuple]],
                              param_host: Optional[torch.Tensor] = None, stream=None,
                              copy_stream=None, d2h_stream=None, groups: Optional[Sequence[tuple]] = None) -> None:
        """Every bucket with its gradients arriving from host memory, pipelined
        over three streams: while bucket b's step runs, bucket b+1's gradients
        are copied in and bucket b-1's bf16 params are copied out.

        h2d[b]: (host_slice, device_slice) tensor pairs that must be resident
        before bucket b's step (pinned host memory for asynchronous copies).
        groups: optional [(first, end)] runs of consecutive buckets covering
        them all in order; then h2d[g] holds group g's pairs, each group is one
        zr_step_direct_range call and one parameter copy, and the pipeline moves
        fewer, larger copies.
        param_host: pinned bf16 [P] receiving the full parameter buffer, or None.
        Work is ordered after everything already queued on `stream`, and
        `stream` waits for all of it at the end."""
        cur = stream or torch.cuda.current_stream(self.device)
        cs = copy_stream or torch.cuda.Stream(self.device)
        ds = d2h_stream or torch.cuda.Stream(self.device)
        cs.wait_stream(cur)
        ds.wait_stream(cur)
        L = self.layout
        spans = self.bucket_flat_spans()
        if groups is None:
            groups = [(b, b + 1) for b in range(L.n_buckets)]
        elif [b for g in groups for b in range(g[0], g[1])] != list(range(L.n_buckets)):
            raise ValueError("groups must cover the buckets in order")
        if len(h2d) != len(groups):
            raise ValueError("h2d needs one entry per bucket (or per group)")
        for g, (b0, b1) in enumerate(groups):
            with torch.cuda.stream(cs):
                for hs, dv in h2d[g]:
                    dv.copy_(hs, non_blocking=True)
            cur.wait_stream(cs)
            if b1 - b0 == 1:
                self.direct(b0, plan, hp, stream=cur)
            else:
                zr.zr_step_direct_range(plan, b0, b1 - b0, self.scale, self._p_master, self._p_m, self._p_v, hp,
                                        self.param, stream=cur)
            if param_host is not None and spans is not None:
                # consecutive buckets hold adjacent param ranges (in either order)
                lo, hi = min(spans[b][0] for b in range(b0, b1)), max(spans[b][1] for b in range(b0, b1))
                ds.wait_stream(cur)
                with torch.cuda.stream(ds):
                    param_host[lo:hi].copy_(self.param[lo:hi], non_blocking=True)
        if param_host is not None and spans is None:  # buckets are not flat ranges: copy out at the end
            ds.wait_stream(cur)
            with torch.cuda.stream(ds):
                param_host[: L.P].copy_(self.param[: L.P], non_blocking=True)
        cur.wait_stream(ds)

    def bucket_flat_spans(self):
        """Per bucket, the flat range [lo, hi) its params (and padding) cover, or
        None when some bucket's params are not one flat range."""
        L = self.layout
        if L.n_buckets == 0:
            return []
        lo = [None] * L.n_buckets
        hi = [0] * L.n_buckets
        count = [0] * L.n_buckets
        for i, n in enumerate(L.numel):
            off, b = L.param(i)
            lo[b] = off if lo[b] is None else min(lo[b], off)
            hi[b] = max(hi[b], off + int(n))
            count[b] += int(n)
        last = L.param(L.n_params - 1)[1]
        hi[last] = max(hi[last], L.P)
        count[last] += L.P - L.T
        if any(hi[b] - lo[b] != count[b] for b in range(L.n_buckets)):
            return None
        return list(zip(lo, hi))

    def main_grad_views(self, main_grad: Sequence[torch.Tensor]) -> List[zr.PtrArray]:
        """Per-bucket pointer arrays into flat [P] per-rank grad buffers (fp32
        main_grad, or a micro-step's 16-bit grads laid out the same way): the
        Megatron-style contiguous buffer is already bucket-ordered, so its
        buckets are read in place without packing."""
        es = main_grad[0].element_size()
        out = []
        for b in range(self.layout.n_buckets):
            start, _ = self.layout.bucket(b)
            out.append(zr.PtrArray([t.data_ptr() + start * es for t in main_grad]))
        return out

    def step_in_place(self, bucket_views: Sequence[zr.PtrArray], hp, stream=None) -> None:
        for b in range(self.layout.n_buckets):
            self.fused(b, hp, bucket_in=bucket_views[b], stream=stream)

    def step_in_place_acc(self, main_views: Sequence[zr.PtrArray], last_views: Sequence[zr.PtrArray], hp,
                          last_dtype=zr.ZR_BF16, stream=None) -> None:
        """The step with the last micro-step folded in: for every bucket, the
        fp32 main_grad (the earlier micro-steps) plus the last micro-step's
        16-bit grads are averaged, and AdamW + cast run, in one pass; the
        accumulated main_grad is never written ("Megatron-LM 分布式训练（四）"
        §"四步接力": micro-step grads are summed into main_grad, then reduced)."""
        for b in range(self.layout.n_buckets):
            zr.zr_rs_adam_fused_acc(self.layout, b, main_views[b], last_views[b], self.scale, self._p_master,
                                    self._p_m, self._p_v, hp, self.param, last_dtype=last_dtype, stream=stream)
