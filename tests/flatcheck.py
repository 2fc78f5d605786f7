"""Whole-array comparison of a full-size step with the oracle (test helper).

Once the flat layout is fixed, every flat element f is computed on its own:
the N replicas' gradients at f are averaged in rank order, AdamW updates
master[f], m[f] and v[f], and the new master is cast to bf16 ("DeepSpeed ZeRO
通信优化深度解析" §三.2: each param's gradient is sliced by partition, the
slices averaged by the reduce-scatter; "Megatron-LM 分布式训练（四）"
§"通信模式": reduce-scatter, the local fp32 update, then the all-gather's
payload). So the flat range [0, P) is cut into disjoint chunks. For each chunk
the device's inputs (copied aside before the step) and outputs are brought to
the host, the oracle's averaging, AdamW and cast run on them, and every element
of master, m, v and the bf16 parameters is compared bit for bit. Chunks are
checked on every host core at once (the oracle is C called through ctypes,
which releases the GIL), while the main thread copies the next chunks from
the device into a ring of pinned buffers.

Where a gradient element sits is the oracle's flat layout (param i holds flat
[o_i, o_i + n_i)); where the test placed that param's gradient tensor is the
test's own arena offset. Nothing here comes from the library under test.
"""
from __future__ import annotations

import contextlib
import os
import queue
import threading
from concurrent.futures import ThreadPoolExecutor
from typing import List, Optional, Sequence

import numpy as np
import torch

import oracle


def host_cores() -> int:
    if hasattr(os, "sched_getaffinity"):
        return max(1, len(os.sched_getaffinity(0)))
    return max(1, os.cpu_count() or 1)


def _np(t: torch.Tensor) -> np.ndarray:
    """A (pinned) CPU tensor as numpy, bf16 as uint16 bits (no arithmetic)."""
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def _on(stream):
    """The copies' stream as a context (none for CPU tensors)."""
    return torch.cuda.stream(stream) if stream is not None else contextlib.nullcontext()


class ArenaGrads:
    """Replica k's gradient of flat position f: the element f - o_i of param i's
    tensor, which the test laid at arena offset arena_off[i] of rank k's arena.
    Positions past T (the padding) have no gradient: zero."""

    def __init__(self, arenas: Sequence[torch.Tensor], lay, arena_off: Sequence[int]):
        self.arenas = list(arenas)
        self.off = np.asarray(lay.offset, dtype=np.int64)
        self.numel = np.asarray(lay.numel, dtype=np.int64)
        self.delta = np.asarray(arena_off, dtype=np.int64) - self.off
        self.T = int(lay.T)
        self.dtype = self.arenas[0].dtype
        self.micro = 1

    def index(self, f0: int, f1: int) -> Optional[torch.Tensor]:
        hi = min(f1, self.T)
        if hi <= f0:
            return None
        i0 = int(np.searchsorted(self.off, f0, "right")) - 1
        i1 = int(np.searchsorted(self.off, hi - 1, "right")) - 1
        lo = np.maximum(self.off[i0:i1 + 1], f0)
        up = np.minimum(self.off[i0:i1 + 1] + self.numel[i0:i1 + 1], hi)
        idx = np.arange(f0, hi, dtype=np.int64) + np.repeat(self.delta[i0:i1 + 1], up - lo)
        return torch.from_numpy(idx).to(self.arenas[0].device)

    def fill(self, f0: int, f1: int, out: List[List[torch.Tensor]], stream) -> None:
        """out[k][0][: f1 - f0] <- replica k's gradients at [f0, f1)."""
        idx = self.index(f0, f1)
        n_real = 0 if idx is None else int(idx.numel())
        with _on(stream):
            for k, a in enumerate(self.arenas):
                dst = out[k][0]
                if n_real:
                    dst[:n_real].copy_(a.index_select(0, idx), non_blocking=True)
                if n_real < f1 - f0:
                    dst[n_real:f1 - f0].zero_()


class FlatGrads:
    """Gradients already in flat order: src[k][s] is rank k's [P] buffer of
    micro-step s (zero past T)."""

    def __init__(self, src: Sequence[Sequence[torch.Tensor]]):
        self.src = [list(r) for r in src]
        self.dtype = self.src[0][0].dtype
        self.micro = len(self.src[0])

    def fill(self, f0: int, f1: int, out, stream) -> None:
        with _on(stream):
            for k, row in enumerate(self.src):
                for s, t in enumerate(row):
                    out[k][s][: f1 - f0].copy_(t[f0:f1], non_blocking=True)


def check_whole(lay, scale: float, hp, grads, before: Sequence[torch.Tensor], after: Sequence[torch.Tensor],
                param: torch.Tensor, *, main_after: Optional[Sequence[torch.Tensor]] = None,
                grad_after: Optional[Sequence[torch.Tensor]] = None, coef: Optional[float] = None,
                integer_avg: bool = False, chunk: Optional[int] = None) -> dict:
    """Compare a step over the whole flat range with the oracle.

    lay: the oracle's layout. grads: an ArenaGrads or FlatGrads. before / after:
    the flat [P] fp32 master, m and v (partition r at offset rS) as the step
    found and left them. param: the device's bf16 [P] output.
    FlatGrads with several micro-steps: each replica's gradient is the fp32
    sum of its micro-steps in order (oracle.grad_accumulate from zero);
    main_after[k], if given, must hold the sum of all but the last one.
    grad_after[r]-as-flat (one [P] fp32 tensor), if given, must hold the
    averaged gradient. coef: the clipped step; AdamW takes the oracle's
    zro_adam_clip_step with this coefficient. integer_avg: the gradients are
    integers, so the average must equal the exact integer sum times the
    scale, at every element.
    Returns the element count and, per output, the mismatch count and the
    first mismatching flat index.
    """
    oracle.lib()  # load before the worker threads start
    P, T, world = int(lay.P), int(lay.T), int(lay.world)
    micro = grads.micro
    es = 2 if grads.dtype in (torch.bfloat16, torch.float16) else 4
    if chunk is None:
        per_elem = world * micro * es + 7 * 4 + 2 + (world * 4 if main_after is not None else 0)
        chunk = max(1 << 18, min(1 << 22, (96 << 20) // per_elem))
    workers = max(1, host_cores() - 1)
    ring = workers + 2
    cuda = param.device.type == "cuda"
    pin = dict(device="cpu", pin_memory=cuda)

    def new_set():
        return {
            "x": [[torch.empty(chunk, dtype=grads.dtype, **pin) for _ in range(micro)] for _ in range(world)],
            "st": [torch.empty(chunk, dtype=torch.float32, **pin) for _ in range(6)],
            "q": torch.empty(chunk, dtype=torch.bfloat16, **pin),
            "main": [torch.empty(chunk, dtype=torch.float32, **pin) for _ in range(world)]
            if main_after is not None else None,
            "g": torch.empty(chunk, dtype=torch.float32, **pin) if grad_after is not None else None,
        }

    sets = [new_set() for _ in range(ring)]
    free: "queue.Queue[int]" = queue.Queue()
    for i in range(ring):
        free.put(i)
    names = ["master", "m", "v", "param", "main_grad", "grad", "integer_avg"]
    total = {n: 0 for n in names}
    first = {n: None for n in names}
    lock = threading.Lock()
    copy_stream = torch.cuda.Stream() if cuda else None

    def note(name, f0, bad):
        n = int(np.count_nonzero(bad))
        if n:
            with lock:
                total[name] += n
                at = f0 + int(np.flatnonzero(bad)[0])
                first[name] = at if first[name] is None else min(first[name], at)

    def work(sid, f0, f1):
        try:
            S_ = sets[sid]
            n = f1 - f0
            xs = [[_np(t)[:n] for t in row] for row in S_["x"]]
            if micro > 1:
                g = []
                for k, row in enumerate(xs):
                    acc = np.zeros(n, np.float32)
                    for s, mb in enumerate(row):
                        oracle.grad_accumulate(acc, np.ascontiguousarray(mb))
                        if main_after is not None and s == micro - 2:
                            note("main_grad", f0, _np(S_["main"][k])[:n].view(np.uint32) != acc.view(np.uint32))
                    g.append(acc)
            else:
                g = [np.ascontiguousarray(row[0]) for row in xs]
            avg = oracle.average(world, g, scale)
            if integer_avg:
                exact = np.zeros(n, np.int64)
                for xk in g:
                    exact += np.rint(oracle.bf16_to_f32(xk)).astype(np.int64)
                want = exact.astype(np.float32) * np.float32(scale)  # |sum| <= 8N: exact in fp32
                note("integer_avg", f0, avg.view(np.uint32) != want.view(np.uint32))
            p, m, v = (_np(S_["st"][i])[:n] for i in range(3))
            if grad_after is not None:
                note("grad", f0, _np(S_["g"])[:n].view(np.uint32) != avg.view(np.uint32))
            t_here = max(0, min(n, T - f0))
            if coef is None:
                oracle.adamw(p, m, v, avg, hp)
                want_q = oracle.f32_to_bf16(p)
                want_q[t_here:] = 0
            else:
                want_q = np.zeros(n, np.uint16)
                oracle.adam_clip_step(_ChunkLayout(n, t_here), [p], [m], [v], [avg], hp, coef, False, want_q)
            for i, name in enumerate(("master", "m", "v")):
                got = _np(S_["st"][3 + i])[:n]
                ref = (p, m, v)[i]
                note(name, f0, got.view(np.uint32) != ref.view(np.uint32))
            note("param", f0, _np(S_["q"])[:n] != want_q)
        finally:
            free.put(sid)

    futures = []
    with ThreadPoolExecutor(workers) as ex:
        for f0 in range(0, P, chunk):
            f1 = min(P, f0 + chunk)
            n = f1 - f0
            sid = free.get()
            S_ = sets[sid]
            if cuda:
                copy_stream.wait_stream(torch.cuda.current_stream())
            grads.fill(f0, f1, S_["x"], copy_stream)
            with _on(copy_stream):
                for i, t in enumerate(list(before) + list(after)):
                    S_["st"][i][:n].copy_(t[f0:f1], non_blocking=True)
                S_["q"][:n].copy_(param[f0:f1], non_blocking=True)
                if main_after is not None:
                    for k, t in enumerate(main_after):
                        S_["main"][k][:n].copy_(t[f0:f1], non_blocking=True)
                if grad_after is not None:
                    S_["g"][:n].copy_(grad_after[0][f0:f1], non_blocking=True)
            if cuda:
                copy_stream.synchronize()
            futures.append(ex.submit(work, sid, f0, f1))
            keep = []
            for f in futures:  # surface a worker's exception early
                if f.done():
                    f.result()
                else:
                    keep.append(f)
            futures = keep
        for f in futures:
            f.result()
    out = {"elements": P, "chunk": chunk, "threads": workers}
    for name in names:
        out[name] = total[name]
        out[name + "_first"] = first[name]
    return out


class _ChunkLayout:
    """The oracle's clipped step over one chunk as a one-partition layout:
    world 1, S = the chunk, T = the chunk's elements below the padding."""

    def __init__(self, n: int, t_here: int):
        self.world, self.S, self.T, self.P = 1, n, t_here, n


def summary(name: str, res: dict, outputs: Sequence[str] = ("master", "m", "v", "param")) -> str:
    bad = {k: res[k] for k in outputs}
    return (f"{name}: {sum(bad.values())} of {res['elements']} elements differ "
            f"({', '.join(f'{k} {v}' for k, v in bad.items())}; chunks of {res['chunk']} on {res['threads']} threads)")
