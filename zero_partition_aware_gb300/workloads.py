"""Synthetic workloads: parameter shapes and seeded input generators.

This module holds the tensor shapes of the five workloads and the seeded random
draws that fill them. It holds none of the method's arithmetic: no flat layout,
no padding, no partitioning, no averaging and no optimizer maths. Both the CUDA
path's harness and the CPU oracle's tests draw their inputs from here, so the
two sides see the same numbers without sharing any code that computes a result.

Shapes follow the models the pages train with data parallelism (GPT-2 small and
Llama-style decoders, "Megatron-LM 分布式训练（四）" §"朴素 DP 的致命浪费") and
the configuration keys of "DeepSpeed ZeRO 通信优化深度解析" §五
(``reduce_bucket_size``). The pages measure no public dataset, so every input is
synthetic; values are drawn as follows, in this order from one seeded generator:
fp32 master ~ N(0, master_std), then replica 0..N-1 gradients (each micro-step in
turn), then m, then v.
"""
from __future__ import annotations

import dataclasses
from typing import List, Optional, Sequence

import numpy as np
import torch


@dataclasses.dataclass(frozen=True)
class AdamW:
    lr: float = 1e-3
    beta1: float = 0.9
    beta2: float = 0.999
    eps: float = 1e-8
    weight_decay: float = 0.01
    step: int = 1


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    numel: tuple            # per-parameter element counts, in layout order
    world: int              # emulated data-parallel replicas
    bucket: int             # reduce_bucket_size in elements
    grad: tuple             # ("normal", std) or ("int", lo, hi)
    master_std: float
    state: tuple            # ("zero",) or ("absnormal", std)
    adam: AdamW
    micro_steps: int = 1    # >1: bf16 micro-step grads summed into an fp32 buffer
    description: str = ""

    @property
    def n_params(self) -> int:
        return len(self.numel)

    @property
    def total(self) -> int:
        return int(sum(self.numel))


def gpt2_small_numel() -> List[int]:
    """wte, wpe, then 12 blocks of (c_attn w/b, c_proj w/b, fc w/b, proj w/b, ln1 w/b, ln2 w/b)."""
    d, v, ctx = 768, 50257, 1024
    out = [v * d, ctx * d]
    for _ in range(12):
        out += [d * 3 * d, 3 * d, d * d, d, d * 4 * d, 4 * d, 4 * d * d, d, d, d, d, d]
    return out


def llama_numel(vocab: int, d: int, layers: int, n_q: int, n_kv: int, ffn: int,
                tied: bool) -> List[int]:
    """embed; per layer [in_norm, q, k, v, o, post_norm, gate, up, down]; norm; lm_head unless tied."""
    head = d // n_q
    kv = n_kv * head
    out = [vocab * d]
    for _ in range(layers):
        out += [d, d * d, d * kv, d * kv, d * d, d, d * ffn, d * ffn, ffn * d]
    out += [d]
    if not tied:
        out += [vocab * d]
    return out


def irregular_numel(n: int = 10_000, hi: float = 1e6, seed: int = 0) -> List[int]:
    """Log-uniform element counts in [1, hi]: clip(rint(exp(U[0, ln hi))), 1, hi)."""
    rng = np.random.default_rng(seed)
    x = np.clip(np.rint(np.exp(rng.uniform(0.0, np.log(hi), n))), 1, hi)
    return [int(t) for t in x]


_STEP10 = AdamW(step=10)

WORKLOADS = {
    "tiny": Workload(
        "tiny", tuple([1000, 333 * 17, 4096, 129 * 65, 10, 2048 * 3, 777]), 4, 8192,
        ("normal", 1e-2), 0.02, ("zero",), AdamW(step=1),
        description="7 params, world=4, bucket 8192"),
    "gpt2_124m": Workload(
        "gpt2_124m", tuple(gpt2_small_numel()), 8, 50_000_000,
        ("normal", 1e-3), 0.02, ("absnormal", 1e-4), _STEP10,
        description="GPT-2 small shapes (124M), world=8, bucket 5e7"),
    "llama_1p1b": Workload(
        "llama_1p1b", tuple(llama_numel(32000, 2048, 22, 32, 4, 5632, tied=False)), 8,
        500_000_000, ("normal", 1e-3), 0.02, ("absnormal", 1e-4), _STEP10, micro_steps=4,
        description="Llama 1.1B shapes, world=8, bucket 5e8, 4 bf16 micro-steps into fp32"),
    "irregular_10k": Workload(
        "irregular_10k", tuple(irregular_numel()), 16, 1 << 24,
        ("int", -8, 8), 0.02, ("zero",), AdamW(step=1),
        description="10,000 log-uniform params in [1,1e6], world=16, bucket 2^24, integer grads"),
    "llama3_3b": Workload(
        "llama3_3b", tuple(llama_numel(128256, 3072, 28, 24, 8, 8192, tied=True)), 8,
        500_000_000, ("normal", 1e-3), 0.02, ("absnormal", 1e-4), _STEP10,
        description="Llama-3.2-3B shapes (tied embedding), world=8, bucket 5e8"),
}


# A small slice of the irregular workload for profiler captures: its first 400
# params (world 16, 2^24 buckets); each bucket's working set still exceeds L2.
WORKLOADS["irregular_prof"] = Workload(
    "irregular_prof", WORKLOADS["irregular_10k"].numel[:400], 16, 1 << 24,
    ("int", -8, 8), 0.02, ("zero",), AdamW(step=1),
    description="first 400 params of irregular_10k, world=16, bucket 2^24 (profiling size)")


# The world sweep's fixed ~1B layout: the Llama 1.1B tensor list with bf16
# gradients straight from one step (no micro-steps).
WORKLOADS["llama_1p1b_bf16"] = dataclasses.replace(
    WORKLOADS["llama_1p1b"], name="llama_1p1b_bf16", micro_steps=1,
    description="Llama 1.1B shapes, bf16 grads of one step (the world sweep's layout)")

# The Llama 1.1B micro-step path at profiling size: the first decoder layer's
# nine tensors (44.0 M elements, one bucket), world 8, 4 bf16 micro-steps.
WORKLOADS["llama_prof"] = Workload(
    "llama_prof", WORKLOADS["llama_1p1b"].numel[1:10], 8, 500_000_000,
    ("normal", 1e-3), 0.02, ("absnormal", 1e-4), _STEP10, micro_steps=4,
    description="first decoder layer of llama_1p1b, world=8, 4 micro-steps (profiling size)")


def replace(wl: Workload, **kw) -> Workload:
    return dataclasses.replace(wl, **kw)


def generator(device, seed: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def draw_grad(wl: Workload, n: int, gen: torch.Generator, device) -> torch.Tensor:
    """One replica's (or one micro-step's) gradient values, n elements, as bf16."""
    kind = wl.grad[0]
    if kind == "normal":
        x = torch.randn(n, generator=gen, device=device, dtype=torch.float32)
        x.mul_(float(wl.grad[1]))
        return x.to(torch.bfloat16)
    if kind == "int":
        lo, hi = int(wl.grad[1]), int(wl.grad[2])
        x = torch.randint(lo, hi + 1, (n,), generator=gen, device=device, dtype=torch.int32)
        return x.to(torch.bfloat16)
    raise ValueError(kind)


def draw_state(wl: Workload, n: int, gen: torch.Generator, device) -> torch.Tensor:
    if wl.state[0] == "zero":
        return torch.zeros(n, device=device, dtype=torch.float32)
    x = torch.randn(n, generator=gen, device=device, dtype=torch.float32)
    return x.mul_(float(wl.state[1])).abs_()


def draw_inputs(wl: Workload, device="cpu", seed: int = 0, n: Optional[int] = None):
    """Draw n (default: all) elements of every input in the fixed order.

    Returns a dict with ``master`` (fp32 [n]), ``grads`` (list over replicas of
    lists over micro-steps of bf16 [n]), ``m`` and ``v`` (fp32 [n]).
    """
    n = wl.total if n is None else int(n)
    gen = generator(device, seed)
    master = torch.randn(n, generator=gen, device=device, dtype=torch.float32)
    master.mul_(float(wl.master_std))
    grads = [[draw_grad(wl, n, gen, device) for _ in range(wl.micro_steps)]
             for _ in range(wl.world)]
    m = draw_state(wl, n, gen, device)
    v = draw_state(wl, n, gen, device)
    return {"master": master, "grads": grads, "m": m, "v": v}


def arena_offsets(numel: Sequence[int], align: int = 256) -> List[int]:
    """Start of each tensor when the tensors are allocated one after another in
    one arena, each start rounded up to `align` elements (as separately
    allocated gradient tensors would sit in memory). align=1 packs them."""
    out, pos = [], 0
    for n in numel:
        pos = -(-pos // align) * align
        out.append(pos)
        pos += int(n)
    return out


def random_numels(rng: np.random.Generator, n: int, lo: int = 1, hi: int = 4000,
                  log: bool = True) -> List[int]:
    """Seeded element counts for small parity layouts (log-uniform by default)."""
    if log:
        x = np.exp(rng.uniform(np.log(lo), np.log(hi + 1), n))
        return [int(min(hi, max(lo, t))) for t in x]
    return [int(t) for t in rng.integers(lo, hi + 1, n)]


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """Raw bf16 bit patterns of a CPU bf16 tensor as uint16 (no arithmetic)."""
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def from_bf16_bits(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16)


__all__ = ["AdamW", "Workload", "WORKLOADS", "draw_inputs", "draw_grad", "draw_state",
           "generator", "replace", "random_numels", "arena_offsets", "bf16_bits", "from_bf16_bits",
           "gpt2_small_numel", "llama_numel", "irregular_numel"]
