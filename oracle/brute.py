"""Pure-Python brute force for tiny cases -- TEST INFRASTRUCTURE.

Independent of ``zr_oracle.c``: it labels every flat element one by one and
sums with exact rationals, so that the C oracle can be pinned to something
other than itself. Only for layouts of a few thousand elements.

Sources: [DS] "DeepSpeed ZeRO 通信优化深度解析：用 reduce-scatter 分区感知规约替代
all-reduce" §二, §三.2, §四; [IQ] "07. 大规模训练时通信瓶颈在哪里？..." §"三种原语".
"""
from __future__ import annotations

from fractions import Fraction
from typing import Dict, List, Sequence, Tuple


def flat_labels(numel: Sequence[int], world: int):
    """Per flat element f: (param index or -1 for padding, owning rank f // S)."""
    T = sum(numel)
    P = -(-T // world) * world
    S = P // world
    param_of = []
    for i, n in enumerate(numel):
        param_of += [i] * n
    param_of += [-1] * (P - T)
    rank_of = [f // S for f in range(P)]
    return T, P, S, param_of, rank_of


def brute_slices(numel: Sequence[int], world: int, bucket_of: Sequence[int],
                 bucket_start: Sequence[int]) -> List[Tuple[int, ...]]:
    """Maximal stretches of constant (param, rank) over [0, T), one element at a time.

    Rows: (param, bucket, dst, param_offset, bucket_offset, partition_offset, numel).
    """
    T, P, S, param_of, rank_of = flat_labels(numel, world)
    offs = [0]
    for n in numel:
        offs.append(offs[-1] + n)
    rows = []
    f = 0
    while f < T:
        i, r = param_of[f], rank_of[f]
        g = f
        while g < T and param_of[g] == i and rank_of[g] == r:
            g += 1
        b = bucket_of[i]
        rows.append((i, b, r, f - offs[i], f - bucket_start[b], f - r * S, g - f))
        f = g
    return rows


def brute_runs(numel: Sequence[int], world: int, bucket_ranges: Sequence[Tuple[int, int]]):
    """Maximal stretches of constant (bucket, rank) over [0, P).

    Rows: (bucket, dst, bucket_offset, partition_offset, numel).
    """
    T, P, S, param_of, rank_of = flat_labels(numel, world)
    bucket_at = [None] * P
    for b, (s, e) in enumerate(bucket_ranges):
        for f in range(s, e):
            bucket_at[f] = b
    rows = []
    f = 0
    while f < P:
        b, r = bucket_at[f], rank_of[f]
        g = f
        while g < P and bucket_at[g] == b and rank_of[g] == r:
            g += 1
        rows.append((b, r, f - bucket_ranges[b][0], f - r * S, g - f))
        f = g
    return rows


def bf16_value(bits: int) -> Fraction:
    """Exact value of a finite bf16 bit pattern."""
    sign = -1 if bits & 0x8000 else 1
    exp = (bits >> 7) & 0xFF
    man = bits & 0x7F
    if exp == 0xFF:
        raise ValueError("non-finite")
    if exp == 0:
        return sign * Fraction(man, 1 << 7) * Fraction(1, 1 << 126)
    return sign * (1 + Fraction(man, 1 << 7)) * (Fraction(2) ** (exp - 127))


def exact_mean(values: Sequence[Fraction]) -> Fraction:
    return sum(values, Fraction(0)) / len(values)


def f32_ulp(x: float) -> float:
    import numpy as np
    x = np.float32(abs(x))
    return float(np.spacing(x)) if x != 0 else float(np.float32(1.4e-45))
