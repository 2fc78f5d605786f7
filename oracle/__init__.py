"""CPU oracle for partition-aware ZeRO averaging + sharded AdamW -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg
may import this package. It wraps ``zr_oracle.c`` (plain single-threaded C, no
FMA contraction) with numpy marshalling, plus ``brute.py`` (pure-Python exact
arithmetic for tiny cases). It shares no code with the CUDA library.

Every function below calls straight into the C file, which cites the passage of
the pages each step follows.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass
from typing import List, NamedTuple, Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "zr_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "libzr_oracle.so")
_CFLAGS = ["-std=c99", "-O2", "-ffp-contract=off", "-fPIC", "-shared", "-Wall"]

BF16, FP32, FP16 = 0, 1, 2

_lib = None


def _foreign(path: str) -> bool:
    """True if an ELF file was built for another machine (x86-64 vs aarch64)."""
    import platform
    want = {"x86_64": 62, "aarch64": 183, "arm64": 183}.get(platform.machine())
    try:
        with open(path, "rb") as f:
            head = f.read(20)
        return want is not None and int.from_bytes(head[18:20], "little") != want
    except OSError:
        return True


def build(force: bool = False) -> str:
    """Compile the oracle with the host C compiler (no FMA contraction)."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_LIB_PATH) or _foreign(_LIB_PATH) or \
            os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".{os.getpid()}.tmp"
        cc = os.environ.get("CC", "gcc")
        subprocess.run([cc, *_CFLAGS, "-o", tmp, _SRC, "-lm"], check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def lib():
    global _lib
    if _lib is None:
        _lib = ctypes.CDLL(build())
        _declare(_lib)
    return _lib


_i64p = ctypes.POINTER(ctypes.c_int64)
_vp = ctypes.c_void_p
_i32 = ctypes.c_int32
_i64 = ctypes.c_int64
_f32 = ctypes.c_float


def _declare(L):
    L.zro_layout.restype = ctypes.c_int
    L.zro_layout.argtypes = [_vp, _i64, _i32, _i64, _vp, _vp, _vp, _vp, _vp, _vp]
    L.zro_layout_ordered.restype = ctypes.c_int
    L.zro_layout_ordered.argtypes = [_vp, _i64, _i32, _i64, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp]
    L.zro_bucket_flat_map.restype = ctypes.c_int
    L.zro_bucket_flat_map.argtypes = [_vp, _i64, _vp, _vp, _i64, _i64, _i64, _i64, _vp]
    L.zro_bucket_pack_ordered.restype = ctypes.c_int
    L.zro_bucket_pack_ordered.argtypes = [_vp, _i64, _i32, _vp, _vp, _i64, _i64, _i64, _vp, _i32, _vp]
    L.zro_reduce_scatter_avg_map.restype = ctypes.c_int
    L.zro_reduce_scatter_avg_map.argtypes = [_i32, _i64, _i64, _vp, _vp, _i32, _f32, _vp]
    L.zro_rs_adam_fused_map.restype = ctypes.c_int
    L.zro_rs_adam_fused_map.argtypes = [_i32, _i64, _i64, _i64, _vp, _vp, _i32, _f32,
                                        _vp, _vp, _vp, _f32, _f32, _f32, _f32, _f32, _i64,
                                        _vp, _vp]
    L.zro_bucket_pack.restype = ctypes.c_int
    L.zro_bucket_pack.argtypes = [_vp, _vp, _i64, _i32, _i64, _i64, _i64, _vp, _i32, _vp]
    L.zro_reduce_scatter_avg.restype = ctypes.c_int
    L.zro_reduce_scatter_avg.argtypes = [_i32, _i64, _i64, _i64, _vp, _i32, _f32, _vp]
    L.zro_allreduce_avg.restype = ctypes.c_int
    L.zro_allreduce_avg.argtypes = [_i32, _i64, _vp, _i32, _f32, _f32, _vp]
    L.zro_f16_to_f32.restype = None
    L.zro_f16_to_f32.argtypes = [_vp, _vp, _i64]
    L.zro_grad_accumulate.restype = ctypes.c_int
    L.zro_grad_accumulate.argtypes = [_i64, _vp, _vp, _i32]
    L.zro_adamw_scalars.restype = ctypes.c_int
    L.zro_adamw_scalars.argtypes = [_f32, _f32, _f32, _f32, _f32, _i64, _vp]
    L.zro_adamw.restype = ctypes.c_int
    L.zro_adamw.argtypes = [_i64, _vp, _vp, _vp, _vp, _f32, _f32, _f32, _f32, _f32, _i64]
    L.zro_gather_cast_bf16.restype = ctypes.c_int
    L.zro_gather_cast_bf16.argtypes = [_i32, _i64, _i64, _vp, _vp]
    L.zro_rs_adam_fused.restype = ctypes.c_int
    L.zro_rs_adam_fused.argtypes = [_i32, _i64, _i64, _i64, _i64, _vp, _i32, _f32,
                                    _vp, _vp, _vp, _f32, _f32, _f32, _f32, _f32, _i64,
                                    _vp, _vp]
    L.zro_grad_check.restype = ctypes.c_int
    L.zro_grad_check.argtypes = [_i32, _i64, _vp, _f32, _vp, _vp, _vp, _vp, _vp]
    L.zro_adam_clip_step.restype = ctypes.c_int
    L.zro_adam_clip_step.argtypes = [_i32, _i64, _i64, _vp, _vp, _vp, _vp, _f32, _i32,
                                     _f32, _f32, _f32, _f32, _f32, _i64, _vp]
    L.zro_comm_bytes.restype = ctypes.c_int
    L.zro_comm_bytes.argtypes = [_i32, _i32, _i64, _i32, ctypes.POINTER(ctypes.c_double)]
    L.zro_layout_bytes.restype = ctypes.c_int
    L.zro_layout_bytes.argtypes = [_i32, _i64, _i64, ctypes.POINTER(ctypes.c_double)]
    L.zro_bf16_to_f32.restype = None
    L.zro_bf16_to_f32.argtypes = [_vp, _vp, _i64]
    L.zro_f32_to_bf16.restype = None
    L.zro_f32_to_bf16.argtypes = [_vp, _vp, _i64]


class OracleError(RuntimeError):
    pass


def _check(rc: int, what: str):
    if rc != 0:
        raise OracleError(f"{what} returned {rc}")


def _ptr(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data


def _ptr_array(arrs: Sequence[np.ndarray]):
    return (ctypes.c_void_p * len(arrs))(*[_ptr(a) for a in arrs])


def _dtype_code(a: np.ndarray) -> int:
    if a.dtype == np.uint16:
        return BF16
    if a.dtype == np.float32:
        return FP32
    if a.dtype == np.float16:
        return FP16
    raise TypeError(f"oracle takes bf16 bit patterns (uint16), float16 or float32, got {a.dtype}")


# ----------------------------------------------------------------------------
# Layout
# ----------------------------------------------------------------------------

@dataclass
class Layout:
    numel: np.ndarray          # [n] int64
    world: int
    bucket_size: int
    T: int
    P: int
    S: int
    offset: np.ndarray         # [n]
    bucket_of: np.ndarray      # [n]
    bucket_range: np.ndarray   # [nb, 2] flat [start, end)
    slices: np.ndarray         # [ns, 7] param, bucket, dst, param_offset, bucket_offset, partition_offset, numel
    runs: np.ndarray           # [nr, 5] bucket, dst, bucket_offset, partition_offset, numel
    order: Optional[np.ndarray] = None        # arrival order (None: the flat order)
    bucket_pos: Optional[np.ndarray] = None   # [n] position of each param in its bucket
    bucket_info: Optional[np.ndarray] = None  # [nb, 3] numel_b, pad_pos (-1), flat_start (-1)

    @property
    def n_params(self) -> int:
        return int(self.numel.shape[0])

    @property
    def n_buckets(self) -> int:
        return int(self.bucket_range.shape[0])

    def bucket(self, b: int):
        """(flat start, numel) of bucket b; the start is -1 when the bucket is not
        one flat range in flat order (an arrival order other than the flat one)."""
        s, e = (int(x) for x in self.bucket_range[b])
        return s, e - s

    def flat_map(self, b: int) -> np.ndarray:
        """The flat index of every position of bucket b."""
        s, nb = self.bucket(b)
        if self.order is None:
            return np.arange(s, s + nb, dtype=np.int64)
        out = np.full(max(nb, 1), -1, dtype=np.int64)
        _check(lib().zro_bucket_flat_map(_ptr(self.numel), self.n_params, _ptr(self.bucket_of),
                                         _ptr(self.bucket_pos), b, self.T, int(self.bucket_info[b, 1]),
                                         self.P, _ptr(out)), "zro_bucket_flat_map")
        return out[:nb]

    def param_partitions(self, i: int):
        """(param_to_partition_ids, grad_start_offset) of param i."""
        rows = self.slices[self.slices[:, 0] == i]
        return [int(r) for r in rows[:, 2]], [int(g) for g in rows[:, 3]]

    def runs_of(self, b: int) -> np.ndarray:
        return self.runs[self.runs[:, 0] == b]


def layout(numel: Sequence[int], world: int, bucket_size: int, order: Optional[Sequence[int]] = None) -> Layout:
    """The layout; `order`: the arrival order of the grads (a permutation of the
    params; None: the flat order)."""
    if order is not None:
        return _layout_ordered(numel, world, bucket_size, order)
    L = lib()
    nm = np.ascontiguousarray(np.asarray(numel, dtype=np.int64))
    n = int(nm.shape[0])
    dims = np.zeros(6, dtype=np.int64)
    _check(L.zro_layout(_ptr(nm) if n else None, n, world, bucket_size, _ptr(dims),
                        None, None, None, None, None), "zro_layout(count)")
    T, P, S, nb, ns, nr = (int(x) for x in dims)
    offset = np.zeros(max(n, 1), dtype=np.int64)
    bucket_of = np.zeros(max(n, 1), dtype=np.int64)
    br = np.zeros((max(nb, 1), 2), dtype=np.int64)
    sl = np.zeros((max(ns, 1), 7), dtype=np.int64)
    ru = np.zeros((max(nr, 1), 5), dtype=np.int64)
    _check(L.zro_layout(_ptr(nm) if n else None, n, world, bucket_size, _ptr(dims),
                        _ptr(offset), _ptr(bucket_of), _ptr(br), _ptr(sl), _ptr(ru)),
           "zro_layout(fill)")
    return Layout(nm, world, bucket_size, T, P, S, offset[:n], bucket_of[:n], br[:nb],
                  sl[:ns], ru[:nr])


def _layout_ordered(numel, world, bucket_size, order) -> Layout:
    L = lib()
    nm = np.ascontiguousarray(np.asarray(numel, dtype=np.int64))
    od = np.ascontiguousarray(np.asarray(order, dtype=np.int64))
    n = int(nm.shape[0])
    assert od.shape == (n,)
    dims = np.zeros(6, dtype=np.int64)
    args = (_ptr(nm) if n else None, n, world, bucket_size, _ptr(od) if n else None)
    _check(L.zro_layout_ordered(*args, _ptr(dims), None, None, None, None, None, None), "zro_layout_ordered(count)")
    T, P, S, nb, ns, nr = (int(x) for x in dims)
    offset = np.zeros(max(n, 1), dtype=np.int64)
    bucket_of = np.zeros(max(n, 1), dtype=np.int64)
    bucket_pos = np.zeros(max(n, 1), dtype=np.int64)
    info = np.zeros((max(nb, 1), 3), dtype=np.int64)
    sl = np.zeros((max(ns, 1), 7), dtype=np.int64)
    ru = np.zeros((max(nr, 1), 5), dtype=np.int64)
    _check(L.zro_layout_ordered(*args, _ptr(dims), _ptr(offset), _ptr(bucket_of), _ptr(bucket_pos), _ptr(info),
                                _ptr(sl), _ptr(ru)), "zro_layout_ordered(fill)")
    info = info[:nb]
    br = np.stack([info[:, 2], info[:, 2] + info[:, 0]], axis=1) if nb else np.zeros((0, 2), np.int64)
    return Layout(nm, world, bucket_size, T, P, S, offset[:n], bucket_of[:n], br, sl[:ns], ru[:nr],
                  order=od, bucket_pos=bucket_pos[:n], bucket_info=info)


# ----------------------------------------------------------------------------
# Numerics
# ----------------------------------------------------------------------------

def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    bits = np.ascontiguousarray(bits, dtype=np.uint16)
    out = np.empty(bits.shape, dtype=np.float32)
    lib().zro_bf16_to_f32(_ptr(bits), _ptr(out), bits.size)
    return out


def f32_to_bf16(x: np.ndarray) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, dtype=np.uint16)
    lib().zro_f32_to_bf16(_ptr(x), _ptr(out), x.size)
    return out


def bucket_pack(lay: Layout, b: int, grads: Sequence[Sequence[np.ndarray]]) -> List[np.ndarray]:
    """grads[k][i]: replica k's grad of param i (uint16 bf16 bits or float32)."""
    start, nb = lay.bucket(b)
    end = start + nb
    dt = grads[0][0].dtype
    es = np.dtype(dt).itemsize
    out = [np.empty(nb, dtype=dt) for _ in range(lay.world)]
    n = lay.n_params
    flat = []
    for k in range(lay.world):
        for i in range(n):
            a = grads[k][i]
            assert a.dtype == dt and a.shape == (int(lay.numel[i]),)
            flat.append(np.ascontiguousarray(a))
    ptrs = _ptr_array(flat)
    if lay.order is not None:
        pad = int(lay.bucket_info[b, 1])
        _check(lib().zro_bucket_pack_ordered(_ptr(lay.numel), n, lay.world, _ptr(lay.bucket_of),
                                             _ptr(lay.bucket_pos), b, pad, lay.P - lay.T, ptrs, es,
                                             _ptr_array(out)), "zro_bucket_pack_ordered")
        return out
    _check(lib().zro_bucket_pack(_ptr(lay.numel), _ptr(lay.offset), n, lay.world, lay.T,
                                 start, end, ptrs, es, _ptr_array(out)), "zro_bucket_pack")
    return out


def reduce_scatter_avg(lay: Layout, b: int, bucket: Sequence[np.ndarray], scale: float,
                       shards: Sequence[np.ndarray]) -> None:
    """Writes the averaged bucket into shards[r] (float32 [S]) in place."""
    start, nb = lay.bucket(b)
    code = _dtype_code(bucket[0])
    for s in shards:
        assert s.dtype == np.float32 and s.shape == (lay.S,)
    if lay.order is not None:
        fm = lay.flat_map(b)
        _check(lib().zro_reduce_scatter_avg_map(lay.world, lay.S, nb, _ptr(fm), _ptr_array(bucket), code,
                                                scale, _ptr_array(shards)), "zro_reduce_scatter_avg_map")
        return
    _check(lib().zro_reduce_scatter_avg(lay.world, lay.S, start, nb, _ptr_array(bucket), code,
                                        scale, _ptr_array(shards)), "zro_reduce_scatter_avg")


def allreduce_avg(world: int, bucket: Sequence[np.ndarray], scale: float, postscale: float = 1.0) -> List[np.ndarray]:
    nb = int(bucket[0].shape[0])
    code = _dtype_code(bucket[0])
    out = [np.empty(nb, dtype=np.float32) for _ in range(world)]
    _check(lib().zro_allreduce_avg(world, nb, _ptr_array(bucket), code, scale, postscale, _ptr_array(out)),
           "zro_allreduce_avg")
    return out


def average(world: int, x: Sequence[np.ndarray], scale: float) -> np.ndarray:
    """The averaged gradient of every position of x[0..world-1] (one array):
    zro_allreduce_avg with postscale 1 and every replica's output the same
    array, so a caller comparing long flat ranges holds one result, not N."""
    n = int(x[0].shape[0])
    code = _dtype_code(x[0])
    out = np.empty(n, dtype=np.float32)
    outs = (ctypes.c_void_p * world)(*([_ptr(out)] * world))
    _check(lib().zro_allreduce_avg(world, n, _ptr_array(x), code, scale, 1.0, outs), "zro_allreduce_avg")
    return out


def f16_to_f32(h: np.ndarray) -> np.ndarray:
    h = np.ascontiguousarray(h, dtype=np.float16)
    out = np.empty(h.shape, dtype=np.float32)
    lib().zro_f16_to_f32(_ptr(h), _ptr(out), h.size)
    return out


def grad_accumulate(main_grad: np.ndarray, g: np.ndarray) -> None:
    assert main_grad.dtype == np.float32 and main_grad.shape == g.shape
    _check(lib().zro_grad_accumulate(main_grad.size, _ptr(main_grad), _ptr(g), _dtype_code(g)),
           "zro_grad_accumulate")


def adamw_scalars(hp) -> np.ndarray:
    out = np.zeros(8, dtype=np.float32)
    _check(lib().zro_adamw_scalars(hp.lr, hp.beta1, hp.beta2, hp.eps, hp.weight_decay,
                                   hp.step, _ptr(out)), "zro_adamw_scalars")
    return out


def adamw(p: np.ndarray, m: np.ndarray, v: np.ndarray, g: np.ndarray, hp) -> None:
    """In-place AdamW step on float32 arrays; hp has lr, beta1, beta2, eps, weight_decay, step."""
    for a in (p, m, v, g):
        assert a.dtype == np.float32 and a.shape == p.shape
    _check(lib().zro_adamw(p.size, _ptr(p), _ptr(m), _ptr(v), _ptr(g), hp.lr, hp.beta1,
                           hp.beta2, hp.eps, hp.weight_decay, hp.step), "zro_adamw")


def gather_cast_bf16(lay: Layout, master: Sequence[np.ndarray]) -> np.ndarray:
    out = np.empty(lay.P, dtype=np.uint16)
    _check(lib().zro_gather_cast_bf16(lay.world, lay.T, lay.S, _ptr_array(master), _ptr(out)),
           "zro_gather_cast_bf16")
    return out


def rs_adam_fused(lay: Layout, b: int, bucket: Sequence[np.ndarray], scale: float,
                  master, m, v, hp, param_bf16: Optional[np.ndarray] = None,
                  grad_out: Optional[Sequence[np.ndarray]] = None) -> None:
    start, nb = lay.bucket(b)
    code = _dtype_code(bucket[0])
    if lay.order is not None:
        fm = lay.flat_map(b)
        _check(lib().zro_rs_adam_fused_map(
            lay.world, lay.T, lay.S, nb, _ptr(fm), _ptr_array(bucket), code, scale,
            _ptr_array(master), _ptr_array(m), _ptr_array(v),
            hp.lr, hp.beta1, hp.beta2, hp.eps, hp.weight_decay, hp.step,
            None if param_bf16 is None else _ptr(param_bf16),
            None if grad_out is None else _ptr_array(grad_out)), "zro_rs_adam_fused_map")
        return
    _check(lib().zro_rs_adam_fused(
        lay.world, lay.T, lay.S, start, nb, _ptr_array(bucket), code, scale,
        _ptr_array(master), _ptr_array(m), _ptr_array(v),
        hp.lr, hp.beta1, hp.beta2, hp.eps, hp.weight_decay, hp.step,
        None if param_bf16 is None else _ptr(param_bf16),
        None if grad_out is None else _ptr_array(grad_out)), "zro_rs_adam_fused")


class GradStats(NamedTuple):
    """The global gradient check's outcome (zro_grad_check)."""
    sumsq: float
    nonfinite: int
    norm: float
    coef: float
    skip: bool


def grad_check(grad: Sequence[np.ndarray], max_norm: float) -> GradStats:
    """Global L2 norm, overflow count and clip coefficient of every rank's averaged shard."""
    S = grad[0].size
    for a in grad:
        assert a.dtype == np.float32 and a.size == S
    sumsq, norm = ctypes.c_double(), ctypes.c_double()
    bad, skip, coef = ctypes.c_int64(), ctypes.c_int32(), ctypes.c_float()
    _check(lib().zro_grad_check(len(grad), S, _ptr_array(grad), max_norm, ctypes.byref(sumsq), ctypes.byref(bad),
                                ctypes.byref(norm), ctypes.byref(coef), ctypes.byref(skip)), "zro_grad_check")
    return GradStats(sumsq.value, bad.value, norm.value, coef.value, bool(skip.value))


def adam_clip_step(lay: Layout, master, m, v, grad, hp, coef: float, skip: bool,
                   param_bf16: Optional[np.ndarray] = None) -> None:
    """The step the check steers: nothing if skip, else AdamW on g * coef and the bf16 cast."""
    for arrs in (master, m, v, grad):
        assert len(arrs) == lay.world and all(a.dtype == np.float32 and a.size == lay.S for a in arrs)
    _check(lib().zro_adam_clip_step(
        lay.world, lay.T, lay.S, _ptr_array(master), _ptr_array(m), _ptr_array(v), _ptr_array(grad),
        coef, int(skip), hp.lr, hp.beta1, hp.beta2, hp.eps, hp.weight_decay, hp.step,
        None if param_bf16 is None else _ptr(param_bf16)), "zro_adam_clip_step")


def comm_bytes(scheme: int, world: int, S: int, elem_bytes: int) -> float:
    out = ctypes.c_double()
    _check(lib().zro_comm_bytes(scheme, world, S, elem_bytes, ctypes.byref(out)), "zro_comm_bytes")
    return out.value


def layout_bytes(stage: int, T: int, S: int) -> float:
    out = ctypes.c_double()
    _check(lib().zro_layout_bytes(stage, T, S, ctypes.byref(out)), "zro_layout_bytes")
    return out.value


# ----------------------------------------------------------------------------
# Convenience: whole-flat-space helpers used by tests and the CPU baseline
# ----------------------------------------------------------------------------

def shards_from_flat(lay: Layout, flat: np.ndarray) -> List[np.ndarray]:
    """Split a flat float32 [T] array into N partition arrays of S, zero padded."""
    full = np.zeros(lay.P, dtype=np.float32)
    full[: lay.T] = flat[: lay.T]
    return [np.ascontiguousarray(full[r * lay.S:(r + 1) * lay.S]) for r in range(lay.world)]


def params_from_flat(lay: Layout, flat: np.ndarray) -> List[np.ndarray]:
    """Views of a flat [T] array as the per-parameter tensors."""
    return [flat[int(o): int(o) + int(n)] for o, n in zip(lay.offset, lay.numel)]
