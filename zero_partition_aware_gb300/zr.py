"""Thin ctypes binding of libzr (include/zr.h), same names as the C entry points.

Argument marshalling only: tensors become device addresses, lists of tensors
become host arrays of device pointers, the current torch stream becomes the
launch stream. Every step runs in libzr's sm_103a kernels; there is no
fallback. Importing this module raises ImportError if libzr.so has not been
built (``python -c "import __graft_entry__ as g; g.build()"``).
"""
from __future__ import annotations

import ctypes
import os
from typing import Iterable, Optional, Sequence

import numpy as np

# ZR_LIB names another build of the library to load (the bounds-checked
# libzr_checked.so, for tests); by default the in-tree libzr.so.
_LIB_PATH = os.environ.get("ZR_LIB") or os.path.join(os.path.dirname(os.path.abspath(__file__)), "_lib", "libzr.so")
if not os.path.exists(_LIB_PATH):
    raise ImportError(f"libzr is not built ({_LIB_PATH} missing); run zero_partition_aware_gb300.build.build()")
_lib = ctypes.CDLL(_LIB_PATH)

ZR_OK = 0
ZR_ERR_INVALID_ARG = -1
ZR_ERR_CUDA = -2
ZR_ERR_OOM = -3
ZR_ERR_ALIGN = -4
ZR_ERR_TIMEOUT = -5
ZR_ERR_STATE = -6
ZR_ERR_UNSUPPORTED = -7
ZR_BF16, ZR_FP32, ZR_FP16 = 0, 1, 2
ZR_MAX_WORLD = 1024
ZR_DEFAULT_REDUCE_BUCKET_SIZE = 500_000_000
ZR_DEFAULT_REDUCE_SCATTER = True
ZR_DEFAULT_CONTIGUOUS_GRADIENTS = True
ZR_DEFAULT_OVERLAP_COMM = False

LIB_PATH = _LIB_PATH


class ZrError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(message)
        self.status = status


class zr_layout_info(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int64), ("P", ctypes.c_int64), ("S", ctypes.c_int64),
                ("n_params", ctypes.c_int64), ("n_buckets", ctypes.c_int64),
                ("n_slices", ctypes.c_int64), ("n_runs", ctypes.c_int64),
                ("reduce_bucket_size", ctypes.c_int64), ("world", ctypes.c_int32)]


class zr_slice(ctypes.Structure):
    _fields_ = [("param", ctypes.c_int64), ("bucket", ctypes.c_int64), ("dst", ctypes.c_int32),
                ("param_offset", ctypes.c_int64), ("bucket_offset", ctypes.c_int64),
                ("partition_offset", ctypes.c_int64), ("numel", ctypes.c_int64)]


class zr_run(ctypes.Structure):
    _fields_ = [("bucket", ctypes.c_int64), ("dst", ctypes.c_int32), ("bucket_offset", ctypes.c_int64),
                ("partition_offset", ctypes.c_int64), ("numel", ctypes.c_int64)]


class zr_adamw(ctypes.Structure):
    _fields_ = [("lr", ctypes.c_float), ("beta1", ctypes.c_float), ("beta2", ctypes.c_float),
                ("eps", ctypes.c_float), ("weight_decay", ctypes.c_float), ("step", ctypes.c_int64)]


class zr_grad_stats(ctypes.Structure):
    _fields_ = [("sumsq", ctypes.c_double), ("norm", ctypes.c_double), ("nonfinite", ctypes.c_uint64),
                ("coef", ctypes.c_float), ("skip", ctypes.c_int32)]


class zr_adamw_scalars(ctypes.Structure):
    _fields_ = [(n, ctypes.c_float) for n in ("beta1", "one_minus_beta1", "beta2", "one_minus_beta2",
                                                "step_size", "bc2_sqrt", "decay", "eps")]


_vp = ctypes.c_void_p
_i32, _i64, _f32 = ctypes.c_int32, ctypes.c_int64, ctypes.c_float
_P = ctypes.POINTER

_SIGS = {
    "zr_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "zr_last_error": (ctypes.c_int, [ctypes.c_char_p, ctypes.c_size_t]),
    "zr_version": (ctypes.c_int, []),
    "zr_launch_count": (ctypes.c_int64, []),
    "zr_layout_create": (ctypes.c_int, [_vp, _i64, _i32, _i64, _P(_vp)]),
    "zr_layout_create_ordered": (ctypes.c_int, [_vp, _i64, _i32, _i64, _vp, _P(_vp)]),
    "zr_layout_destroy": (ctypes.c_int, [_vp]),
    "zr_layout_query": (ctypes.c_int, [_vp, _P(zr_layout_info)]),
    "zr_layout_param_partitions": (ctypes.c_int, [_vp, _i64, _vp, _vp, _i32, _P(_i32)]),
    "zr_layout_slices": (ctypes.c_int, [_vp, _vp, _i64, _P(_i64)]),
    "zr_layout_runs": (ctypes.c_int, [_vp, _vp, _i64, _P(_i64)]),
    "zr_layout_bucket": (ctypes.c_int, [_vp, _i64, _P(_i64), _P(_i64)]),
    "zr_layout_param": (ctypes.c_int, [_vp, _i64, _P(_i64), _P(_i64)]),
    "zr_layout_bucket_positions": (ctypes.c_int, [_vp, _vp, _i64, _P(_i64)]),
    "zr_bucket_pack": (ctypes.c_int, [_vp, _i64, _vp, ctypes.c_int, _vp, _vp]),
    "zr_pack_plan_create": (ctypes.c_int, [_vp, _vp, ctypes.c_int, _vp, _P(_vp)]),
    "zr_pack_plan_destroy": (ctypes.c_int, [_vp]),
    "zr_bucket_pack_planned": (ctypes.c_int, [_vp, _i64, _vp]),
    "zr_bucket_pack_noalloc": (ctypes.c_int, [_vp, _i64, _vp, ctypes.c_int, _vp, _vp]),
    "zr_host_mapped": (ctypes.c_int, [_vp, ctypes.POINTER(ctypes.c_int32)]),
    "zr_rs_adam_fused_range": (ctypes.c_int, [_vp, _i64, _i64, _vp, ctypes.c_int, _f32, _vp, _vp, _vp, _vp, _vp,
                                              _vp, _vp]),
    "zr_grad_accumulate": (ctypes.c_int, [_vp, _vp, ctypes.c_int, _i64, _vp]),
    "zr_grad_accumulate_first": (ctypes.c_int, [_vp, _vp, ctypes.c_int, _i64, _vp]),
    "zr_reduce_scatter_avg": (ctypes.c_int, [_vp, _i64, _vp, ctypes.c_int, _f32, _vp, _vp]),
    "zr_reduce_scatter_avg_range": (ctypes.c_int, [_vp, _i64, _i64, _vp, ctypes.c_int, _f32, _vp, _vp]),
    "zr_adam_shard_step": (ctypes.c_int, [_vp, _i32, _vp, _vp, _vp, _vp, _P(zr_adamw), _vp]),
    "zr_gather_cast_bf16": (ctypes.c_int, [_vp, _vp, _vp, _vp]),
    "zr_rs_adam_fused": (ctypes.c_int, [_vp, _i64, _vp, ctypes.c_int, _f32, _vp, _vp, _vp,
                                        _P(zr_adamw), _vp, _vp, _vp]),
    "zr_rs_adam_fused_acc": (ctypes.c_int, [_vp, _i64, _vp, _vp, ctypes.c_int, _f32, _vp, _vp, _vp,
                                            _P(zr_adamw), _vp, _vp, _vp]),
    "zr_allreduce_avg": (ctypes.c_int, [_vp, _i64, _vp, ctypes.c_int, _f32, _f32, _vp, _vp]),
    "zr_allreduce_avg_range": (ctypes.c_int, [_vp, _i64, _i64, _vp, ctypes.c_int, _f32, _f32, _vp, _vp]),
    "zr_direct_plan_create": (ctypes.c_int, [_vp, _vp, ctypes.c_int, _P(_vp)]),
    "zr_direct_plan_destroy": (ctypes.c_int, [_vp]),
    "zr_step_direct": (ctypes.c_int, [_vp, _i64, _f32, _vp, _vp, _vp, _P(zr_adamw), _vp, _vp, _vp]),
    "zr_step_direct_range": (ctypes.c_int, [_vp, _i64, _i64, _f32, _vp, _vp, _vp, _P(zr_adamw), _vp, _vp, _vp]),
    "zr_rs_direct_norm_range": (ctypes.c_int, [_vp, _i64, _i64, _f32, _vp, _vp, _vp]),
    "zr_gradcheck_create": (ctypes.c_int, [_P(_vp)]),
    "zr_gradcheck_destroy": (ctypes.c_int, [_vp]),
    "zr_gradcheck_reset": (ctypes.c_int, [_vp, _vp]),
    "zr_reduce_scatter_avg_norm": (ctypes.c_int, [_vp, _i64, _vp, ctypes.c_int, _f32, _vp, _vp, _vp]),
    "zr_rs_direct_norm": (ctypes.c_int, [_vp, _i64, _f32, _vp, _vp, _vp]),
    "zr_grad_check_finalize": (ctypes.c_int, [_vp, _f32, _vp]),
    "zr_adam_clip_step": (ctypes.c_int, [_vp, _vp, _vp, _vp, _vp, _P(zr_adamw), _vp, _vp, _vp]),
    "zr_gradcheck_read": (ctypes.c_int, [_vp, _vp, _P(zr_grad_stats)]),
    "zr_adamw_prepare": (ctypes.c_int, [_P(zr_adamw), _P(zr_adamw_scalars)]),
    "zr_debug_checks": (ctypes.c_int, [_i32, _P(ctypes.c_uint64), _P(_i32), _P(_i64)]),
    "zr_arith_check": (ctypes.c_int, [_i32, ctypes.c_uint64, ctypes.c_uint64, _P(zr_adamw),
                                      _P(ctypes.c_uint64), _P(ctypes.c_uint64), _i32]),
    "zr_comm_bytes": (ctypes.c_int, [_vp, _i32, _i32, _P(ctypes.c_double)]),
    "zr_layout_bytes": (ctypes.c_int, [_vp, _i32, _P(ctypes.c_double)]),
}
for _name, (_res, _args) in _SIGS.items():
    _fn = getattr(_lib, _name)
    _fn.restype = _res
    _fn.argtypes = _args

EXPORTED = tuple(_SIGS)


def last_error() -> str:
    buf = ctypes.create_string_buffer(1024)
    _lib.zr_last_error(buf, len(buf))
    return buf.value.decode(errors="replace")


def _check(rc: int, what: str):
    if rc != ZR_OK:
        raise ZrError(rc, f"{what}: {last_error() or _lib.zr_status_string(rc).decode()}")


# ----------------------------------------------------------------------------
# Marshalling helpers
# ----------------------------------------------------------------------------

_MAPPED = {}  # host page -> mapped into the device's address space (checked once per page)


def _check_mapped(ptr: int) -> None:
    page = ptr >> 21
    ok = _MAPPED.get(page)
    if ok is None:
        m = ctypes.c_int32(0)
        _check(_lib.zr_host_mapped(ptr, ctypes.byref(m)), "zr_host_mapped")
        ok = _MAPPED[page] = bool(m.value)
    if not ok:
        raise ValueError("pinned host memory at this address is not mapped into the device's address space")


def _addr(x) -> Optional[int]:
    """Device address of a tensor, or an int address, or None. A pinned
    (page-locked) CPU tensor counts: pinned host memory is mapped into the
    device's address space at the same address, so kernels read and write it in
    place over the host link."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if hasattr(x, "data_ptr"):
        if not x.is_cuda:
            if not x.is_pinned():
                raise ValueError("libzr takes CUDA tensors or pinned CPU tensors; got a pageable CPU tensor")
            _check_mapped(x.data_ptr())
        if not x.is_contiguous():
            raise ValueError("libzr takes contiguous tensors")
        return x.data_ptr()
    raise TypeError(f"cannot take a device address of {type(x)}")


class PtrArray:
    """A host array of device pointers, built once and reusable across calls."""

    def __init__(self, items: Iterable):
        if not isinstance(items, np.ndarray):
            items = list(items)  # one pass: a generator's tensors must be both addressed and kept alive
        vals = [_addr(t) or 0 for t in items]
        self.array = np.asarray(vals, dtype=np.uint64)
        self._keep = items if not isinstance(items, np.ndarray) else None

    @property
    def ptr(self) -> int:
        return self.array.ctypes.data

    def __len__(self):
        return int(self.array.shape[0])


def _ptrs(x) -> Optional[PtrArray]:
    if x is None:
        return None
    if isinstance(x, PtrArray):
        return x
    return PtrArray(x)


def _dtype_of(x, dtype) -> int:
    if dtype is not None:
        return int(dtype)
    import torch
    seq = x
    while isinstance(seq, (list, tuple)):
        seq = next((s for s in seq if s is not None), None)
    if isinstance(seq, PtrArray):
        raise ValueError("dtype is required with a prebuilt PtrArray")
    if seq is not None and hasattr(seq, "dtype"):
        if seq.dtype == torch.bfloat16:
            return ZR_BF16
        if seq.dtype == torch.float32:
            return ZR_FP32
        if seq.dtype == torch.float16:
            return ZR_FP16
    raise ValueError("cannot infer dtype: pass dtype=ZR_BF16, ZR_FP32 or ZR_FP16")


def _stream(stream) -> int:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _hp(hp) -> zr_adamw:
    if isinstance(hp, zr_adamw):
        return hp
    return zr_adamw(hp.lr, hp.beta1, hp.beta2, hp.eps, hp.weight_decay, int(hp.step))


# ----------------------------------------------------------------------------
# Layout
# ----------------------------------------------------------------------------

class Layout:
    """Owns a zr_layout handle (host memory only)."""

    def __init__(self, numel: Sequence[int], world: int,
                 reduce_bucket_size: int = ZR_DEFAULT_REDUCE_BUCKET_SIZE, arrival: Optional[Sequence[int]] = None):
        arr = np.ascontiguousarray(np.asarray(numel, dtype=np.int64))
        h = ctypes.c_void_p()
        if arrival is None:
            _check(_lib.zr_layout_create(arr.ctypes.data if arr.size else None, int(arr.size), int(world),
                                         int(reduce_bucket_size), ctypes.byref(h)), "zr_layout_create")
        else:
            order = np.ascontiguousarray(np.asarray(arrival, dtype=np.int64))
            _check(_lib.zr_layout_create_ordered(arr.ctypes.data if arr.size else None, int(arr.size), int(world),
                                                 int(reduce_bucket_size), order.ctypes.data if order.size else None,
                                                 ctypes.byref(h)), "zr_layout_create_ordered")
        self.arrival = None if arrival is None else [int(x) for x in arrival]
        self._h = h
        info = zr_layout_info()
        _check(_lib.zr_layout_query(h, ctypes.byref(info)), "zr_layout_query")
        self.info = info
        self.numel = arr
        self._bucket_cache = {}

    @property
    def handle(self):
        return self._h

    def close(self):
        if getattr(self, "_h", None) is not None and self._h.value:
            _lib.zr_layout_destroy(self._h)
            self._h = ctypes.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    T = property(lambda s: int(s.info.T))
    P = property(lambda s: int(s.info.P))
    S = property(lambda s: int(s.info.S))
    world = property(lambda s: int(s.info.world))
    n_params = property(lambda s: int(s.info.n_params))
    n_buckets = property(lambda s: int(s.info.n_buckets))
    n_slices = property(lambda s: int(s.info.n_slices))
    n_runs = property(lambda s: int(s.info.n_runs))
    reduce_bucket_size = property(lambda s: int(s.info.reduce_bucket_size))

    def bucket(self, b: int):
        """(flat_start, numel) of bucket b."""
        if b not in self._bucket_cache:
            s, n = ctypes.c_int64(), ctypes.c_int64()
            _check(_lib.zr_layout_bucket(self._h, int(b), ctypes.byref(s), ctypes.byref(n)), "zr_layout_bucket")
            self._bucket_cache[b] = (s.value, n.value)
        return self._bucket_cache[b]

    def param(self, i: int):
        """(flat_offset, bucket) of param i."""
        o, b = ctypes.c_int64(), ctypes.c_int64()
        _check(_lib.zr_layout_param(self._h, int(i), ctypes.byref(o), ctypes.byref(b)), "zr_layout_param")
        return o.value, b.value

    def param_partitions(self, i: int):
        """(param_to_partition_ids, grad_start_offset) of param i."""
        n = ctypes.c_int32()
        _check(_lib.zr_layout_param_partitions(self._h, int(i), None, None, 0, ctypes.byref(n)),
               "zr_layout_param_partitions")
        ids = np.zeros(max(n.value, 1), np.int32)
        gso = np.zeros(max(n.value, 1), np.int64)
        _check(_lib.zr_layout_param_partitions(self._h, int(i), ids.ctypes.data, gso.ctypes.data,
                                               n.value, ctypes.byref(n)), "zr_layout_param_partitions")
        return [int(x) for x in ids[: n.value]], [int(x) for x in gso[: n.value]]

    def slices(self) -> np.ndarray:
        """[n_slices, 7]: param, bucket, dst, param_offset, bucket_offset, partition_offset, numel."""
        n = ctypes.c_int64()
        _check(_lib.zr_layout_slices(self._h, None, 0, ctypes.byref(n)), "zr_layout_slices")
        buf = (zr_slice * max(n.value, 1))()
        _check(_lib.zr_layout_slices(self._h, buf, n.value, ctypes.byref(n)), "zr_layout_slices")
        return np.array([[s.param, s.bucket, s.dst, s.param_offset, s.bucket_offset, s.partition_offset,
                          s.numel] for s in buf[: n.value]], dtype=np.int64).reshape(-1, 7)

    def runs(self) -> np.ndarray:
        """[n_runs, 5]: bucket, dst, bucket_offset, partition_offset, numel."""
        n = ctypes.c_int64()
        _check(_lib.zr_layout_runs(self._h, None, 0, ctypes.byref(n)), "zr_layout_runs")
        buf = (zr_run * max(n.value, 1))()
        _check(_lib.zr_layout_runs(self._h, buf, n.value, ctypes.byref(n)), "zr_layout_runs")
        return np.array([[r.bucket, r.dst, r.bucket_offset, r.partition_offset, r.numel]
                         for r in buf[: n.value]], dtype=np.int64).reshape(-1, 5)

    def bucket_positions(self) -> np.ndarray:
        """[n_params]: where each param's gradient starts inside its bucket."""
        out = np.zeros(max(self.n_params, 1), np.int64)
        n = ctypes.c_int64()
        _check(_lib.zr_layout_bucket_positions(self._h, out.ctypes.data, out.size, ctypes.byref(n)),
               "zr_layout_bucket_positions")
        return out[: n.value]

    def offsets(self) -> np.ndarray:
        return np.array([self.param(i)[0] for i in range(self.n_params)], dtype=np.int64)


def zr_layout_create_ordered(numel: Sequence[int], world: int, reduce_bucket_size: int,
                             arrival: Sequence[int]) -> Layout:
    return Layout(numel, world, reduce_bucket_size, arrival)


def zr_layout_create(numel: Sequence[int], world: int,
                     reduce_bucket_size: int = ZR_DEFAULT_REDUCE_BUCKET_SIZE) -> Layout:
    return Layout(numel, world, reduce_bucket_size)


def zr_layout_destroy(layout: Layout) -> None:
    layout.close()


# ----------------------------------------------------------------------------
# Device steps
# ----------------------------------------------------------------------------

def zr_bucket_pack(layout: Layout, bucket: int, grads, bucket_out, dtype=None, stream=None) -> None:
    """grads: [world][n_params] tensors (or a flat PtrArray of world*n_params);
    bucket_out: [world] tensors of numel_b elements."""
    if isinstance(grads, PtrArray):
        g = grads
    else:
        g = PtrArray([t for row in grads for t in row])
    d = _dtype_of(bucket_out, dtype)
    o = _ptrs(bucket_out)
    _check(_lib.zr_bucket_pack(layout.handle, int(bucket), g.ptr, d, o.ptr, _stream(stream)), "zr_bucket_pack")


def zr_bucket_pack_noalloc(layout: Layout, bucket: int, grads, bucket_out, dtype=None, stream=None) -> None:
    """zr_bucket_pack that allocates no device memory (see include/zr.h)."""
    g = grads if isinstance(grads, PtrArray) else PtrArray([t for row in grads for t in row])
    d = _dtype_of(bucket_out, dtype)
    o = _ptrs(bucket_out)
    _check(_lib.zr_bucket_pack_noalloc(layout.handle, int(bucket), g.ptr, d, o.ptr, _stream(stream)),
           "zr_bucket_pack_noalloc")


class PackPlan:
    """Owns a zr_pack_plan: device-resident packing descriptors for fixed
    gradient tensors and bucket buffers (one launch per bucket)."""

    def __init__(self, layout: Layout, grads, bucket_out, dtype=None):
        g = grads if isinstance(grads, PtrArray) else PtrArray([t for row in grads for t in row])
        o = _ptrs(bucket_out)
        d = _dtype_of(bucket_out, dtype)
        h = ctypes.c_void_p()
        _check(_lib.zr_pack_plan_create(layout.handle, g.ptr, d, o.ptr, ctypes.byref(h)), "zr_pack_plan_create")
        self._h = h
        self._keep = (layout, g, o)

    @property
    def handle(self):
        return self._h

    def close(self):
        if getattr(self, "_h", None) is not None and self._h.value:
            _lib.zr_pack_plan_destroy(self._h)
            self._h = ctypes.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def zr_pack_plan_create(layout: Layout, grads, bucket_out, dtype=None) -> PackPlan:
    return PackPlan(layout, grads, bucket_out, dtype)


def zr_pack_plan_destroy(plan: PackPlan) -> None:
    plan.close()


def zr_bucket_pack_planned(plan: PackPlan, bucket: int, stream=None) -> None:
    _check(_lib.zr_bucket_pack_planned(plan.handle, int(bucket), _stream(stream)), "zr_bucket_pack_planned")


def zr_grad_accumulate(main_grad, g, n: Optional[int] = None, dtype=None, stream=None) -> None:
    if n is None:
        n = int(main_grad.numel())
        if int(g.numel()) != n:
            raise ValueError("main_grad and g sizes differ")
    d = _dtype_of([g], dtype)
    _check(_lib.zr_grad_accumulate(_addr(main_grad), _addr(g), d, int(n), _stream(stream)), "zr_grad_accumulate")


def zr_grad_accumulate_first(main_grad, g, n: Optional[int] = None, dtype=None, stream=None) -> None:
    if n is None:
        n = int(main_grad.numel())
        if int(g.numel()) != n:
            raise ValueError("main_grad and g sizes differ")
    d = _dtype_of([g], dtype)
    _check(_lib.zr_grad_accumulate_first(_addr(main_grad), _addr(g), d, int(n), _stream(stream)),
           "zr_grad_accumulate_first")


def zr_reduce_scatter_avg(layout: Layout, bucket: int, bucket_in, scale: float, shard_grad,
                          dtype=None, stream=None) -> None:
    d = _dtype_of(bucket_in, dtype)
    x, g = _ptrs(bucket_in), _ptrs(shard_grad)
    _check(_lib.zr_reduce_scatter_avg(layout.handle, int(bucket), x.ptr, d, float(scale), g.ptr,
                                      _stream(stream)), "zr_reduce_scatter_avg")


def zr_reduce_scatter_avg_range(layout: Layout, bucket_first: int, bucket_count: int, grad_buf, scale: float,
                                shard_grad, dtype=None, stream=None) -> None:
    """grad_buf: [world] buffers holding the buckets back to back in bucket order."""
    d = _dtype_of(grad_buf, dtype)
    x, g = _ptrs(grad_buf), _ptrs(shard_grad)
    _check(_lib.zr_reduce_scatter_avg_range(layout.handle, int(bucket_first), int(bucket_count), x.ptr, d,
                                            float(scale), g.ptr, _stream(stream)), "zr_reduce_scatter_avg_range")


def zr_adam_shard_step(layout: Layout, rank: int, master, m, v, grad, hp, stream=None) -> None:
    h = _hp(hp)
    # the host pointer tables must outlive the call: keep them in locals
    pm, pmm, pv, pg = _ptrs(master), _ptrs(m), _ptrs(v), _ptrs(grad)
    _check(_lib.zr_adam_shard_step(layout.handle, int(rank), pm.ptr, pmm.ptr, pv.ptr, pg.ptr,
                                   ctypes.byref(h), _stream(stream)), "zr_adam_shard_step")


def zr_gather_cast_bf16(layout: Layout, master, param_bf16, stream=None) -> None:
    pm = _ptrs(master)
    _check(_lib.zr_gather_cast_bf16(layout.handle, pm.ptr, _addr(param_bf16), _stream(stream)),
           "zr_gather_cast_bf16")


def zr_rs_adam_fused(layout: Layout, bucket: int, bucket_in, scale: float, master, m, v, hp,
                     param_bf16=None, shard_grad_out=None, dtype=None, stream=None) -> None:
    d = _dtype_of(bucket_in, dtype)
    h = _hp(hp)
    px, pm, pmm, pv, go = _ptrs(bucket_in), _ptrs(master), _ptrs(m), _ptrs(v), _ptrs(shard_grad_out)
    _check(_lib.zr_rs_adam_fused(layout.handle, int(bucket), px.ptr, d, float(scale), pm.ptr, pmm.ptr, pv.ptr,
                                 ctypes.byref(h), _addr(param_bf16), go.ptr if go is not None else None,
                                 _stream(stream)), "zr_rs_adam_fused")


def zr_rs_adam_fused_range(layout: Layout, bucket_first: int, bucket_count: int, grad_buf, scale: float, master,
                           m, v, hp, param_bf16=None, shard_grad_out=None, dtype=None, stream=None) -> None:
    """grad_buf: [world] buffers holding the buckets back to back in bucket order."""
    d = _dtype_of(grad_buf, dtype)
    h = _hp(hp)
    px, pm, pmm, pv, go = _ptrs(grad_buf), _ptrs(master), _ptrs(m), _ptrs(v), _ptrs(shard_grad_out)
    _check(_lib.zr_rs_adam_fused_range(layout.handle, int(bucket_first), int(bucket_count), px.ptr, d, float(scale),
                                       pm.ptr, pmm.ptr, pv.ptr, ctypes.byref(h), _addr(param_bf16),
                                       go.ptr if go is not None else None, _stream(stream)),
           "zr_rs_adam_fused_range")


def zr_rs_adam_fused_acc(layout: Layout, bucket: int, main_in, last_in, scale: float, master, m, v, hp,
                         param_bf16=None, shard_grad_out=None, last_dtype=None, stream=None) -> None:
    d = _dtype_of(last_in, last_dtype)
    h = _hp(hp)
    px, py, pm, pmm, pv, go = _ptrs(main_in), _ptrs(last_in), _ptrs(master), _ptrs(m), _ptrs(v), _ptrs(shard_grad_out)
    _check(_lib.zr_rs_adam_fused_acc(layout.handle, int(bucket), px.ptr, py.ptr, d, float(scale), pm.ptr, pmm.ptr,
                                     pv.ptr, ctypes.byref(h), _addr(param_bf16), go.ptr if go is not None else None,
                                     _stream(stream)), "zr_rs_adam_fused_acc")


class DirectPlan:
    """Owns a zr_direct_plan: where every replica's per-parameter gradients live,
    in device memory, for zr_step_direct (steps 1-4 without a bucket buffer)."""

    def __init__(self, layout: Layout, grads, dtype=None):
        g = grads if isinstance(grads, PtrArray) else PtrArray([t for row in grads for t in row])
        if dtype is None:
            if isinstance(grads, PtrArray):
                raise ValueError("dtype is required with a prebuilt PtrArray")
            dtype = _dtype_of([t for row in grads for t in row], None)
        h = ctypes.c_void_p()
        _check(_lib.zr_direct_plan_create(layout.handle, g.ptr, int(dtype), ctypes.byref(h)), "zr_direct_plan_create")
        self._h = h
        self._keep = (layout, g)

    @property
    def handle(self):
        return self._h

    def close(self):
        if getattr(self, "_h", None) is not None and self._h.value:
            _lib.zr_direct_plan_destroy(self._h)
            self._h = ctypes.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def zr_direct_plan_create(layout: Layout, grads, dtype=None) -> DirectPlan:
    return DirectPlan(layout, grads, dtype)


def zr_direct_plan_destroy(plan: DirectPlan) -> None:
    plan.close()


def zr_step_direct(plan: DirectPlan, bucket: int, scale: float, master, m, v, hp, param_bf16=None,
                   shard_grad_out=None, stream=None) -> None:
    h = _hp(hp)
    pm, pmm, pv, go = _ptrs(master), _ptrs(m), _ptrs(v), _ptrs(shard_grad_out)
    _check(_lib.zr_step_direct(plan.handle, int(bucket), float(scale), pm.ptr, pmm.ptr, pv.ptr, ctypes.byref(h),
                               _addr(param_bf16), go.ptr if go is not None else None, _stream(stream)),
           "zr_step_direct")


def zr_step_direct_range(plan: DirectPlan, bucket_first: int, bucket_count: int, scale: float, master, m, v, hp,
                         param_bf16=None, shard_grad_out=None, stream=None) -> None:
    h = _hp(hp)
    pm, pmm, pv, go = _ptrs(master), _ptrs(m), _ptrs(v), _ptrs(shard_grad_out)
    _check(_lib.zr_step_direct_range(plan.handle, int(bucket_first), int(bucket_count), float(scale), pm.ptr,
                                     pmm.ptr, pv.ptr, ctypes.byref(h), _addr(param_bf16),
                                     go.ptr if go is not None else None, _stream(stream)), "zr_step_direct_range")


def zr_allreduce_avg(layout: Layout, bucket: int, bucket_in, scale: float, out, dtype=None, stream=None,
                     postscale: float = 1.0) -> None:
    d = _dtype_of(bucket_in, dtype)
    px, po = _ptrs(bucket_in), _ptrs(out)
    _check(_lib.zr_allreduce_avg(layout.handle, int(bucket), px.ptr, d, float(scale), float(postscale), po.ptr,
                                 _stream(stream)), "zr_allreduce_avg")


def zr_allreduce_avg_range(layout: Layout, bucket_first: int, bucket_count: int, grad_buf, scale: float, out,
                           dtype=None, stream=None, postscale: float = 1.0) -> None:
    d = _dtype_of(grad_buf, dtype)
    px, po = _ptrs(grad_buf), _ptrs(out)
    _check(_lib.zr_allreduce_avg_range(layout.handle, int(bucket_first), int(bucket_count), px.ptr, d, float(scale),
                                       float(postscale), po.ptr, _stream(stream)), "zr_allreduce_avg_range")


class GradCheck:
    """Owns a zr_gradcheck: the device-side sums and outcome of the global
    gradient check (norm, overflow, clip coefficient) between the averaging
    of every bucket and the optimizer step."""

    def __init__(self):
        h = ctypes.c_void_p()
        _check(_lib.zr_gradcheck_create(ctypes.byref(h)), "zr_gradcheck_create")
        self._h = h

    @property
    def handle(self):
        return self._h

    def close(self):
        if getattr(self, "_h", None) is not None and self._h.value:
            _lib.zr_gradcheck_destroy(self._h)
            self._h = ctypes.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def zr_gradcheck_create() -> GradCheck:
    return GradCheck()


def zr_gradcheck_destroy(chk: GradCheck) -> None:
    chk.close()


def zr_gradcheck_reset(chk: GradCheck, stream=None) -> None:
    _check(_lib.zr_gradcheck_reset(chk.handle, _stream(stream)), "zr_gradcheck_reset")


def zr_reduce_scatter_avg_norm(layout: Layout, bucket: int, bucket_in, scale: float, shard_grad, chk: GradCheck,
                               dtype=None, stream=None) -> None:
    d = _dtype_of(bucket_in, dtype)
    x, g = _ptrs(bucket_in), _ptrs(shard_grad)
    _check(_lib.zr_reduce_scatter_avg_norm(layout.handle, int(bucket), x.ptr, d, float(scale), g.ptr, chk.handle,
                                           _stream(stream)), "zr_reduce_scatter_avg_norm")


def zr_rs_direct_norm(plan: DirectPlan, bucket: int, scale: float, shard_grad, chk: GradCheck, stream=None) -> None:
    g = _ptrs(shard_grad)
    _check(_lib.zr_rs_direct_norm(plan.handle, int(bucket), float(scale), g.ptr, chk.handle, _stream(stream)),
           "zr_rs_direct_norm")


def zr_rs_direct_norm_range(plan: DirectPlan, bucket_first: int, bucket_count: int, scale: float, shard_grad,
                            chk: GradCheck, stream=None) -> None:
    g = _ptrs(shard_grad)
    _check(_lib.zr_rs_direct_norm_range(plan.handle, int(bucket_first), int(bucket_count), float(scale), g.ptr,
                                        chk.handle, _stream(stream)), "zr_rs_direct_norm_range")


def zr_grad_check_finalize(chk: GradCheck, max_norm: float, stream=None) -> None:
    _check(_lib.zr_grad_check_finalize(chk.handle, float(max_norm), _stream(stream)), "zr_grad_check_finalize")


def zr_adam_clip_step(layout: Layout, master, m, v, grad, hp, chk: GradCheck, param_bf16=None, stream=None) -> None:
    h = _hp(hp)
    pm, pmm, pv, pg = _ptrs(master), _ptrs(m), _ptrs(v), _ptrs(grad)
    _check(_lib.zr_adam_clip_step(layout.handle, pm.ptr, pmm.ptr, pv.ptr, pg.ptr, ctypes.byref(h), chk.handle,
                                  _addr(param_bf16), _stream(stream)), "zr_adam_clip_step")


def zr_gradcheck_read(chk: GradCheck, stream=None) -> dict:
    """The last finalized outcome (waits for the stream)."""
    st = zr_grad_stats()
    _check(_lib.zr_gradcheck_read(chk.handle, _stream(stream), ctypes.byref(st)), "zr_gradcheck_read")
    return {"sumsq": st.sumsq, "norm": st.norm, "nonfinite": int(st.nonfinite), "coef": st.coef,
            "skip": bool(st.skip)}


# ----------------------------------------------------------------------------
# Accounting
# ----------------------------------------------------------------------------

def zr_arith_check(which: int, begin: int, count: int, hp=None):
    """(mismatches, first offending indices) of the device arithmetic check."""
    h = _hp(hp) if hp is not None else zr_adamw(1e-3, 0.9, 0.999, 1e-8, 0.0, 1)
    n = ctypes.c_uint64()
    bad = (ctypes.c_uint64 * 8)()
    _check(_lib.zr_arith_check(int(which), int(begin), int(count), ctypes.byref(h), ctypes.byref(n), bad, 8),
           "zr_arith_check")
    return n.value, list(bad[: min(n.value, 8)])


def zr_debug_checks(reset: bool = False):
    """(failed checks, first check code, first element) of the bounds-checked
    build (ZrError ZR_ERR_UNSUPPORTED from the ordinary one)."""
    n, code, where = ctypes.c_uint64(), ctypes.c_int32(), ctypes.c_int64()
    _check(_lib.zr_debug_checks(int(bool(reset)), ctypes.byref(n), ctypes.byref(code), ctypes.byref(where)),
           "zr_debug_checks")
    return n.value, code.value, where.value


def zr_adamw_prepare(hp) -> dict:
    h = _hp(hp)
    out = zr_adamw_scalars()
    _check(_lib.zr_adamw_prepare(ctypes.byref(h), ctypes.byref(out)), "zr_adamw_prepare")
    return {n: getattr(out, n) for n, _ in zr_adamw_scalars._fields_}


def zr_comm_bytes(layout: Layout, scheme: int, elem_bytes: int) -> float:
    out = ctypes.c_double()
    _check(_lib.zr_comm_bytes(layout.handle, int(scheme), int(elem_bytes), ctypes.byref(out)), "zr_comm_bytes")
    return out.value


def zr_layout_bytes(layout: Layout, stage: int) -> float:
    out = ctypes.c_double()
    _check(_lib.zr_layout_bytes(layout.handle, int(stage), ctypes.byref(out)), "zr_layout_bytes")
    return out.value


def zr_status_string(status: int) -> str:
    return _lib.zr_status_string(int(status)).decode()


def zr_version() -> int:
    return int(_lib.zr_version())


def zr_launch_count() -> int:
    return int(_lib.zr_launch_count())
