"""Host-side checks of libzr (CPU only, no kernel launches).

The library loads, exports every entry point include/zr.h declares, and its
host code -- layout, slices, runs, AdamW scalars, byte accounting -- agrees
bit-exactly with the oracle. Argument errors come back as status codes.
"""
import ctypes
import os
import re

import numpy as np
import pytest

import oracle
from zero_partition_aware_gb300 import workloads as W

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def zr():
    from zero_partition_aware_gb300 import build
    build.build()
    from zero_partition_aware_gb300 import zr as mod
    return mod


def _declared_entry_points():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            src = open(os.path.join(ROOT, "include", fn)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names |= set(re.findall(r"\b(zr_\w+)\s*\(", src))
    return names


def test_library_exports_every_declared_symbol(zr):
    declared = _declared_entry_points()
    assert declared, "no declarations found"
    lib = ctypes.CDLL(zr.LIB_PATH)
    missing = [n for n in sorted(declared) if not hasattr(lib, n)]
    assert not missing, missing
    assert declared == set(zr.EXPORTED)


def test_status_strings(zr):
    assert zr.zr_status_string(0) == "ZR_OK"
    assert zr.zr_status_string(-4) == "ZR_ERR_ALIGN"
    assert zr.zr_version() >= 1


def _same_layout(lib_lay, orc):
    assert (lib_lay.T, lib_lay.P, lib_lay.S) == (orc.T, orc.P, orc.S)
    assert lib_lay.n_buckets == orc.n_buckets
    assert np.array_equal(lib_lay.slices(), orc.slices)
    assert np.array_equal(lib_lay.runs(), orc.runs)
    for b in range(orc.n_buckets):
        assert lib_lay.bucket(b) == orc.bucket(b)
    for i in range(orc.n_params):
        assert lib_lay.param(i) == (int(orc.offset[i]), int(orc.bucket_of[i]))
        assert lib_lay.param_partitions(i) == orc.param_partitions(i)


@pytest.mark.parametrize("name", list(W.WORKLOADS))
def test_layout_matches_oracle_on_workloads(zr, name):
    wl = W.WORKLOADS[name]
    _same_layout(zr.Layout(list(wl.numel), wl.world, wl.bucket), oracle.layout(list(wl.numel), wl.world, wl.bucket))


@pytest.mark.parametrize("seed", range(20))
def test_ordered_layout_matches_oracle(zr, seed):
    """Buckets filled in a gradient arrival order (reverse, random, or pairs swapped)."""
    rng = np.random.default_rng(1000 + seed)
    n = int(rng.integers(1, 50))
    world = int(rng.choice([1, 2, 3, 4, 8, 16, 32]))
    numel = W.random_numels(rng, n, 1, 6000)
    B = int(rng.integers(1, 30000))
    kind = seed % 3
    if kind == 0:
        order = list(range(n - 1, -1, -1))
    elif kind == 1:
        order = [int(x) for x in rng.permutation(n)]
    else:
        order = list(range(n))
        for i in range(0, n - 1, 2):
            order[i], order[i + 1] = order[i + 1], order[i]
    _same_layout(zr.Layout(numel, world, B, arrival=order), oracle.layout(numel, world, B, order=order))


def test_ordered_layout_rejects_non_permutations(zr):
    for bad in ([0, 0, 2], [0, 1, 3], [-1, 1, 2]):
        with pytest.raises(zr.ZrError) as e:
            zr.Layout([3, 4, 5], 2, 10, arrival=bad)
        assert e.value.status == zr.ZR_ERR_INVALID_ARG


@pytest.mark.parametrize("seed", range(30))
def test_layout_matches_oracle_random(zr, seed):
    rng = np.random.default_rng(seed)
    n = int(rng.integers(1, 40))
    world = int(rng.choice([1, 2, 3, 5, 8, 16, 31, 64, 100]))
    numel = W.random_numels(rng, n, 1, 5000)
    B = int(rng.integers(1, 20000))
    _same_layout(zr.Layout(numel, world, B), oracle.layout(numel, world, B))


def test_layout_edges(zr):
    for numel, world, B in [([1], 1, 1), ([1], 1024, 1), ([5, 1, 1, 1], 8, 2), ([3, 3, 3], 3, 3),
                            ([10] * 7, 4, 1), ([7], 4, 1000)]:
        _same_layout(zr.Layout(numel, world, B), oracle.layout(numel, world, B))
    empty = zr.Layout([], 4, 10)
    assert (empty.T, empty.P, empty.S, empty.n_buckets) == (0, 0, 0, 0)


def test_layout_rejects_bad_arguments(zr):
    for args in [([0], 2, 4), ([1, -3], 2, 4), ([4], 0, 4), ([4], 2, 0), ([4], zr.ZR_MAX_WORLD + 1, 4)]:
        with pytest.raises(zr.ZrError) as ei:
            zr.Layout(*args)
        assert ei.value.status == zr.ZR_ERR_INVALID_ARG
    lay = zr.Layout([10, 20], 2, 15)
    with pytest.raises(zr.ZrError):
        lay.bucket(5)
    with pytest.raises(zr.ZrError):
        lay.param(-1)


def test_defaults_match_config_table(zr):
    import json
    g = json.load(open(os.path.join(ROOT, "tests", "golden", "config_defaults.json")))
    assert zr.ZR_DEFAULT_REDUCE_BUCKET_SIZE == g["reduce_bucket_size"]
    assert zr.ZR_DEFAULT_REDUCE_SCATTER == g["reduce_scatter"]
    assert zr.ZR_DEFAULT_CONTIGUOUS_GRADIENTS == g["contiguous_gradients"]
    assert zr.ZR_DEFAULT_OVERLAP_COMM == g["overlap_comm"]
    hdr = open(os.path.join(ROOT, "include", "zr.h")).read()
    assert re.search(r"ZR_DEFAULT_REDUCE_BUCKET_SIZE\s+500000000LL", hdr)


@pytest.mark.parametrize("step", [1, 2, 10, 1000, 100000])
def test_adamw_scalars_match_oracle(zr, step):
    hp = W.AdamW(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01, step=step)
    mine = zr.zr_adamw_prepare(hp)
    ref = oracle.adamw_scalars(hp)
    got = np.array([mine[k] for k in ("beta1", "one_minus_beta1", "beta2", "one_minus_beta2", "step_size",
                                      "bc2_sqrt", "decay", "eps")], np.float32)
    assert np.array_equal(got.view(np.uint32), ref.view(np.uint32))


def test_adamw_scalars_reject_bad_hyperparameters(zr):
    for hp in [W.AdamW(step=0), W.AdamW(beta1=1.0), W.AdamW(eps=0.0), W.AdamW(lr=float("nan"))]:
        with pytest.raises(zr.ZrError):
            zr.zr_adamw_prepare(hp)


@pytest.mark.parametrize("name", list(W.WORKLOADS))
def test_accounting_matches_oracle(zr, name):
    wl = W.WORKLOADS[name]
    lay = zr.Layout(list(wl.numel), wl.world, wl.bucket)
    for scheme in range(4):
        for e in (2, 4):
            assert zr.zr_comm_bytes(lay, scheme, e) == oracle.comm_bytes(scheme, wl.world, lay.S, e)
    for stage in (0, 1, 15, 3):
        assert zr.zr_layout_bytes(lay, stage) == oracle.layout_bytes(stage, lay.T, lay.S)
    with pytest.raises(zr.ZrError):
        zr.zr_comm_bytes(lay, 4, 2)
    with pytest.raises(zr.ZrError):
        zr.zr_layout_bytes(lay, 2)


def test_device_steps_validate_before_launch(zr):
    """NULL and misaligned pointers are rejected on the host; nothing is launched."""
    lay = zr.Layout([100, 200], 2, 1000)
    L = zr._lib
    two = (ctypes.c_void_p * 2)(0x1000, 0x2000)
    odd = (ctypes.c_void_p * 2)(0x1001, 0x2000)
    nul = (ctypes.c_void_p * 2)(0, 0x2000)
    hp = zr.zr_adamw(1e-3, 0.9, 0.999, 1e-8, 0.01, 1)
    assert L.zr_reduce_scatter_avg(lay.handle, 0, nul, zr.ZR_BF16, 0.5, two, None) == zr.ZR_ERR_INVALID_ARG
    assert L.zr_reduce_scatter_avg(lay.handle, 0, odd, zr.ZR_BF16, 0.5, two, None) == zr.ZR_ERR_ALIGN
    assert L.zr_reduce_scatter_avg(lay.handle, 7, two, zr.ZR_BF16, 0.5, two, None) == zr.ZR_ERR_INVALID_ARG
    assert L.zr_reduce_scatter_avg(lay.handle, 0, two, 9, 0.5, two, None) == zr.ZR_ERR_INVALID_ARG
    assert L.zr_reduce_scatter_avg(lay.handle, 0, two, zr.ZR_BF16, float("inf"), two, None) == zr.ZR_ERR_INVALID_ARG
    assert L.zr_rs_adam_fused(lay.handle, 0, two, zr.ZR_BF16, 0.5, two, two, two, None, None, None,
                              None) == zr.ZR_ERR_INVALID_ARG
    bad = zr.zr_adamw(1e-3, 0.9, 0.999, 1e-8, 0.01, 0)
    assert L.zr_rs_adam_fused(lay.handle, 0, two, zr.ZR_BF16, 0.5, two, two, two, ctypes.byref(bad), None,
                              None, None) == zr.ZR_ERR_INVALID_ARG
    assert L.zr_rs_adam_fused(lay.handle, 0, two, zr.ZR_BF16, 0.5, two, two, two, ctypes.byref(hp),
                              ctypes.c_void_p(0x1001), None, None) == zr.ZR_ERR_ALIGN
    assert L.zr_adam_shard_step(lay.handle, 2, two, two, two, two, ctypes.byref(hp), None) == zr.ZR_ERR_INVALID_ARG
    assert L.zr_gather_cast_bf16(lay.handle, two, ctypes.c_void_p(0x1001), None) == zr.ZR_ERR_ALIGN
    assert L.zr_grad_accumulate(ctypes.c_void_p(0x1002), ctypes.c_void_p(0x2000), zr.ZR_BF16, 10,
                                None) == zr.ZR_ERR_ALIGN
    assert L.zr_grad_accumulate(None, None, zr.ZR_BF16, 0, None) == zr.ZR_OK  # empty: nothing to do
    assert L.zr_grad_accumulate(None, None, zr.ZR_BF16, -1, None) == zr.ZR_ERR_INVALID_ARG
    grads = (ctypes.c_void_p * 4)(0x1000, 0x2001, 0x3000, 0x4000)
    assert L.zr_bucket_pack(lay.handle, 0, grads, zr.ZR_BF16, two, None) == zr.ZR_ERR_ALIGN
    assert "grads" in zr.last_error()


def test_launch_without_device_reports_state(zr):
    """With no usable GPU a well-formed call fails with ZR_ERR_STATE (never run where a GPU exists)."""
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present: this check only runs on a machine without one")
    lay = zr.Layout([100, 200], 2, 1000)
    two = (ctypes.c_void_p * 2)(0x1000, 0x2000)
    rc = zr._lib.zr_reduce_scatter_avg(lay.handle, 0, two, zr.ZR_BF16, 0.5, two, None)
    assert rc in (zr.ZR_ERR_STATE, zr.ZR_ERR_CUDA)


def test_gradient_check_validates_before_launch(zr):
    """The global gradient check's entry points reject bad arguments on the host."""
    lay = zr.Layout([100, 200], 2, 1000)
    L = zr._lib
    two = (ctypes.c_void_p * 2)(0x1000, 0x2000)
    odd = (ctypes.c_void_p * 2)(0x1001, 0x2000)
    hp = zr.zr_adamw(1e-3, 0.9, 0.999, 1e-8, 0.01, 1)
    assert L.zr_gradcheck_create(None) == zr.ZR_ERR_INVALID_ARG
    assert L.zr_gradcheck_destroy(None) == zr.ZR_OK
    assert L.zr_gradcheck_reset(None, None) == zr.ZR_ERR_INVALID_ARG
    assert L.zr_grad_check_finalize(None, 1.0, None) == zr.ZR_ERR_INVALID_ARG
    assert L.zr_gradcheck_read(None, None, None) == zr.ZR_ERR_INVALID_ARG
    assert L.zr_rs_direct_norm(None, 0, 0.5, two, None, None) == zr.ZR_ERR_INVALID_ARG
    # the layout and pointer checks come before the check object's
    assert L.zr_reduce_scatter_avg_norm(lay.handle, 0, odd, zr.ZR_BF16, 0.5, two, None, None) == zr.ZR_ERR_ALIGN
    assert L.zr_reduce_scatter_avg_norm(lay.handle, 5, two, zr.ZR_BF16, 0.5, two, None, None) == zr.ZR_ERR_INVALID_ARG
    assert L.zr_reduce_scatter_avg_norm(lay.handle, 0, two, zr.ZR_BF16, 0.5, two, None, None) == zr.ZR_ERR_INVALID_ARG
    assert L.zr_adam_clip_step(None, two, two, two, two, ctypes.byref(hp), None, None, None) == zr.ZR_ERR_INVALID_ARG
    assert L.zr_adam_clip_step(lay.handle, two, two, two, None, ctypes.byref(hp), None, None,
                               None) == zr.ZR_ERR_INVALID_ARG
    assert L.zr_adam_clip_step(lay.handle, two, two, two, two, ctypes.byref(hp), None, None,
                               None) == zr.ZR_ERR_INVALID_ARG
    assert "gradient check" in zr.last_error()


def test_gradient_check_create_without_device_reports_state(zr):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present: this check only runs on a machine without one")
    h = ctypes.c_void_p()
    assert zr._lib.zr_gradcheck_create(ctypes.byref(h)) in (zr.ZR_ERR_STATE, zr.ZR_ERR_OOM, zr.ZR_ERR_CUDA)
    assert not h.value


def test_range_folded_and_first_validate_before_launch(zr):
    """zr_step_direct_range, zr_rs_direct_norm_range, zr_rs_adam_fused_acc and
    zr_grad_accumulate_first reject bad arguments on the host."""
    lay = zr.Layout([100, 200], 2, 1000)
    L = zr._lib
    two = (ctypes.c_void_p * 2)(0x1000, 0x2000)
    odd = (ctypes.c_void_p * 2)(0x1002, 0x2000)
    hp = zr.zr_adamw(1e-3, 0.9, 0.999, 1e-8, 0.01, 1)
    assert L.zr_step_direct_range(None, 0, 1, 0.5, two, two, two, ctypes.byref(hp), None, None,
                                  None) == zr.ZR_ERR_INVALID_ARG
    assert L.zr_rs_direct_norm_range(None, 0, 1, 0.5, two, None, None) == zr.ZR_ERR_INVALID_ARG
    # the folded step: bucket, dtype, pointers, world cap, scale
    assert L.zr_rs_adam_fused_acc(lay.handle, 3, two, two, zr.ZR_BF16, 0.5, two, two, two, ctypes.byref(hp),
                                  None, None, None) == zr.ZR_ERR_INVALID_ARG
    assert L.zr_rs_adam_fused_acc(lay.handle, 0, two, two, zr.ZR_FP32, 0.5, two, two, two, ctypes.byref(hp),
                                  None, None, None) == zr.ZR_ERR_INVALID_ARG
    assert L.zr_rs_adam_fused_acc(lay.handle, 0, odd, two, zr.ZR_BF16, 0.5, two, two, two, ctypes.byref(hp),
                                  None, None, None) == zr.ZR_ERR_ALIGN
    assert L.zr_rs_adam_fused_acc(lay.handle, 0, two, None, zr.ZR_BF16, 0.5, two, two, two, ctypes.byref(hp),
                                  None, None, None) == zr.ZR_ERR_INVALID_ARG
    assert L.zr_rs_adam_fused_acc(lay.handle, 0, two, two, zr.ZR_BF16, float("nan"), two, two, two,
                                  ctypes.byref(hp), None, None, None) == zr.ZR_ERR_INVALID_ARG
    big = zr.Layout([100, 200], 40, 1000)
    forty = (ctypes.c_void_p * 40)(*([0x1000] * 40))
    assert L.zr_rs_adam_fused_acc(big.handle, 0, forty, forty, zr.ZR_BF16, 0.5, forty, forty, forty,
                                  ctypes.byref(hp), None, None, None) == zr.ZR_ERR_UNSUPPORTED
    # the first micro-step
    assert L.zr_grad_accumulate_first(None, None, zr.ZR_BF16, -1, None) == zr.ZR_ERR_INVALID_ARG
    assert L.zr_grad_accumulate_first(None, None, zr.ZR_BF16, 0, None) == zr.ZR_OK
    assert L.zr_grad_accumulate_first(ctypes.c_void_p(0x1002), ctypes.c_void_p(0x2000), zr.ZR_BF16, 10,
                                      None) == zr.ZR_ERR_ALIGN


@pytest.mark.parametrize("kind", ["flat", "reverse", "random"])
def test_bucket_positions_match_the_oracle(zr, kind):
    """zr_layout_bucket_positions: each param's first element inside its bucket,
    as the oracle's layout places it (the flat offset minus the bucket's flat
    start, or its bucket position)."""
    rng = np.random.default_rng(sum(map(ord, kind)))
    numel = W.random_numels(rng, 300, 1, 50_000)
    n = len(numel)
    order = None if kind == "flat" else (list(range(n - 1, -1, -1)) if kind == "reverse"
                                         else [int(x) for x in rng.permutation(n)])
    for world, B in ((8, 200_000), (16, 1), (3, 1 << 22)):
        got = zr.Layout(numel, world, B, arrival=order).bucket_positions()
        lay = oracle.layout(numel, world, B, order=order)
        if order is None:
            want = lay.offset - lay.bucket_range[lay.bucket_of, 0]
        else:
            want = lay.bucket_pos
        assert np.array_equal(got, want), (world, B)
    L = zr._lib
    lay = zr.Layout(numel, 4, 1000)
    cnt = ctypes.c_int64()
    assert L.zr_layout_bucket_positions(lay.handle, None, 0, ctypes.byref(cnt)) == zr.ZR_OK and cnt.value == n
    assert L.zr_layout_bucket_positions(None, None, 0, ctypes.byref(cnt)) == zr.ZR_ERR_INVALID_ARG
    assert L.zr_layout_bucket_positions(lay.handle, None, -1, ctypes.byref(cnt)) == zr.ZR_ERR_INVALID_ARG


def test_grouped_calls_validate_before_launch(zr):
    """zr_reduce_scatter_avg_range and zr_allreduce_avg_range reject bad ranges,
    pointers and scales on the host."""
    lay = zr.Layout([100, 200, 300], 2, 250)
    L = zr._lib
    two = (ctypes.c_void_p * 2)(0x1000, 0x2000)
    odd = (ctypes.c_void_p * 2)(0x1001, 0x2000)
    nb = lay.n_buckets
    for first, count in ((-1, 1), (0, nb + 1), (1, -1)):
        assert L.zr_reduce_scatter_avg_range(lay.handle, first, count, two, zr.ZR_BF16, 0.5, two,
                                             None) == zr.ZR_ERR_INVALID_ARG
        assert L.zr_allreduce_avg_range(lay.handle, first, count, two, zr.ZR_BF16, 0.5, 1.0, two,
                                        None) == zr.ZR_ERR_INVALID_ARG
    assert L.zr_reduce_scatter_avg_range(lay.handle, 0, 1, odd, zr.ZR_BF16, 0.5, two, None) == zr.ZR_ERR_ALIGN
    assert L.zr_reduce_scatter_avg_range(lay.handle, 0, 1, two, zr.ZR_BF16, float("nan"), two,
                                         None) == zr.ZR_ERR_INVALID_ARG
    assert L.zr_reduce_scatter_avg_range(lay.handle, 0, 1, two, zr.ZR_BF16, 0.5, None, None) == zr.ZR_ERR_INVALID_ARG
    assert L.zr_allreduce_avg_range(lay.handle, 0, 1, two, zr.ZR_BF16, 0.5, float("inf"), two,
                                    None) == zr.ZR_ERR_INVALID_ARG
    assert L.zr_allreduce_avg_range(lay.handle, 0, 1, two, zr.ZR_FP32, 0.5, 1.0, odd, None) == zr.ZR_ERR_ALIGN
    assert L.zr_allreduce_avg_range(None, 0, 1, two, zr.ZR_BF16, 0.5, 1.0, two, None) == zr.ZR_ERR_INVALID_ARG
    # an empty range is valid and launches nothing
    assert L.zr_reduce_scatter_avg_range(lay.handle, 1, 0, two, zr.ZR_BF16, 0.5, two, None) == zr.ZR_OK
    assert L.zr_allreduce_avg_range(lay.handle, 1, 0, two, zr.ZR_BF16, 0.5, 1.0, two, None) == zr.ZR_OK


def test_bounds_checked_build_exports_the_same_calls(zr):
    """libzr_checked.so exports every declared call too; only it answers
    zr_debug_checks (the ordinary build refuses with ZR_ERR_UNSUPPORTED)."""
    from zero_partition_aware_gb300 import build
    chk = ctypes.CDLL(build.LIB_CHECKED)
    for name in zr.EXPORTED:
        assert hasattr(chk, name), name
    n = ctypes.c_uint64()
    assert zr._lib.zr_debug_checks(0, ctypes.byref(n), None, None) == zr.ZR_ERR_UNSUPPORTED
    import torch
    if not torch.cuda.is_available():  # the checked build reaches for the device
        chk.zr_debug_checks.argtypes = [ctypes.c_int32, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]
        assert chk.zr_debug_checks(0, ctypes.byref(n), None, None) in (zr.ZR_ERR_CUDA, zr.ZR_ERR_STATE)
