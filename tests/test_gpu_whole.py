"""Every element of every full-size workload against the oracle (GPU).

Each full-size workload runs as bench.py runs it: each rank's gradients are
separately placed per-parameter tensors (512-byte aligned starts in one arena
per rank), the state is flat [P] buffers whose partitions are views. Then
every flat position of master, m, v and the bf16 parameters is compared with
the oracle, bit for bit, chunk by chunk over the flat range on every host core
(tests/flatcheck.py). With integer gradients the averaged gradient must also
equal the exact integer sum times 1/N at every element. Each test prints
"<name>: 0 of P elements differ" on success.
"""
import numpy as np
import pytest
import torch

import oracle
from zero_partition_aware_gb300 import workloads as W

import flatcheck

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def zr():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from zero_partition_aware_gb300 import build
    build.build()
    from zero_partition_aware_gb300 import zr as mod
    return mod


def _group(wl, lay, **kw):
    """The group with its state loaded from the seeded draw, and each rank's
    gradients moved param by param into its arena (then the flat draw freed)."""
    from zero_partition_aware_gb300.engine import DPGroup
    torch.cuda.empty_cache()
    inp = W.draw_inputs(wl, "cuda", seed=0)
    grp = DPGroup(list(wl.numel), wl.world, wl.bucket, **kw)
    grp.load_flat(inp["master"], inp["m"], inp["v"])
    del inp["master"], inp["m"], inp["v"]
    return grp, inp


def _arenas(wl, lay, inp):
    offs = W.arena_offsets(wl.numel, 256)
    size = offs[-1] + wl.numel[-1]
    arenas, rows = [], []
    for k in range(wl.world):
        arena = torch.zeros(size, dtype=torch.bfloat16, device="cuda")
        src = inp["grads"][k][0]
        views = [arena[o:o + n] for o, n in zip(offs, wl.numel)]
        for i, v in enumerate(views):
            v.copy_(src[int(lay.offset[i]): int(lay.offset[i]) + wl.numel[i]])
        inp["grads"][k][0] = None
        arenas.append(arena)
        rows.append(views)
    return arenas, rows, offs


def _report(capsys, name, res, outputs=("master", "m", "v", "param")):
    line = flatcheck.summary(name, res, outputs)
    with capsys.disabled():
        print("\n" + line, flush=True)
    for k in outputs:
        assert res[k] == 0, f"{line}; first {k} mismatch at flat {res[k + '_first']}"


@pytest.mark.parametrize("name,path", [("gpt2_124m", "direct"), ("gpt2_124m", "packed"),
                                       ("irregular_10k", "direct"), ("irregular_10k", "packed"),
                                       ("llama3_3b", "direct"), ("llama3_3b", "packed")])
def test_whole_workload(zr, capsys, name, path):
    """The one-pass step (zr_step_direct_range, the bench's step) or the two-kernel
    step (planned pack + zr_rs_adam_fused per bucket) over a whole full-size
    workload == the oracle at every element."""
    wl = W.WORKLOADS[name]
    lay = oracle.layout(list(wl.numel), wl.world, wl.bucket)
    grp, inp = _group(wl, lay, allocate_buckets=path == "packed")
    arenas, rows, offs = _arenas(wl, lay, inp)
    table = grp.grad_table(rows)
    before = [t.clone() for t in grp.flat_state()]
    if path == "direct":
        grp.step_direct(grp.direct_plan(table), wl.adam)
    else:
        grp.step(table, wl.adam, plan=grp.pack_plan(table))
    torch.cuda.synchronize()
    integer = wl.grad[0] == "int"
    res = flatcheck.check_whole(lay, grp.scale, wl.adam, flatcheck.ArenaGrads(arenas, lay, offs), before,
                                grp.flat_state(), grp.param, integer_avg=integer)
    _report(capsys, f"{name} {path}", res, ("master", "m", "v", "param") + (("integer_avg",) if integer else ()))


@pytest.mark.parametrize("folded", [True, False], ids=["last_folded", "unfolded"])
def test_whole_llama_micro_steps(zr, capsys, folded):
    """Llama 1.1B at full size, world 8, 4 bf16 micro-steps per rank in flat [P]
    buffers, summed into an fp32 main_grad as the bench runs it: micro-step 0
    by zr_grad_accumulate_first, then zr_grad_accumulate; folded: the last one
    added inside zr_rs_adam_fused_acc; unfolded: all four accumulated, then
    zr_rs_adam_fused on main_grad in place. Every element == the oracle's
    accumulation, average, AdamW and cast; the main_grad the step leaves too."""
    wl = W.WORKLOADS["llama_1p1b"]
    lay = oracle.layout(list(wl.numel), wl.world, wl.bucket)
    grp, inp = _group(wl, lay, grad_dtype=torch.float32, allocate_buckets=False)
    P, T, S_ = lay.P, lay.T, wl.micro_steps
    mb = []
    for k in range(wl.world):
        row = []
        for s in range(S_):
            g = inp["grads"][k][s]
            if P > T:
                t = torch.zeros(P, dtype=torch.bfloat16, device="cuda")
                t[:T].copy_(g)
                g = t
            row.append(g)
            inp["grads"][k][s] = None
        mb.append(row)
    main = [torch.empty(P, dtype=torch.float32, device="cuda") for _ in range(wl.world)]
    upto = S_ - 1 if folded else S_
    for k in range(wl.world):
        zr.zr_grad_accumulate_first(main[k], mb[k][0])
        for s in range(1, upto):
            zr.zr_grad_accumulate(main[k], mb[k][s])
    before = [t.clone() for t in grp.flat_state()]
    if folded:
        grp.step_in_place_acc(grp.main_grad_views(main), grp.main_grad_views([row[-1] for row in mb]), wl.adam)
    else:
        grp.step_in_place(grp.main_grad_views(main), wl.adam)
    torch.cuda.synchronize()
    res = flatcheck.check_whole(lay, grp.scale, wl.adam, flatcheck.FlatGrads(mb), before, grp.flat_state(),
                                grp.param, main_after=main if folded else None)
    outs = ("master", "m", "v", "param") + (("main_grad",) if folded else ())
    _report(capsys, f"llama_1p1b micro-steps {'folded' if folded else 'unfolded'}", res, outs)


@pytest.mark.parametrize("name,max_norm", [("irregular_10k", 100.0), ("gpt2_124m", 0.05)])
def test_whole_clipped(zr, capsys, name, max_norm):
    """The step with the global gradient check, launched as the bench's clipped
    step: the averaged gradient at every element == the oracle's average; the
    check's outcome from the oracle over that gradient (bit for bit with
    integer gradients, within the check's stated bound otherwise); then every
    element of the clipped AdamW and cast == the oracle's clipped step with the
    device's coefficient."""
    wl = W.WORKLOADS[name]
    lay = oracle.layout(list(wl.numel), wl.world, wl.bucket)
    grp, inp = _group(wl, lay, allocate_buckets=False)
    arenas, rows, offs = _arenas(wl, lay, inp)
    plan = grp.direct_plan(grp.grad_table(rows))
    before = [t.clone() for t in grp.flat_state()]
    grp.step_direct_clipped(plan, wl.adam, max_norm)
    torch.cuda.synchronize()
    got = zr.zr_gradcheck_read(grp.check)
    ref = oracle.grad_check([t.cpu().numpy() for t in grp.grad_shards()], max_norm)
    assert not got["skip"] and got["nonfinite"] == 0 and got["coef"] < 1.0
    if wl.grad[0] == "int":
        assert got["sumsq"] == ref.sumsq and got["coef"] == ref.coef
    else:
        assert abs(got["sumsq"] - ref.sumsq) <= 1e-6 * ref.sumsq
        assert abs(got["coef"] - ref.coef) <= 2e-6 * ref.coef
    res = flatcheck.check_whole(lay, grp.scale, wl.adam, flatcheck.ArenaGrads(arenas, lay, offs), before,
                                grp.flat_state(), grp.param, grad_after=[grp._grad_flat], coef=got["coef"],
                                integer_avg=wl.grad[0] == "int")
    outs = ("grad", "master", "m", "v", "param") + (("integer_avg",) if wl.grad[0] == "int" else ())
    _report(capsys, f"{name} clipped (max_norm {max_norm})", res, outs)
