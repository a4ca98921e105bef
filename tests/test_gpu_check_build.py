"""The checking build (libarnorm_check.so, compiled with AR_CHECK=1).

Every kernel of that build tests the indices it derives from its launch
shape -- the row, the pack range of a CTA and that its threads cover it, the
cluster rank, the shared-memory ring against the launch's size, the rank
counts of stage 1 and of the signal pads -- and a failed test records
AR_ERR_BOUNDS in the device status word and skips the access.  compute-
sanitizer is closed on this machine; this build, the canaries around outputs
and tiny shapes stand in for it.

Here every kernel form runs on tiny and ragged shapes in both modes through
the checking build: no check fires (the status word stays AR_OK) and the
results are bit-identical to the normal build's.  A kernel whose only work
is one failing check shows that the checks are live in the checking build
and compiled away in the normal one.
"""
import ctypes

import pytest
import torch

import allreduce_sum_residual_gb300 as arn
import synth
from gpu_helpers import compare, device_inputs, oracle_rows

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def checklib():
    from allreduce_sum_residual_gb300 import _build
    L = arn.load(_build.build(check=True))
    assert L.ar_checks_bounds() == 1
    torch.cuda.set_device(0)
    assert L.ar_reserve_workspace(1 << 22, 0) == arn.AR_OK
    assert L.ar_device_status(0, 1) == arn.AR_OK
    return L


def _run(L, inp, mode, plan):
    m, H = inp.residual.shape
    out = torch.empty_like(inp.residual)
    rout = torch.empty_like(inp.residual)
    s = torch.empty((m, H), dtype=torch.float32, device="cuda")
    arr = (ctypes.c_void_p * len(inp.partials))(*[p.data_ptr() for p in inp.partials])
    p = ctypes.pointer(arn.ar_plan_t(0, *plan, 0, 0, 0, 0, 0)) if plan else None
    st = L.ar_rmsnorm_ex(arr, len(inp.partials), inp.residual.data_ptr(), inp.weight.data_ptr(),
                         inp.eps, m, H, out.data_ptr(), rout.data_ptr(), mode,
                         torch.cuda.current_stream().cuda_stream, s.data_ptr(), p)
    assert st == arn.AR_OK, (st, plan)
    return out, rout, s


SHAPES = [(1, 1, 8), (3, 3, 24), (2, 7, 1032), (8, 19, 7168), (4, 300, 4104), (3, 2, 16384),
          (16, 5, 2048), (1, 64, 4096)]
PLANS = [None, (arn.AR_KERNEL_REGISTER, 1, 1), (arn.AR_KERNEL_REGISTER, 4, 2),
         (arn.AR_KERNEL_REGISTER, 16, 1), (arn.AR_KERNEL_REGISTER_LATE_W, 1, 4),
         (arn.AR_KERNEL_STREAM, 0, 0)]


@pytest.mark.parametrize("n,m,H", SHAPES)
@pytest.mark.parametrize("mode", [arn.AR_MODE_ONE_STAGE, arn.AR_MODE_TWO_STAGE])
def test_no_check_fires_and_results_match_the_normal_build(checklib, n, m, H, mode):
    w = synth.Workload("check", n=n, H=H, ms=(m,), p_std=0.5, res_std=1.0, seed=n * m + H)
    inp = device_inputs(w, m)
    if arn.ar_workspace_elems(0) < m * H:
        arn.ar_reserve_workspace(m * H, 0)
    ran = 0
    for plan in PLANS:
        if plan and plan[0] == arn.AR_KERNEL_REGISTER and -(-(H // 8) // plan[1]) > 1024:
            continue                                   # a row slice must fit one CTA
        if plan and plan[0] == arn.AR_KERNEL_REGISTER and plan[1] > 1 and plan[1] > H // 8:
            continue
        if plan and plan[0] == arn.AR_KERNEL_REGISTER_LATE_W and H // 8 > 1024:
            continue                                   # one CTA per row only
        got = _run(checklib, inp, mode, plan)
        ref = _run(arn.lib(), inp, mode, plan)
        torch.cuda.synchronize()
        assert checklib.ar_device_status(0, 1) == arn.AR_OK, plan
        for a, b in zip(got, ref):
            assert torch.equal(a.view(torch.int16) if a.dtype == torch.bfloat16 else
                               a.view(torch.int32),
                               b.view(torch.int16) if b.dtype == torch.bfloat16 else
                               b.view(torch.int32)), plan
        ran += 1
    assert ran >= 3
    compare(got, oracle_rows(inp, None, mode == arn.AR_MODE_TWO_STAGE), f"checking build n={n}")


def test_stage_and_cross_rank_kernels_pass_their_checks(checklib):
    torch.cuda.set_device(0)
    m = ctypes.c_int(-1)
    assert checklib.ar_selftest_barrier(0, 4, 200, 1_000_000, ctypes.byref(m)) == arn.AR_OK
    assert m.value == 0
    w = synth.Workload("check_rs", n=4, H=1032, ms=(7,), p_std=0.5, res_std=1.0)
    inp = device_inputs(w, 7)
    temps = [torch.zeros((7, 1032), dtype=torch.bfloat16, device="cuda") for _ in range(4)]
    arr = (ctypes.c_void_p * 4)(*[p.data_ptr() for p in inp.partials])
    tarr = (ctypes.c_void_p * 4)(*[t.data_ptr() for t in temps])
    for r in range(4):
        assert checklib.ar_reduce_scatter_store(arr, 4, 7 * 1032, r, 4, tarr, None) == arn.AR_OK
    torch.cuda.synchronize()
    assert checklib.ar_device_status(0, 1) == arn.AR_OK
    for t in temps[1:]:
        assert torch.equal(t.view(torch.int16), temps[0].view(torch.int16))


def test_one_and_two_shot_calls_pass_their_checks(checklib):
    """Both cross-rank entry points of the checking build, rank 0 of 4 with
    the other ranks' posts (and stage-1 slices) run first: no check fires
    and the results are the oracle's."""
    torch.cuda.set_device(0)
    world, m, H = 4, 9, 2056
    w = synth.Workload("check_shots", n=world, H=H, ms=(m,), p_std=0.5, res_std=1.0)
    inp = device_inputs(w, m)
    arr = (ctypes.c_void_p * world)(*[p.data_ptr() for p in inp.partials])
    pads = [torch.zeros(arn.AR_SIGNAL_PAD_BYTES // 4, dtype=torch.int32, device="cuda")
            for _ in range(world)]
    parr = (ctypes.c_void_p * world)(*[p.data_ptr() for p in pads])
    temps = [torch.zeros((m, H), dtype=torch.bfloat16, device="cuda") for _ in range(world)]
    tarr = (ctypes.c_void_p * world)(*[t.data_ptr() for t in temps])
    out = torch.empty_like(inp.residual)
    rout = torch.empty_like(inp.residual)
    args = (inp.residual.data_ptr(), inp.weight.data_ptr(), inp.eps, m, H, out.data_ptr(),
            rout.data_ptr(), 0, world)
    for r in range(1, world):
        assert checklib.ar_signal_post(parr, world, r, 1, None) == arn.AR_OK
        assert checklib.ar_signal_post(parr, world, r, 2, None) == arn.AR_OK
    assert checklib.ar_rmsnorm_one_shot(arr, world, *args, parr, 1, 1_000_000, 1,
                                        None) == arn.AR_OK
    torch.cuda.synchronize()
    assert checklib.ar_device_status(0, 1) == arn.AR_OK
    compare((out, rout, None), oracle_rows(inp, None, False), "checking build, one-shot")
    for r in range(1, world):
        assert checklib.ar_signal_post(parr, world, r, 3, None) == arn.AR_OK
        assert checklib.ar_reduce_scatter_store(arr, world, m * H, r, world, tarr, None) == arn.AR_OK
        assert checklib.ar_signal_post(parr, world, r, 4, None) == arn.AR_OK
    assert checklib.ar_rmsnorm_two_shot(arr, world, *args, tarr, parr, 3, 1_000_000,
                                        None) == arn.AR_OK
    torch.cuda.synchronize()
    assert checklib.ar_device_status(0, 1) == arn.AR_OK
    compare((out, rout, None), oracle_rows(inp, None, True), "checking build, two-shot")


def test_checks_are_live_only_in_the_checking_build(checklib):
    assert checklib.ar_selftest_bounds(0) == arn.AR_ERR_BOUNDS
    assert checklib.ar_device_status(0, 0) == arn.AR_OK       # the self-test cleared it
    assert arn.lib().ar_checks_bounds() == 0
    assert arn.lib().ar_selftest_bounds(0) == arn.AR_OK
