"""ar_rmsnorm_mapped: the kernels read and write pinned host buffers over
the host link.  Against the CPU oracle (sum path: residual_out bit-exact,
out within 2^-7 |ref| + 1e-3) and against the device-memory path with the
same register-kernel launch shape (bit-identical outputs), for host-only and
mixed host/device buffers, one- and two-stage, the decode cluster path, and
the pointer checks that refuse memory the device cannot reach."""
import ctypes

import pytest
import torch

import allreduce_sum_residual_gb300 as arn
import synth
from gpu_helpers import compare, device_inputs, oracle_rows

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def workspace(arlib):
    torch.cuda.set_device(0)
    arn.ar_reserve_workspace(2048 * 8192, 0)
    yield


def pinned(t):
    return t.cpu().pin_memory()


def _host_inputs(inp, which):
    parts = [pinned(p) if "partials" in which else p for p in inp.partials]
    res = pinned(inp.residual) if "residual" in which else inp.residual
    w = pinned(inp.weight) if "weight" in which else inp.weight
    return parts, res, w


@pytest.mark.parametrize("n,m,H,mode", [(2, 4, 1024, "one_stage"), (8, 16, 7168, "auto"),
                                        (3, 300, 4096, "auto"), (4, 257, 2056, "two_stage"),
                                        (8, 1024, 6144, "auto"), (4, 1024, 7168, "auto")])
def test_host_buffers_match_oracle_and_device_path(n, m, H, mode):
    w = synth.Workload("mapped", n=n, H=H, ms=(m,), p_std=0.5, res_std=1.0)
    inp = device_inputs(w, m, seed=11)
    parts, res, wt = _host_inputs(inp, ("partials", "residual", "weight"))
    out, rout = arn.ar_rmsnorm_mapped(parts, res, wt, inp.eps, mode=mode)
    assert not out.is_cuda and out.is_pinned() and not rout.is_cuda
    torch.cuda.synchronize()
    two = mode == "two_stage"
    orc = oracle_rows(inp, None, two)
    compare((out, rout, None), orc, f"mapped n={n} m={m} H={H} {mode}")
    # the same register-kernel shape on device memory gives the same bits
    plan = arn.ar_get_plan(n, m, H, {"one_stage": 1, "two_stage": 2, "auto": 0}[mode])
    if plan["kernel"] in (arn.AR_KERNEL_REGISTER, arn.AR_KERNEL_REGISTER_LATE_W):
        d_out, d_rout, _ = arn.ar_rmsnorm_ex(inp.partials, inp.residual, inp.weight, inp.eps,
                                             mode=mode, cluster=plan["cluster"], vpt=plan["vpt"],
                                             kernel="register")
        torch.cuda.synchronize()
        assert torch.equal(d_rout.cpu(), rout)
        assert torch.equal(d_out.cpu(), out)


@pytest.mark.parametrize("which", [("partials",), ("residual", "weight"), ("partials", "residual")])
def test_mixed_host_and_device_buffers(which):
    n, m, H = 4, 96, 4096
    w = synth.Workload("mixed", n=n, H=H, ms=(m,), p_std=0.5, res_std=1.0)
    inp = device_inputs(w, m, seed=5)
    parts, res, wt = _host_inputs(inp, which)
    out = torch.empty((m, H), dtype=torch.bfloat16).pin_memory()
    rout = torch.empty((m, H), dtype=torch.bfloat16, device="cuda")
    arn.ar_rmsnorm_mapped(parts, res, wt, inp.eps, out=out, residual_out=rout, device="cuda:0")
    torch.cuda.synchronize()
    compare((out, rout, None), oracle_rows(inp, None, False), f"mixed {which}")


def test_in_place_residual_on_the_host():
    n, m, H = 2, 40, 2048
    w = synth.Workload("inplace", n=n, H=H, ms=(m,), p_std=0.5, res_std=1.0)
    inp = device_inputs(w, m, seed=9)
    orc = oracle_rows(inp, None, False)
    parts, res, wt = _host_inputs(inp, ("partials", "residual", "weight"))
    out, rout = arn.ar_rmsnorm_mapped(parts, res, wt, inp.eps, residual_out=res)
    torch.cuda.synchronize()
    assert rout.data_ptr() == res.data_ptr()
    compare((out, rout, None), orc, "in place on the host")


def test_pageable_host_memory_is_refused_before_any_launch():
    n, m, H = 2, 8, 1024
    w = synth.Workload("pageable", n=n, H=H, ms=(m,), p_std=0.5, res_std=1.0)
    inp = device_inputs(w, m, seed=1)
    pageable = inp.partials[0].cpu()           # not pinned
    assert not pageable.is_pinned()
    with pytest.raises(ValueError):
        arn.ar_rmsnorm_mapped([pageable, inp.partials[1]], inp.residual, inp.weight, inp.eps)
    # the C ABI's own check: AR_ERR_ARG, nothing launched
    out = torch.full((m, H), 7.0, dtype=torch.bfloat16, device="cuda")
    rout = torch.full((m, H), 7.0, dtype=torch.bfloat16, device="cuda")
    arr = (ctypes.c_void_p * 2)(pageable.data_ptr(), inp.partials[1].data_ptr())
    st = arn.lib().ar_rmsnorm_mapped(arr, 2, ctypes.c_void_p(inp.residual.data_ptr()),
                                     ctypes.c_void_p(inp.weight.data_ptr()), ctypes.c_float(inp.eps),
                                     m, H, ctypes.c_void_p(out.data_ptr()),
                                     ctypes.c_void_p(rout.data_ptr()), 1,
                                     ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    torch.cuda.synchronize()
    assert st == arn.AR_ERR_ARG
    assert bool((out == 7.0).all()) and bool((rout == 7.0).all())


def test_empty_batch_with_host_buffers():
    H = 1024
    e = torch.empty((0, H), dtype=torch.bfloat16).pin_memory()
    wt = torch.ones(H, dtype=torch.bfloat16).pin_memory()
    out, rout = arn.ar_rmsnorm_mapped([e, e], e, wt, 1e-6)
    torch.cuda.synchronize()
    assert out.shape == (0, H) and rout.shape == (0, H)


def _random_mapped_shapes(count, seed):
    import numpy as np
    rng = np.random.default_rng(seed)
    out = []
    while len(out) < count:
        n = int(rng.integers(1, 17))
        H = int(rng.choice([int(rng.integers(1, 1025)) * 8, 2560, 4096, 7168, 12288]))
        m = int(rng.integers(1, 17)) if rng.random() < 0.3 else int(rng.integers(64, 1025))
        if m * H <= 2_000_000:
            out.append((n, m, H, str(rng.choice(["auto", "two_stage"]))))
    return out


@pytest.mark.parametrize("n,m,H,mode", _random_mapped_shapes(12, 7))
def test_random_shapes_from_host_buffers(n, m, H, mode):
    """The plain-load plans (the best register-kernel form of the table, no
    bulk prefetch) on seeded shapes off every grid, all buffers in pinned
    host memory: the oracle's results."""
    w = synth.Workload("mapped_random", n=n, H=H, ms=(m,), p_std=0.5, res_std=1.0, seed=m + H + n)
    inp = device_inputs(w, m, seed=3)
    if arn.ar_workspace_elems(0) < m * H:
        arn.ar_reserve_workspace(m * H, 0)
    parts, res, wt = _host_inputs(inp, ("partials", "residual", "weight"))
    out, rout = arn.ar_rmsnorm_mapped(parts, res, wt, inp.eps, mode=mode)
    torch.cuda.synchronize()
    assert arn.ar_device_status(0) == arn.AR_OK
    compare((out, rout, None), oracle_rows(inp, None, mode == "two_stage"),
            f"mapped random n={n} m={m} H={H} {mode}")
