"""ar_rmsnorm_two_stage_static: the two-stage epilogue for callers that cannot
allocate device memory (a plug-in whose host program owns all device memory,
a process whose memory a framework's pool already holds, a path that cannot
take cudaMalloc's implicit synchronisation).  Its temporary is a fixed array
inside the library instead of a reserved workspace.

Called through the raw C ABI on two calls in a row with different inputs,
and checked three ways: against the CPU oracle's two-stage result (sum
path: residual_out bit-exact; out within 2^-7 |ref| + 1e-3), bit for bit
against the existing two-stage entry point (ar_rmsnorm with a reserved
workspace: the same kernels and launch plan), and for what it must not do
(write outside its outputs, allocate device memory).  One case fills the
array exactly (m * H = AR_STATIC_SCRATCH_ELEMS).  This file is named to be
collected last.
"""
import ctypes

import numpy as np
import pytest
import torch

import allreduce_sum_residual_gb300 as arn
import synth
from gpu_helpers import compare, oracle_rows, sample_rows

pytestmark = pytest.mark.gpu

GUARD = 2048          # bf16 canaries on each side of an output
CANARY = 0x5A5A


def _inputs(w, m, seed):
    inp = synth.make_inputs(w, m, seed=seed, backend="torch" if m * w.H * w.n > (1 << 24) else
                            "numpy", device="cuda" if m * w.H * w.n > (1 << 24) else "cpu")
    return synth.Inputs([p.cuda() for p in inp.partials], inp.residual.cuda(), inp.weight.cuda(),
                        inp.eps)


def _guarded(m, H):
    buf = torch.full((m * H + 2 * GUARD,), CANARY, dtype=torch.int16, device="cuda")
    return buf, buf[GUARD:GUARD + m * H].view(torch.bfloat16).view(m, H)


def _guards_intact(buf, m, H):
    return bool(torch.all(buf[:GUARD] == CANARY)) and bool(torch.all(buf[GUARD + m * H:] == CANARY))


def _static_call(inp, out, rout):
    L = arn.lib()
    m, H = inp.residual.shape
    arr = (ctypes.c_void_p * len(inp.partials))(*[p.data_ptr() for p in inp.partials])
    return L.ar_rmsnorm_two_stage_static(arr, len(inp.partials), inp.residual.data_ptr(),
                                         inp.weight.data_ptr(), inp.eps, m, H, out.data_ptr(),
                                         rout.data_ptr(), torch.cuda.current_stream().cuda_stream)


CASES = [(synth.TWO_STAGE, 256), (synth.DECODE, 16), (synth.PREFILL, 1024),
         # m * H exactly AR_STATIC_SCRATCH_ELEMS: the whole array is used
         (synth.Workload("limit", n=8, H=8192, ms=(1024,), p_std=0.5, res_std=1.0), 1024)]


@pytest.mark.parametrize("w,m", CASES, ids=lambda x: getattr(x, "name", x))
def test_static_scratch_matches_oracle_and_workspace_path_twice(arlib, w, m):
    torch.cuda.set_device(0)
    H = w.H
    assert m * H <= arn.AR_STATIC_SCRATCH_ELEMS
    arn.ar_reserve_workspace(m * H, 0)            # only the comparison path allocates
    bo, out = _guarded(m, H)
    br, rout = _guarded(m, H)
    for seed in (11, 12):                         # two calls in a row, different inputs
        inp = _inputs(w, m, seed)
        assert _static_call(inp, out, rout) == arn.AR_OK
        ref_out, ref_rout = arn.ar_rmsnorm(inp.partials, inp.residual, inp.weight, inp.eps,
                                           mode="two_stage")
        torch.cuda.synchronize()
        assert _guards_intact(bo, m, H) and _guards_intact(br, m, H)
        # same kernels, same plan: bit for bit the workspace path's results
        assert torch.equal(rout.view(torch.int16), ref_rout.view(torch.int16))
        assert torch.equal(out.view(torch.int16), ref_out.view(torch.int16))
        # and the oracle's two-stage result (sampled rows at the larger sizes)
        rows = None if m <= 256 else sample_rows(m, 40, seed)
        sel = slice(None) if rows is None else torch.as_tensor(rows, device="cuda")
        compare((out[sel], rout[sel], None), oracle_rows(inp, rows, True),
                f"static {w.name} m={m} seed={seed}")
    assert arn.ar_device_status(0) == arn.AR_OK


def test_static_scratch_allocates_no_device_memory(arlib):
    """After a first call (which looks up the array's address), further calls
    leave the device's free memory unchanged: nothing is allocated."""
    torch.cuda.set_device(0)
    w = synth.Workload("noalloc", n=4, H=7168, ms=(512,), p_std=0.5, res_std=1.0)
    m = 512
    inp = _inputs(w, m, 5)
    out = torch.empty_like(inp.residual)
    rout = torch.empty_like(inp.residual)
    assert _static_call(inp, out, rout) == arn.AR_OK
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info(0)
    for _ in range(3):
        assert _static_call(inp, out, rout) == arn.AR_OK
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info(0)
    assert free1 == free0, (free0, free1)
    compare((out, rout, None), oracle_rows(inp, None, True), "static no-alloc")


def test_static_scratch_rejects_sizes_beyond_its_limit(arlib):
    torch.cuda.set_device(0)
    H = 8192
    m = arn.AR_STATIC_SCRATCH_ELEMS // H + 1
    L = arn.lib()
    fake = (ctypes.c_void_p * 2)(0, 0)
    # refused on the size alone, before any pointer is looked at or anything launched
    assert L.ar_rmsnorm_two_stage_static(fake, 2, None, None, 1e-6, m, H, None, None,
                                         None) == arn.AR_ERR_SCRATCH_LIMIT
    assert "scratch" in arn.ar_strerror(arn.AR_ERR_SCRATCH_LIMIT)
    # one row less fits exactly; nothing is read for m == 0
    assert L.ar_rmsnorm_two_stage_static(fake, 2, None, None, 1e-6, 0, H, None, None,
                                         None) == arn.AR_OK
    assert np.int64(arn.AR_STATIC_SCRATCH_ELEMS // H) * H <= arn.AR_STATIC_SCRATCH_ELEMS
