"""ar_rmsnorm_two_stage_static: the two-stage epilogue for callers that cannot
allocate device memory (a plug-in whose host program owns all device memory,
a process whose memory a framework's pool already holds, a path that cannot
take cudaMalloc's implicit synchronisation).  Its temporary is a fixed array
inside the library instead of a reserved workspace.

Called through the raw C ABI and compared, on two calls in a row with
different inputs, with the existing two-stage entry point (ar_rmsnorm with a
reserved workspace): residual_out bit-exact and out within the tolerance the
other parity tests use.  This file is named to be collected last.
"""
import ctypes

import numpy as np
import pytest
import torch

import allreduce_sum_residual_gb300 as arn
import synth
from gpu_helpers import OUT_ABS, OUT_REL, to_f32

pytestmark = pytest.mark.gpu


def _inputs(w, m, seed):
    inp = synth.make_inputs(w, m, seed=seed)
    return synth.Inputs([p.cuda() for p in inp.partials], inp.residual.cuda(), inp.weight.cuda(),
                        inp.eps)


def _static_call(inp, out, rout):
    L = arn.lib()
    m, H = inp.residual.shape
    arr = (ctypes.c_void_p * len(inp.partials))(*[p.data_ptr() for p in inp.partials])
    return L.ar_rmsnorm_two_stage_static(arr, len(inp.partials), inp.residual.data_ptr(),
                                         inp.weight.data_ptr(), inp.eps, m, H, out.data_ptr(),
                                         rout.data_ptr(), torch.cuda.current_stream().cuda_stream)


@pytest.mark.parametrize("w,m", [(synth.TWO_STAGE, 256), (synth.DECODE, 16), (synth.PREFILL, 1024)])
def test_static_scratch_matches_workspace_path_twice(arlib, w, m):
    torch.cuda.set_device(0)
    arn.ar_reserve_workspace(m * w.H, 0)          # only the reference path allocates
    for seed in (11, 12):                         # two calls in a row, different inputs
        inp = _inputs(w, m, seed)
        out = torch.empty_like(inp.residual)
        rout = torch.empty_like(inp.residual)
        assert _static_call(inp, out, rout) == arn.AR_OK
        ref_out, ref_rout = arn.ar_rmsnorm(inp.partials, inp.residual, inp.weight, inp.eps,
                                           mode="two_stage")
        torch.cuda.synchronize()
        assert torch.equal(rout.view(torch.int16), ref_rout.view(torch.int16))
        a = to_f32(synth.bits(out)).astype(np.float64)
        b = to_f32(synth.bits(ref_out)).astype(np.float64)
        assert np.all(np.abs(a - b) <= OUT_REL * np.abs(b) + OUT_ABS)


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
