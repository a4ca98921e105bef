"""Shared pieces of the GPU parity tests: run the CUDA path through the C ABI
and the CPU oracle on the same seeded inputs, compare element by element.

Contract: the reduced sum and residual_out bit-exact; out within
|gpu - oracle| <= 2^-7 |oracle| + 1e-3 (one bf16 ulp is 2^-8 relative).
"""
import numpy as np
import torch

import allreduce_sum_residual_gb300 as arn
import oracle
import synth

OUT_REL = 2.0 ** -7
OUT_ABS = 1e-3


def host_threads():
    return oracle.host_threads()


def to_f32(bits):
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def device_inputs(w, m, seed=None, big=None):
    """Workload inputs on cuda:0; numpy generator for small, torch for big."""
    if big is None:
        big = m * w.H * w.n > 64 * 1024 * 1024
    if big:
        return synth.make_inputs(w, m, backend="torch", device="cuda", seed=seed)
    inp = synth.make_inputs(w, m, backend="numpy", seed=seed)
    return synth.Inputs([p.cuda() for p in inp.partials], inp.residual.cuda(), inp.weight.cuda(),
                        inp.eps)


def run_gpu(inp, mode, cluster=0, vpt=0, with_sum=True, stream=None, kernel=0, prefetch=0):
    m, H = inp.residual.shape
    s = torch.empty((m, H), dtype=torch.float32, device=inp.residual.device) if with_sum else None
    out, rout, s = arn.ar_rmsnorm_ex(inp.partials, inp.residual, inp.weight, inp.eps, mode=mode,
                                     sum_out=s, cluster=cluster, vpt=vpt, stream=stream,
                                     kernel=kernel, prefetch=prefetch)
    return out, rout, s


def is_two_stage(n, m, H, mode):
    if mode in ("two_stage", 2):
        return True
    if mode in ("one_stage", 1):
        return False
    return arn.ar_get_plan(n, m, H, 0)["mode"] == 2


def oracle_rows(inp, rows, two_stage):
    """Oracle results for the given rows (None = all), from the inputs' bits."""
    sel = slice(None) if rows is None else torch.as_tensor(rows, device=inp.residual.device)
    parts = [synth.bits(p[sel]) for p in inp.partials]
    res = synth.bits(inp.residual[sel])
    w = synth.bits(inp.weight)
    return oracle.ar_rmsnorm(parts, res, w, inp.eps, two_stage=two_stage,
                             threads=host_threads())


def compare(gpu, orc, tag=""):
    """gpu = (out, rout, sum) tensors restricted to the compared rows."""
    g_out, g_rout, g_sum = gpu
    o_out, o_rout, o_sum = orc
    if g_sum is not None:
        gs = g_sum.cpu().numpy()
        bad = np.nonzero(gs.view(np.uint32) != o_sum.view(np.uint32))
        assert bad[0].size == 0, (f"{tag}: reduced sum not bit-exact at {bad[0].size} elements, "
                                  f"first {tuple(b[0] for b in bad)}: gpu {gs[bad][0]!r} "
                                  f"oracle {o_sum[bad][0]!r}")
    gr = synth.bits(g_rout)
    bad = np.nonzero(gr != o_rout)
    assert bad[0].size == 0, (f"{tag}: residual_out not bit-exact at {bad[0].size} elements, "
                              f"first {tuple(b[0] for b in bad)}")
    go = to_f32(synth.bits(g_out)).astype(np.float64)
    oo = to_f32(o_out).astype(np.float64)
    err = np.abs(go - oo)
    tol = OUT_REL * np.abs(oo) + OUT_ABS
    assert np.all(err <= tol), (f"{tag}: out outside tolerance at {int(np.sum(err > tol))} elements,"
                                f" worst excess {float(np.max(err - tol))}")
    return float(np.mean(synth.bits(g_out) == o_out))


def sample_rows(m, k=48, seed=0):
    """First, last and k random rows (sorted, unique)."""
    if m <= k + 2:
        return list(range(m))
    rng = np.random.default_rng(seed)
    rows = set(rng.choice(m, size=k, replace=False).tolist()) | {0, m - 1}
    return sorted(rows)
