"""CUDA path (through the C ABI) against the CPU oracle, element by element.

The reduced sum and residual_out must be bit-exact, out within
2^-7 |ref| + 1e-3.  Covers the five workloads at their full sizes (small ones
compared in full, large ones on sampled rows), every rank count, every
launch shape, ragged and degenerate shapes, in-place residual, graph
capture, non-default streams, guard bands around outputs and the argument
errors that need a device.
"""
import ctypes

import numpy as np
import pytest
import torch

import allreduce_sum_residual_gb300 as arn
import synth
from gpu_helpers import (compare, device_inputs, is_two_stage, oracle_rows, run_gpu,
                         sample_rows, to_f32)

pytestmark = pytest.mark.gpu

MAX_WS = 16384 * 8192


@pytest.fixture(scope="module", autouse=True)
def workspace(arlib):
    torch.cuda.set_device(0)
    arn.ar_reserve_workspace(MAX_WS, 0)
    yield


def check_full(inp, mode, tag, **kw):
    n, (m, H) = len(inp.partials), inp.residual.shape
    gpu = run_gpu(inp, mode, **kw)
    torch.cuda.synchronize()
    orc = oracle_rows(inp, None, is_two_stage(n, m, H, mode))
    return compare(gpu, orc, tag)


def check_sampled(inp, mode, tag, k=48):
    n, (m, H) = len(inp.partials), inp.residual.shape
    out, rout, s = run_gpu(inp, mode)
    torch.cuda.synchronize()
    rows = sample_rows(m, k)
    idx = torch.as_tensor(rows, device=out.device)
    orc = oracle_rows(inp, rows, is_two_stage(n, m, H, mode))
    return compare((out[idx], rout[idx], s[idx]), orc, tag)


# ------------------------------------------------------------------ workloads

@pytest.mark.parametrize("mode", ["one_stage", "two_stage", "auto"])
def test_tiny(mode):
    w = synth.TINY
    check_full(device_inputs(w, w.ms[0]), mode, f"tiny/{mode}")


@pytest.mark.parametrize("m", synth.DECODE.ms)
@pytest.mark.parametrize("mode", ["one_stage", "auto"])
def test_decode(m, mode):
    check_full(device_inputs(synth.DECODE, m), mode, f"decode m={m}/{mode}")


@pytest.mark.parametrize("m", synth.TWO_STAGE.ms)
@pytest.mark.parametrize("mode", ["two_stage", "one_stage", "auto"])
def test_two_stage_workload(m, mode):
    check_full(device_inputs(synth.TWO_STAGE, m), mode, f"two_stage m={m}/{mode}")


@pytest.mark.parametrize("mode", ["one_stage", "two_stage", "auto"])
def test_prefill_full(mode):
    w = synth.PREFILL
    same = check_full(device_inputs(w, w.ms[0]), mode, f"prefill/{mode}")
    # fp32 + rsqrtf against the fp64 oracle: beyond the tolerance, almost
    # every output rounds to the very same bf16
    assert same >= 0.999, f"only {same:.5f} of out bit-identical to the oracle"


@pytest.mark.parametrize("m", [1, 16])
def test_decode_out_mostly_bit_identical(m):
    same = check_full(device_inputs(synth.DECODE, m), "auto", f"decode m={m}")
    assert same >= 0.999, f"only {same:.5f} of out bit-identical to the oracle"


@pytest.mark.parametrize("w", synth.SWEEP, ids=lambda w: w.name)
def test_sweep_auto(w):
    for m in w.ms:
        inp = device_inputs(w, m, seed=m)
        if m * w.H <= 1024 * 8192:
            check_full(inp, "auto", f"{w.name} m={m}")
        else:
            check_sampled(inp, "auto", f"{w.name} m={m}")
        del inp
        torch.cuda.empty_cache()


# ------------------------------------------------------------------ structure

@pytest.mark.parametrize("n", range(1, 17))
@pytest.mark.parametrize("mode", ["one_stage", "two_stage"])
def test_every_rank_count(n, mode):
    w = synth.Workload("ranks", n=n, H=1032, ms=(7,), p_std=0.5, res_std=1.0, seed=n)
    check_full(device_inputs(w, 7), mode, f"n={n}/{mode}")


def wide_range_inputs(n, m, H, seed):
    """Magnitudes spread over 2^-16 .. 2^16 so that the order of the fp32 adds
    changes the result in many elements."""
    rng = np.random.default_rng(seed)
    parts = []
    for _ in range(n):
        x = rng.standard_normal((m, H)).astype(np.float32) * np.exp2(
            rng.integers(-16, 17, (m, H))).astype(np.float32)
        parts.append(torch.from_numpy(x).to(torch.bfloat16).cuda())
    res = torch.from_numpy(rng.standard_normal((m, H)).astype(np.float32)).to(torch.bfloat16).cuda()
    wt = torch.from_numpy((1 + 0.1 * rng.standard_normal(H)).astype(np.float32)).to(torch.bfloat16).cuda()
    return synth.Inputs(parts, res, wt, 1e-6)


@pytest.mark.parametrize("n", [3, 8, 16])
@pytest.mark.parametrize("mode", ["one_stage", "two_stage"])
def test_order_sensitive_inputs(n, mode):
    inp = wide_range_inputs(n, 33, 2048, seed=n)
    # the data really is order sensitive: a reversed-order fp32 sum differs
    f = [synth.bits(p).astype(np.uint32) << 16 for p in inp.partials]
    fwd = f[0].view(np.float32).copy()
    for x in f[1:]:
        fwd = fwd + x.view(np.float32)
    rev = f[-1].view(np.float32).copy()
    for x in f[-2::-1]:
        rev = rev + x.view(np.float32)
    assert np.mean(fwd != rev) > 0.01
    check_full(inp, mode, f"order-sensitive n={n}/{mode}")


SHAPES = [(c, v) for c in (1, 2, 4, 8, 16) for v in (1, 2, 4, 8)]


@pytest.mark.parametrize("cluster,vpt", SHAPES)
def test_launch_shape_does_not_change_results(cluster, vpt):
    inp = wide_range_inputs(8, 5, 7168, seed=1)
    m, H = inp.residual.shape
    if -(-(H // 8) // cluster) > 1024:
        pytest.skip("a CTA holds at most 1024 packs")
    ref = run_gpu(inp, "one_stage")
    got = run_gpu(inp, "one_stage", cluster=cluster, vpt=vpt)
    torch.cuda.synchronize()
    assert torch.equal(ref[2].view(torch.int32), got[2].view(torch.int32))
    assert torch.equal(ref[1].view(torch.int16), got[1].view(torch.int16))
    check_full(inp, "one_stage", f"cluster={cluster} vpt={vpt}", cluster=cluster, vpt=vpt)


@pytest.mark.parametrize("n,m,H,vpt", [(1, 300, 2056, 1), (4, 257, 7168, 1), (5, 64, 6144, 2),
                                       (8, 100, 4104, 4), (3, 7, 1024, 8), (16, 130, 8192, 2),
                                       (6, 1000, 8, 1)])
@pytest.mark.parametrize("mode", ["one_stage", "two_stage"])
def test_late_weight_register_kernel(n, m, H, vpt, mode):
    """The register kernel that loads the weight after the sums: against the
    oracle, and bit for bit against the same shape with the weight loaded
    up front (only the load order differs)."""
    w = synth.Workload("late", n=n, H=H, ms=(m,), p_std=0.5, res_std=1.0)
    inp = device_inputs(w, m, seed=3)
    late = run_gpu(inp, mode, cluster=1, vpt=vpt, kernel="register_late")
    early = run_gpu(inp, mode, cluster=1, vpt=vpt, kernel="register")
    torch.cuda.synchronize()
    for a, b in zip(late, early):
        assert torch.equal(a.view(torch.int16 if a.dtype == torch.bfloat16 else torch.int32),
                           b.view(torch.int16 if b.dtype == torch.bfloat16 else torch.int32))
    orc = oracle_rows(inp, None, mode == "two_stage")
    compare(late, orc, f"late weight n={n} m={m} H={H} vpt={vpt} {mode}")


def test_late_weight_needs_one_cta_per_row():
    inp = device_inputs(synth.Workload("late2", n=2, H=1024, ms=(4,), p_std=0.5, res_std=1.0), 4)
    with pytest.raises(arn.ArError):
        run_gpu(inp, "one_stage", cluster=2, vpt=1, kernel="register_late")


@pytest.mark.parametrize("m,H", [(1, 8), (3, 24), (2, 1032), (5, 7176), (153, 4104), (1, 131072),
                                 (2, 65544), (300, 8)])
@pytest.mark.parametrize("mode", ["one_stage", "two_stage"])
def test_ragged_and_extreme_shapes(m, H, mode):
    w = synth.Workload("ragged", n=3, H=H, ms=(m,), p_std=0.5, res_std=1.0, seed=H)
    check_full(device_inputs(w, m), mode, f"m={m} H={H}/{mode}")


@pytest.mark.parametrize("mode", ["one_stage", "two_stage"])
def test_many_rows_of_a_very_wide_hidden_size(mode):
    """H = 65536 (beyond the stream kernel) at 600 rows: register kernel,
    8-CTA clusters of 2 packs per thread; compared on sampled rows."""
    w = synth.Workload("wide", n=5, H=65536, ms=(600,), p_std=0.5, res_std=1.0)
    inp = device_inputs(w, 600)
    p = arn.ar_get_plan(5, 600, 65536, mode)
    assert p["kernel"] == arn.AR_KERNEL_REGISTER and p["cluster"] == 8
    check_sampled(inp, mode, f"wide/{mode}", k=24)


@pytest.mark.parametrize("n,m,H", [(4, 1024, 16384), (8, 300, 12288), (2, 700, 16384),
                                   (16, 200, 12288), (3, 96, 12296)])
@pytest.mark.parametrize("mode", ["one_stage", "two_stage"])
def test_wide_rows_planned_from_the_table(n, m, H, mode):
    """Rows of 1025-2048 packs are planned from the table's widest columns:
    the register kernel over a 2-CTA cluster per row (prefetching one wave
    ahead when the rows need more than one wave), or the stream kernel."""
    w = synth.Workload("wide_table", n=n, H=H, ms=(m,), p_std=0.5, res_std=1.0, seed=m + n)
    inp = device_inputs(w, m)
    p = arn.ar_get_plan(n, m, H, mode)
    assert p["kernel"] == arn.AR_KERNEL_STREAM or p["cluster"] == 2, p
    check_sampled(inp, mode, f"wide table n={n} m={m} H={H}/{mode}", k=32)
    assert arn.ar_device_status(0) == arn.AR_OK


PREFETCH_CASES = [
    # (n, m, H, kernel, cluster, vpt): one CTA per row, late weight, cluster, wide rows, stream
    (8, 400, 4096, "register", 1, 1), (4, 700, 7168, "register_late", 1, 1),
    (8, 9, 7168, "register", 8, 1), (4, 500, 16384, "register", 2, 2),
    (8, 300, 6144, "stream", 0, 0), (1, 1000, 2056, "register", 1, 2)]


@pytest.mark.parametrize("n,m,H,kernel,cluster,vpt", PREFETCH_CASES)
@pytest.mark.parametrize("mode", ["one_stage", "two_stage"])
def test_prefetch_never_changes_results(n, m, H, kernel, cluster, vpt, mode):
    """The L2 prefetch is only a hint: with it off, on the own row, or also one
    wave (stream kernel: one row) ahead, every output bit is the same."""
    w = synth.Workload("prefetch", n=n, H=H, ms=(m,), p_std=0.5, res_std=1.0, seed=3 * m + n)
    inp = device_inputs(w, m)
    runs = [run_gpu(inp, mode, cluster=cluster, vpt=vpt, kernel=kernel, prefetch=pf)
            for pf in ("none", "row", "row_ahead")]
    torch.cuda.synchronize()
    for other in runs[1:]:
        for a, b in zip(runs[0], other):
            assert torch.equal(a.view(torch.int16) if a.dtype == torch.bfloat16 else
                               a.view(torch.int32),
                               b.view(torch.int16) if b.dtype == torch.bfloat16 else
                               b.view(torch.int32))
    rows = sample_rows(m, 16)
    idx = torch.as_tensor(rows, device="cuda")
    out, rout, s = runs[2]
    compare((out[idx], rout[idx], s[idx]), oracle_rows(inp, rows, mode == "two_stage"),
            f"prefetch {kernel} n={n} m={m} H={H}/{mode}")
    assert arn.ar_device_status(0) == arn.AR_OK


def guarded(m, H):
    """An [m, H] bf16 view inside a buffer with 4 KiB guard bands each side,
    every guard element holding the pattern 0x5A5A."""
    g = 2048
    buf = torch.full((m * H + 2 * g,), 0x5A5A, dtype=torch.int16, device="cuda")
    return buf, buf[g:g + m * H].view(torch.bfloat16).view(m, H), g


@pytest.mark.parametrize("mode", ["one_stage", "two_stage"])
@pytest.mark.parametrize("m,H", [(1, 8), (7, 1032), (19, 7168), (300, 4104)])
@pytest.mark.parametrize("kernel,cluster", [(0, 0), ("stream", 0), ("register_late", 1),
                                            ("register", 4)])
def test_outputs_stay_inside_their_buffers(mode, m, H, kernel, cluster):
    """Canaries around every output, for every kernel form (the plan's
    choice, the stream kernel, the late-weight kernel, a forced cluster)."""
    w = synth.Workload("guard", n=4, H=H, ms=(m,), p_std=0.5, res_std=1.0)
    inp = device_inputs(w, m)
    bo, out, g = guarded(m, H)
    br, rout, _ = guarded(m, H)
    bs = torch.full((m * H + 2 * 1024,), 7.0, dtype=torch.float32, device="cuda")
    s = bs[1024:1024 + m * H].view(m, H)
    arn.ar_rmsnorm_ex(inp.partials, inp.residual, inp.weight, inp.eps, out=out, residual_out=rout,
                      mode=mode, sum_out=s, kernel=kernel, cluster=cluster)
    torch.cuda.synchronize()
    for b in (bo, br):
        assert torch.all(b[:g] == 0x5A5A) and torch.all(b[g + m * H:] == 0x5A5A)
    assert torch.all(bs[:1024] == 7.0) and torch.all(bs[1024 + m * H:] == 7.0)
    orc = oracle_rows(inp, None, mode == "two_stage")
    compare((out, rout, s), orc, f"guarded {mode}")


def test_empty_batch_launches_nothing():
    w = synth.DECODE
    inp = device_inputs(w, 1)
    z = [torch.empty((0, w.H), dtype=torch.bfloat16, device="cuda") for _ in range(w.n)]
    res = torch.empty((0, w.H), dtype=torch.bfloat16, device="cuda")
    out, rout = arn.ar_rmsnorm(z, res, inp.weight, w.eps)
    assert out.shape == (0, w.H) and rout.shape == (0, w.H)


@pytest.mark.parametrize("mode", ["one_stage", "two_stage"])
def test_in_place_residual(mode):
    w = synth.DECODE
    inp = device_inputs(w, 16)
    orc = oracle_rows(inp, None, mode == "two_stage")
    res_copy = inp.residual.clone()
    out, rout = arn.ar_rmsnorm(inp.partials, inp.residual, inp.weight, w.eps,
                               residual_out=inp.residual, mode=mode)
    torch.cuda.synchronize()
    assert rout.data_ptr() == inp.residual.data_ptr()
    assert not torch.equal(res_copy, inp.residual)
    compare((out, rout, None), orc, f"in-place {mode}")


@pytest.mark.parametrize("mode", ["one_stage", "two_stage"])
@pytest.mark.parametrize("n,m,H,kernel,cluster,vpt,prefetch", [
    (4, 300, 4104, "register", 1, 1, "row_ahead"), (4, 1024, 7168, "register_late", 1, 1, "row_ahead"),
    (8, 700, 4096, "register", 1, 2, "row_ahead"), (8, 96, 12288, "register", 2, 1, "row"),
    (16, 600, 4096, "stream", 0, 0, "row"), (8, 19, 7168, "register", 8, 1, "row")])
def test_in_place_residual_every_kernel_form(mode, n, m, H, kernel, cluster, vpt, prefetch):
    """residual_out == residual for every kernel form, with the L2 prefetch of
    the own row and one wave ahead: a row's residual is read before its
    residual_out overwrites it, and no row is read after another row's CTA
    has written it."""
    w = synth.Workload("inplace_forms", n=n, H=H, ms=(m,), p_std=0.5, res_std=1.0, seed=n + m)
    inp = device_inputs(w, m)
    if arn.ar_workspace_elems(0) < m * H:
        arn.ar_reserve_workspace(m * H, 0)
    orc = oracle_rows(inp, None, mode == "two_stage")
    out, rout, _ = arn.ar_rmsnorm_ex(inp.partials, inp.residual, inp.weight, w.eps,
                                     residual_out=inp.residual, mode=mode, kernel=kernel,
                                     cluster=cluster, vpt=vpt, prefetch=prefetch)
    torch.cuda.synchronize()
    assert rout.data_ptr() == inp.residual.data_ptr()
    assert arn.ar_device_status(0) == arn.AR_OK
    compare((out, rout, None), orc, f"in-place {kernel} n={n} m={m} H={H} {mode}")


def test_n1_two_stage_equals_one_stage():
    w = synth.Workload("n1", n=1, H=4096, ms=(64,), p_std=0.5, res_std=1.0)
    inp = device_inputs(w, 64)
    a = run_gpu(inp, "one_stage")
    b = run_gpu(inp, "two_stage")
    torch.cuda.synchronize()
    for x, y in zip(a, b):
        assert torch.equal(x.view(torch.int16) if x.dtype == torch.bfloat16 else x.view(torch.int32),
                           y.view(torch.int16) if y.dtype == torch.bfloat16 else y.view(torch.int32))


@pytest.mark.parametrize("scale", [1e15, 1e-15])
def test_large_and_small_magnitudes_and_zero_rows(scale):
    """Magnitudes far from 1 (the fp32 square sum stays finite while
    H * max r^2 < 3.4e38, so 1e15 is in range) and an all-zero row."""
    w = synth.Workload("big", n=4, H=1024, ms=(4,), p_std=scale, res_std=scale)
    inp = device_inputs(w, 4)
    for p in inp.partials:
        p[2].zero_()
    inp.residual[2].zero_()
    check_full(inp, "one_stage", "large magnitudes")
    check_full(inp, "two_stage", "large magnitudes two-stage")


# ------------------------------------------------------------------ kernels

STREAM_CASES = [(8, 8192, 6144), (4, 2048, 7168), (8, 300, 8192), (1, 7, 1032), (3, 151, 7176),
                (16, 40, 4096), (2, 1000, 24), (5, 64, 16384), (8, 19, 32768), (12, 500, 2048)]


@pytest.mark.parametrize("n,m,H", STREAM_CASES)
@pytest.mark.parametrize("mode", ["one_stage", "two_stage"])
def test_stream_kernel_against_oracle_and_register_kernel(n, m, H, mode):
    w = synth.Workload("stream", n=n, H=H, ms=(m,), p_std=0.5, res_std=1.0, seed=m + H)
    inp = device_inputs(w, m)
    a = run_gpu(inp, mode, kernel="stream")
    b = run_gpu(inp, mode, kernel="register")
    torch.cuda.synchronize()
    assert torch.equal(a[2].view(torch.int32), b[2].view(torch.int32))
    assert torch.equal(a[1].view(torch.int16), b[1].view(torch.int16))
    rows = sample_rows(m, 64)
    idx = torch.as_tensor(rows, device="cuda")
    compare((a[0][idx], a[1][idx], a[2][idx]), oracle_rows(inp, rows, mode == "two_stage"),
            f"stream n={n} m={m} H={H}/{mode}")
    assert arn.ar_device_status(0) == arn.AR_OK


@pytest.mark.parametrize("n", range(1, 17))
def test_stream_kernel_every_rank_count(n):
    w = synth.Workload("stream_ranks", n=n, H=7168, ms=(33,), p_std=0.5, res_std=1.0, seed=n)
    check_full(device_inputs(w, 33), "one_stage", f"stream n={n}", kernel="stream")


def test_stream_kernel_order_sensitive():
    inp = wide_range_inputs(8, 320, 6144, seed=3)
    check_full(inp, "one_stage", "stream order-sensitive", kernel="stream")


def test_bounded_wait_gives_up_and_reports():
    assert arn.ar_device_status(0, reset=True) == arn.AR_OK
    assert arn.ar_selftest_bounded_wait(0, 2000) == arn.AR_ERR_TIMEOUT
    assert arn.ar_device_status(0) == arn.AR_OK      # the self-test clears it
    check_full(device_inputs(synth.TINY, 4), "one_stage", "after the self-test")


# ------------------------------------------------------------------ stages

def test_stage_entry_points():
    w = synth.TWO_STAGE
    inp = device_inputs(w, 64)
    m, H = inp.residual.shape
    temp = torch.empty((m, H), dtype=torch.bfloat16, device="cuda")
    arn.ar_reduce_scatter_flat(inp.partials, temp)
    out, rout = arn.ar_load_rmsnorm(temp, inp.residual, inp.weight, w.eps)
    torch.cuda.synchronize()
    o_out, o_rout, o_sum = oracle_rows(inp, None, two_stage=True)
    assert np.array_equal(to_f32(synth.bits(temp)), o_sum)       # stage 1 bit-exact
    compare((out, rout, None), (o_out, o_rout, o_sum), "stage 2")


@pytest.mark.parametrize("world", [1, 2, 3, 4, 8, 16])
def test_reduce_scatter_store_every_rank_fills_every_temp(world):
    """All `world` ranks of the reduce-scatter with gather-by-stores: each
    temp ends up holding the whole bf16 sum bit-exactly, and stage 2 on any
    of them gives the two-stage result."""
    w = synth.Workload("rs", n=4, H=1032, ms=(7,), p_std=0.5, res_std=1.0, seed=world)
    inp = device_inputs(w, 7)
    m, H = inp.residual.shape
    temps = [torch.full((m, H), 0x5A5A, dtype=torch.int16, device="cuda").view(torch.bfloat16)
             for _ in range(world)]
    for r in range(world):
        arn.ar_reduce_scatter_store(inp.partials, temps, r)
    torch.cuda.synchronize()
    o_out, o_rout, o_sum = oracle_rows(inp, None, two_stage=True)
    for t in temps:
        assert np.array_equal(to_f32(synth.bits(t)).view(np.uint32), o_sum.view(np.uint32))
    out, rout = arn.ar_load_rmsnorm(temps[-1], inp.residual, inp.weight, w.eps)
    torch.cuda.synchronize()
    compare((out, rout, None), (o_out, o_rout, o_sum), f"gathered temp, world={world}")


def test_reduce_scatter_store_writes_only_its_slice():
    w = synth.Workload("rs", n=3, H=4104, ms=(5,), p_std=0.5, res_std=1.0)
    inp = device_inputs(w, 5)
    m, H = inp.residual.shape
    world, rank = 4, 2
    temps = [torch.full((m, H), 0x5A5A, dtype=torch.int16, device="cuda").view(torch.bfloat16)
             for _ in range(world)]
    arn.ar_reduce_scatter_store(inp.partials, temps, rank)
    torch.cuda.synchronize()
    npacks = m * H // 8
    per = -(-npacks // world)
    lo, hi = rank * per * 8, min(npacks, (rank + 1) * per) * 8
    _, _, o_sum = oracle_rows(inp, None, two_stage=True)
    want = o_sum.ravel()[lo:hi].view(np.uint32)
    for t in temps:
        bits = synth.bits(t).ravel()
        assert np.all(bits[:lo] == 0x5A5A) and np.all(bits[hi:] == 0x5A5A)
        assert np.array_equal(to_f32(bits[lo:hi]).view(np.uint32), want)


# ------------------------------------------------------------------ runtime

def test_graph_capture_and_replay():
    w = synth.DECODE
    inp = device_inputs(w, 8)
    s = torch.cuda.Stream()
    out = torch.empty_like(inp.residual)
    rout = torch.empty_like(inp.residual)
    s.wait_stream(torch.cuda.current_stream())  # the inputs were made on the default stream
    with torch.cuda.stream(s):
        arn.ar_rmsnorm(inp.partials, inp.residual, inp.weight, w.eps, out=out, residual_out=rout,
                       mode="two_stage")
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        for mode in ("one_stage", "two_stage"):
            arn.ar_rmsnorm(inp.partials, inp.residual, inp.weight, w.eps, out=out,
                           residual_out=rout, mode=mode)
    out.zero_()
    rout.zero_()
    g.replay()
    torch.cuda.synchronize()
    compare((out, rout, None), oracle_rows(inp, None, True), "graph replay")


@pytest.mark.parametrize("mode", ["one_stage", "two_stage"])
def test_stream_kernel_in_a_graph_matches_eager(mode):
    """The persistent stream kernel (and two-stage) captured in a CUDA graph
    gives the same bits as the same call launched eagerly."""
    w = synth.Workload("graph", n=8, H=6144, ms=(1536,), p_std=0.5, res_std=1.0)
    inp = device_inputs(w, 1536)
    kernel = "stream" if mode == "one_stage" else "auto"

    def call(out=None, rout=None):
        return arn.ar_rmsnorm_ex(inp.partials, inp.residual, inp.weight, w.eps, out=out,
                                 residual_out=rout, mode=mode, kernel=kernel)[:2]

    ref_out, ref_rout = call()
    s = torch.cuda.Stream()
    out = torch.empty_like(inp.residual)
    rout = torch.empty_like(inp.residual)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        for _ in range(3):
            call(out, rout)
    out.zero_()
    rout.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), ref_out.view(torch.int16))
    assert torch.equal(rout.view(torch.int16), ref_rout.view(torch.int16))
    assert arn.ar_device_status(0) == arn.AR_OK


def test_non_default_stream():
    w = synth.DECODE
    inp = device_inputs(w, 4)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        out, rout, sm = run_gpu(inp, "one_stage")
    s.synchronize()
    compare((out, rout, sm), oracle_rows(inp, None, False), "side stream")


def test_workspace_errors():
    w = synth.TWO_STAGE
    inp = device_inputs(w, 32)
    arn.ar_release_workspace(0)
    assert arn.ar_workspace_elems(0) == 0
    with pytest.raises(arn.ArError) as e:
        arn.ar_rmsnorm(inp.partials, inp.residual, inp.weight, w.eps, mode="two_stage")
    assert e.value.status == arn.AR_ERR_WORKSPACE
    arn.ar_reserve_workspace(16 * w.H, 0)
    with pytest.raises(arn.ArError) as e:
        arn.ar_rmsnorm(inp.partials, inp.residual, inp.weight, w.eps, mode="two_stage")
    assert e.value.status == arn.AR_ERR_WORKSPACE
    arn.ar_reserve_workspace(MAX_WS, 0)
    assert arn.ar_workspace_elems(0) >= MAX_WS
    check_full(inp, "two_stage", "after re-reserve")


def test_plan_matches_device():
    p = arn.ar_get_plan(8, 1, 7168, 0)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert p == arn.ar_get_plan(8, 1, 7168, 0, sm_count=sms)


def test_device_plan_respects_wave_boundaries():
    """Between rows columns of the plan table the device plan uses each
    register kernel's occupancy on the device (how many rows one wave of
    CTAs holds): on random shapes it equals the host planner fed with the
    device's own occupancy figures, and differs from the plain
    interpolation somewhere.  On a grid point every plan agrees."""
    import random
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    arn.ar_get_plan(4, 256, 7168, 1)                      # the device is ready
    assert arn.ar_register_occupancy(4, 1, 0, 896) >= 1
    occ = arn.lib().ar_register_occupancy
    rng = random.Random(5)
    differ = 0
    for _ in range(400):
        n = rng.randint(1, 16)
        H = 8 * rng.randint(16, 1024)
        m = int(round(10 ** rng.uniform(1.81, 4.2)))
        dev = arn.ar_get_plan(n, m, H, 1)
        assert dev == arn.ar_get_plan_ex(n, m, H, 1, sms, occ), (n, m, H)
        plain = arn.ar_get_plan(n, m, H, 1, sm_count=sms)
        differ += {k: dev[k] for k in ("kernel", "vpt")} != {k: plain[k] for k in ("kernel", "vpt")}
    assert differ > 0
    assert arn.ar_get_plan(4, 256, 7168, 1)["kernel"] == arn.ar_get_plan(4, 256, 7168, 1,
                                                                          sm_count=sms)["kernel"]


def _plant_nonfinite(inp, rng):
    """Plant +inf, -inf and NaN in a few partial and residual elements
    (bf16 patterns), one kind per chosen row; returns the planted rows."""
    m, H = inp.residual.shape
    rows = rng.choice(m, size=min(m, 6), replace=False)
    pats = [0x7F80, 0xFF80, 0x7FC0]
    for i, r in enumerate(rows):
        col = int(rng.integers(H))
        t = inp.partials[i % len(inp.partials)] if i % 2 == 0 else inp.residual
        t.view(torch.int16)[r, col] = torch.tensor(pats[i % 3], dtype=torch.int32).to(torch.int16)
    return rows


def _compare_nonfinite(gpu, orc, tag):
    """NaN where the oracle has NaN (any payload), every other element as in
    compare(): sum and residual_out bit-exact, out within the tolerance."""
    g_out, g_rout, g_sum = gpu
    o_out, o_rout, o_sum = orc
    gs = g_sum.cpu().numpy()
    assert np.array_equal(np.isnan(gs), np.isnan(o_sum)), tag
    ok = ~np.isnan(o_sum)
    assert np.array_equal(gs[ok].view(np.uint32), o_sum[ok].view(np.uint32)), tag
    gr, orr = to_f32(synth.bits(g_rout)), to_f32(o_rout)
    assert np.array_equal(np.isnan(gr), np.isnan(orr)), tag
    ok = ~np.isnan(orr)
    assert np.array_equal(synth.bits(g_rout)[ok], o_rout[ok]), tag
    go, oo = to_f32(synth.bits(g_out)).astype(np.float64), to_f32(o_out).astype(np.float64)
    assert np.array_equal(np.isnan(go), np.isnan(oo)), tag
    ok = ~np.isnan(oo)
    assert np.all(np.abs(go[ok] - oo[ok]) <= 2.0 ** -7 * np.abs(oo[ok]) + 1e-3), tag


@pytest.mark.parametrize("m,kernel,mode", [(40, 0, "one_stage"), (300, 0, "one_stage"),
                                           (300, "stream", "one_stage"),
                                           (300, "register_late", "one_stage"),
                                           (300, 0, "two_stage")])
def test_inf_and_nan_propagate_as_in_the_oracle(m, kernel, mode):
    """Non-finite inputs are not special-cased: inf and NaN flow through the
    sum, residual_out and the norm (a row with an inf gets inv = 0, one with
    a NaN is NaN throughout), exactly as in the oracle."""
    w = synth.Workload("nonfinite", n=3, H=7168, ms=(m,), p_std=0.5, res_std=1.0)
    inp = device_inputs(w, m, seed=21)
    rows = _plant_nonfinite(inp, np.random.default_rng(5))
    cluster = 1 if kernel == "register_late" else 0
    gpu = run_gpu(inp, mode, cluster=cluster, kernel=kernel)
    torch.cuda.synchronize()
    orc = oracle_rows(inp, None, mode == "two_stage")
    assert np.isnan(to_f32(orc[0][rows])).any()   # the plant reached the outputs
    _compare_nonfinite(gpu, orc, f"non-finite m={m} {kernel} {mode}")


def test_raw_c_abi_call():
    """The plain C entry point with raw pointers (no binding helpers)."""
    w = synth.TINY
    inp = device_inputs(w, 4)
    out = torch.empty_like(inp.residual)
    rout = torch.empty_like(inp.residual)
    L = arn.lib()
    arr = (ctypes.c_void_p * w.n)(*[p.data_ptr() for p in inp.partials])
    st = L.ar_rmsnorm(arr, w.n, inp.residual.data_ptr(), inp.weight.data_ptr(), w.eps, 4, w.H,
                      out.data_ptr(), rout.data_ptr(), 1,
                      torch.cuda.current_stream().cuda_stream)
    assert st == 0
    torch.cuda.synchronize()
    compare((out, rout, None), oracle_rows(inp, None, False), "raw C ABI")


def _random_shapes(count, seed):
    """Seeded shapes across the planner's whole range: n 1..16, H any
    multiple of 8 up to 16384 (biased to model-like widths and to odd pack
    counts), m 1..16 or 64..2048 with m*H kept small enough for the oracle."""
    rng = np.random.default_rng(seed)
    shapes = []
    while len(shapes) < count:
        n = int(rng.integers(1, 17))
        H = int(rng.choice([int(rng.integers(1, 2049)) * 8,
                            int(rng.choice([2560, 2880, 3584, 4608, 5632, 10240, 14336]))]))
        m = int(rng.integers(1, 17)) if rng.random() < 0.3 else int(rng.integers(64, 2049))
        if m * H <= 4_000_000:
            shapes.append((n, m, H, str(rng.choice(["auto", "two_stage"]))))
    return shapes


@pytest.mark.parametrize("n,m,H,mode", _random_shapes(40, 2026))
def test_random_shapes_against_the_oracle(n, m, H, mode):
    """Whatever plan AUTO makes for a shape off every grid (kernel form,
    cluster, packs per thread, prefetch), the results match the oracle."""
    w = synth.Workload("random", n=n, H=H, ms=(m,), p_std=0.5, res_std=1.0, seed=n * 7919 + m + H)
    inp = device_inputs(w, m)
    if arn.ar_workspace_elems(0) < m * H:
        arn.ar_reserve_workspace(m * H, 0)
    out, rout, s = run_gpu(inp, mode)
    torch.cuda.synchronize()
    assert arn.ar_device_status(0) == arn.AR_OK
    compare((out, rout, s), oracle_rows(inp, None, is_two_stage(n, m, H, mode)),
            f"random n={n} m={m} H={H} {mode} plan={arn.ar_get_plan(n, m, H, mode)}")
