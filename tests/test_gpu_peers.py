"""The cross-rank data plane on one GPU.

* The bounded flag barrier: a wait on a flag that nothing sets gives up with
  AR_ERR_TIMEOUT and leaves the context usable; flags posted by earlier
  kernels on the stream let it pass; epochs compare modulo 2^32.
* All ranks of a barrier inside one cooperative kernel (they run at the same
  time), checking that data written before a post is seen after the wait.
* The two-shot path (barrier, stage 1 stored into every rank's temporary,
  barrier, stage 2) with the other ranks' parts run earlier on the stream,
  so that no kernel waits on a later one: against the oracle's two-stage
  result.
* The one-shot call (barrier, epilogue over every rank's partial, barrier)
  with the other ranks' posts run earlier: against the oracle's one-stage
  result; a rank that never reaches the end barrier; graph replay.
* Two processes on this GPU sharing their buffers through CUDA IPC handles
  exchanged over a gloo group: the one-shot path (every rank reads both
  partials through the mappings) and the two-shot path (stores into both
  ranks' temporaries, synchronised on the host, then stage 2), each rank
  against the oracle; and the collective decline when one rank's IPC setup
  fails.  Kernels of the two processes never wait on one another.
"""
import multiprocessing as mp
import os
import socket
import sys

import pytest
import torch

import allreduce_sum_residual_gb300 as arn
import synth
from gpu_helpers import compare, device_inputs, oracle_rows

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _pads(world):
    return [torch.zeros(arn.AR_SIGNAL_PAD_BYTES // 4, dtype=torch.int32, device="cuda")
            for _ in range(world)]


def _flags(pad, world):
    return [int(x) & 0xFFFFFFFF for x in pad[:world].tolist()]


def test_wait_on_a_flag_nobody_sets_times_out():
    torch.cuda.set_device(0)
    arn.ar_device_status(0, reset=True)
    pads = _pads(2)
    arn.ar_barrier(pads, 0, 1, limit_us=2000)          # rank 1 never arrives
    assert arn.ar_device_status(0, reset=True) == arn.AR_ERR_TIMEOUT
    assert _flags(pads[0], 2) == [1, 0] and _flags(pads[1], 2) == [1, 0]   # rank 0 did post
    arn.ar_signal_wait(pads[1], 2, 1, limit_us=2000)   # rank 1's own flag is still unset
    assert arn.ar_device_status(0, reset=True) == arn.AR_ERR_TIMEOUT
    x = torch.arange(8, device="cuda", dtype=torch.float32)
    assert float(x.sum()) == 28.0                      # the context is still usable
    assert arn.ar_device_status(0) == arn.AR_OK


def test_wait_passes_on_flags_posted_by_earlier_kernels():
    torch.cuda.set_device(0)
    arn.ar_device_status(0, reset=True)
    pads = _pads(4)
    for r in (1, 2, 3):
        arn.ar_signal_post(pads, r, 7)
    arn.ar_barrier(pads, 0, 7, limit_us=1_000_000)
    assert arn.ar_device_status(0, reset=True) == arn.AR_OK
    for p in pads:
        assert _flags(p, 4) == [7, 7, 7, 7]
    # a flag of an older epoch does not satisfy a newer wait
    arn.ar_signal_post(pads, 1, 8)
    arn.ar_signal_post(pads, 2, 8)
    arn.ar_barrier(pads, 0, 8, limit_us=2000)          # rank 3 is still at 7
    assert arn.ar_device_status(0, reset=True) == arn.AR_ERR_TIMEOUT
    # epochs compare modulo 2^32: 0xFFFFFFFF, then 1 and 2 after the wrap (0
    # is AR_EPOCH_AUTO)
    pads = _pads(2)
    for e in (0xFFFFFFFE, 0xFFFFFFFF, 1, 2):
        arn.ar_signal_post(pads, 1, e)
        arn.ar_barrier(pads, 0, e, limit_us=1_000_000)
        assert arn.ar_device_status(0, reset=True) == arn.AR_OK, hex(e)
    assert _flags(pads[0], 2) == [2, 2]


def test_automatic_epochs_advance_per_call_and_across_the_wrap():
    """AR_EPOCH_AUTO: each post moves this rank's counter (in its own pad) on
    by one, skipping 0, and a wait alone uses the counter as it stands."""
    torch.cuda.set_device(0)
    arn.ar_device_status(0, reset=True)
    pads = _pads(3)
    for k in range(1, 4):
        for r in (1, 2):
            arn.ar_signal_post(pads, r)                 # epoch = ++counter of pad r
        arn.ar_barrier(pads, 0, limit_us=1_000_000)
        assert arn.ar_device_status(0, reset=True) == arn.AR_OK, k
        for p in pads:
            assert _flags(p, 3) == [k, k, k] and int(p[arn.AR_MAX_RANKS]) == k
    arn.ar_signal_wait(pads[1], 3, limit_us=1_000_000)  # counter 3: every flag is there
    assert arn.ar_device_status(0, reset=True) == arn.AR_OK
    # across the wrap: counters at 0xFFFFFFFF move on to 1, not to 0
    for p in pads:
        p[arn.AR_MAX_RANKS] = -1
    for r in (1, 2):
        arn.ar_signal_post(pads, r)
    arn.ar_barrier(pads, 0, limit_us=1_000_000)
    assert arn.ar_device_status(0, reset=True) == arn.AR_OK
    assert all(int(p[arn.AR_MAX_RANKS]) == 1 for p in pads)
    # one rank missing: rank 2 does not post, so rank 0 times out
    arn.ar_signal_post(pads, 1)
    arn.ar_barrier(pads, 0, limit_us=2000)
    assert arn.ar_device_status(0, reset=True) == arn.AR_ERR_TIMEOUT


@pytest.mark.parametrize("world", [1, 2, 3, 8, 16])
def test_all_ranks_of_a_barrier_in_one_cooperative_kernel(world):
    st, stale = arn.ar_selftest_barrier(0, world, rounds=2000, limit_us=1_000_000)
    assert st == arn.AR_OK and stale == 0


@pytest.mark.parametrize("world,m,H", [(1, 64, 4096), (2, 77, 4104), (4, 300, 7168),
                                       (8, 16, 6144), (3, 5, 24)])
def test_two_shot_with_the_other_ranks_run_first(world, m, H):
    """Ranks 1 .. world-1 post the first epoch, run their stage 1 and post
    the second before rank 0's whole two-shot call: both its barriers find
    every flag set (nothing waits on a later launch), and its results are
    the two-stage results."""
    torch.cuda.set_device(0)
    arn.ar_device_status(0, reset=True)
    w = synth.Workload("two_shot", n=world, H=H, ms=(m,), p_std=0.5, res_std=1.0, seed=world + m)
    inp = device_inputs(w, m)
    temps = [torch.zeros((m, H), dtype=torch.bfloat16, device="cuda") for _ in range(world)]
    pads = _pads(world)
    for r in range(1, world):
        arn.ar_signal_post(pads, r, 1)                 # its partial is written
        arn.ar_reduce_scatter_store(inp.partials, temps, r)
        arn.ar_signal_post(pads, r, 2)                 # its stores have landed
    out, rout = arn.ar_rmsnorm_two_shot(inp.partials, inp.residual, inp.weight, inp.eps, temps,
                                        pads, 0, 1)
    if arn.ar_workspace_elems(0) < m * H:
        arn.ar_reserve_workspace(m * H, 0)
    ref_out, ref_rout = arn.ar_rmsnorm(inp.partials, inp.residual, inp.weight, inp.eps,
                                       mode="two_stage")
    torch.cuda.synchronize()
    assert arn.ar_device_status(0, reset=True) == arn.AR_OK
    for t in temps[1:]:                                 # every rank's temporary holds the sum
        assert torch.equal(t.view(torch.int16), temps[0].view(torch.int16))
    compare((out, rout, temps[0].float()), oracle_rows(inp, None, True), f"two-shot world={world}")
    assert torch.equal(out.view(torch.int16), ref_out.view(torch.int16))
    assert torch.equal(rout.view(torch.int16), ref_rout.view(torch.int16))


@pytest.mark.parametrize("kind", ["one_shot", "two_shot"])
def test_an_explicit_epoch_at_the_wrap_takes_one_next(kind):
    """A call given epoch 2^32 - 1 runs its second barrier on epoch 1 (0 is
    the automatic-epoch value): the other ranks post those two epochs and
    rank 0's call passes both barriers."""
    torch.cuda.set_device(0)
    arn.ar_device_status(0, reset=True)
    world, m, H = 2, 8, 1024
    w = synth.Workload("wrap", n=world, H=H, ms=(m,), p_std=0.5, res_std=1.0)
    inp = device_inputs(w, m)
    pads = _pads(world)
    temps = [torch.zeros((m, H), dtype=torch.bfloat16, device="cuda") for _ in range(world)]
    last = 0xFFFFFFFF
    arn.ar_signal_post(pads, 1, last)
    if kind == "two_shot":
        arn.ar_reduce_scatter_store(inp.partials, temps, 1)
    arn.ar_signal_post(pads, 1, 1)
    if kind == "one_shot":
        out, rout = arn.ar_rmsnorm_one_shot(inp.partials, inp.residual, inp.weight, inp.eps, pads,
                                            0, last, limit_us=100_000)
    else:
        out, rout = arn.ar_rmsnorm_two_shot(inp.partials, inp.residual, inp.weight, inp.eps, temps,
                                            pads, 0, last, limit_us=100_000)
    torch.cuda.synchronize()
    assert arn.ar_device_status(0, reset=True) == arn.AR_OK
    assert _flags(pads[1], world) == [1, 1]
    compare((out, rout, None), oracle_rows(inp, None, kind == "two_shot"), f"{kind} at the wrap")


def test_two_shot_replays_from_a_cuda_graph_with_fresh_epochs():
    """The emulated ranks' calls (the other ranks' two posts around their
    stage 1, then rank 0's two-shot call), captured once in a CUDA graph
    with automatic epochs and replayed on new inputs: every replay
    synchronises on two new epochs and matches the oracle."""
    torch.cuda.set_device(0)
    arn.ar_device_status(0, reset=True)
    world, m, H = 4, 48, 2056
    w = synth.Workload("two_shot_graph", n=world, H=H, ms=(m,), p_std=0.5, res_std=1.0)
    inp = device_inputs(w, m)
    temps = [torch.zeros((m, H), dtype=torch.bfloat16, device="cuda") for _ in range(world)]
    pads = _pads(world)
    out = torch.empty_like(inp.residual)
    rout = torch.empty_like(inp.residual)
    stream = torch.cuda.Stream()

    def call():
        for r in range(1, world):
            arn.ar_signal_post(pads, r, stream=stream)
            arn.ar_reduce_scatter_store(inp.partials, temps, r, stream=stream)
            arn.ar_signal_post(pads, r, stream=stream)
        arn.ar_rmsnorm_two_shot(inp.partials, inp.residual, inp.weight, inp.eps, temps, pads, 0,
                                out=out, residual_out=rout, stream=stream)

    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        call()                                         # eager: epochs 1 and 2
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        call()
    for replay in range(3):                            # epochs 3-4, 5-6, 7-8
        fresh = device_inputs(synth.Workload("two_shot_graph", n=world, H=H, ms=(m,), p_std=0.5,
                                             res_std=1.0, seed=100 + replay), m)
        for dst, src in zip(inp.partials + [inp.residual], fresh.partials + [fresh.residual]):
            dst.copy_(src)
        torch.cuda.synchronize()
        with torch.cuda.stream(stream):
            g.replay()
        torch.cuda.synchronize()
        assert arn.ar_device_status(0, reset=True) == arn.AR_OK, replay
        compare((out, rout, temps[0].float()), oracle_rows(inp, None, True), f"replay {replay}")
        for p in pads:
            assert int(p[arn.AR_MAX_RANKS]) == 2 * (replay + 2)


def _mapped_one_stage(inp):
    out = torch.empty_like(inp.residual)
    rout = torch.empty_like(inp.residual)
    arn.ar_rmsnorm_mapped(inp.partials, inp.residual, inp.weight, inp.eps, out=out,
                          residual_out=rout, mode="one_stage")
    return out, rout


@pytest.mark.parametrize("world,m,H", [(1, 64, 4096), (2, 77, 4104), (4, 300, 7168),
                                       (8, 16, 7168), (3, 5, 24), (16, 2, 1024),
                                       (2, 100, 12288), (4, 1024, 7168)])
def test_one_shot_with_the_other_ranks_posted_first(world, m, H):
    """Ranks 1 .. world-1 post both barriers' epochs before rank 0's one-shot
    call (nothing waits on a later launch): its results are the oracle's
    one-stage results and ar_rmsnorm_mapped's bits, and both barriers left
    every flag at the second epoch."""
    torch.cuda.set_device(0)
    arn.ar_device_status(0, reset=True)
    w = synth.Workload("one_shot", n=world, H=H, ms=(m,), p_std=0.5, res_std=1.0, seed=world + m)
    inp = device_inputs(w, m)
    pads = _pads(world)
    for r in range(1, world):
        arn.ar_signal_post(pads, r, 5)
        arn.ar_signal_post(pads, r, 6)
    out, rout = arn.ar_rmsnorm_one_shot(inp.partials, inp.residual, inp.weight, inp.eps, pads, 0, 5)
    ref_out, ref_rout = _mapped_one_stage(inp)
    torch.cuda.synchronize()
    assert arn.ar_device_status(0, reset=True) == arn.AR_OK
    for p in pads:
        assert _flags(p, world) == [6] * world
    compare((out, rout, None), oracle_rows(inp, None, False), f"one-shot world={world}")
    assert torch.equal(out.view(torch.int16), ref_out.view(torch.int16))
    assert torch.equal(rout.view(torch.int16), ref_rout.view(torch.int16))


def test_one_shot_end_barrier_gives_up_when_a_rank_never_finishes():
    """Rank 1 posts only the first epoch: rank 0's results are complete, its
    second barrier records AR_ERR_TIMEOUT and the context stays usable.
    Without the end barrier the same call passes."""
    torch.cuda.set_device(0)
    arn.ar_device_status(0, reset=True)
    world, m, H = 2, 24, 2048
    w = synth.Workload("one_shot_timeout", n=world, H=H, ms=(m,), p_std=0.5, res_std=1.0)
    inp = device_inputs(w, m)
    pads = _pads(world)
    arn.ar_signal_post(pads, 1, 1)
    out, rout = arn.ar_rmsnorm_one_shot(inp.partials, inp.residual, inp.weight, inp.eps, pads, 0, 1,
                                        limit_us=2000)
    torch.cuda.synchronize()
    assert arn.ar_device_status(0, reset=True) == arn.AR_ERR_TIMEOUT
    assert _flags(pads[1], world) == [2, 1]            # rank 0 did post its second epoch
    compare((out, rout, None), oracle_rows(inp, None, False), "one-shot, end barrier timed out")
    arn.ar_signal_post(pads, 1, 3)
    out2, rout2 = arn.ar_rmsnorm_one_shot(inp.partials, inp.residual, inp.weight, inp.eps, pads, 0,
                                          3, limit_us=1_000_000, end_barrier=False)
    torch.cuda.synchronize()
    assert arn.ar_device_status(0, reset=True) == arn.AR_OK
    assert _flags(pads[1], world) == [3, 3]
    assert torch.equal(out2.view(torch.int16), out.view(torch.int16))
    assert torch.equal(rout2.view(torch.int16), rout.view(torch.int16))


def test_one_shot_replays_from_a_cuda_graph_with_fresh_epochs():
    """The other ranks' posts and rank 0's one-shot call, captured once with
    automatic epochs and replayed on new inputs: every call advances every
    pad's counter by two and matches the oracle."""
    torch.cuda.set_device(0)
    arn.ar_device_status(0, reset=True)
    world, m, H = 4, 40, 3072
    w = synth.Workload("one_shot_graph", n=world, H=H, ms=(m,), p_std=0.5, res_std=1.0)
    inp = device_inputs(w, m)
    pads = _pads(world)
    out = torch.empty_like(inp.residual)
    rout = torch.empty_like(inp.residual)
    stream = torch.cuda.Stream()

    def call():
        for r in range(1, world):
            arn.ar_signal_post(pads, r, stream=stream)
            arn.ar_signal_post(pads, r, stream=stream)
        arn.ar_rmsnorm_one_shot(inp.partials, inp.residual, inp.weight, inp.eps, pads, 0,
                                out=out, residual_out=rout, stream=stream)

    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        call()                                         # eager: epochs 1 and 2
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        call()
    for replay in range(3):
        fresh = device_inputs(synth.Workload("one_shot_graph", n=world, H=H, ms=(m,), p_std=0.5,
                                             res_std=1.0, seed=200 + replay), m)
        for dst, src in zip(inp.partials + [inp.residual], fresh.partials + [fresh.residual]):
            dst.copy_(src)
        torch.cuda.synchronize()
        with torch.cuda.stream(stream):
            g.replay()
        torch.cuda.synchronize()
        assert arn.ar_device_status(0, reset=True) == arn.AR_OK, replay
        compare((out, rout, None), oracle_rows(inp, None, False), f"replay {replay}")
        for p in pads:
            assert int(p[arn.AR_MAX_RANKS]) == 2 * (replay + 2)


def test_tp_group_object_on_one_rank():
    """FusedAllReduceRMSNorm without a process group (one rank): the layer
    writes into partial(m), then one-shot calls (m <= 32) and two-shot calls
    each give the oracle's result, with automatic epochs, eagerly and
    replayed from a CUDA graph."""
    from allreduce_sum_residual_gb300 import peers
    torch.cuda.set_device(0)
    arn.ar_device_status(0, reset=True)
    H = 4096
    g = peers.FusedAllReduceRMSNorm.create(256, H)
    assert g is not None and (g.rank, g.world, g.one_shot_rows) == (0, 1, 32)
    for m, seed in ((8, 1), (100, 2), (100, 3), (32, 4), (256, 5)):
        w = synth.Workload("tp_group", n=1, H=H, ms=(m,), p_std=0.5, res_std=1.0, seed=seed)
        inp = device_inputs(w, m)
        g.partial(m).copy_(inp.partials[0])
        out, rout = g(inp.residual, inp.weight, inp.eps)
        torch.cuda.synchronize()
        assert arn.ar_device_status(0, reset=True) == arn.AR_OK, m
        compare((out, rout, None), oracle_rows(inp, None, g.path(m) == "two_shot"),
                f"tp group m={m} {g.path(m)}")
    assert g.calls == 5
    # two calls (one-shot, two-shot) captured once and replayed on new inputs
    stream = torch.cuda.Stream()
    ins = [device_inputs(synth.Workload("tp_graph", n=1, H=H, ms=(m,), p_std=0.5, res_std=1.0,
                                       seed=10 + m), m) for m in (16, 64)]
    outs = [(torch.empty_like(i.residual), torch.empty_like(i.residual)) for i in ins]

    def step():
        for i, (o, r) in zip(ins, outs):
            g.partial(i.residual.shape[0]).copy_(i.partials[0])
            g(i.residual, i.weight, i.eps, out=o, residual_out=r, stream=stream)
        g.barrier(stream=stream)

    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        step()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        step()
    for replay in range(2):
        for k, i in enumerate(ins):
            fresh = device_inputs(synth.Workload("tp_graph", n=1, H=H, ms=(i.residual.shape[0],),
                                                 p_std=0.5, res_std=1.0, seed=50 + 2 * replay + k),
                                  i.residual.shape[0])
            i.partials[0].copy_(fresh.partials[0])
            i.residual.copy_(fresh.residual)
        torch.cuda.synchronize()
        with torch.cuda.stream(stream):
            graph.replay()
        torch.cuda.synchronize()
        assert arn.ar_device_status(0, reset=True) == arn.AR_OK
        for i, (o, r) in zip(ins, outs):
            m = i.residual.shape[0]
            compare((o, r, None), oracle_rows(i, None, g.path(m) == "two_shot"),
                    f"tp group graph replay {replay} m={m}")
    g.close()


# ---------------------------------------------------------------- two processes, CUDA IPC

def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _ipc_rank(rank, world, port, m, H, fail_open_rank, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK="0")
    sys.path[:0] = [ROOT, os.path.join(ROOT, "tests")]
    try:
        import torch.distributed as dist
        import allreduce_sum_residual_gb300 as arn
        from allreduce_sum_residual_gb300 import peers
        import synth
        from gpu_helpers import compare, oracle_rows
        torch.cuda.set_device(0)
        dist.init_process_group("gloo")
        w = synth.Workload("ipc", n=world, H=H, ms=(m,), p_std=0.5, res_std=1.0, seed=m + H)
        inp = synth.make_inputs(w, m)              # the same seeded inputs on every rank
        mine = inp.partials[rank].cuda()           # this rank's partial, its own allocation
        temp = torch.zeros((m, H), dtype=torch.bfloat16, device="cuda")
        residual, weight = inp.residual.cuda(), inp.weight.cuda()

        def open_handle(h, off):
            if rank == fail_open_rank:
                raise RuntimeError("IPC open failure injected on this rank")
            return arn.ar_ipc_open(h, off)

        pm = peers.map_peer_buffers([mine, temp], open_handle=open_handle)
        if pm is None:
            dist.barrier()
            q.put((rank, "declined"))
            dist.destroy_process_group()
            return
        torch.cuda.synchronize()
        dist.barrier()                             # every partial is written
        full = synth.Inputs([p.cuda() for p in inp.partials], residual, weight, inp.eps)
        # one-shot: every rank reads every rank's partial through the mappings
        out, rout = peers.ar_rmsnorm_peers(pm[0], residual, weight, inp.eps, mode="one_stage")
        torch.cuda.synchronize()
        compare((out, rout, None), oracle_rows(full, None, False), f"one-shot rank {rank}")
        # two-shot: this rank's slice into both temporaries, a host barrier, stage 2
        peers.ar_reduce_scatter_store_peers(pm[0], pm[1], m * H, rank)
        torch.cuda.synchronize()
        dist.barrier()                             # every rank's stores have landed
        out2, rout2 = arn.ar_load_rmsnorm(temp, residual, weight, inp.eps)
        torch.cuda.synchronize()
        compare((out2, rout2, temp.float()), oracle_rows(full, None, True), f"two-shot rank {rank}")
        assert arn.ar_device_status(0) == arn.AR_OK
        dist.barrier()                             # no rank still reads a peer's buffer
        pm.close()
        dist.destroy_process_group()
        q.put((rank, "ok"))
    except Exception as e:  # report instead of hanging the parent
        q.put((rank, f"error: {type(e).__name__}: {e}"))
        raise


@pytest.mark.parametrize("m,H,fail_open_rank", [(64, 4096, None), (77, 4104, None),
                                                (16, 1024, 1)])
def test_two_processes_share_buffers_through_ipc(m, H, fail_open_rank):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_ipc_rank, args=(r, 2, port, m, H, fail_open_rank, q))
             for r in range(2)]
    for p in procs:
        p.start()
    got = sorted(q.get(timeout=300) for _ in procs)
    for p in procs:
        p.join(timeout=120)
    want = "ok" if fail_open_rank is None else "declined"
    assert got == [(0, want), (1, want)], got
    assert all(p.exitcode == 0 for p in procs)
