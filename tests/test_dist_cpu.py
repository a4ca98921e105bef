"""The bench's multi-rank host logic on CPU ranks (gloo, world size 2):
barrier, max and sum over ranks, and the rank-0-only reference arm under
torchrun.  No GPU is involved."""
import json
import multiprocessing as mp
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank), ARN_DIST_BACKEND="gloo")
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    w, r, _ = bench.dist_setup(None)
    bench.barrier(w)
    mx = bench.max_over_ranks(w, 10.0 * (r + 1))
    sm = bench.sum_over_ranks(w, 10.0 * (r + 1))
    bench.barrier(w)
    q.put((r, w, mx, sm))
    dist.destroy_process_group()


def test_max_and_sum_over_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert got == [(0, 2, 20.0, 30.0), (1, 2, 20.0, 30.0)]


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(1, 3.5) == 3.5
    assert bench.sum_over_ranks(1, 3.5) == 3.5
    bench.barrier(1)


@pytest.mark.slow
def test_reference_arm_under_torchrun_prints_one_line():
    port = free_port()
    env = dict(os.environ, OMP_NUM_THREADS="1")
    r = subprocess.run(
        [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
         "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py", "--impl",
         "reference", "--gpus", "2", "--steps", "3", "--warmup", "3", "--quick"],
        cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle"
    assert d["e2e"]["h2d_bytes_per_step"] == 0


def _consensus_rank(rank, world, port, fail_rank, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    from allreduce_sum_residual_gb300 import consensus
    dist.init_process_group("gloo")
    held = []

    def reserve(elems, device):
        if rank == fail_rank:
            raise MemoryError("allocation failure injected on this rank")
        held.append(elems)

    def release(device):
        held.clear()

    ok = consensus.reserve_two_stage_workspace(1 << 20, rank, reserve=reserve, release=release)
    # every rank then takes the same path; a collective after the decision
    # completes on all ranks (no split between two different collectives)
    dist.barrier()
    q.put((rank, ok, list(held)))
    dist.destroy_process_group()


@pytest.mark.parametrize("fail_rank", [None, 0, 1])
def test_decline_is_collective(fail_rank):
    """An allocation failure injected on one rank makes every rank decline
    the two-stage path and hold no workspace; without a failure every rank
    keeps it."""
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = free_port()
    procs = [ctx.Process(target=_consensus_rank, args=(r, 2, port, fail_rank, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    if fail_rank is None:
        assert got == [(0, True, [1 << 20]), (1, True, [1 << 20])]
    else:
        assert got == [(0, False, []), (1, False, [])]


def test_agree_without_a_process_group():
    sys.path.insert(0, ROOT)
    from allreduce_sum_residual_gb300 import consensus
    assert consensus.agree(True) is True and consensus.agree(False) is False


def _peer_map_rank(rank, world, port, fail_rank, fail_at, q):
    """One gloo rank mapping two fake buffers: handles are (rank, index)
    pairs, 'opening' one yields a made-up address; a failure is injected on
    `fail_rank` while getting its handles or while opening a peer's."""
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    from allreduce_sum_residual_gb300 import peers
    dist.init_process_group("gloo")
    opened = []

    class Buf:
        def __init__(self, i):
            self.i = i

        def data_ptr(self):
            return 1000 * rank + self.i

    def get_handle(t):
        if rank == fail_rank and fail_at == "handle":
            raise RuntimeError("IPC handle failure injected on this rank")
        return bytes([rank, t.i]) + bytes(62), 16 * t.i

    def open_handle(h, off):
        if rank == fail_rank and fail_at == "open":
            raise RuntimeError("IPC open failure injected on this rank")
        opened.append(h)
        return 1000 * h[0] + h[1] + off

    def close_handle(h):
        opened.remove(h)

    pm = peers.map_peer_buffers([Buf(0), Buf(1)], get_handle=get_handle, open_handle=open_handle,
                                close_handle=close_handle)
    dist.barrier()   # every rank reached the same decision: a collective still completes
    q.put((rank, None if pm is None else pm.addrs, len(opened)))
    if pm is not None:
        pm.close()
        assert not opened
    dist.destroy_process_group()


@pytest.mark.parametrize("fail_rank,fail_at", [(None, None), (0, "handle"), (1, "handle"),
                                               (1, "open"), (0, "open")])
def test_peer_mapping_is_collective(fail_rank, fail_at):
    """Every rank maps every other rank's buffers, in rank order, or -- when
    one rank's IPC setup fails -- every rank declines and keeps nothing open."""
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = free_port()
    procs = [ctx.Process(target=_peer_map_rank, args=(r, 2, port, fail_rank, fail_at, q))
             for r in range(2)]
    for p in procs:
        p.start()
    got = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    if fail_rank is None:
        # buffer i of rank r: this rank's own pointer, or the peer's handle
        # opened at its offset (1000 r + i + 16 i)
        assert got[0] == (0, [[0, 1000], [1, 1001 + 16]], 2)
        assert got[1] == (1, [[0, 1000], [1 + 16, 1001]], 2)
    else:
        assert got == [(0, None, 0), (1, None, 0)]


def _tp_group_rank(rank, world, port, fail_rank, q):
    """One gloo rank setting up FusedAllReduceRMSNorm on CPU tensors with fake
    IPC handles, then making a sequence of calls whose library entry points
    are replaced by recorders: which path each call takes and which
    buffers it passes."""
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import torch
    import torch.distributed as dist
    import allreduce_sum_residual_gb300 as arn
    from allreduce_sum_residual_gb300 import peers
    dist.init_process_group("gloo")

    def fake_map(tensors, group=None):
        index = {id(t): i for i, t in enumerate(tensors)}

        def get_handle(t):
            if rank == fail_rank:
                raise RuntimeError("IPC handle failure injected on this rank")
            return bytes([rank, index[id(t)]]) + bytes(62), 0

        return peers.map_peer_buffers(tensors, group, get_handle=get_handle,
                                      open_handle=lambda h, off: 1000 * (1 + h[0]) + h[1],
                                      close_handle=lambda h: None)

    g = peers.FusedAllReduceRMSNorm.create(64, 1024, device="cpu", map_buffers=fake_map)
    dist.barrier()
    if g is None:
        q.put((rank, None))
        dist.destroy_process_group()
        return
    calls = []
    arn.ar_rmsnorm_one_shot = lambda p, res, w, eps, pads, r, **kw: calls.append(
        ("one_shot", res.shape[0], list(p), list(pads), r, kw.get("end_barrier", True)))
    arn.ar_rmsnorm_two_shot = lambda p, res, w, eps, temps, pads, r, **kw: calls.append(
        ("two_shot", res.shape[0], list(p), list(temps), r))
    w = torch.ones(1024, dtype=torch.bfloat16)
    written = []
    for m in (8, 40, 40, 32, 33, 64):
        written.append(g.partial(m).data_ptr())      # the buffer this call reads as this rank's
        g(torch.zeros((m, 1024), dtype=torch.bfloat16), w, 1e-6)
    bad = []
    for m in (65, 0):
        try:
            g.partial(m)
        except ValueError:
            bad.append(m)
    own = [c[2][rank] for c in calls]
    q.put((rank, (g.rank, g.world, g.one_shot_rows, tuple(g.partial(5).shape), calls, bad,
                  written == own)))
    g.close()
    dist.destroy_process_group()


@pytest.mark.parametrize("fail_rank", [None, 1])
def test_tp_group_picks_paths_and_alternates_partials(fail_rank):
    """FusedAllReduceRMSNorm on two gloo ranks: one-shot up to 32 rows
    (2 ranks) without an end barrier, two-shot above; the two partials in
    turn call by call (partial(m) hands out the one the next call reads),
    the other rank's buffers in rank order; or, when one rank's setup
    fails, None on both."""
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = free_port()
    procs = [ctx.Process(target=_tp_group_rank, args=(r, 2, port, fail_rank, q))
             for r in range(2)]
    for p in procs:
        p.start()
    got = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    if fail_rank is not None:
        assert got == [(0, None), (1, None)]
        return
    for rank, (r, world, rows, shape, calls, bad, own_partial_ok) in got:
        assert (r, world, rows, shape, bad, own_partial_ok) == (rank, 2, 32, (5, 1024), [65],
                                                                True)
        assert [c[:2] for c in calls] == [("one_shot", 8), ("two_shot", 40), ("two_shot", 40),
                                          ("one_shot", 32), ("two_shot", 33), ("two_shot", 64)]
        peer = 1 - rank
        addr = lambda i: 1000 * (1 + peer) + i     # the peer's buffer i, as this rank sees it
        # buffers 0 and 1: the partials, alternating call by call
        assert [c[2][peer] for c in calls] == [addr(0), addr(1)] * 3
        for c in calls:
            if c[0] == "one_shot":        # the pads, this rank, and no end barrier
                assert c[3][peer] == addr(3) and c[4] == rank and c[5] is False
            else:                         # buffer 2: the temporaries, every time
                assert c[3][peer] == addr(2) and c[4] == rank


def _tp_cache_rank(rank, world, port, q):
    """One gloo rank asking for the group object three times: the first ask
    fails on rank 1 (both decline), the later asks return None at once on
    both ranks without another setup; another size sets up afresh."""
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    from allreduce_sum_residual_gb300 import peers
    dist.init_process_group("gloo")
    setups = []

    def fake_map(tensors, group=None, fail=False):
        setups.append(len(tensors))
        index = {id(t): i for i, t in enumerate(tensors)}

        def get_handle(t):
            if fail and rank == 1:
                raise RuntimeError("IPC handle failure injected on this rank")
            return bytes([rank, index[id(t)]]) + bytes(62), 0

        return peers.map_peer_buffers(tensors, group, get_handle=get_handle,
                                      open_handle=lambda h, off: 1000 * (1 + h[0]) + h[1],
                                      close_handle=lambda h: None)

    F = peers.FusedAllReduceRMSNorm
    failing = lambda t, group=None: fake_map(t, group, fail=True)
    a = [F.for_group(32, 1024, device="cpu", map_buffers=failing) for _ in range(3)]
    b = [F.for_group(64, 1024, device="cpu", map_buffers=fake_map) for _ in range(2)]
    q.put((rank, [x is None for x in a], b[0] is not None and b[0] is b[1], setups))
    dist.destroy_process_group()


def test_tp_group_decline_is_kept():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = free_port()
    procs = [ctx.Process(target=_tp_cache_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    # one setup for the declined size, one for the other, on both ranks
    assert got == [(0, [True, True, True], True, [4, 4]), (1, [True, True, True], True, [4, 4])]
