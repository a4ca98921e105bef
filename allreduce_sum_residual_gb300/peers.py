"""Mapping the ranks' buffers into each other's processes for the all-reduce.

lightseekorg/tokenspeed #968 "perf(comm): add opt-in Triton AR+RMSNorm
backend", Summary: the ranks' coarse buffers are shared through IPC handles
and the backend falls back collectively when IPC setup fails; its review of
the state creation adds that a rank which fails alone must not leave the
group split between two paths.  ``map_peer_buffers`` exchanges this rank's
CUDA IPC handles (``ar_ipc_get_handle``) with every rank over the process
group (``all_gather_object``), opens the other ranks' (``ar_ipc_open``),
and lets every rank keep the mapping only if every rank succeeded
(``consensus.agree``); otherwise every rank closes what it opened and gets
``None``.  It is setup: call it once, outside graph capture, and keep the
result (or the decline) for good.

The returned ``PeerMap`` gives, per buffer, the device addresses of all
ranks' copies in rank order, ready for the peer-pointer calls
``ar_rmsnorm_peers`` (one-shot: every rank reads every rank's partial) and
``ar_reduce_scatter_store_peers`` (stage 1 of the two-shot path: stores into
every rank's temporary).  Before stage 1 (or the one-shot epilogue) and
between the stages the ranks synchronise: on separate GPUs with
``ar_barrier`` on signal pads mapped the same way (``ar_rmsnorm_one_shot``
and ``ar_rmsnorm_two_shot`` do it themselves), or, for ranks sharing one
GPU, on the host (stream synchronisation and a process-group barrier),
since kernels of ranks on one GPU must never wait on one another.

``FusedAllReduceRMSNorm`` puts it together for a tensor-parallel group:
setup (buffers, mapping, collective decline) once, then one call per layer
that picks the one-shot or the two-shot path by the number of rows.
"""
from typing import Callable, List, Optional, Sequence

from . import consensus


class PeerMap:
    """Device addresses of every rank's copy of each mapped buffer."""

    def __init__(self, addrs: List[List[int]], opened: list, close: Callable):
        self.addrs = addrs        # addrs[i][r]: buffer i of rank r, as seen by this process
        self._opened = opened     # handles opened here, one entry per ar_ipc_open
        self._close = close

    def __getitem__(self, i):
        return self.addrs[i]

    def close(self):
        """Unmap the other ranks' buffers (after every use has completed)."""
        while self._opened:
            self._close(self._opened.pop())


def map_peer_buffers(tensors: Sequence, group=None,
                     get_handle: Optional[Callable] = None,
                     open_handle: Optional[Callable] = None,
                     close_handle: Optional[Callable] = None) -> Optional[PeerMap]:
    """Map every rank's copy of each of ``tensors`` (this rank's buffers, the
    same list on every rank) into this process.  Returns a PeerMap on every
    rank, or None on every rank when any rank failed (nothing left open).
    ``get_handle(t) -> (handle, offset)``, ``open_handle(handle, offset) ->
    address`` and ``close_handle(handle)`` default to the library's IPC
    calls."""
    import torch.distributed as dist
    if get_handle is None or open_handle is None or close_handle is None:
        from . import ar_ipc_close, ar_ipc_get_handle, ar_ipc_open
        get_handle = get_handle or ar_ipc_get_handle
        open_handle = open_handle or ar_ipc_open
        close_handle = close_handle or ar_ipc_close
    if not (dist.is_available() and dist.is_initialized()):
        # one process, no group: every buffer is this rank's own
        return PeerMap([[int(t.data_ptr()) if hasattr(t, "data_ptr") else int(t)]
                        for t in tensors], [], close_handle)
    rank = dist.get_rank(group)
    world = dist.get_world_size(group)
    ok = True
    local = []
    try:
        for t in tensors:
            h, off = get_handle(t)
            local.append((bytes(h), int(off)))
    except Exception:   # a rank-local failure must not leave the group
        ok = False
    gathered = [None] * world
    dist.all_gather_object(gathered, local if ok else None, group=group)
    ok = ok and all(g is not None and len(g) == len(tensors) for g in gathered)
    opened, addrs = [], []
    if ok:
        try:
            for i, t in enumerate(tensors):
                row = []
                for r in range(world):
                    if r == rank:
                        row.append(int(t.data_ptr()) if hasattr(t, "data_ptr") else int(t))
                    else:
                        h, off = gathered[r][i]
                        row.append(int(open_handle(h, off)))
                        opened.append(h)
                addrs.append(row)
        except Exception:
            ok = False
    if not consensus.agree(ok, group):
        while opened:
            close_handle(opened.pop())
        return None
    return PeerMap(addrs, opened, close_handle)


def ar_rmsnorm_peers(partials: Sequence[int], residual, weight, eps, out=None, residual_out=None,
                     mode=0, stream=None):
    """ar_rmsnorm over partials given as device addresses in rank order (this
    rank's and the other ranks' mapped copies): the one-shot all-reduce with
    the epilogue fused.  Runs through ar_rmsnorm_mapped (plain loads on the
    register kernel).  Returns (out, residual_out)."""
    import torch
    from . import MODES, _check, _ptr, _stream_ptr, _VP, lib
    m, H = residual.shape
    if out is None:
        out = torch.empty_like(residual)
    if residual_out is None:
        residual_out = torch.empty_like(residual)
    arr = (_VP * len(partials))(*[int(p) for p in partials])
    st = lib().ar_rmsnorm_mapped(arr, len(partials), _ptr(residual), _ptr(weight), float(eps), m, H,
                                 _ptr(out), _ptr(residual_out), int(MODES.get(mode, mode)),
                                 _stream_ptr(stream, residual.device))
    _check(st, "ar_rmsnorm_mapped")
    return out, residual_out


def ar_reduce_scatter_store_peers(partials: Sequence[int], temps: Sequence[int], count: int,
                                  rank: int, stream=None, device=None):
    """Stage 1 of the two-shot path with device addresses: this rank's slice of
    the count elements, reduced over the partials and stored into every
    rank's temporary temps[0 .. world-1]."""
    import torch
    from . import _check, _VP, lib
    if stream is None:
        stream = torch.cuda.current_stream(device)
    parr = (_VP * len(partials))(*[int(p) for p in partials])
    tarr = (_VP * len(temps))(*[int(t) for t in temps])
    st = lib().ar_reduce_scatter_store(parr, len(partials), int(count), int(rank), len(temps), tarr,
                                       _VP(stream.cuda_stream))
    _check(st, "ar_reduce_scatter_store")


def one_shot_max_rows(world: int) -> int:
    """Rows up to which a tensor-parallel group of ``world`` ranks takes the
    one-shot path (every rank reads every rank's partial) rather than the
    two-shot path: 32 up to 4 ranks and 16 from 8, the rule ROCm/aiter #3817
    keeps for MI355X across GPUs (Test Results, thresholds from #3458); 5 to
    7 ranks take the 8-rank value.  No measurement across GB300s backs it
    yet; one would replace it."""
    return 32 if world <= 4 else 16


class FusedAllReduceRMSNorm:
    """The fused all-reduce + residual + RMSNorm of one tensor-parallel group.

    ``create`` (every rank, once, outside graph capture) allocates this
    rank's buffers -- two partials that the layer writes its output into
    (``partial(m)``), a temporary for the two-shot path and a signal pad --
    and maps every rank's copies (``map_peer_buffers``), or returns None on
    every rank when any rank failed (tokenspeed #968's collective
    fallback).  A call then runs, on the caller's stream, the one-shot path
    (``ar_rmsnorm_one_shot``: barrier, epilogue) up to ``one_shot_rows``
    rows and the two-shot path (``ar_rmsnorm_two_shot``: barrier, stage 1,
    barrier, stage 2) above, with epochs from the signal pads.  Every rank
    must make the same sequence of calls.

    Why two partials.  Calls alternate between them, so the one-shot path
    needs no second barrier: a rank writes a partial again two calls
    later, after it has passed the first barrier of the call in between,
    which every rank reaches only once it has finished reading that
    partial.  (The two-shot path's own barriers make one temporary enough.)
    A CUDA graph fixes the alternation it captured, so a graph that is
    replayed back to back must capture an even number of calls, or end
    with ``barrier()``.
    """

    def __init__(self, pm, partials, own, rank, world, one_shot_rows):
        self._pm = pm                    # 0, 1: partials; 2: temporaries; 3: signal pads
        self._partials = partials        # this rank's two [max_rows, H] partials
        self._own = own                  # this rank's other tensors, kept alive while mapped
        self.rank, self.world = rank, world
        self.max_rows, self.hidden = partials[0].shape
        self.one_shot_rows = one_shot_rows
        self.calls = 0

    @classmethod
    def create(cls, max_rows: int, hidden: int, group=None, device=None,
               one_shot_rows: Optional[int] = None, map_buffers: Optional[Callable] = None):
        """Set up on every rank of ``group``; None on every rank if any failed."""
        import torch
        import torch.distributed as dist
        from . import AR_SIGNAL_PAD_BYTES
        if max_rows < 1 or hidden < 8 or hidden % 8:
            raise ValueError("max_rows >= 1 and hidden a positive multiple of 8 are required")
        dev = torch.device("cuda", torch.cuda.current_device()) if device is None else \
            torch.device(device)
        bufs = [torch.zeros((max_rows, hidden), dtype=torch.bfloat16, device=dev)
                for _ in range(3)]
        pad = torch.zeros(AR_SIGNAL_PAD_BYTES // 4, dtype=torch.int32, device=dev)
        pm = (map_buffers or map_peer_buffers)(bufs + [pad], group=group)
        if pm is None:
            return None
        on = dist.is_available() and dist.is_initialized()
        rank = dist.get_rank(group) if on else 0
        world = dist.get_world_size(group) if on else 1
        rows = one_shot_max_rows(world) if one_shot_rows is None else int(one_shot_rows)
        return cls(pm, bufs[:2], (bufs[2:], pad), rank, world, rows)

    _cache = {}                          # key -> group object, or _DECLINED
    _DECLINED = object()

    @classmethod
    def for_group(cls, max_rows: int, hidden: int, group=None, device=None,
                  one_shot_rows: Optional[int] = None, map_buffers: Optional[Callable] = None):
        """``create`` once per (group, max_rows, hidden, device), then the same
        object -- or, after a decline, None without trying again: the
        permanent decline tokenspeed #968's review asks for (a setup that
        failed is not retried on every call, so no rank takes the collective
        setup path alone).  Every rank must call it with the same arguments
        in the same order, as for ``create``."""
        import torch
        dev = torch.device("cuda", torch.cuda.current_device()) if device is None else \
            torch.device(device)
        key = (id(group), max_rows, hidden, str(dev), one_shot_rows)
        hit = cls._cache.get(key)
        if hit is None:
            made = cls.create(max_rows, hidden, group=group, device=dev,
                              one_shot_rows=one_shot_rows, map_buffers=map_buffers)
            hit = cls._cache[key] = made if made is not None else cls._DECLINED
        return None if hit is cls._DECLINED else hit

    def partial(self, m: int):
        """This rank's partial for the next call, with m rows: the [m, H]
        tensor the layer writes its output into before that call."""
        if not 0 <= m <= self.max_rows:
            raise ValueError(f"m = {m} is outside 0 .. {self.max_rows}")
        return self._partials[self.calls % 2][:m]

    def path(self, m: int) -> str:
        return "one_shot" if m <= self.one_shot_rows else "two_shot"

    def __call__(self, residual, weight, eps, out=None, residual_out=None, stream=None):
        """out, residual_out for this rank, from every rank's partial(m)."""
        from . import ar_rmsnorm_one_shot, ar_rmsnorm_two_shot
        m = residual.shape[0]
        if m > self.max_rows or residual.shape[1] != self.hidden:
            raise ValueError(f"residual {tuple(residual.shape)} does not fit "
                             f"[<= {self.max_rows}, {self.hidden}]")
        partials, pads = self._pm[self.calls % 2], self._pm[3]
        self.calls += 1
        if self.path(m) == "one_shot":
            return ar_rmsnorm_one_shot(partials, residual, weight, eps, pads, self.rank, out=out,
                                       residual_out=residual_out, end_barrier=False,
                                       stream=stream)
        return ar_rmsnorm_two_shot(partials, residual, weight, eps, self._pm[2], pads, self.rank,
                                   out=out, residual_out=residual_out, stream=stream)

    def barrier(self, limit_us: int = 1000000, stream=None):
        """A barrier of the group on the signal pads (the next epoch)."""
        from . import ar_barrier
        ar_barrier(self._pm[3], self.rank, limit_us=limit_us, stream=stream)

    def close(self):
        """Unmap the other ranks' buffers, after every call has completed on
        every rank."""
        self._pm.close()


__all__ = ["PeerMap", "map_peer_buffers", "ar_rmsnorm_peers", "ar_reduce_scatter_store_peers",
           "one_shot_max_rows", "FusedAllReduceRMSNorm"]
