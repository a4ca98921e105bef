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
every rank's temporary).  Between the stages the ranks synchronise: on
separate GPUs with ``ar_barrier`` on signal pads mapped the same way, or,
for ranks sharing one GPU, on the host (stream synchronisation and a
process-group barrier), since kernels of ranks on one GPU must never wait
on one another.
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


__all__ = ["PeerMap", "map_peer_buffers", "ar_rmsnorm_peers", "ar_reduce_scatter_store_peers"]
