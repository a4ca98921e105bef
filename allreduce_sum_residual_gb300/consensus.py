"""Collective agreement on the two-stage path across the ranks of a group.

lightseekorg/tokenspeed #968 "perf(comm): add opt-in Triton AR+RMSNorm
backend", review comments on state creation: when setup (an allocation, a
runtime call) fails on one rank only, that rank falls back while its peers
keep the fused path, the group splits between two collectives and hangs.
The review's remedy is for the ranks to share whether their setup worked,
so that all of them take the same path -- the allocation included.

Here the setup that can fail rank-locally is the reservation of the
two-stage workspace.  ``reserve_two_stage_workspace`` has every rank try it,
then all-reduces (MIN) a success flag; if any rank failed, every rank
releases what it reserved and returns False, so the whole group uses the
one-stage path (which needs no workspace).  The decision is made once, at
setup, outside graph capture, and the caller keeps it for good (the same
review asks that a failed setup not be retried on every call).
"""
from typing import Callable, Optional


def agree(ok: bool, group=None) -> bool:
    """True on every rank iff ``ok`` is true on every rank of ``group``."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return bool(ok)
    backend = dist.get_backend(group)
    dev = torch.device("cuda", torch.cuda.current_device()) if backend == "nccl" else "cpu"
    flag = torch.tensor([1 if ok else 0], dtype=torch.int32, device=dev)
    dist.all_reduce(flag, op=dist.ReduceOp.MIN, group=group)
    return bool(flag.item())


def reserve_two_stage_workspace(max_elems: int, device: int, group=None,
                                reserve: Optional[Callable[[int, int], None]] = None,
                                release: Optional[Callable[[int], None]] = None) -> bool:
    """Reserve the two-stage workspace on every rank, or on none.

    Returns True when every rank of ``group`` holds a workspace of
    ``max_elems`` elements, False (on every rank, with nothing held) when any
    rank failed.  ``reserve`` / ``release`` default to the library's
    ar_reserve_workspace / ar_release_workspace.
    """
    if reserve is None or release is None:
        from . import ar_release_workspace, ar_reserve_workspace
        reserve = reserve or ar_reserve_workspace
        release = release or ar_release_workspace
    try:
        reserve(max_elems, device)
        ok = True
    except Exception:  # a rank-local failure must not leave the group
        ok = False
    everyone = agree(ok, group)
    if not everyone and ok:
        release(device)
    return everyone
