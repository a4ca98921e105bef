"""Python binding of libarnorm.so: fused AllReduce + residual-add + RMSNorm.

Argument marshalling only.  Every step of the computation runs in the CUDA
kernels of libarnorm.so (the C ABI declared in include/ar_rmsnorm.h); this
module checks tensor shapes, dtypes and devices, turns tensors into raw
device pointers and passes the current CUDA stream.  There is no CPU or
PyTorch fallback: if the library is missing, importing ``lib()`` raises.

Names follow the C ABI:

    ar_rmsnorm(partials, residual, weight, eps, out=None, residual_out=None,
               mode=AR_MODE_AUTO, stream=None) -> (out, residual_out)
    ar_rmsnorm_ex(..., sum_out=None, cluster=0, vpt=0)
    ar_rmsnorm_mapped(partials, residual, weight, eps, out=None,
                      residual_out=None, mode=AR_MODE_AUTO, stream=None, device=None)
    ar_reduce_scatter_flat(partials, temp, stream=None)
    ar_reduce_scatter_store(partials, temps, rank, stream=None)
    ar_load_rmsnorm(temp, residual, weight, eps, out=None, residual_out=None)
    ar_reserve_workspace(max_elems, device) / ar_release_workspace(device)
    ar_workspace_elems(device), ar_select_mode(n, m, H),
    ar_get_plan(n, m, H, mode, sm_count=0), ar_get_plan_ex(n, m, H, mode, sm_count, ctas_per_sm),
    ar_device_status(device, reset),
    ar_selftest_bounded_wait(device, limit_us), ar_strerror(status), ar_version()
"""
import ctypes
import os

AR_OK = 0
AR_ERR_ARG = 1
AR_ERR_ALIGN = 2
AR_ERR_ALIAS = 3
AR_ERR_WORKSPACE = 4
AR_ERR_CUDA = 5
AR_ERR_TIMEOUT = 6
AR_ERR_UNSUPPORTED = 7
AR_ERR_SCRATCH_LIMIT = 8
AR_ERR_BOUNDS = 9
AR_STATIC_SCRATCH_ELEMS = 8 * 1024 * 1024

AR_MODE_AUTO = 0
AR_MODE_ONE_STAGE = 1
AR_MODE_TWO_STAGE = 2
MODES = {"auto": AR_MODE_AUTO, "one_stage": AR_MODE_ONE_STAGE, "two_stage": AR_MODE_TWO_STAGE}

AR_MAX_RANKS = 16
AR_MAX_HIDDEN = 131072

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libarnorm.so")
# The checking build (device-side bounds checks compiled in; for tests):
# ARN_CHECK_BUILD=1 makes lib() load it instead.
CHECK_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libarnorm_check.so")


class ArError(RuntimeError):
    def __init__(self, status, what):
        self.status = status
        super().__init__(f"{what}: status {status} ({_strerror(status)})")


AR_KERNEL_AUTO = 0
AR_KERNEL_REGISTER = 1
AR_KERNEL_STREAM = 2
AR_KERNEL_REGISTER_LATE_W = 3
KERNELS = {"auto": AR_KERNEL_AUTO, "register": AR_KERNEL_REGISTER, "stream": AR_KERNEL_STREAM,
           "register_late": AR_KERNEL_REGISTER_LATE_W}


AR_PREFETCH_AUTO = 0
AR_PREFETCH_NONE = 1
AR_PREFETCH_ROW = 2
AR_PREFETCH_ROW_AHEAD = 3
PREFETCHES = {"auto": AR_PREFETCH_AUTO, "none": AR_PREFETCH_NONE, "row": AR_PREFETCH_ROW,
              "row_ahead": AR_PREFETCH_ROW_AHEAD}


class ar_plan_t(ctypes.Structure):
    _fields_ = [("mode", ctypes.c_int), ("kernel", ctypes.c_int), ("cluster", ctypes.c_int),
                ("vpt", ctypes.c_int), ("threads", ctypes.c_int), ("stages", ctypes.c_int),
                ("ctas", ctypes.c_int64), ("launches", ctypes.c_int), ("prefetch", ctypes.c_int)]


_lib = None

_VP = ctypes.c_void_p
_I64 = ctypes.c_int64
_SIGS = {
    "ar_rmsnorm": (ctypes.c_int, [ctypes.POINTER(_VP), ctypes.c_int, _VP, _VP, ctypes.c_float,
                                  _I64, _I64, _VP, _VP, ctypes.c_int, _VP]),
    "ar_rmsnorm_ex": (ctypes.c_int, [ctypes.POINTER(_VP), ctypes.c_int, _VP, _VP, ctypes.c_float,
                                     _I64, _I64, _VP, _VP, ctypes.c_int, _VP, _VP,
                                     ctypes.POINTER(ar_plan_t)]),
    "ar_rmsnorm_mapped": (ctypes.c_int, [ctypes.POINTER(_VP), ctypes.c_int, _VP, _VP,
                                         ctypes.c_float, _I64, _I64, _VP, _VP, ctypes.c_int, _VP]),
    "ar_get_plan": (ctypes.c_int, [ctypes.c_int, _I64, _I64, ctypes.c_int, ctypes.c_int,
                                   ctypes.POINTER(ar_plan_t)]),
    "ar_get_plan_ex": (ctypes.c_int, [ctypes.c_int, _I64, _I64, ctypes.c_int, ctypes.c_int,
                                      _VP, ctypes.POINTER(ar_plan_t)]),
    "ar_reduce_scatter_flat": (ctypes.c_int, [ctypes.POINTER(_VP), ctypes.c_int, _I64, _VP, _VP]),
    "ar_reduce_scatter_store": (ctypes.c_int, [ctypes.POINTER(_VP), ctypes.c_int, _I64, ctypes.c_int,
                                               ctypes.c_int, ctypes.POINTER(_VP), _VP]),
    "ar_load_rmsnorm": (ctypes.c_int, [_VP, _VP, _VP, ctypes.c_float, _I64, _I64, _VP, _VP, _VP]),
    "ar_reserve_workspace": (ctypes.c_int, [_I64, ctypes.c_int]),
    "ar_release_workspace": (ctypes.c_int, [ctypes.c_int]),
    "ar_workspace_elems": (_I64, [ctypes.c_int]),
    "ar_select_mode": (ctypes.c_int, [ctypes.c_int, _I64, _I64]),
    "ar_rmsnorm_two_stage_static": (ctypes.c_int, [ctypes.POINTER(_VP), ctypes.c_int, _VP, _VP,
                                                   ctypes.c_float, _I64, _I64, _VP, _VP, _VP]),
    "ar_device_status": (ctypes.c_int, [ctypes.c_int, ctypes.c_int]),
    "ar_selftest_bounded_wait": (ctypes.c_int, [ctypes.c_int, ctypes.c_uint]),
    "ar_signal_post": (ctypes.c_int, [ctypes.POINTER(_VP), ctypes.c_int, ctypes.c_int,
                                      ctypes.c_uint32, _VP]),
    "ar_signal_wait": (ctypes.c_int, [_VP, ctypes.c_int, ctypes.c_uint32, ctypes.c_uint, _VP]),
    "ar_barrier": (ctypes.c_int, [ctypes.POINTER(_VP), ctypes.c_int, ctypes.c_int, ctypes.c_uint32,
                                  ctypes.c_uint, _VP]),
    "ar_rmsnorm_two_shot": (ctypes.c_int, [ctypes.POINTER(_VP), ctypes.c_int, _VP, _VP,
                                           ctypes.c_float, _I64, _I64, _VP, _VP, ctypes.c_int,
                                           ctypes.c_int, ctypes.POINTER(_VP), ctypes.POINTER(_VP),
                                           ctypes.c_uint32, ctypes.c_uint, _VP]),
    "ar_rmsnorm_one_shot": (ctypes.c_int, [ctypes.POINTER(_VP), ctypes.c_int, _VP, _VP,
                                           ctypes.c_float, _I64, _I64, _VP, _VP, ctypes.c_int,
                                           ctypes.c_int, ctypes.POINTER(_VP), ctypes.c_uint32,
                                           ctypes.c_uint, ctypes.c_int, _VP]),
    "ar_ipc_get_handle": (ctypes.c_int, [_VP, ctypes.c_char_p, ctypes.POINTER(_I64)]),
    "ar_ipc_open": (ctypes.c_int, [ctypes.c_char_p, _I64, ctypes.POINTER(_VP)]),
    "ar_ipc_close": (ctypes.c_int, [ctypes.c_char_p]),
    "ar_selftest_barrier": (ctypes.c_int, [ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_uint,
                                           ctypes.POINTER(ctypes.c_int)]),
    "ar_register_occupancy": (ctypes.c_int, [ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                             ctypes.c_int]),
    "ar_checks_bounds": (ctypes.c_int, []),
    "ar_selftest_bounds": (ctypes.c_int, [ctypes.c_int]),
    "ar_strerror": (ctypes.c_char_p, [ctypes.c_int]),
    "ar_version": (ctypes.c_int, []),
}


def load(path):
    """A build of the library at `path` (ctypes), with argument types set."""
    handle = ctypes.CDLL(path)
    for name, (res, args) in _SIGS.items():
        fn = getattr(handle, name)
        fn.restype = res
        fn.argtypes = args
    return handle


def lib():
    """The loaded libarnorm.so (ctypes), with argument types set; with
    ARN_CHECK_BUILD=1 in the environment, the checking build instead."""
    global _lib
    if _lib is None:
        checking = os.environ.get("ARN_CHECK_BUILD", "0") == "1"
        path = CHECK_LIB_PATH if checking else LIB_PATH
        if not os.path.exists(path):
            how = ("python -m allreduce_sum_residual_gb300._build --check" if checking else
                   "python -c \"import __graft_entry__ as g; g.build()\"")
            raise RuntimeError(f"{path} is not built: run `{how}` (the CUDA library is required; "
                               "there is no fallback)")
        _lib = load(path)
    return _lib


def _strerror(status):
    try:
        return lib().ar_strerror(int(status)).decode()
    except Exception:  # pragma: no cover - only while the library is unavailable
        return "unknown"


def _check(status, what):
    if status != AR_OK:
        raise ArError(status, what)


def _stream_ptr(stream, device):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return _VP(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _ptr(t):
    return _VP(t.data_ptr())


def _check_tensor(t, name, shape, device):
    import torch
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != torch.bfloat16:
        raise TypeError(f"{name} must be bfloat16, got {t.dtype}")
    if not t.is_cuda or (device is not None and t.device != device):
        raise ValueError(f"{name} must be on {device or 'a CUDA device'}, got {t.device}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _prepare(partials, residual, weight, out, residual_out):
    import torch
    if len(partials) < 1:
        raise ValueError("need at least one partial")
    if residual.dim() != 2:
        raise ValueError("residual must be [m, H]")
    m, H = residual.shape
    dev = residual.device
    _check_tensor(residual, "residual", (m, H), None)
    for k, p in enumerate(partials):
        _check_tensor(p, f"partials[{k}]", (m, H), dev)
    _check_tensor(weight, "weight", (H,), dev)
    if out is None:
        out = torch.empty_like(residual)
    if residual_out is None:
        residual_out = torch.empty_like(residual)
    _check_tensor(out, "out", (m, H), dev)
    _check_tensor(residual_out, "residual_out", (m, H), dev)
    arr = (_VP * len(partials))(*[p.data_ptr() for p in partials])
    return m, H, dev, out, residual_out, arr


def ar_rmsnorm(partials, residual, weight, eps, out=None, residual_out=None,
               mode=AR_MODE_AUTO, stream=None):
    """Fused epilogue on the current (or given) stream; returns (out, residual_out).

    partials: sequence of n bf16 [m, H] CUDA tensors, rank order = reduce order.
    mode: AR_MODE_AUTO / AR_MODE_ONE_STAGE / AR_MODE_TWO_STAGE or "auto" /
    "one_stage" / "two_stage".
    """
    mode = MODES.get(mode, mode)
    m, H, dev, out, residual_out, arr = _prepare(partials, residual, weight, out, residual_out)
    st = lib().ar_rmsnorm(arr, len(partials), _ptr(residual), _ptr(weight), float(eps), m, H,
                          _ptr(out), _ptr(residual_out), int(mode), _stream_ptr(stream, dev))
    _check(st, "ar_rmsnorm")
    return out, residual_out


def _check_mapped_tensor(t, name, shape, device):
    import torch
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != torch.bfloat16:
        raise TypeError(f"{name} must be bfloat16, got {t.dtype}")
    if t.is_cuda:
        if t.device != device:
            raise ValueError(f"{name} must be on {device} or in pinned host memory, got {t.device}")
    elif t.numel() > 0 and not t.is_pinned():
        raise ValueError(f"{name} must be a CUDA tensor or in pinned host memory")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def ar_rmsnorm_mapped(partials, residual, weight, eps, out=None, residual_out=None,
                      mode=AR_MODE_AUTO, stream=None, device=None):
    """ar_rmsnorm where any tensor may be in pinned host memory (CPU tensors
    with ``is_pinned()``): the kernels on ``device`` (default: the CUDA
    tensors' device, else the current device) read and write those buffers
    over the host link.  Missing outputs are allocated pinned on the host
    when the residual is on the host, else on its device.  Asynchronous on
    the stream: host outputs are valid once the stream has passed the call.
    Returns (out, residual_out)."""
    import torch
    mode = MODES.get(mode, mode)
    if len(partials) < 1:
        raise ValueError("need at least one partial")
    if residual.dim() != 2:
        raise ValueError("residual must be [m, H]")
    m, H = residual.shape
    tensors = list(partials) + [residual, weight] + [t for t in (out, residual_out) if t is not None]
    if device is None:
        cuda = [t.device for t in tensors if isinstance(t, torch.Tensor) and t.is_cuda]
        device = cuda[0] if cuda else torch.device("cuda", torch.cuda.current_device())
    device = torch.device(device)
    for k, p in enumerate(partials):
        _check_mapped_tensor(p, f"partials[{k}]", (m, H), device)
    _check_mapped_tensor(residual, "residual", (m, H), device)
    _check_mapped_tensor(weight, "weight", (H,), device)
    if out is None:
        out = torch.empty((m, H), dtype=torch.bfloat16, device=residual.device,
                          pin_memory=not residual.is_cuda)
    if residual_out is None:
        residual_out = torch.empty((m, H), dtype=torch.bfloat16, device=residual.device,
                                   pin_memory=not residual.is_cuda)
    _check_mapped_tensor(out, "out", (m, H), device)
    _check_mapped_tensor(residual_out, "residual_out", (m, H), device)
    arr = (_VP * len(partials))(*[p.data_ptr() for p in partials])
    with torch.cuda.device(device):
        st = lib().ar_rmsnorm_mapped(arr, len(partials), _ptr(residual), _ptr(weight), float(eps),
                                     m, H, _ptr(out), _ptr(residual_out), int(mode),
                                     _stream_ptr(stream, device))
    _check(st, "ar_rmsnorm_mapped")
    return out, residual_out


def ar_rmsnorm_ex(partials, residual, weight, eps, out=None, residual_out=None,
                  mode=AR_MODE_AUTO, stream=None, sum_out=None, cluster=0, vpt=0, kernel=0,
                  threads=0, stages=0, ctas=0, prefetch=0):
    """ar_rmsnorm plus the reduced sum (fp32 [m, H] ``sum_out``) and a forced
    kernel ("register" / "register_late" / "stream") and launch shape: register kernel
    ``cluster`` CTAs per row and ``vpt`` packs per thread; stream kernel
    ``threads`` (32 + consumers), ring ``stages`` and grid ``ctas``; L2
    ``prefetch`` ("none" / "row" / "row_ahead").  0 = library's choice.
    Returns (out, residual_out, sum_out)."""
    import torch
    mode = MODES.get(mode, mode)
    m, H, dev, out, residual_out, arr = _prepare(partials, residual, weight, out, residual_out)
    if sum_out is not None:
        if sum_out.dtype != torch.float32 or tuple(sum_out.shape) != (m, H) or \
                not sum_out.is_contiguous() or sum_out.device != dev:
            raise ValueError("sum_out must be a contiguous float32 [m, H] tensor on the inputs' device")
    plan = None
    kernel = KERNELS.get(kernel, kernel)
    prefetch = PREFETCHES.get(prefetch, prefetch)
    if cluster or vpt or kernel or threads or stages or ctas or prefetch:
        plan = ctypes.pointer(ar_plan_t(0, int(kernel), int(cluster), int(vpt), int(threads),
                                        int(stages), int(ctas), 0, int(prefetch)))
    st = lib().ar_rmsnorm_ex(arr, len(partials), _ptr(residual), _ptr(weight), float(eps), m, H,
                             _ptr(out), _ptr(residual_out), int(mode), _stream_ptr(stream, dev),
                             _VP(sum_out.data_ptr()) if sum_out is not None else None, plan)
    _check(st, "ar_rmsnorm_ex")
    return out, residual_out, sum_out


def ar_rmsnorm_two_stage_static(partials, residual, weight, eps, out=None, residual_out=None,
                                stream=None):
    """Two-stage epilogue that allocates no device memory: its temporary is a
    fixed 16 MiB array inside the library (m * H <= AR_STATIC_SCRATCH_ELEMS).
    For callers that may not call cudaMalloc; calls share that array, so
    calls overlapping on the GPU race.  Returns (out, residual_out)."""
    m, H, dev, out, residual_out, arr = _prepare(partials, residual, weight, out, residual_out)
    st = lib().ar_rmsnorm_two_stage_static(arr, len(partials), _ptr(residual), _ptr(weight),
                                           float(eps), m, H, _ptr(out), _ptr(residual_out),
                                           _stream_ptr(stream, dev))
    _check(st, "ar_rmsnorm_two_stage_static")
    return out, residual_out


def ar_reduce_scatter_flat(partials, temp, stream=None):
    """Stage 1 alone: temp = bf16(rank-order fp32 sum of the partials)."""
    count = temp.numel()
    for k, p in enumerate(partials):
        _check_tensor(p, f"partials[{k}]", tuple(temp.shape), temp.device)
    _check_tensor(temp, "temp", tuple(temp.shape), temp.device)
    arr = (_VP * len(partials))(*[p.data_ptr() for p in partials])
    st = lib().ar_reduce_scatter_flat(arr, len(partials), count, _ptr(temp),
                                      _stream_ptr(stream, temp.device))
    _check(st, "ar_reduce_scatter_flat")
    return temp


def ar_reduce_scatter_store(partials, temps, rank, stream=None):
    """Stage 1 as rank `rank` of len(temps) ranks: reduce this rank's slice
    of the packs and store bf16(sum) into every buffer of `temps`."""
    shape = tuple(temps[0].shape)
    dev = temps[0].device
    for k, p in enumerate(partials):
        _check_tensor(p, f"partials[{k}]", shape, dev)
    for d, t in enumerate(temps):
        _check_tensor(t, f"temps[{d}]", shape, dev)
    arr = (_VP * len(partials))(*[p.data_ptr() for p in partials])
    tarr = (_VP * len(temps))(*[t.data_ptr() for t in temps])
    st = lib().ar_reduce_scatter_store(arr, len(partials), temps[0].numel(), int(rank), len(temps),
                                       tarr, _stream_ptr(stream, dev))
    _check(st, "ar_reduce_scatter_store")
    return temps


def ar_load_rmsnorm(temp, residual, weight, eps, out=None, residual_out=None, stream=None):
    """Stage 2 alone: residual add and RMSNorm of an already reduced ``temp``."""
    m, H, dev, out, residual_out, _ = _prepare([temp], residual, weight, out, residual_out)
    st = lib().ar_load_rmsnorm(_ptr(temp), _ptr(residual), _ptr(weight), float(eps), m, H,
                               _ptr(out), _ptr(residual_out), _stream_ptr(stream, dev))
    _check(st, "ar_load_rmsnorm")
    return out, residual_out


def ar_reserve_workspace(max_elems, device=0):
    _check(lib().ar_reserve_workspace(int(max_elems), int(device)), "ar_reserve_workspace")


def ar_release_workspace(device=0):
    _check(lib().ar_release_workspace(int(device)), "ar_release_workspace")


def ar_workspace_elems(device=0):
    return int(lib().ar_workspace_elems(int(device)))


def ar_select_mode(n, m, H):
    r = lib().ar_select_mode(int(n), int(m), int(H))
    if r < 0:
        raise ArError(-r, "ar_select_mode")
    return r


def ar_get_plan(n, m, H, mode=AR_MODE_AUTO, sm_count=0):
    """The launch plan as a dict (pure host logic when sm_count > 0)."""
    p = ar_plan_t()
    _check(lib().ar_get_plan(int(n), int(m), int(H), int(MODES.get(mode, mode)), int(sm_count),
                             ctypes.byref(p)), "ar_get_plan")
    return {f: getattr(p, f) for f, _ in ar_plan_t._fields_}


OCCUPANCY_FN = ctypes.CFUNCTYPE(ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int)


def ar_get_plan_ex(n, m, H, mode, sm_count, ctas_per_sm=None):
    """ar_get_plan for a GPU of ``sm_count`` SMs with the caller's occupancy
    figures: ``ctas_per_sm(inputs, vpt, late_weight, threads) -> int`` (or
    None for plain interpolation).  Pure host logic."""
    p = ar_plan_t()
    fn = OCCUPANCY_FN(lambda a, b, c, d: int(ctas_per_sm(a, b, c, d))) if ctas_per_sm else None
    _check(lib().ar_get_plan_ex(int(n), int(m), int(H), int(MODES.get(mode, mode)), int(sm_count),
                                ctypes.cast(fn, _VP) if fn else None, ctypes.byref(p)),
           "ar_get_plan_ex")
    return {f: getattr(p, f) for f, _ in ar_plan_t._fields_}


def ar_register_occupancy(inputs, vpt, late_weight, threads):
    """CTAs per SM of the one-CTA register kernel on the current device (0 if
    unknown)."""
    return int(lib().ar_register_occupancy(int(inputs), int(vpt), int(late_weight), int(threads)))


def ar_device_status(device=0, reset=False):
    """AR_OK, or AR_ERR_TIMEOUT after a bounded in-kernel wait gave up
    (synchronises the device)."""
    return int(lib().ar_device_status(int(device), int(bool(reset))))


def ar_selftest_bounded_wait(device=0, limit_us=1000):
    """Run the bounded-wait self-test kernel; returns the status it left."""
    return int(lib().ar_selftest_bounded_wait(int(device), int(limit_us)))


# ---------------------------------------------------------------- cross-rank data plane

AR_SIGNAL_PAD_BYTES = 128
AR_EPOCH_AUTO = 0
AR_IPC_HANDLE_BYTES = 64


def _addr(x):
    """A device address from a tensor or an int."""
    return int(x.data_ptr()) if hasattr(x, "data_ptr") else int(x)


def _addrs(xs):
    return (_VP * len(xs))(*[_addr(x) for x in xs])


def _cur_stream(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return _VP(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def ar_signal_post(pads, rank, epoch=AR_EPOCH_AUTO, stream=None):
    """Post `epoch` of `rank` into every rank's signal pad (tensors or addresses)."""
    _check(lib().ar_signal_post(_addrs(pads), len(pads), int(rank), int(epoch) & 0xFFFFFFFF,
                                _cur_stream(stream)), "ar_signal_post")


def ar_signal_wait(pad, world, epoch=AR_EPOCH_AUTO, limit_us=1000000, stream=None):
    """Wait (bounded) until flags 0..world-1 of `pad` reach `epoch`."""
    _check(lib().ar_signal_wait(_VP(_addr(pad)), int(world), int(epoch) & 0xFFFFFFFF,
                                int(limit_us), _cur_stream(stream)), "ar_signal_wait")


def ar_barrier(pads, rank, epoch=AR_EPOCH_AUTO, limit_us=1000000, stream=None):
    """Post, then wait on pads[rank]: a bounded barrier of len(pads) ranks."""
    _check(lib().ar_barrier(_addrs(pads), len(pads), int(rank), int(epoch) & 0xFFFFFFFF,
                            int(limit_us), _cur_stream(stream)), "ar_barrier")


def ar_rmsnorm_two_shot(partials, residual, weight, eps, temps, pads, rank,
                        epoch=AR_EPOCH_AUTO, out=None, residual_out=None, limit_us=1000000,
                        stream=None):
    """Two-stage epilogue of rank `rank` of len(temps) ranks: its stage-1 slice
    stored into every rank's temporary, a barrier, stage 2 on temps[rank].
    `partials`, `temps` and `pads` are tensors or device addresses (peer or
    IPC mappings for other ranks); residual, weight and the outputs are
    tensors of this device.  Returns (out, residual_out)."""
    import torch
    m, H = residual.shape
    _check_tensor(residual, "residual", (m, H), None)
    _check_tensor(weight, "weight", (H,), residual.device)
    if out is None:
        out = torch.empty_like(residual)
    if residual_out is None:
        residual_out = torch.empty_like(residual)
    _check_tensor(out, "out", (m, H), residual.device)
    _check_tensor(residual_out, "residual_out", (m, H), residual.device)
    st = lib().ar_rmsnorm_two_shot(_addrs(partials), len(partials), _ptr(residual), _ptr(weight),
                                   float(eps), m, H, _ptr(out), _ptr(residual_out), int(rank),
                                   len(temps), _addrs(temps), _addrs(pads),
                                   int(epoch) & 0xFFFFFFFF, int(limit_us),
                                   _stream_ptr(stream, residual.device))
    _check(st, "ar_rmsnorm_two_shot")
    return out, residual_out


def ar_rmsnorm_one_shot(partials, residual, weight, eps, pads, rank, epoch=AR_EPOCH_AUTO,
                        out=None, residual_out=None, limit_us=1000000, end_barrier=True,
                        stream=None):
    """One-stage epilogue of rank `rank` of len(pads) ranks: a barrier, the
    epilogue over every rank's partial (plain loads), and with `end_barrier`
    a second barrier.  An explicit `epoch` e takes e and e + 1.  `partials`
    and `pads` are tensors or device addresses (peer or IPC mappings for
    other ranks); residual, weight and the outputs are tensors of this
    device.  Returns (out, residual_out)."""
    import torch
    m, H = residual.shape
    _check_tensor(residual, "residual", (m, H), None)
    _check_tensor(weight, "weight", (H,), residual.device)
    if out is None:
        out = torch.empty_like(residual)
    if residual_out is None:
        residual_out = torch.empty_like(residual)
    _check_tensor(out, "out", (m, H), residual.device)
    _check_tensor(residual_out, "residual_out", (m, H), residual.device)
    st = lib().ar_rmsnorm_one_shot(_addrs(partials), len(partials), _ptr(residual), _ptr(weight),
                                   float(eps), m, H, _ptr(out), _ptr(residual_out), int(rank),
                                   len(pads), _addrs(pads), int(epoch) & 0xFFFFFFFF,
                                   int(limit_us), 1 if end_barrier else 0,
                                   _stream_ptr(stream, residual.device))
    _check(st, "ar_rmsnorm_one_shot")
    return out, residual_out


def ar_ipc_get_handle(x):
    """(handle bytes, byte offset) of the allocation holding tensor/address x."""
    h = ctypes.create_string_buffer(AR_IPC_HANDLE_BYTES)
    off = _I64(0)
    _check(lib().ar_ipc_get_handle(_VP(_addr(x)), h, ctypes.byref(off)), "ar_ipc_get_handle")
    return h.raw, int(off.value)


def ar_ipc_open(handle, offset):
    """Device address of byte `offset` of another process's allocation."""
    p = _VP()
    _check(lib().ar_ipc_open(bytes(handle), int(offset), ctypes.byref(p)), "ar_ipc_open")
    return int(p.value)


def ar_ipc_close(handle):
    _check(lib().ar_ipc_close(bytes(handle)), "ar_ipc_close")


def ar_selftest_barrier(device=0, world=8, rounds=1000, limit_us=1000000):
    """All ranks of a barrier in one cooperative kernel; returns (status,
    stale reads)."""
    mism = ctypes.c_int(-1)
    st = int(lib().ar_selftest_barrier(int(device), int(world), int(rounds), int(limit_us),
                                       ctypes.byref(mism)))
    return st, int(mism.value)


def ar_strerror(status):
    return _strerror(status)


def ar_version():
    return int(lib().ar_version())
