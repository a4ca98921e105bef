"""CPU oracle for the fused AllReduce + residual-add + RMSNorm epilogue.

TEST INFRASTRUCTURE ONLY: the test suite, the smoke check and the bench's
CPU-baseline / reference arm may import this package; the product path
(``allreduce_sum_residual_gb300``) never does, and this package never
imports it.  The arithmetic lives in ``ar_rmsnorm_oracle.c`` (plain C,
compiled by ``oracle/build.py``); this module only marshals numpy arrays.

bf16 tensors are handled as their raw 16-bit patterns (numpy ``uint16``).

Definitions followed (see the C file for the step-by-step statement):
  * reduced sum: fp32, strictly in rank order p_0, p_1, ..., p_{n-1}
    (ROCm/aiter #3817 "perf: optimize fused AllReduce + RMSNorm
    (custom_all_reduce)", Technical Details, 2stage, reduce-scatter);
  * two-stage: the sum is rounded to bf16 before the residual add (same
    section: stage 1 downcasts to bf16 into the temporary buffer);
  * residual_out = bf16(sum + residual), out = bf16(r / sqrt(mean(r^2) + eps) * w)
    with the RMSNorm part in fp64.

Parity status: every function here is pinned by tests/test_oracle_pins.py.
"""
import ctypes
import os

import numpy as np

from . import build as _build

class Oracle:
    """The oracle library at ``path`` (default: the committed C source, built)."""

    def __init__(self, path=None):
        lib = ctypes.CDLL(path or _build.build())
        lib.oracle_bf16_to_f32.argtypes = [ctypes.c_uint16]
        lib.oracle_bf16_to_f32.restype = ctypes.c_float
        lib.oracle_bf16_from_f64.argtypes = [ctypes.c_double]
        lib.oracle_bf16_from_f64.restype = ctypes.c_uint16
        lib.oracle_ar_rmsnorm.argtypes = [
            ctypes.POINTER(ctypes.c_void_p), ctypes.c_int,
            ctypes.c_void_p, ctypes.c_void_p, ctypes.c_double,
            ctypes.c_int64, ctypes.c_int64, ctypes.c_int,
            ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int]
        lib.oracle_ar_rmsnorm.restype = ctypes.c_int
        self._lib = lib

    def bf16_to_f32(self, bits) -> np.ndarray:
        """Widen bf16 patterns to float32 (exact)."""
        flat = np.ascontiguousarray(bits, dtype=np.uint16).ravel()
        f = self._lib.oracle_bf16_to_f32
        out = np.fromiter((f(int(b)) for b in flat), dtype=np.float32, count=flat.size)
        return out.reshape(np.shape(bits))

    def bf16_from_f64(self, x) -> np.ndarray:
        """Round float64 values to bf16 patterns, nearest-even, one rounding."""
        flat = np.ascontiguousarray(x, dtype=np.float64).ravel()
        f = self._lib.oracle_bf16_from_f64
        out = np.fromiter((f(float(v)) for v in flat), dtype=np.uint16, count=flat.size)
        return out.reshape(np.shape(x))

    def ar_rmsnorm(self, partials, residual, weight, eps, two_stage=False, threads=1):
        """Run the oracle over m rows.

        partials: sequence of n uint16 arrays [m, H] (or one [n, m, H] array),
                  in rank order; residual: uint16 [m, H]; weight: uint16 [H].
        eps:      taken as the fp32 value a caller hands the library.
        Returns (out uint16 [m, H], residual_out uint16 [m, H], sum float32
        [m, H]) where ``sum`` is the reduced sum that feeds the residual add
        (the fp32 accumulator for one-stage, the widened bf16 temporary for
        two-stage).
        """
        ps = [np.ascontiguousarray(p, dtype=np.uint16) for p in partials]
        n = len(ps)
        res = np.ascontiguousarray(residual, dtype=np.uint16)
        w = np.ascontiguousarray(weight, dtype=np.uint16)
        if res.ndim != 2:
            raise ValueError("residual must be [m, H]")
        m, H = res.shape
        for p in ps:
            if p.shape != (m, H):
                raise ValueError("every partial must have the residual's shape")
        if w.shape != (H,):
            raise ValueError("weight must be [H]")
        out = np.empty((m, H), dtype=np.uint16)
        rout = np.empty((m, H), dtype=np.uint16)
        s = np.empty((m, H), dtype=np.float32)
        arr = (ctypes.c_void_p * n)(*[p.ctypes.data for p in ps])
        rc = self._lib.oracle_ar_rmsnorm(
            arr, n, res.ctypes.data, w.ctypes.data, float(np.float32(eps)), m, H,
            int(bool(two_stage)), out.ctypes.data, rout.ctypes.data, s.ctypes.data,
            int(threads))
        if rc != 0:
            raise RuntimeError(f"oracle_ar_rmsnorm failed with status {rc}")
        return out, rout, s


_default = None


def _get():
    global _default
    if _default is None:
        _default = Oracle()
    return _default


def bf16_to_f32(bits):
    return _get().bf16_to_f32(bits)


def bf16_from_f64(x):
    return _get().bf16_from_f64(x)


def ar_rmsnorm(partials, residual, weight, eps, two_stage=False, threads=1):
    return _get().ar_rmsnorm(partials, residual, weight, eps, two_stage, threads)


def host_threads() -> int:
    """Cores this process may run on (what a row-parallel oracle run uses)."""
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1
