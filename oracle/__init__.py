"""Plain CPU oracle for the KDA decode projections (test infrastructure).

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline /
reference leg may import this package. The product library never loads it,
and it shares no code with the CUDA path: the arithmetic lives in
``kda_oracle.c`` (double-precision triple loop, see that file's header for the
passages it follows), and this module only compiles it with gcc, loads it with
ctypes and moves numpy arrays in and out.

Inputs are raw bf16 (or, for ``gemm_ex``, fp16) bit patterns
(``numpy.uint16``); outputs are float64.

Comparison criterion (the build's stated tolerance for bf16 outputs with fp32
accumulation): ``|gpu - ref| <= 4 * ulp_bf16(|ref|) + 1e-3`` element-wise, with
``ulp_bf16(v) = 2^(floor(log2 v) - 7)`` for normal ``v`` (bf16 keeps 8
significant bits) and ``2^-133`` below the normal range. fp16 outputs use the
same rule with fp16's unit in the last place: ``2^(floor(log2 v) - 10)`` (11
significant bits), ``2^-24`` below ``2^-14``.

Parity pins: closed forms, one-hot selection, power-of-two scaling, row
independence, exact rational brute force and hand-derived bf16 rounding cases
(``tests/test_oracle_pins.py``). Nothing here is "parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kda_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_SO = os.path.join(_BUILD, "libkdaoracle.so")
_lock = threading.Lock()
_lib = None

CFLAGS = ["-O2", "-fPIC", "-shared", "-pthread", "-ffp-contract=off", "-fno-fast-math"]


def _compile(src: str, out: str) -> str:
    tmp = out + f".tmp{os.getpid()}"
    subprocess.run(["gcc", *CFLAGS, "-o", tmp, src, "-lm"], check=True)
    os.replace(tmp, out)
    return out


def build(force: bool = False) -> str:
    """Compile ``kda_oracle.c`` into ``oracle/_build/libkdaoracle.so``."""
    os.makedirs(_BUILD, exist_ok=True)
    if (not force and os.path.exists(_SO)
            and os.path.getmtime(_SO) >= os.path.getmtime(_SRC)):
        return _SO
    return _compile(_SRC, _SO)


def _u16(a) -> np.ndarray:
    a = np.ascontiguousarray(a)
    if a.dtype != np.uint16:
        raise TypeError(f"expected bf16 bit patterns as uint16, got {a.dtype}")
    return a


def _p(a, ctype):
    return a.ctypes.data_as(ctypes.POINTER(ctype))


class Oracle:
    """ctypes front end of one compiled copy of ``kda_oracle.c``."""

    def __init__(self, so_path: str):
        lib = ctypes.CDLL(so_path)
        u16p = ctypes.POINTER(ctypes.c_uint16)
        f64p = ctypes.POINTER(ctypes.c_double)
        i64 = ctypes.c_int64
        ci = ctypes.c_int
        lib.kdo_bf16_to_f64.argtypes = [ctypes.c_uint16]
        lib.kdo_bf16_to_f64.restype = ctypes.c_double
        lib.kdo_f64_to_bf16_rne.argtypes = [ctypes.c_double]
        lib.kdo_f64_to_bf16_rne.restype = ctypes.c_uint16
        lib.kdo_round_bf16.argtypes = [f64p, u16p, i64]
        lib.kdo_round_bf16.restype = None
        lib.kdo_widen_bf16.argtypes = [u16p, f64p, i64]
        lib.kdo_widen_bf16.restype = None
        lib.kdo_gemm.argtypes = [u16p, i64, u16p, i64, f64p, i64, ci, ci, ci, ci]
        lib.kdo_gemm.restype = ci
        lib.kdo_gemm_ex.argtypes = [u16p, i64, u16p, i64, u16p, i64, ci, f64p, i64, ci, ci, ci, ci]
        lib.kdo_gemm_ex.restype = ci
        lib.kdo_fp16_to_f64.argtypes = [ctypes.c_uint16]
        lib.kdo_fp16_to_f64.restype = ctypes.c_double
        lib.kdo_widen_fp16.argtypes = [u16p, f64p, i64]
        lib.kdo_widen_fp16.restype = None
        lib.kdo_kda_proj.argtypes = [u16p, u16p, u16p, f64p, f64p, u16p, f64p,
                                     ci, ci, ci, ci, ci, ci, ci]
        lib.kdo_kda_proj.restype = ci
        self.lib = lib
        self.path = so_path

    @classmethod
    def from_source(cls, c_text: str, workdir: str) -> "Oracle":
        """Compile C source text (e.g. a deliberately broken copy, for the
        tests that check the pins catch mistakes) and load it."""
        os.makedirs(workdir, exist_ok=True)
        src = os.path.join(workdir, "oracle_variant.c")
        with open(src, "w") as f:
            f.write(c_text)
        return cls(_compile(src, os.path.join(workdir, "liboracle_variant.so")))

    def bf16_to_f64(self, bits) -> np.ndarray:
        """Exact widening of bf16 bit patterns to float64."""
        b = _u16(bits)
        out = np.empty(b.shape, dtype=np.float64)
        self.lib.kdo_widen_bf16(_p(b, ctypes.c_uint16), _p(out, ctypes.c_double), b.size)
        return out

    def fp16_to_f64(self, bits) -> np.ndarray:
        """Exact widening of fp16 bit patterns to float64."""
        b = _u16(bits)
        out = np.empty(b.shape, dtype=np.float64)
        self.lib.kdo_widen_fp16(_p(b, ctypes.c_uint16), _p(out, ctypes.c_double), b.size)
        return out

    def f64_to_bf16(self, v) -> np.ndarray:
        """float64 -> bf16 bit patterns, round to nearest, ties to even."""
        a = np.ascontiguousarray(v, dtype=np.float64)
        out = np.empty(a.shape, dtype=np.uint16)
        self.lib.kdo_round_bf16(_p(a, ctypes.c_double), _p(out, ctypes.c_uint16), a.size)
        return out

    def gemm(self, x_bits, w_bits, nthreads: int = 1) -> np.ndarray:
        """``y[m, n] = sum_k x[m, k] * W[n, k]`` in double; x ``[M, K]``, W ``[N, K]``."""
        x = _u16(x_bits)
        w = _u16(w_bits)
        if x.ndim != 2 or w.ndim != 2 or x.shape[1] != w.shape[1]:
            raise ValueError(f"shape mismatch {x.shape} vs {w.shape}")
        M, K = x.shape
        N = w.shape[0]
        y = np.empty((M, N), dtype=np.float64)
        rc = self.lib.kdo_gemm(_p(x, ctypes.c_uint16), K, _p(w, ctypes.c_uint16), K,
                               _p(y, ctypes.c_double), N, M, N, K, int(nthreads))
        if rc:
            raise ValueError("kdo_gemm rejected its arguments")
        return y

    def gemm_ex(self, x_bits, w_bits, res_bits=None, dtype: str = "bf16",
                nthreads: int = 1) -> np.ndarray:
        """``y[m, n] = sum_k x[m, k] * W[n, k] + res[m, n]`` in double, inputs of
        type ``dtype`` ("bf16" or "fp16"); ``res`` ``[M, N]`` or None."""
        x = _u16(x_bits)
        w = _u16(w_bits)
        if x.ndim != 2 or w.ndim != 2 or x.shape[1] != w.shape[1]:
            raise ValueError(f"shape mismatch {x.shape} vs {w.shape}")
        M, K = x.shape
        N = w.shape[0]
        code = {"bf16": 0, "fp16": 1}[dtype]
        r = None
        if res_bits is not None:
            r = _u16(res_bits)
            if r.shape != (M, N):
                raise ValueError(f"residual shape {r.shape} != {(M, N)}")
        y = np.empty((M, N), dtype=np.float64)
        rc = self.lib.kdo_gemm_ex(_p(x, ctypes.c_uint16), K, _p(w, ctypes.c_uint16), K,
                                  _p(r, ctypes.c_uint16) if r is not None else None, N, code,
                                  _p(y, ctypes.c_double), N, M, N, K, int(nthreads))
        if rc:
            raise ValueError("kdo_gemm_ex rejected its arguments")
        return y

    def kda_proj(self, x_bits, wp_bits, wfb_bits, n_qkvg: int, n_fab: int,
                 n_fa: int = 128, nthreads: int = 1):
        """The full projection: returns ``(qkvg, fab, fa_bf16_bits, fb)``."""
        x = _u16(x_bits)
        wp = _u16(wp_bits)
        wfb = _u16(wfb_bits)
        M, K = x.shape
        if wp.shape != (n_qkvg + n_fab, K):
            raise ValueError(f"packed weight shape {wp.shape} != {(n_qkvg + n_fab, K)}")
        if wfb.ndim != 2 or wfb.shape[1] != n_fa:
            raise ValueError(f"W_fb shape {wfb.shape} must be [N_fb, {n_fa}]")
        n_fb = wfb.shape[0]
        qkvg = np.empty((M, n_qkvg), dtype=np.float64)
        fab = np.empty((M, n_fab), dtype=np.float64)
        fa = np.empty((M, n_fa), dtype=np.uint16)
        fb = np.empty((M, n_fb), dtype=np.float64)
        rc = self.lib.kdo_kda_proj(_p(x, ctypes.c_uint16), _p(wp, ctypes.c_uint16),
                                   _p(wfb, ctypes.c_uint16), _p(qkvg, ctypes.c_double),
                                   _p(fab, ctypes.c_double), _p(fa, ctypes.c_uint16),
                                   _p(fb, ctypes.c_double), M, K, n_qkvg, n_fab, n_fa,
                                   n_fb, int(nthreads))
        if rc:
            raise ValueError("kdo_kda_proj rejected its arguments")
        return qkvg, fab, fa, fb


def default() -> Oracle:
    """The oracle built from ``kda_oracle.c`` (compiled on first use)."""
    global _lib
    with _lock:
        if _lib is None:
            _lib = Oracle(build())
    return _lib


def bf16_to_f64(bits) -> np.ndarray:
    return default().bf16_to_f64(bits)


def fp16_to_f64(bits) -> np.ndarray:
    return default().fp16_to_f64(bits)


def f64_to_bf16(v) -> np.ndarray:
    return default().f64_to_bf16(v)


def gemm_ex(x_bits, w_bits, res_bits=None, dtype: str = "bf16", nthreads: int = 1) -> np.ndarray:
    return default().gemm_ex(x_bits, w_bits, res_bits, dtype, nthreads)


def gemm(x_bits, w_bits, nthreads: int = 1) -> np.ndarray:
    return default().gemm(x_bits, w_bits, nthreads)


def kda_proj(x_bits, wp_bits, wfb_bits, n_qkvg: int, n_fab: int, n_fa: int = 128,
             nthreads: int = 1):
    return default().kda_proj(x_bits, wp_bits, wfb_bits, n_qkvg, n_fab, n_fa, nthreads)


# ---- comparison -----------------------------------------------------------

def ulp_bf16(v) -> np.ndarray:
    """bf16 unit in the last place at |v|: 2^(floor(log2|v|) - 7), 2^-133 below 2^-126."""
    a = np.abs(np.asarray(v, dtype=np.float64))
    with np.errstate(divide="ignore"):
        _, e = np.frexp(a)            # a = f * 2^e, f in [0.5, 1)
    E = e.astype(np.int64) - 1
    u = np.ldexp(1.0, (E - 7).astype(np.int32))
    return np.where(a < 2.0 ** -126, 2.0 ** -133, u)


def ulp_fp16(v) -> np.ndarray:
    """fp16 unit in the last place at |v|: 2^(floor(log2|v|) - 10), 2^-24 below 2^-14."""
    a = np.abs(np.asarray(v, dtype=np.float64))
    with np.errstate(divide="ignore"):
        _, e = np.frexp(a)
    E = e.astype(np.int64) - 1
    u = np.ldexp(1.0, (E - 10).astype(np.int32))
    return np.where(a < 2.0 ** -14, 2.0 ** -24, u)


def ulp(v, dtype: str = "bf16") -> np.ndarray:
    return {"bf16": ulp_bf16, "fp16": ulp_fp16}[dtype](v)


def tolerance(ref, ulps: float = 4.0, abs_tol: float = 1e-3, dtype: str = "bf16") -> np.ndarray:
    """Per-element bound ``ulps * ulp(|ref|) + abs_tol`` for outputs of type ``dtype``."""
    return ulps * ulp(ref, dtype) + abs_tol


def compare(got, ref, ulps: float = 4.0, abs_tol: float = 1e-3, extra=None,
            dtype: str = "bf16") -> dict:
    """Element-wise check of ``got`` (float array) against ``ref`` (double).

    Non-finite values in ``got`` always fail. ``extra`` (optional, same shape)
    widens the bound element-wise. Returns a dict with ``ok``, the worst
    excess over the bound, the max abs error and the cosine similarity.
    """
    g = np.asarray(got, dtype=np.float64)
    r = np.asarray(ref, dtype=np.float64)
    if g.shape != r.shape:
        raise ValueError(f"shape mismatch {g.shape} vs {r.shape}")
    bound = tolerance(r, ulps, abs_tol, dtype)
    if extra is not None:
        bound = bound + np.asarray(extra, dtype=np.float64)
    finite = np.isfinite(g)
    err = np.where(finite, np.abs(g - r), np.inf)
    excess = err - bound
    worst = int(np.argmax(excess)) if excess.size else 0
    gn = float(np.linalg.norm(g[finite])) if finite.all() else float("nan")
    rn = float(np.linalg.norm(r))
    cos = float(np.dot(g.ravel(), r.ravel()) / (gn * rn)) if gn > 0 and rn > 0 else float("nan")
    return {
        "ok": bool(finite.all() and (excess <= 0).all()),
        "n_bad": int(np.count_nonzero(~(excess <= 0))),
        "max_abs_err": float(err.max()) if err.size else 0.0,
        "worst_index": np.unravel_index(worst, g.shape) if g.size else (),
        "worst_excess": float(excess.ravel()[worst]) if excess.size else 0.0,
        "cosine": cos,
    }
