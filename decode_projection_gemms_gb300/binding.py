"""ctypes binding of ``libkdaproj.so`` (argument marshalling only).

Every computation runs in the library's CUDA kernels; this module checks
tensor types and shapes, passes ``data_ptr()`` / stream handles through the C
ABI declared in ``include/kdaproj.h`` and turns non-zero status codes into
``KdaProjError``. There is no CPU or PyTorch fallback: if the library is not
built, importing the functions below raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libkdaproj.so")
TABLE_PATH = os.path.join(_HERE, "tune", "gb300_table.txt")

# enum kp_status
(KP_OK, KP_EINVAL, KP_EALIGN, KP_ESHAPE, KP_ENOPLAN, KP_ECUDA, KP_ETOOBIG, KP_ENODEV, KP_ECONFIG,
 KP_EIO, KP_EDEVICE) = (0, -1, -2, -3, -4, -5, -6, -7, -8, -9, -10)
STATUS_NAMES = {0: "KP_OK", -1: "KP_EINVAL", -2: "KP_EALIGN", -3: "KP_ESHAPE", -4: "KP_ENOPLAN",
                -5: "KP_ECUDA", -6: "KP_ETOOBIG", -7: "KP_ENODEV", -8: "KP_ECONFIG", -9: "KP_EIO",
                -10: "KP_EDEVICE"}
# enum kp_kind
KIND_AUTO, KIND_CC, KIND_TC05, KIND_SMALLK = 0, 1, 2, 3
KIND_NAMES = {0: "auto", 1: "cc", 2: "tc05", 3: "smallk"}
FLAG_PDL = 1
FLAG_FUSE_FB = 2
DTYPE_BF16, DTYPE_FP16 = 0, 1
BRANCH_QKVG, BRANCH_FAB, BRANCH_FB = 0, 1, 2

# exported symbols (must match include/kdaproj.h)
EXPORTS = (
    "skinny_gemm", "kp_select_config", "kp_table_load", "kp_table_clear", "kp_table_size",
    "kda_proj_plan", "kda_proj_set_overlap", "kda_proj_get_config", "kda_proj_set_config",
    "kda_proj_overlap_at", "kda_proj_run", "kda_proj_destroy", "kp_last_error", "kp_version",
    "kp_device_error", "kp_scratch_bytes", "skinny_gemm_noalloc", "skinny_gemm_ex",
    "kp_selftest_timeout", "kp_pdl_consumer_checksum",
)
DEV_SELFTEST = 5   # device error code of kp_selftest_timeout


class KdaProjError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"{STATUS_NAMES.get(code, code)}: {msg}")
        self.code = code


class KpCfg(ctypes.Structure):
    _fields_ = [("kind", ctypes.c_int32), ("split_k", ctypes.c_int32), ("block", ctypes.c_int32),
                ("rows", ctypes.c_int32), ("k_unroll", ctypes.c_int32), ("producers", ctypes.c_int32),
                ("stages", ctypes.c_int32), ("flags", ctypes.c_int32)]

    def as_dict(self) -> dict:
        d = {f: int(getattr(self, f)) for f, _ in self._fields_}
        d["kind"] = KIND_NAMES.get(d["kind"], d["kind"])
        return d

    @classmethod
    def make(cls, kind, split_k=1, block=256, rows=4, k_unroll=2, producers=1, stages=0,
             flags=FLAG_PDL):
        if isinstance(kind, str):
            kind = {v: k for k, v in KIND_NAMES.items()}[kind]
        return cls(int(kind), int(split_k), int(block), int(rows), int(k_unroll), int(producers),
                   int(stages), int(flags))


_lock = threading.Lock()
_lib = None


def load(path: str | None = None):
    """Load the library (once) and declare its signatures. Raises if absent."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        p = path or LIB_PATH
        if not os.path.exists(p):
            raise ImportError(f"{p} is missing: build it with decode_projection_gemms_gb300.build.build()")
        lib = ctypes.CDLL(p)
        vp, ci, cfgp = ctypes.c_void_p, ctypes.c_int, ctypes.POINTER(KpCfg)
        sig = {
            "skinny_gemm": [vp, vp, vp, ci, ci, ci, cfgp, vp],
            "kp_select_config": [ci, ci, ci, ci, cfgp],
            "kp_table_load": [ctypes.c_char_p],
            "kp_table_clear": [],
            "kp_table_size": [],
            "kda_proj_plan": [ci, ci, ci, ci, ci, ctypes.POINTER(vp)],
            "kda_proj_set_overlap": [vp, ci],
            "kda_proj_get_config": [vp, ci, ci, cfgp],
            "kda_proj_set_config": [vp, ci, ci, cfgp],
            "kda_proj_overlap_at": [vp, ci],
            "kda_proj_run": [vp, vp, vp, vp, vp, vp, vp, ci, vp, vp, ctypes.POINTER(vp)],
            "kda_proj_destroy": [vp],
            "kp_last_error": [],
            "kp_version": [],
            "kp_device_error": [ctypes.POINTER(ci)],
            "kp_scratch_bytes": [ci, ci, ci, cfgp, ci, ctypes.POINTER(ctypes.c_size_t)],
            "skinny_gemm_noalloc": [vp, vp, vp, ci, ci, ci, cfgp, vp],
            "skinny_gemm_ex": [vp, vp, vp, vp, ci, ci, ci, ci, cfgp, vp],
            "kp_selftest_timeout": [ci, vp],
            "kp_pdl_consumer_checksum": [vp, ctypes.c_int64, vp, ci, vp],
        }
        for name, args in sig.items():
            fn = getattr(lib, name)
            fn.argtypes = args
            fn.restype = ctypes.c_char_p if name == "kp_last_error" else ci
        _lib = lib
        if os.path.exists(TABLE_PATH):
            rc = lib.kp_table_load(TABLE_PATH.encode())
            if rc:
                raise KdaProjError(rc, lib.kp_last_error().decode())
        return _lib


def _check(rc: int):
    if rc != KP_OK:
        raise KdaProjError(rc, load().kp_last_error().decode())


def last_error() -> str:
    return load().kp_last_error().decode()


def _bf16_2d(t: torch.Tensor, name: str):
    # the common case in a few cheap checks; the rest only to name the problem
    if type(t) is torch.Tensor and t.dtype is torch.bfloat16 and t.is_cuda and t.dim() == 2 \
            and t.is_contiguous():
        return
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != torch.bfloat16:
        raise TypeError(f"{name} must be bfloat16, got {t.dtype}")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dim() != 2 or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous 2-D tensor")


def _stream_handle(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream)


def table_load(path: str = TABLE_PATH):
    _check(load().kp_table_load(str(path).encode()))


def table_clear():
    _check(load().kp_table_clear())


def table_size() -> int:
    return int(load().kp_table_size())


def select_config(M: int, N: int, K: int, num_sms: int = 0) -> KpCfg:
    c = KpCfg()
    _check(load().kp_select_config(M, N, K, num_sms, ctypes.byref(c)))
    return c


def scratch_bytes(M: int, N: int, K: int, cfg: KpCfg, num_sms: int) -> int:
    b = ctypes.c_size_t()
    _check(load().kp_scratch_bytes(M, N, K, ctypes.byref(cfg), num_sms, ctypes.byref(b)))
    return int(b.value)


def selftest_timeout(timeout_us: int = 2000, stream=None):
    """Launch the failure-path self-test (a wait that must run out)."""
    _check(load().kp_selftest_timeout(int(timeout_us), _stream_handle(stream)))


def pdl_consumer_checksum(t: torch.Tensor, out: torch.Tensor, pdl: bool = True, stream=None):
    """Launch the dependent checksum kernel on ``t`` (bf16/fp16, contiguous)
    adding into ``out`` (a CUDA int64 tensor of one element); ``pdl`` launches
    it with programmatic stream serialisation."""
    if t.dtype not in _DTYPES or not t.is_contiguous() or not t.is_cuda:
        raise TypeError("t must be a contiguous CUDA bf16/fp16 tensor")
    if out.dtype != torch.int64 or out.numel() != 1 or not out.is_cuda:
        raise TypeError("out must be a one-element CUDA int64 tensor")
    _check(load().kp_pdl_consumer_checksum(t.data_ptr(), t.numel(), out.data_ptr(), int(bool(pdl)),
                                           _stream_handle(stream)))


def device_error() -> int:
    """Read and clear the current device's error word (0: no kernel wait ran
    out). Does not wait for the device."""
    v = ctypes.c_int()
    _check(load().kp_device_error(ctypes.byref(v)))
    return int(v.value)


def check_device(stream=None):
    """Wait for ``stream`` (default: the current stream), then raise
    ``KdaProjError(KP_EDEVICE)`` if a kernel wait ran out meanwhile (the
    outputs of that work are undefined). Reading clears the code."""
    (stream or torch.cuda.current_stream()).synchronize()
    code = device_error()
    if code:
        raise KdaProjError(KP_EDEVICE, f"a kernel wait ran out (device error code {code}); "
                                       "the outputs of the work just run are undefined")


def skinny_gemm(x: torch.Tensor, W: torch.Tensor, y: torch.Tensor | None = None,
                cfg: KpCfg | None = None, stream=None) -> torch.Tensor:
    """``y = bf16(x @ W.T)`` with fp32 accumulation, in the library's kernels."""
    _bf16_2d(x, "x")
    _bf16_2d(W, "W")
    M, K = x.shape
    N = W.shape[0]
    if W.shape[1] != K:
        raise ValueError(f"W has K={W.shape[1]}, x has K={K}")
    if y is None:
        y = torch.empty((M, N), dtype=torch.bfloat16, device=x.device)
    _bf16_2d(y, "y")
    if tuple(y.shape) != (M, N):
        raise ValueError(f"y must be {(M, N)}")
    _check(load().skinny_gemm(x.data_ptr(), W.data_ptr(), y.data_ptr(), M, N, K,
                              ctypes.byref(cfg) if cfg is not None else None,
                              _stream_handle(stream)))
    return y


_DTYPES = {torch.bfloat16: DTYPE_BF16, torch.float16: DTYPE_FP16}


def _half_2d(t: torch.Tensor, name: str, dtype=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype not in _DTYPES or (dtype is not None and t.dtype != dtype):
        raise TypeError(f"{name} must be {dtype or 'bfloat16 or float16'}, got {t.dtype}")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dim() != 2 or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous 2-D tensor")


def skinny_gemm_ex(x: torch.Tensor, W: torch.Tensor, residual: torch.Tensor | None = None,
                   y: torch.Tensor | None = None, cfg: KpCfg | None = None,
                   stream=None) -> torch.Tensor:
    """``y = round(x @ W.T + residual)`` with fp32 accumulation; x, W, residual
    and y all bfloat16 or all float16 (the element type is x's). ``residual``
    may be ``y`` itself."""
    _half_2d(x, "x")
    _half_2d(W, "W", x.dtype)
    M, K = x.shape
    N = W.shape[0]
    if W.shape[1] != K:
        raise ValueError(f"W has K={W.shape[1]}, x has K={K}")
    if y is None:
        y = torch.empty((M, N), dtype=x.dtype, device=x.device)
    _half_2d(y, "y", x.dtype)
    if tuple(y.shape) != (M, N):
        raise ValueError(f"y must be {(M, N)}")
    if residual is not None:
        _half_2d(residual, "residual", x.dtype)
        if tuple(residual.shape) != (M, N):
            raise ValueError(f"residual must be {(M, N)}")
    _check(load().skinny_gemm_ex(x.data_ptr(), W.data_ptr(),
                                 residual.data_ptr() if residual is not None else None,
                                 y.data_ptr(), M, N, K, _DTYPES[x.dtype],
                                 ctypes.byref(cfg) if cfg is not None else None,
                                 _stream_handle(stream)))
    return y


def skinny_gemm_noalloc(x: torch.Tensor, W: torch.Tensor, y: torch.Tensor,
                        cfg: KpCfg | None = None, stream=None) -> torch.Tensor:
    """``y = bf16(x @ W.T)`` without any allocation by the library: the
    CUDA-core split-K kernel keeps its partial sums in a fixed device array
    (for callers that cannot allocate, e.g. during graph capture). ``y`` must
    be given; M <= 16. Concurrent calls on one device race."""
    _bf16_2d(x, "x")
    _bf16_2d(W, "W")
    _bf16_2d(y, "y")
    M, K = x.shape
    N = W.shape[0]
    if W.shape[1] != K or tuple(y.shape) != (M, N):
        raise ValueError("shape mismatch")
    _check(load().skinny_gemm_noalloc(x.data_ptr(), W.data_ptr(), y.data_ptr(), M, N, K,
                                      ctypes.byref(cfg) if cfg is not None else None,
                                      _stream_handle(stream)))
    return y


class KdaPlan:
    """Owns a ``kda_plan`` (scratch per branch + per-M configurations)."""

    def __init__(self, K: int = 7168, N_qkvg: int = 4096, N_fab: int = 136, N_fb: int = 1024,
                 max_M: int = 256):
        self.K, self.N_qkvg, self.N_fab, self.N_fb, self.max_M = K, N_qkvg, N_fab, N_fb, max_M
        self._lib = load()
        self._run = self._lib.kda_proj_run
        self._ev_key, self._ev_arr = None, None
        h = ctypes.c_void_p()
        _check(self._lib.kda_proj_plan(K, N_qkvg, N_fab, N_fb, max_M, ctypes.byref(h)))
        self._h = h

    @property
    def handle(self) -> int:
        return int(self._h.value or 0)

    def set_overlap(self, mode: int):
        _check(self._lib.kda_proj_set_overlap(self._h, int(mode)))

    def overlap_at(self, M: int) -> int:
        """Mode at M: 0 sequential, 1 overlapped, 2 single launch."""
        return int(self._lib.kda_proj_overlap_at(self._h, M))

    def get_config(self, branch: int, M: int) -> KpCfg:
        c = KpCfg()
        _check(self._lib.kda_proj_get_config(self._h, branch, M, ctypes.byref(c)))
        return c

    def set_config(self, branch: int, M: int, cfg: KpCfg):
        _check(self._lib.kda_proj_set_config(self._h, branch, M, ctypes.byref(cfg)))

    def outputs(self, M: int, device=None):
        dev = device or torch.device("cuda", torch.cuda.current_device())
        return (torch.empty((M, self.N_qkvg), dtype=torch.bfloat16, device=dev),
                torch.empty((M, self.N_fab), dtype=torch.bfloat16, device=dev),
                torch.empty((M, self.N_fb), dtype=torch.bfloat16, device=dev))

    def run(self, x: torch.Tensor, W_packed: torch.Tensor, W_fb: torch.Tensor,
            out_qkvg=None, out_fab=None, out_fb=None, aux_stream=None, events=None,
            stream=None, check: bool = False):
        """Enqueue the projection; returns ``(out_qkvg, out_fab, out_fb)``.

        ``aux_stream`` (torch.cuda.Stream) and ``events`` (two
        torch.cuda.Event) enable the two-stream overlap; ``stream`` is the
        main stream (default: the current stream). ``check=True`` waits for
        the main stream and raises ``KdaProjError(KP_EDEVICE)`` if a kernel
        wait ran out during the call (not usable under graph capture)."""
        _bf16_2d(x, "x")
        _bf16_2d(W_packed, "W_packed")
        _bf16_2d(W_fb, "W_fb")
        M, kx = x.shape
        if kx != self.K:
            raise ValueError(f"x must be [M, {self.K}]")
        if W_packed.shape != (self.N_qkvg + self.N_fab, self.K):
            raise ValueError(f"W_packed must be {(self.N_qkvg + self.N_fab, self.K)}")
        if W_fb.shape != (self.N_fb, 128):
            raise ValueError(f"W_fb must be {(self.N_fb, 128)}")
        if out_qkvg is None or out_fab is None or out_fb is None:
            oq, of, ob = self.outputs(M, x.device)
            out_qkvg = oq if out_qkvg is None else out_qkvg
            out_fab = of if out_fab is None else out_fab
            out_fb = ob if out_fb is None else out_fb
        for t, n, shape in ((out_qkvg, "out_qkvg", (M, self.N_qkvg)), (out_fab, "out_fab", (M, self.N_fab)),
                            (out_fb, "out_fb", (M, self.N_fb))):
            _bf16_2d(t, n)
            if t.shape != shape:
                raise ValueError(f"{n} must be {shape}")
        ev = None
        aux = None
        if aux_stream is not None and events is not None:
            aux = aux_stream.cuda_stream
            key = (events[0].cuda_event, events[1].cuda_event)
            if self._ev_key != key:   # the handle array, reused while the events are
                self._ev_key = key
                self._ev_arr = (ctypes.c_void_p * 2)(*key)
            ev = self._ev_arr
        rc = self._run(self._h, x.data_ptr(), W_packed.data_ptr(), W_fb.data_ptr(),
                       out_qkvg.data_ptr(), out_fab.data_ptr(), out_fb.data_ptr(), M,
                       _stream_handle(stream), aux, ev)
        if rc:
            _check(rc)
        if check:
            check_device(stream)
        return out_qkvg, out_fab, out_fb

    def close(self):
        if self._h is not None and self._h.value:
            self._lib.kda_proj_destroy(self._h)
            self._h = ctypes.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def make_events():
    """Two timing-free CUDA events, created eagerly (a fresh torch Event only
    gets its handle when first recorded)."""
    evs = (torch.cuda.Event(enable_timing=False), torch.cuda.Event(enable_timing=False))
    for e in evs:
        e.record()
    return evs
