"""Python binding of libfp8mp, the GB300 FP8 delayed-scaling linear layer.

Argument marshalling only: every function below forwards to the C entry
point of the same name in ``libfp8mp.so`` (declared in ``include/fp8mp.h``),
passing device pointers, sizes and the CUDA stream. All computation runs in
the library's CUDA kernels. torch is used for device memory and streams.
If the library has not been built, ``load()`` raises: there is no fallback.
"""

from __future__ import annotations

import ctypes
import os

import torch

E4M3, E5M2 = 0, 1
F32, BF16 = 0, 1
AMAX_MAX, AMAX_MOST_RECENT = 0, 1
MAX_HISTORY = 8192
FMT_MAX = {E4M3: 448.0, E5M2: 57344.0}

OK, ERR_INVALID, ERR_DEVICE, ERR_LAUNCH, ERR_TIMEOUT = 0, -1, -2, -3, -4

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libfp8mp.so")
EXPORTS = ("fp8_quantize", "fp8_quantize_ex", "fp8_quantize_current", "fp8_quantize_dbias",
           "fp8_quantize_dbias_workspace_bytes", "fp8_quantize_dbias_noalloc", "fp8_linear_fwd", "fp8_linear_fwd_fp8out", "fp8_linear_dgrad", "fp8_linear_wgrad",
           "fp8_linear_bwd", "fp8_linear_bwd_rowmajor", "fp8_linear_bwd_rowmajor_ex", "delayed_scaling_update",
           "delayed_scaling_update_ex", "mp_master_step", "mp_master_step_adam", "mp_master_step_prescanned", "mp_master_step_adam_prescanned",
           "mp_master_step_prescanned_ex", "mp_master_step_adam_prescanned_ex",
           "mp_master_step_prescanned_scaling_ex", "mp_master_step_adam_prescanned_scaling_ex", "fp8mp_check",
           "fp8mp_last_error",
           "fp8mp_version", "fp8mp_selftest_timeout", "fp8mp_selftest_barrier_timeout")

_lib = None


class Fp8mpError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"libfp8mp error {code}: {msg}")
        self.code = code


class fp8mp_meta(ctypes.Structure):
    """Mirror of the C struct fp8mp_meta (device pointers + two int32)."""

    _fields_ = [("amax_history", ctypes.c_void_p), ("scale", ctypes.c_void_p),
                ("scale_inv", ctypes.c_void_p), ("cur_amax", ctypes.c_void_p),
                ("history_len", ctypes.c_int32), ("fmt", ctypes.c_int32)]


def build(force: bool = False) -> str:
    from . import buildlib

    return buildlib.build(force=force)


def load(path: str | None = None):
    """Loads libfp8mp.so (raises if it is missing) and declares the signatures."""
    global _lib
    if _lib is not None:
        return _lib
    path = path or LIB_PATH
    if not os.path.exists(path):
        raise Fp8mpError(ERR_LAUNCH, f"{path} is missing: build it with "
                         "fp8_mixed_precision_reduce_gb300.build() (no CPU fallback exists)")
    L = ctypes.CDLL(path)
    P, I64, I32, F = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_float
    L.fp8_quantize.argtypes = [P, I32, I64, I64, I32, P, P, P, P, P]
    L.fp8_quantize_ex.argtypes = [P, I32, I64, I64, I32, P, P, P, P, ctypes.c_uint32, P]
    L.fp8_quantize_current.argtypes = [P, I32, I64, I64, I32, I32, P, P, P, P, P, P]
    L.fp8_quantize_dbias.argtypes = [P, I32, I64, I64, I32, P, P, P, P, P, I32, P, I64, P]
    L.fp8_quantize_dbias_noalloc.argtypes = [P, I32, I64, I64, I32, P, P, P, P, P, I32, P]
    L.fp8_quantize_dbias_workspace_bytes.argtypes = [I64, I64]
    L.fp8_quantize_dbias_workspace_bytes.restype = I64
    L.fp8_linear_fwd.argtypes = [P, P, I64, I64, I64, P, P, P, I32, P, I32, P, P]
    L.fp8_linear_fwd_fp8out.argtypes = [P, P, I64, I64, I64, P, P, P, I32, P, I32, P, P, P]
    L.fp8_linear_dgrad.argtypes = [P, P, I64, I64, I64, I32, P, P, P, I32, P]
    L.fp8_linear_wgrad.argtypes = [P, P, I64, I64, I64, I32, P, P, P, I32, P]
    L.fp8_linear_bwd.argtypes = [P, P, P, P, I64, I64, I64, I32, P, P, P, P, I32, P, I32, P]
    L.fp8_linear_bwd_rowmajor.argtypes = [P, P, P, I64, I64, I64, I32, P, P, P, P, I32, P, I32, P, P]
    L.fp8_linear_bwd_rowmajor_ex.argtypes = [P, P, P, I64, I64, I64, I32, P, P, P, P, I32, P, I32, P,
                                             ctypes.c_uint32, P]
    L.delayed_scaling_update.argtypes = [ctypes.POINTER(fp8mp_meta), I32, I32, I32, P]
    L.delayed_scaling_update_ex.argtypes = [ctypes.POINTER(fp8mp_meta), I32, I32, I32, P, P]
    L.mp_master_step.argtypes = [P, I64, P, P, P, P, P, P, P, P, F, F, F, F, I32, P]
    L.mp_master_step_adam.argtypes = [P, I64, P, P, P, P, P, P, P, P, P, P, F, F, F, F, F, F, I32, P]
    L.mp_master_step_prescanned.argtypes = [P, I64, P, P, P, P, P, P, P, P, P, F, F, F, F, I32, P]
    L.mp_master_step_adam_prescanned.argtypes = [P, I64, P, P, P, P, P, P, P, P, P, P, P, F, F, F, F, F, F, I32, P]
    U32 = ctypes.c_uint32
    L.mp_master_step_prescanned_ex.argtypes = [P, I64, P, P, P, P, P, P, P, P, P, P, F, F, F, F, I32, U32, P]
    L.mp_master_step_adam_prescanned_ex.argtypes = [P, I64, P, P, P, P, P, P, P, P, P, P, P, P, F, F, F, F, F, F,
                                                    I32, U32, P]
    M = ctypes.POINTER(fp8mp_meta)
    L.mp_master_step_prescanned_scaling_ex.argtypes = [P, I64, P, P, P, P, P, P, P, P, P, P, F, F, F, F, I32,
                                                       M, I32, I32, I32, U32, P]
    L.mp_master_step_adam_prescanned_scaling_ex.argtypes = [P, I64, P, P, P, P, P, P, P, P, P, P, P, P, F, F, F,
                                                            F, F, F, I32, M, I32, I32, I32, U32, P]
    L.fp8mp_check.argtypes = [P]
    L.fp8mp_selftest_timeout.argtypes = [P]
    L.fp8mp_selftest_barrier_timeout.argtypes = [P]
    L.fp8mp_last_error.restype = ctypes.c_char_p
    L.fp8mp_version.restype = I32
    for name in ("fp8_quantize", "fp8_quantize_ex", "fp8_quantize_current", "fp8_quantize_dbias", "fp8_quantize_dbias_noalloc",
                 "fp8_linear_fwd", "fp8_linear_fwd_fp8out", "fp8_linear_dgrad", "fp8_linear_wgrad",
                 "fp8_linear_bwd", "fp8_linear_bwd_rowmajor", "fp8_linear_bwd_rowmajor_ex", "delayed_scaling_update",
                 "delayed_scaling_update_ex", "mp_master_step", "mp_master_step_adam", "mp_master_step_prescanned", "mp_master_step_adam_prescanned",
                 "mp_master_step_prescanned_ex", "mp_master_step_adam_prescanned_ex", "fp8mp_check",
                 "fp8mp_selftest_timeout", "fp8mp_selftest_barrier_timeout"):
        getattr(L, name).restype = ctypes.c_int
    _lib = L
    return L


def last_error() -> str:
    return load().fp8mp_last_error().decode()


def _check(rc: int) -> None:
    if rc != OK:
        raise Fp8mpError(rc, last_error())


def _ptr(t) -> int | None:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream) -> int | None:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return F32
    if t.dtype == torch.bfloat16:
        return BF16
    raise TypeError(f"unsupported dtype {t.dtype}")


def _rows_cols(t: torch.Tensor):
    if t.dim() == 2:
        return t.shape[0], t.shape[1]
    return 1, t.numel()


# ------------------------------------------------------------- entry points


def fp8_quantize(x: torch.Tensor, fmt: int, scale: torch.Tensor, out: torch.Tensor,
                 out_t: torch.Tensor | None = None, amax: torch.Tensor | None = None,
                 stream=None) -> None:
    """out = sat_rne(x * scale) as FP8 codes (uint8), out_t its transpose,
    amax = max(amax, max|x|). x is 2-D (rows, cols) or flat, contiguous."""
    rows, cols = _rows_cols(x)
    _check(load().fp8_quantize(_ptr(x), _dtype_code(x), rows, cols, fmt, _ptr(scale), _ptr(out),
                               _ptr(out_t), _ptr(amax), _stream(stream)))


OVERLAP_PREVIOUS = 1  # FP8MP_OVERLAP_PREVIOUS: fp8_quantize_ex, mp_master_step(_adam) with w8_in
SIGNAL_DW_DONE = 2  # FP8MP_SIGNAL_DW_DONE: fp8_linear_bwd_rowmajor
WAIT_DW_DONE = 4  # FP8MP_WAIT_DW_DONE: mp_master_step(_adam) with grad_nonfinite and OVERLAP_PREVIOUS


def fp8_quantize_ex(x: torch.Tensor, fmt: int, scale: torch.Tensor, out: torch.Tensor,
                    out_t: torch.Tensor | None = None, amax: torch.Tensor | None = None, flags: int = 0,
                    stream=None) -> None:
    """fp8_quantize with flags. OVERLAP_PREVIOUS: the caller guarantees that the
    work enqueued before this call neither writes nor reads x, out, out_t or
    amax, so the cast may run while the previous kernel is still running; the
    call still completes after it."""
    rows, cols = _rows_cols(x)
    _check(load().fp8_quantize_ex(_ptr(x), _dtype_code(x), rows, cols, fmt, _ptr(scale), _ptr(out),
                                  _ptr(out_t), _ptr(amax), flags, _stream(stream)))


def fp8_quantize_current(x: torch.Tensor, fmt: int, scale: torch.Tensor, scale_inv: torch.Tensor,
                         amax: torch.Tensor, out: torch.Tensor, out_t: torch.Tensor | None = None,
                         margin: int = 0, stream=None) -> None:
    """Just-in-time scaling: amax = max|x|, scale from it (kept when the amax
    is 0 / not finite), then out = sat_rne(x * scale) and its transpose."""
    rows, cols = _rows_cols(x)
    _check(load().fp8_quantize_current(_ptr(x), _dtype_code(x), rows, cols, fmt, margin, _ptr(scale),
                                       _ptr(scale_inv), _ptr(amax), _ptr(out), _ptr(out_t), _stream(stream)))


def fp8_quantize_dbias_workspace_bytes(rows: int, cols: int) -> int:
    return int(load().fp8_quantize_dbias_workspace_bytes(rows, cols))


def fp8_quantize_dbias(dy: torch.Tensor, fmt: int, scale: torch.Tensor, out: torch.Tensor,
                       out_t: torch.Tensor | None, dbias: torch.Tensor, workspace: torch.Tensor,
                       amax: torch.Tensor | None = None, stream=None) -> None:
    """Cast of an output gradient (+ optional transposed copy, + amax) that
    also writes the bias gradient dbias = column sums of dy, in one launch.
    `workspace` is a device buffer of at least
    fp8_quantize_dbias_workspace_bytes(rows, cols) bytes, zero-filled before
    its first use; every call leaves it zero again."""
    rows, cols = _rows_cols(dy)
    _check(load().fp8_quantize_dbias(_ptr(dy), _dtype_code(dy), rows, cols, fmt, _ptr(scale), _ptr(out),
                                     _ptr(out_t), _ptr(amax), _ptr(dbias), _dtype_code(dbias),
                                     _ptr(workspace), workspace.numel() * workspace.element_size(),
                                     _stream(stream)))


NOALLOC_DBIAS_SCRATCH_FLOATS = 1 << 20


def fp8_quantize_dbias_noalloc(dy: torch.Tensor, fmt: int, scale: torch.Tensor, out: torch.Tensor,
                               out_t: torch.Tensor, dbias: torch.Tensor, amax: torch.Tensor | None = None,
                               stream=None) -> None:
    """fp8_quantize_dbias without a workspace, for callers that cannot
    allocate device memory: the partial sums and counters live in a fixed
    4 MiB array in the library (fp8_quantize_dbias_workspace_bytes(rows, cols)
    <= 4 MiB). The first call on a device looks up that array's address;
    calls that overlap on the GPU race on it."""
    rows, cols = _rows_cols(dy)
    _check(load().fp8_quantize_dbias_noalloc(_ptr(dy), _dtype_code(dy), rows, cols, fmt, _ptr(scale), _ptr(out),
                                             _ptr(out_t), _ptr(amax), _ptr(dbias), _dtype_code(dbias),
                                             _stream(stream)))


def fp8_linear_fwd(x8: torch.Tensor, w8: torch.Tensor, sinv_x: torch.Tensor, sinv_w: torch.Tensor,
                   y: torch.Tensor, bias: torch.Tensor | None = None,
                   y_amax: torch.Tensor | None = None, stream=None) -> None:
    """y[M, N] = (x8[M, K] . w8[N, K]^T) * sinv_x * sinv_w + bias."""
    M, K = x8.shape
    N = w8.shape[0]
    _check(load().fp8_linear_fwd(_ptr(x8), _ptr(w8), M, N, K, _ptr(sinv_x), _ptr(sinv_w), _ptr(bias),
                                 _dtype_code(bias) if bias is not None else F32, _ptr(y), _dtype_code(y),
                                 _ptr(y_amax), _stream(stream)))


def fp8_linear_fwd_fp8out(x8: torch.Tensor, w8: torch.Tensor, sinv_x: torch.Tensor, sinv_w: torch.Tensor,
                          y_scale: torch.Tensor, y8: torch.Tensor, y_fmt: int = E4M3,
                          bias: torch.Tensor | None = None, y_amax: torch.Tensor | None = None,
                          stream=None) -> None:
    """y8 = FP8 codes of ((x8 . w8^T) * sinv_x * sinv_w + bias) * y_scale."""
    M, K = x8.shape
    N = w8.shape[0]
    _check(load().fp8_linear_fwd_fp8out(_ptr(x8), _ptr(w8), M, N, K, _ptr(sinv_x), _ptr(sinv_w), _ptr(bias),
                                        _dtype_code(bias) if bias is not None else F32, _ptr(y_scale), y_fmt,
                                        _ptr(y8), _ptr(y_amax), _stream(stream)))


def fp8_linear_dgrad(dy8: torch.Tensor, w8t: torch.Tensor, sinv_dy: torch.Tensor,
                     sinv_w: torch.Tensor, dx: torch.Tensor, dy_fmt: int = E5M2, stream=None) -> None:
    """dx[M, K] = (dy8[M, N] . w8t[K, N]^T) * sinv_dy * sinv_w."""
    M, N = dy8.shape
    K = w8t.shape[0]
    _check(load().fp8_linear_dgrad(_ptr(dy8), _ptr(w8t), M, N, K, dy_fmt, _ptr(sinv_dy), _ptr(sinv_w),
                                   _ptr(dx), _dtype_code(dx), _stream(stream)))


def fp8_linear_wgrad(dy8t: torch.Tensor, x8t: torch.Tensor, sinv_dy: torch.Tensor,
                     sinv_x: torch.Tensor, dw: torch.Tensor, dy_fmt: int = E5M2, stream=None) -> None:
    """dw[N, K] = (dy8t[N, M] . x8t[K, M]^T) * sinv_dy * sinv_x."""
    N, M = dy8t.shape
    K = x8t.shape[0]
    _check(load().fp8_linear_wgrad(_ptr(dy8t), _ptr(x8t), M, N, K, dy_fmt, _ptr(sinv_dy), _ptr(sinv_x),
                                   _ptr(dw), _dtype_code(dw), _stream(stream)))


def fp8_linear_bwd(dy8: torch.Tensor, dy8t: torch.Tensor, w8t: torch.Tensor, x8t: torch.Tensor,
                   sinv_dy: torch.Tensor, sinv_w: torch.Tensor, sinv_x: torch.Tensor, dx: torch.Tensor,
                   dw: torch.Tensor, dy_fmt: int = E5M2, stream=None) -> None:
    """fp8_linear_dgrad and fp8_linear_wgrad in one launch:
    dx[M, K] = (dy8 . w8t^T) * sinv_dy * sinv_w, dw[N, K] = (dy8t . x8t^T) * sinv_dy * sinv_x."""
    M, N = dy8.shape
    K = w8t.shape[0]
    _check(load().fp8_linear_bwd(_ptr(dy8), _ptr(dy8t), _ptr(w8t), _ptr(x8t), M, N, K, dy_fmt, _ptr(sinv_dy),
                                 _ptr(sinv_w), _ptr(sinv_x), _ptr(dx), _dtype_code(dx), _ptr(dw), _dtype_code(dw),
                                 _stream(stream)))


def fp8_linear_bwd_rowmajor(dy8: torch.Tensor, w8: torch.Tensor | None, x8: torch.Tensor | None,
                            sinv_dy: torch.Tensor, sinv_w: torch.Tensor | None, sinv_x: torch.Tensor | None,
                            dx: torch.Tensor | None, dw: torch.Tensor | None, dy_fmt: int = E5M2,
                            dw_nonfinite: torch.Tensor | None = None, stream=None, flags: int = 0) -> None:
    """Both backward GEMMs from the forward's row-major FP8 copies, one launch:
    dx[M, K] = (dy8 . w8) * sinv_dy * sinv_w, dw[N, K] = (dy8^T . x8) * sinv_dy * sinv_x.
    dx or dw may be None to skip that gradient. dw_nonfinite (int32[1] on the
    device) gets 1 OR-ed in when a stored element of dw is Inf or NaN. flags
    (SIGNAL_DW_DONE) selects fp8_linear_bwd_rowmajor_ex."""
    M, N = dy8.shape
    K = (w8 if w8 is not None else x8).shape[1]
    args = (_ptr(dy8), _ptr(w8), _ptr(x8), M, N, K, dy_fmt, _ptr(sinv_dy), _ptr(sinv_w), _ptr(sinv_x), _ptr(dx),
            _dtype_code(dx) if dx is not None else F32, _ptr(dw), _dtype_code(dw) if dw is not None else F32,
            _ptr(dw_nonfinite))
    if flags:
        _check(load().fp8_linear_bwd_rowmajor_ex(*args, int(flags), _stream(stream)))
    else:
        _check(load().fp8_linear_bwd_rowmajor(*args, _stream(stream)))


class Meta:
    """One tensor's delayed-scaling state in device memory (fp32)."""

    def __init__(self, history_len: int, fmt: int, device="cuda"):
        self.fmt = fmt
        self.history_len = history_len
        self.amax_history = torch.zeros(history_len, dtype=torch.float32, device=device)
        self.scale = torch.ones(1, dtype=torch.float32, device=device)
        self.scale_inv = torch.ones(1, dtype=torch.float32, device=device)
        self.cur_amax = torch.zeros(1, dtype=torch.float32, device=device)

    def c_struct(self) -> fp8mp_meta:
        return fp8mp_meta(self.amax_history.data_ptr(), self.scale.data_ptr(),
                          self.scale_inv.data_ptr(), self.cur_amax.data_ptr(),
                          self.history_len, self.fmt)


def delayed_scaling_update(metas, algo: int, margin: int = 0, stream=None,
                           prev_scale_inv: torch.Tensor | None = None) -> None:
    """Rolls each meta's history, picks the amax and refreshes scale/scale_inv.
    With prev_scale_inv (fp32[len(metas)] on the device) each meta's
    scale_inv from before the update is kept there (delayed_scaling_update_ex)."""
    metas = list(metas)
    arr = (fp8mp_meta * max(1, len(metas)))(*[m.c_struct() for m in metas])
    if prev_scale_inv is not None:
        if prev_scale_inv.numel() < len(metas) or prev_scale_inv.dtype != torch.float32:
            raise Fp8mpError(ERR_INVALID, "prev_scale_inv must be float32 with one entry per meta")
        _check(load().delayed_scaling_update_ex(arr, len(metas), algo, margin, _ptr(prev_scale_inv),
                                                _stream(stream)))
        return
    _check(load().delayed_scaling_update(arr, len(metas), algo, margin, _stream(stream)))


def mp_master_step(grad_bf16: torch.Tensor, master: torch.Tensor, momentum: torch.Tensor,
                   w8: torch.Tensor, scale_w: torch.Tensor, amax_w: torch.Tensor,
                   loss_scale: torch.Tensor, growth_tracker: torch.Tensor, found_inf: torch.Tensor,
                   lr: float, momentum_coef: float, backoff: float = 0.5, growth_factor: float = 2.0,
                   growth_interval: int = 2000, stream=None, grad_nonfinite: torch.Tensor | None = None,
                   w8_in: torch.Tensor | None = None, flags: int = 0, metas=None, amax_algo: int = AMAX_MOST_RECENT,
                   margin: int = 0) -> None:
    """Unscale, overflow skip, FP32 SGD-momentum update and E4M3 re-cast, in place.
    With grad_nonfinite (int32[1] on the device holding 0 or 1, set by the
    gradients' producer, e.g. fp8_linear_bwd_rowmajor's dw_nonfinite) the step
    reads that flag instead of scanning the gradients, writes it to found_inf
    and resets it to 0. With it, w8_in (the current E4M3 copy; the new one goes
    to w8, which a skipped step fills with w8_in) and flags
    (OVERLAP_PREVIOUS) select mp_master_step_prescanned_ex; metas (with
    amax_algo, margin; flags OVERLAP_PREVIOUS | WAIT_DW_DONE) select
    mp_master_step_prescanned_scaling_ex, which also runs the metas'
    delayed-scaling update."""
    n = grad_bf16.numel()
    if metas is not None:
        if grad_nonfinite is None:
            raise Fp8mpError(ERR_INVALID, "metas need grad_nonfinite (the prescanned step)")
        metas = list(metas)
        arr = (fp8mp_meta * max(1, len(metas)))(*[m.c_struct() for m in metas])
        _check(load().mp_master_step_prescanned_scaling_ex(
            _ptr(grad_bf16), n, _ptr(master), _ptr(momentum), _ptr(w8_in), _ptr(w8), _ptr(scale_w), _ptr(amax_w),
            _ptr(loss_scale), _ptr(growth_tracker), _ptr(found_inf), _ptr(grad_nonfinite), float(lr),
            float(momentum_coef), float(backoff), float(growth_factor), int(growth_interval), arr, len(metas),
            int(amax_algo), int(margin), int(flags), _stream(stream)))
        return
    if w8_in is not None or flags:
        if grad_nonfinite is None:
            raise Fp8mpError(ERR_INVALID, "w8_in and flags need grad_nonfinite (the prescanned step)")
        _check(load().mp_master_step_prescanned_ex(
            _ptr(grad_bf16), n, _ptr(master), _ptr(momentum), _ptr(w8_in), _ptr(w8), _ptr(scale_w), _ptr(amax_w),
            _ptr(loss_scale), _ptr(growth_tracker), _ptr(found_inf), _ptr(grad_nonfinite), float(lr),
            float(momentum_coef), float(backoff), float(growth_factor), int(growth_interval), int(flags),
            _stream(stream)))
        return
    if grad_nonfinite is not None:
        _check(load().mp_master_step_prescanned(_ptr(grad_bf16), n, _ptr(master), _ptr(momentum), _ptr(w8),
                                                _ptr(scale_w), _ptr(amax_w), _ptr(loss_scale), _ptr(growth_tracker),
                                                _ptr(found_inf), _ptr(grad_nonfinite), float(lr),
                                                float(momentum_coef), float(backoff), float(growth_factor),
                                                int(growth_interval), _stream(stream)))
        return
    _check(load().mp_master_step(_ptr(grad_bf16), n, _ptr(master), _ptr(momentum), _ptr(w8),
                                 _ptr(scale_w), _ptr(amax_w), _ptr(loss_scale), _ptr(growth_tracker),
                                 _ptr(found_inf), float(lr), float(momentum_coef), float(backoff),
                                 float(growth_factor), int(growth_interval), _stream(stream)))


def mp_master_step_adam(grad_bf16: torch.Tensor, master: torch.Tensor, exp_avg: torch.Tensor,
                        exp_avg_sq: torch.Tensor, w8: torch.Tensor, scale_w: torch.Tensor, amax_w: torch.Tensor,
                        loss_scale: torch.Tensor, growth_tracker: torch.Tensor, found_inf: torch.Tensor,
                        beta_pows: torch.Tensor, lr: float, beta1: float = 0.9, beta2: float = 0.999,
                        eps: float = 1e-8, backoff: float = 0.5, growth_factor: float = 2.0,
                        growth_interval: int = 2000, stream=None, grad_nonfinite: torch.Tensor | None = None,
                        w8_in: torch.Tensor | None = None, flags: int = 0, metas=None, amax_algo: int = AMAX_MOST_RECENT,
                        margin: int = 0) -> None:
    """Unscale, overflow skip, FP32 Adam update and E4M3 re-cast, in place
    (grad_nonfinite, w8_in, flags, metas, amax_algo, margin: as mp_master_step)."""
    n = grad_bf16.numel()
    if metas is not None:
        if grad_nonfinite is None:
            raise Fp8mpError(ERR_INVALID, "metas need grad_nonfinite (the prescanned step)")
        metas = list(metas)
        arr = (fp8mp_meta * max(1, len(metas)))(*[m.c_struct() for m in metas])
        _check(load().mp_master_step_adam_prescanned_scaling_ex(
            _ptr(grad_bf16), n, _ptr(master), _ptr(exp_avg), _ptr(exp_avg_sq), _ptr(w8_in), _ptr(w8),
            _ptr(scale_w), _ptr(amax_w), _ptr(loss_scale), _ptr(growth_tracker), _ptr(found_inf),
            _ptr(grad_nonfinite), _ptr(beta_pows), float(lr), float(beta1), float(beta2), float(eps),
            float(backoff), float(growth_factor), int(growth_interval), arr, len(metas), int(amax_algo),
            int(margin), int(flags), _stream(stream)))
        return
    if w8_in is not None or flags:
        if grad_nonfinite is None:
            raise Fp8mpError(ERR_INVALID, "w8_in and flags need grad_nonfinite (the prescanned step)")
        _check(load().mp_master_step_adam_prescanned_ex(
            _ptr(grad_bf16), n, _ptr(master), _ptr(exp_avg), _ptr(exp_avg_sq), _ptr(w8_in), _ptr(w8),
            _ptr(scale_w), _ptr(amax_w), _ptr(loss_scale), _ptr(growth_tracker), _ptr(found_inf),
            _ptr(grad_nonfinite), _ptr(beta_pows), float(lr), float(beta1), float(beta2), float(eps),
            float(backoff), float(growth_factor), int(growth_interval), int(flags), _stream(stream)))
        return
    if grad_nonfinite is not None:
        _check(load().mp_master_step_adam_prescanned(
            _ptr(grad_bf16), n, _ptr(master), _ptr(exp_avg), _ptr(exp_avg_sq), _ptr(w8), _ptr(scale_w),
            _ptr(amax_w), _ptr(loss_scale), _ptr(growth_tracker), _ptr(found_inf), _ptr(grad_nonfinite),
            _ptr(beta_pows), float(lr), float(beta1), float(beta2), float(eps), float(backoff), float(growth_factor),
            int(growth_interval), _stream(stream)))
        return
    _check(load().mp_master_step_adam(_ptr(grad_bf16), n, _ptr(master), _ptr(exp_avg), _ptr(exp_avg_sq), _ptr(w8),
                                      _ptr(scale_w), _ptr(amax_w), _ptr(loss_scale), _ptr(growth_tracker),
                                      _ptr(found_inf), _ptr(beta_pows), float(lr), float(beta1), float(beta2),
                                      float(eps), float(backoff), float(growth_factor), int(growth_interval),
                                      _stream(stream)))


def fp8mp_check(stream=None) -> int:
    """Synchronises the stream and returns the library's check code (0 = OK)."""
    return int(load().fp8mp_check(_stream(stream)))


def fp8mp_selftest_timeout(stream=None) -> None:
    """Enqueues the kernel whose bounded wait runs out (about 2 s); the next
    fp8mp_check() on the stream then returns ERR_TIMEOUT."""
    _check(load().fp8mp_selftest_timeout(_stream(stream)))


def fp8mp_selftest_barrier_timeout(stream=None) -> None:
    """Enqueues the one-block kernel whose grid-barrier wait (the master
    step's) runs out (about 2 s); the next fp8mp_check() returns ERR_TIMEOUT."""
    _check(load().fp8mp_selftest_barrier_timeout(_stream(stream)))


def fp8mp_version() -> int:
    return int(load().fp8mp_version())
