"""CPU oracle for the FP8 delayed-scaling linear layer (test infrastructure).

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package. The product path (the CUDA library and
its Python binding) never imports, links or calls it, and this package imports
nothing from the product path. The arithmetic lives in ``fp8_oracle.c``; this
file only loads that library and marshals numpy arrays into it.

Functions (each one restates a step the pages describe; the C file cites the
passage):

* ``decode(fmt, codes)`` / ``encode(fmt, x_f32)``: bit-level E4M3 / E5M2 codec.
* ``cast(x, scale, fmt)``: q = encode(fl32(x * scale)); x fp32 or bf16 bits.
* ``amax(x)``: max |x| ignoring NaN, from +0.
* ``transpose_u8(q)``: the transposed copy.
* ``scale_update(hist, scale, scale_inv, cur_amax, fmt, algo, margin)``.
* ``gemm_ref(A, fa, B, fb, sinv_a, sinv_b, bias, rows)``: fp64 reference.
* ``master_step(...)``: unscale, overflow skip, SGD-momentum, E4M3 re-cast.
* ``dbias(dy)``: the bias gradient (fp64 column sums) and column abs sums.
* ``adam_step(...)``: the Adam variant of the master step.
* ``cast_current(x, fmt, margin)``: just-in-time scaling then the cast.
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import sys

import numpy as np

E4M3, E5M2 = 0, 1
AMAX_MAX, AMAX_MOST_RECENT = 0, 1

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "fp8_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lib = None


def build(force: bool = False, quiet: bool = True) -> str:
    """Compile fp8_oracle.c into liboracle.so with gcc (OpenMP when present)."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    base = ["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
            "-shared", _SRC, "-o", _LIB_PATH + ".tmp", "-lm"]
    for extra in (["-fopenmp"], []):
        r = subprocess.run(base[:1] + extra + base[1:], capture_output=True, text=True)
        if r.returncode == 0:
            os.replace(_LIB_PATH + ".tmp", _LIB_PATH)
            return _LIB_PATH
        if not quiet:
            print(r.stderr, file=sys.stderr)
    raise RuntimeError("could not compile the oracle: " + r.stderr)


def _bind(path: str):
    L = ctypes.CDLL(path)
    P, I64, I32, F, D = (ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32,
                         ctypes.c_float, ctypes.c_double)
    L.orc_decode.restype = D
    L.orc_decode.argtypes = [ctypes.c_int, ctypes.c_uint8]
    L.orc_encode.restype = ctypes.c_uint8
    L.orc_encode.argtypes = [ctypes.c_int, F]
    L.orc_fmt_max.restype = D
    L.orc_fmt_max.argtypes = [ctypes.c_int]
    L.orc_num_threads.restype = ctypes.c_int
    L.orc_cast_f32.argtypes = [P, I64, F, ctypes.c_int, P]
    L.orc_cast_bf16.argtypes = [P, I64, F, ctypes.c_int, P]
    L.orc_transpose_u8.argtypes = [P, I64, I64, P]
    L.orc_amax_f32.restype = F
    L.orc_amax_f32.argtypes = [P, I64]
    L.orc_amax_bf16.restype = F
    L.orc_amax_bf16.argtypes = [P, I64]
    L.orc_scale_update.argtypes = [P, I32, P, P, P, ctypes.c_int, ctypes.c_int, I32]
    L.orc_gemm_ref.argtypes = [P, ctypes.c_int, P, ctypes.c_int, I64, I64, I64, P, I64, D, D,
                               P, P, P]
    L.orc_master_step.argtypes = [P, I64, P, P, P, F, P, P, P, P, F, F, F, F, I32]
    L.orc_dbias.argtypes = [P, ctypes.c_int, I64, I64, P, P]
    L.orc_adam_step.argtypes = [P, I64, P, P, P, P, F, P, P, P, P, P, P, F, F, F, F, F, F, I32]
    return L


def lib():
    global _lib
    if _lib is None:
        build()
        _lib = _bind(_LIB_PATH)
    return _lib


class swapped_library:
    """Context manager: route every call through another build of the oracle
    (used by the mutation test, which compiles planted mistakes)."""

    def __init__(self, path: str):
        self.path = path

    def __enter__(self):
        global _lib
        self.saved = lib()
        _lib = _bind(self.path)
        return self

    def __exit__(self, *exc):
        global _lib
        _lib = self.saved
        return False


def num_threads() -> int:
    return int(lib().orc_num_threads())


def _ptr(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"], "oracle inputs must be C-contiguous"
    return a.ctypes.data_as(ctypes.c_void_p)


def fmt_max(fmt: int) -> float:
    return float(lib().orc_fmt_max(fmt))


def decode(fmt: int, codes) -> np.ndarray:
    codes = np.asarray(codes, dtype=np.uint8)
    L = lib()
    out = np.empty(codes.shape, dtype=np.float64)
    flat_in, flat_out = codes.reshape(-1), out.reshape(-1)
    for i in range(flat_in.size):
        flat_out[i] = L.orc_decode(fmt, int(flat_in[i]))
    return out


def encode(fmt: int, x) -> np.ndarray:
    """Encode fp32 values (no scale); the same as cast(x, 1.0, fmt)."""
    x = np.ascontiguousarray(np.asarray(x, dtype=np.float32))
    return cast(x, 1.0, fmt)


def cast(x: np.ndarray, scale: float, fmt: int) -> np.ndarray:
    """q = encode(fl32(x * scale)); x is float32, or uint16 holding bf16 bits."""
    x = np.ascontiguousarray(x)
    q = np.empty(x.shape, dtype=np.uint8)
    if x.dtype == np.float32:
        lib().orc_cast_f32(_ptr(x), x.size, ctypes.c_float(scale), fmt, _ptr(q))
    elif x.dtype in (np.uint16, np.int16):
        lib().orc_cast_bf16(_ptr(x), x.size, ctypes.c_float(scale), fmt, _ptr(q))
    else:
        raise TypeError(f"unsupported input dtype {x.dtype}")
    return q


def transpose_u8(q: np.ndarray) -> np.ndarray:
    q = np.ascontiguousarray(q)
    rows, cols = q.shape
    qt = np.empty((cols, rows), dtype=np.uint8)
    lib().orc_transpose_u8(_ptr(q), rows, cols, _ptr(qt))
    return qt


def amax(x: np.ndarray) -> np.float32:
    x = np.ascontiguousarray(x)
    if x.dtype == np.float32:
        return np.float32(lib().orc_amax_f32(_ptr(x), x.size))
    if x.dtype in (np.uint16, np.int16):
        return np.float32(lib().orc_amax_bf16(_ptr(x), x.size))
    raise TypeError(f"unsupported input dtype {x.dtype}")


class Meta:
    """One tensor's delayed-scaling state on the host (all fp32)."""

    def __init__(self, history_len: int):
        self.hist = np.zeros(history_len, dtype=np.float32)
        self.scale = np.ones(1, dtype=np.float32)
        self.scale_inv = np.ones(1, dtype=np.float32)
        self.cur_amax = np.zeros(1, dtype=np.float32)

    def copy(self) -> "Meta":
        m = Meta(self.hist.size)
        m.hist[:] = self.hist
        m.scale[:] = self.scale
        m.scale_inv[:] = self.scale_inv
        m.cur_amax[:] = self.cur_amax
        return m

    def record_amax(self, a) -> None:
        """cur_amax = max(cur_amax, a): what the cast's amax output does."""
        a = np.float32(a)
        if a > self.cur_amax[0]:
            self.cur_amax[0] = a


def scale_update(meta: Meta, fmt: int, algo: int, margin: int) -> Meta:
    lib().orc_scale_update(_ptr(meta.hist), meta.hist.size, _ptr(meta.scale), _ptr(meta.scale_inv),
                           _ptr(meta.cur_amax), fmt, algo, margin)
    return meta


def gemm_ref(A: np.ndarray, fmt_a: int, B: np.ndarray, fmt_b: int, sinv_a: float, sinv_b: float,
             bias: np.ndarray | None = None, rows: np.ndarray | None = None,
             with_abs: bool = True):
    """fp64 reference of (A_dec @ B_dec.T) * sinv_a * sinv_b + bias.

    A is (rows_a, kc) and B is (rows_b, kc) uint8 codes. ``rows`` selects rows
    of A (all when None). Returns (ref, abs_sum) with shapes (len(rows), rows_b).
    """
    A = np.ascontiguousarray(A, dtype=np.uint8)
    B = np.ascontiguousarray(B, dtype=np.uint8)
    rows_a, kc = A.shape
    rows_b, kc2 = B.shape
    assert kc == kc2
    if rows is None:
        idx_p, n_rows = None, rows_a
    else:
        rows = np.ascontiguousarray(rows, dtype=np.int64)
        idx_p, n_rows = _ptr(rows), rows.size
    out = np.empty((n_rows, rows_b), dtype=np.float64)
    abs_out = np.empty((n_rows, rows_b), dtype=np.float64) if with_abs else None
    if bias is not None:
        bias = np.ascontiguousarray(bias, dtype=np.float64)
        assert bias.size == rows_b
    lib().orc_gemm_ref(_ptr(A), fmt_a, _ptr(B), fmt_b, rows_a, rows_b, kc, idx_p, n_rows,
                       ctypes.c_double(sinv_a), ctypes.c_double(sinv_b),
                       _ptr(bias) if bias is not None else None, _ptr(out),
                       _ptr(abs_out) if abs_out is not None else None)
    return out, abs_out


def dbias(dy: np.ndarray):
    """(column sums, column abs sums) in fp64; dy is float32 or bf16 bits."""
    dy = np.ascontiguousarray(dy)
    rows, cols = dy.shape
    out = np.empty(cols, dtype=np.float64)
    ab = np.empty(cols, dtype=np.float64)
    is_bf16 = 1 if dy.dtype in (np.uint16, np.int16) else 0
    assert is_bf16 or dy.dtype == np.float32
    lib().orc_dbias(_ptr(dy), is_bf16, rows, cols, _ptr(out), _ptr(ab))
    return out, ab


def cast_current(x: np.ndarray, fmt: int, margin: int = 0, scale0: float = 1.0):
    """Just-in-time scaling: amax of this tensor, the scale rule on a one-entry
    history (most_recent), then the cast. Returns (codes, meta)."""
    m = Meta(1)
    m.scale[0] = scale0
    m.record_amax(amax(x))
    a = np.float32(m.cur_amax[0])
    scale_update(m, fmt, AMAX_MOST_RECENT, margin)
    m.cur_amax[0] = a  # report this tensor's amax, as the cast does
    return cast(x, float(m.scale[0]), fmt), m


class AdamState:
    """Adam's beta powers beta1^(t-1), beta2^(t-1) (both start at 1)."""

    def __init__(self):
        self.b1p = np.ones(1, dtype=np.float32)
        self.b2p = np.ones(1, dtype=np.float32)


def adam_step(g_bits, w, m, v, w8, scale_w, cur_amax_w, st, ad: AdamState, lr, beta1=0.9, beta2=0.999,
              eps=1e-8, backoff=0.5, growth_factor=2.0, growth_interval=2000):
    """In-place reference of one Adam master step (w, m, v, w8, amax, st, ad)."""
    n = g_bits.size
    for a in (w, m, v):
        assert a.dtype == np.float32 and a.size == n and a.flags["C_CONTIGUOUS"]
    lib().orc_adam_step(_ptr(g_bits), n, _ptr(w), _ptr(m), _ptr(v), _ptr(w8), ctypes.c_float(scale_w),
                        _ptr(cur_amax_w), _ptr(st.S), _ptr(st.growth), _ptr(st.found_inf), _ptr(ad.b1p),
                        _ptr(ad.b2p), ctypes.c_float(lr), ctypes.c_float(beta1), ctypes.c_float(beta2),
                        ctypes.c_float(eps), ctypes.c_float(backoff), ctypes.c_float(growth_factor),
                        int(growth_interval))


class LossScaleState:
    def __init__(self, S: float = 2.0 ** 16, growth: int = 0):
        self.S = np.array([S], dtype=np.float32)
        self.growth = np.array([growth], dtype=np.int32)
        self.found_inf = np.zeros(1, dtype=np.int32)


def master_step(g_bits: np.ndarray, w: np.ndarray, v: np.ndarray, w8: np.ndarray, scale_w: float,
                cur_amax_w: np.ndarray, st: LossScaleState, lr: float, mu: float,
                backoff: float = 0.5, growth_factor: float = 2.0,
                growth_interval: int = 2000) -> None:
    """In-place reference of one master step (w, v, w8, cur_amax_w, st)."""
    for a, dt in ((g_bits, (np.uint16, np.int16)), (w, (np.float32,)), (v, (np.float32,)),
                  (w8, (np.uint8,)), (cur_amax_w, (np.float32,))):
        assert a.dtype in dt and a.flags["C_CONTIGUOUS"]
    n = g_bits.size
    assert w.size == n and v.size == n and w8.size == n
    lib().orc_master_step(_ptr(g_bits), n, _ptr(w), _ptr(v), _ptr(w8), ctypes.c_float(scale_w),
                          _ptr(cur_amax_w), _ptr(st.S), _ptr(st.growth), _ptr(st.found_inf),
                          ctypes.c_float(lr), ctypes.c_float(mu), ctypes.c_float(backoff),
                          ctypes.c_float(growth_factor), int(growth_interval))
