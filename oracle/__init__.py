"""CPU oracle for the NVFP4 training quantizer -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` may import this package.  The product
path (``tensor_quantization_gb300``) never imports it and shares no code with it.

The arithmetic lives in ``nvfp4_oracle.c`` (plain single-threaded C, fp32 IEEE,
no FMA contraction); this module compiles it with gcc on first use and wraps it
with ctypes.  Inputs are numpy arrays: bf16 data is passed as its uint16 bit
pattern, fp32 as float32.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from concurrent.futures import ThreadPoolExecutor

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "nvfp4_oracle.c")
_SO = os.path.join(_HERE, "_liboracle.so")
_LOCK = threading.Lock()
_LIB = None

MODES = {"rne": 0, "sr": 1, "4o6": 2}


def build(force: bool = False) -> str:
    """Compile the oracle into ``oracle/_liboracle.so`` (gcc, no fast math)."""
    with _LOCK:
        fresh = os.path.exists(_SO) and os.path.getmtime(_SO) >= os.path.getmtime(_SRC)
        if force or not fresh:
            tmp = _SO + f".{os.getpid()}.tmp"
            cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math",
                   "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"]
            subprocess.run(cmd, check=True)
            os.replace(tmp, _SO)
    return _SO


def _lib():
    global _LIB
    if _LIB is None:
        lib = ctypes.CDLL(build())
        i64, i32, u32, u64, vp = ctypes.c_int64, ctypes.c_int, ctypes.c_uint32, ctypes.c_uint64, ctypes.c_void_p
        lib.ora_quantize.argtypes = [vp, i32, i64, i64, i64, i32, i32, i32, i32, i32, i32, u32,
                                     u64, u64, i64, i64, vp, vp, vp, vp, vp, u64]
        lib.ora_quantize.restype = i32
        lib.ora_dequantize.argtypes = [vp, vp, vp, i64, i64, i32, i32, vp, i32]
        lib.ora_dequantize.restype = i32
        lib.ora_amax.argtypes = [vp, i32, i64, i64, i64, i32, i32, u32, i32, vp, vp]
        lib.ora_amax.restype = i32
        lib.ora_e2m1_value.argtypes = [i32]
        lib.ora_e2m1_value.restype = ctypes.c_float
        lib.ora_e2m1_rne.argtypes = [ctypes.c_float]
        lib.ora_e2m1_rne.restype = i32
        lib.ora_e2m1_sr.argtypes = [ctypes.c_float, ctypes.c_uint]
        lib.ora_e2m1_sr.restype = i32
        lib.ora_e4m3_value.argtypes = [ctypes.c_uint]
        lib.ora_e4m3_value.restype = ctypes.c_float
        lib.ora_e4m3_rn.argtypes = [ctypes.c_float]
        lib.ora_e4m3_rn.restype = ctypes.c_uint
        lib.ora_philox4x32_10.argtypes = [vp, vp, vp]
        lib.ora_philox4x32_10.restype = None
        lib.ora_rht16.argtypes = [vp, u32]
        lib.ora_rht16.restype = None
        lib.ora_swizzle_offset.argtypes = [i64, i64, i64]
        lib.ora_swizzle_offset.restype = i64
        lib.ora_scale_bytes.argtypes = [i64, i64, i32]
        lib.ora_scale_bytes.restype = i64
        lib.ora_e2m1_rne_n.argtypes = [vp, i64, vp]
        lib.ora_e2m1_rne_n.restype = None
        lib.ora_e2m1_sr_n.argtypes = [vp, vp, i64, vp]
        lib.ora_e2m1_sr_n.restype = None
        lib.ora_e4m3_rn_n.argtypes = [vp, i64, vp]
        lib.ora_e4m3_rn_n.restype = None
        lib.ora_inverse_rht16.argtypes = [vp, u32]
        lib.ora_inverse_rht16.restype = None
        lib.ora_dequantize_rht.argtypes = [vp, vp, vp, i64, i64, i32, i32, u32, vp, i32]
        lib.ora_dequantize_rht.restype = i32
        lib.ora_candidate_error_n.argtypes = [vp, vp, vp, vp, i64, vp]
        lib.ora_candidate_error_n.restype = None
        lib.ora_f32_to_bf16.argtypes = [ctypes.c_float]
        lib.ora_f32_to_bf16.restype = ctypes.c_uint16
        _LIB = lib
    return _LIB


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _input(x: np.ndarray):
    if x.ndim != 2:
        raise ValueError("oracle input must be 2-D")
    if x.dtype == np.uint16:
        dtype = 0
    elif x.dtype == np.float32:
        dtype = 1
    else:
        raise ValueError("oracle input must be uint16 (bf16 bits) or float32")
    if x.strides[1] != x.itemsize or x.strides[0] % x.itemsize:
        x = np.ascontiguousarray(x)
    ld = x.strides[0] // x.itemsize if x.shape[0] > 1 else x.shape[1]
    return x, dtype, ld


def scale_bytes(rows_out: int, cols_out: int, swizzled: bool) -> int:
    return int(_lib().ora_scale_bytes(rows_out, cols_out, int(swizzled)))


def quantize(x: np.ndarray, *, colwise: bool = False, mode: str = "rne", block2d: bool = False,
             per_row: bool = False, swizzled: bool = False, rht: bool = False, sign_mask: int = 0,
             seed: int = 0, offset: int = 0, row_range: tuple[int, int] | None = None,
             amax_given: float | None = None, block_base: int = 0) -> dict:
    """Quantize one orientation of ``x``; returns codes, scales, amax, global_scale.

    ``colwise`` works on X^T.  ``row_range`` restricts encoding to output rows
    [r0, r1) (the per-tensor amax still covers the whole tensor); rows outside
    the range are left zero.  ``amax_given`` replaces the per-tensor amax.
    ``block_base`` is added to every block number of the Philox counter: the
    number of this input's first block when it is a shard of a larger tensor.
    """
    x, dtype, ld = _input(x)
    rows, cols = x.shape
    R, C = (cols, rows) if colwise else (rows, cols)
    r0, r1 = row_range if row_range is not None else (0, R)
    codes = np.zeros((R, C // 2), np.uint8)
    scales = np.zeros(scale_bytes(R, C, swizzled), np.uint8)
    n_g = R if per_row else 1
    amax = np.zeros(n_g, np.float32)
    gs = np.zeros(n_g, np.float32)
    given = None if amax_given is None else np.array([amax_given], np.float32)
    rc = _lib().ora_quantize(_ptr(x), dtype, rows, cols, ld, int(colwise), MODES[mode], int(block2d),
                             int(per_row), int(swizzled), int(rht), sign_mask & 0xFFFF, seed, offset,
                             r0, r1, None if given is None else _ptr(given),
                             _ptr(codes), _ptr(scales), _ptr(amax), _ptr(gs), block_base)
    if rc != 0:
        raise ValueError(f"oracle quantize rejected the arguments (status {rc})")
    if not swizzled:
        scales = scales.reshape(R, C // 16)
    return {"codes": codes, "scales": scales, "amax": amax, "global_scale": gs}


def host_threads() -> int:
    """Host cores this process may run on."""
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def amax_parallel(x: np.ndarray, *, colwise: bool = False, rht: bool = False, sign_mask: int = 0,
                  threads: int | None = None) -> float:
    """The per-tensor amax of ``amax`` computed on slices in parallel threads:
    row ranges for rowwise blocks, column ranges for columnwise ones (so every
    block lies in one slice), combined by the same unsigned maximum of magnitude
    bits, hence equal to the single call bit for bit (NaN included)."""
    x, _, _ = _input(x)
    rows, cols = x.shape
    n = max(1, min(threads or host_threads(), (cols if colwise else rows)))
    cuts = np.linspace(0, cols if colwise else rows, n + 1).astype(int)

    def one(i):
        part = x[:, cuts[i]:cuts[i + 1]] if colwise else x[cuts[i]:cuts[i + 1]]
        return amax(part, colwise=colwise, rht=rht, sign_mask=sign_mask)[0]

    with ThreadPoolExecutor(n) as ex:
        parts = [p for p in ex.map(one, range(n)) if p.size]
    bits = max(int(p.view(np.uint32)[0]) & 0x7FFFFFFF for p in parts)
    return float(np.array([bits], np.uint32).view(np.float32)[0])


def quantize_parallel(x: np.ndarray, *, threads: int | None = None, colwise: bool = False, mode: str = "rne",
                      block2d: bool = False, per_row: bool = False, swizzled: bool = False, rht: bool = False,
                      sign_mask: int = 0, seed: int = 0, offset: int = 0,
                      amax_given: float | None = None, row_range: tuple[int, int] | None = None) -> dict:
    """``quantize`` of the whole tensor with its output rows split over threads.

    Orchestration only (the arithmetic is the same C code): the per-tensor
    amax comes from ``amax_parallel`` (or ``amax_given``), then each thread
    encodes a range of output rows into the shared code and scale arrays (whole
    16-row bands in 2D mode; only ``row_range`` if given, as ``quantize``).  An
    output row depends only on the input, the global scale and its own Philox
    blocks, so the result equals a single call bit for bit."""
    x, dtype, ld = _input(x)
    rows, cols = x.shape
    R, C = (cols, rows) if colwise else (rows, cols)
    n = threads or host_threads()
    if not per_row and amax_given is None:
        amax_given = amax_parallel(x, colwise=colwise, rht=rht, sign_mask=sign_mask, threads=n)
    codes = np.zeros((R, C // 2), np.uint8)
    scales = np.zeros(scale_bytes(R, C, swizzled), np.uint8)
    n_g = R if per_row else 1
    amax_out = np.zeros(n_g, np.float32)
    gs_out = np.zeros(n_g, np.float32)
    step = 16 if block2d else 1
    lo, hi = row_range if row_range is not None else (0, R)
    units = (hi - lo) // step
    cuts = (lo + np.linspace(0, units, max(1, min(units, 4 * n)) + 1).astype(int) * step).tolist()
    given = None if amax_given is None else np.array([amax_given], np.float32)
    lib = _lib()

    def one(i):
        r0, r1 = cuts[i], cuts[i + 1]
        a, g = (amax_out, gs_out) if per_row else (np.zeros(1, np.float32), np.zeros(1, np.float32))
        rc = lib.ora_quantize(_ptr(x), dtype, rows, cols, ld, int(colwise), MODES[mode], int(block2d),
                              int(per_row), int(swizzled), int(rht), sign_mask & 0xFFFF, seed, offset,
                              r0, r1, None if given is None else _ptr(given),
                              _ptr(codes), _ptr(scales), _ptr(a), _ptr(g), 0)
        return rc, a, g

    with ThreadPoolExecutor(n) as ex:
        results = list(ex.map(one, range(len(cuts) - 1)))
    for rc, _, _ in results:
        if rc != 0:
            raise ValueError(f"oracle quantize rejected the arguments (status {rc})")
    if not per_row:
        amax_out[:], gs_out[:] = results[0][1], results[0][2]
    if not swizzled:
        scales = scales.reshape(R, C // 16)
    return {"codes": codes, "scales": scales, "amax": amax_out, "global_scale": gs_out}


def dequantize(codes: np.ndarray, scales: np.ndarray, global_scale: np.ndarray, rows: int, cols: int,
               *, swizzled: bool = False, per_row: bool = False, out_dtype: str = "fp32") -> np.ndarray:
    codes = np.ascontiguousarray(codes, np.uint8)
    scales = np.ascontiguousarray(scales, np.uint8)
    gsc = np.ascontiguousarray(global_scale, np.float32)
    out = np.zeros((rows, cols), np.uint16 if out_dtype == "bf16" else np.float32)
    rc = _lib().ora_dequantize(_ptr(codes), _ptr(scales), _ptr(gsc), rows, cols, int(swizzled),
                               int(per_row), _ptr(out), 0 if out_dtype == "bf16" else 1)
    if rc != 0:
        raise ValueError(f"oracle dequantize rejected the arguments (status {rc})")
    return out


def amax(x: np.ndarray, *, colwise: bool = False, rht: bool = False, sign_mask: int = 0,
         per_row: bool = False) -> tuple[np.ndarray, np.ndarray]:
    x, dtype, ld = _input(x)
    rows, cols = x.shape
    R = cols if colwise else rows
    n = R if per_row else 1
    a = np.zeros(n, np.float32)
    g = np.zeros(n, np.float32)
    rc = _lib().ora_amax(_ptr(x), dtype, rows, cols, ld, int(colwise), int(rht), sign_mask & 0xFFFF,
                         int(per_row), _ptr(a), _ptr(g))
    if rc != 0:
        raise ValueError(f"oracle amax rejected the arguments (status {rc})")
    return a, g


# ---- scalar building blocks (exposed for the pin tests) ----
def e2m1_value(code: int) -> float:
    return float(_lib().ora_e2m1_value(code))


def e2m1_rne(q: float) -> int:
    return int(_lib().ora_e2m1_rne(q))


def e2m1_sr(q: float, r: int) -> int:
    return int(_lib().ora_e2m1_sr(q, r))


def e4m3_value(b: int) -> float:
    return float(_lib().ora_e4m3_value(b))


def e4m3_rn(s: float) -> int:
    return int(_lib().ora_e4m3_rn(s))


def philox4x32_10(ctr, key) -> list[int]:
    c = np.array(ctr, np.uint32)
    k = np.array(key, np.uint32)
    o = np.zeros(4, np.uint32)
    _lib().ora_philox4x32_10(_ptr(c), _ptr(k), _ptr(o))
    return [int(v) for v in o]


def rht16(v, sign_mask: int) -> np.ndarray:
    a = np.array(v, np.float32).copy()
    _lib().ora_rht16(_ptr(a), sign_mask & 0xFFFF)
    return a


def swizzle_offset(r: int, j: int, cs_padded: int) -> int:
    return int(_lib().ora_swizzle_offset(r, j, cs_padded))


def f32_to_bf16(f: float) -> int:
    return int(_lib().ora_f32_to_bf16(f))


def e2m1_rne_array(q: np.ndarray) -> np.ndarray:
    q = np.ascontiguousarray(q, np.float32)
    out = np.zeros(q.size, np.uint8)
    _lib().ora_e2m1_rne_n(_ptr(q), q.size, _ptr(out))
    return out


def e2m1_sr_array(q: np.ndarray, r: np.ndarray) -> np.ndarray:
    q = np.ascontiguousarray(q, np.float32)
    r = np.ascontiguousarray(r, np.uint8)
    out = np.zeros(q.size, np.uint8)
    _lib().ora_e2m1_sr_n(_ptr(q), _ptr(r), q.size, _ptr(out))
    return out


def e4m3_rn_array(s: np.ndarray) -> np.ndarray:
    s = np.ascontiguousarray(s, np.float32)
    out = np.zeros(s.size, np.uint8)
    _lib().ora_e4m3_rn_n(_ptr(s), s.size, _ptr(out))
    return out


def candidate_error_array(y: np.ndarray, codes: np.ndarray, S: np.ndarray, g: np.ndarray) -> np.ndarray:
    """Four-over-six squared-error of each 16-value block (y [n,16], codes
    [n,16] 4-bit, block scale bytes S [n], global scales g [n])."""
    y = np.ascontiguousarray(y, np.float32).reshape(-1, 16)
    codes = np.ascontiguousarray(codes, np.int32).reshape(-1, 16)
    S = np.ascontiguousarray(S, np.uint32).ravel()
    g = np.ascontiguousarray(g, np.float32).ravel()
    out = np.zeros(len(y), np.float32)
    _lib().ora_candidate_error_n(_ptr(y), _ptr(codes), _ptr(S), _ptr(g), len(y), _ptr(out))
    return out


def inverse_rht16(y, sign_mask: int) -> np.ndarray:
    """Inverse of rht16: signs on the inputs, the butterfly, then x 0.25."""
    y = np.ascontiguousarray(y, np.float32).copy()
    _lib().ora_inverse_rht16(_ptr(y), sign_mask & 0xFFFF)
    return y


def dequantize_rht(codes: np.ndarray, scales: np.ndarray, global_scale: np.ndarray, rows: int, cols: int, *,
                   sign_mask: int, swizzled: bool = False, per_row: bool = False,
                   out_dtype: str = "fp32") -> np.ndarray:
    """Standard decode followed by the inverse RHT of every 16-block."""
    codes = np.ascontiguousarray(codes, np.uint8)
    scales = np.ascontiguousarray(scales, np.uint8)
    gs = np.ascontiguousarray(global_scale, np.float32)
    out = np.zeros((rows, cols), np.uint16 if out_dtype == "bf16" else np.float32)
    rc = _lib().ora_dequantize_rht(_ptr(codes), _ptr(scales), _ptr(gs), rows, cols, int(swizzled), int(per_row),
                                   sign_mask & 0xFFFF, _ptr(out), 0 if out_dtype == "bf16" else 1)
    if rc != 0:
        raise ValueError(f"ora_dequantize_rht failed ({rc})")
    return out
