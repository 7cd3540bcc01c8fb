"""Python binding of libnvfp4.so (include/nvfp4.h): argument marshalling only.

The functions named ``nvfp4_*`` mirror the C entry points one to one; they take
torch CUDA tensors for the buffers, pass their device pointers and the current
(or given) CUDA stream, and raise ``NVFP4Error`` on a non-OK status.  Every
step of the computation runs in the library's kernels.  There is no fallback:
if the library cannot be loaded, every call raises.

``quantize`` / ``dequantize`` are conveniences that allocate the outputs with
torch (device memory only) and call the matching entry point.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass

import torch

_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libnvfp4.so")
_lib = None

OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_CUDA, ERR_TIMEOUT = 0, 1, 2, 3, 4
IN_BF16, IN_FP32 = 0, 1
ROWWISE, COLWISE, BLOCK_2D, SCALE_PER_ROW, SWIZZLED, AMAX_GIVEN, FAST_MATH = 1, 2, 4, 8, 16, 32, 64


class NVFP4Error(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_string(status)} (status {status})")


class Input(ctypes.Structure):
    _fields_ = [("x", ctypes.c_void_p), ("dtype", ctypes.c_int32), ("rows", ctypes.c_int64),
                ("cols", ctypes.c_int64), ("ld", ctypes.c_int64), ("row0", ctypes.c_int64),
                ("col0", ctypes.c_int64)]


class Output(ctypes.Structure):
    _fields_ = [("codes_row", ctypes.c_void_p), ("scales_row", ctypes.c_void_p),
                ("codes_col", ctypes.c_void_p), ("scales_col", ctypes.c_void_p),
                ("amax", ctypes.c_void_p), ("global_scale", ctypes.c_void_p)]


EXPORTS = ("nvfp4_workspace_bytes", "nvfp4_scale_bytes", "nvfp4_amax", "nvfp4_quantize_rne",
           "nvfp4_quantize_sr", "nvfp4_quantize_rht_sr", "nvfp4_quantize_four_over_six",
           "nvfp4_dequantize", "nvfp4_status_string", "nvfp4_quantize_rht_sr_static", "nvfp4_quantize_grouped",
           "nvfp4_dequantize_rht", "nvfp4_workspace_status", "nvfp4_set_wait_limit")
MODE_RNE, MODE_SR, MODE_RHT_SR, MODE_FOUR_OVER_SIX = 0, 1, 2, 3


def lib_path() -> str:
    return _LIB_PATH


def load(path: str | None = None):
    """Load libnvfp4.so (raises OSError if it is missing or unloadable)."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or _LIB_PATH
    if not os.path.exists(p):
        raise OSError(f"libnvfp4.so not found at {p}; build it with "
                      "`python -m tensor_quantization_gb300.build`")
    L = ctypes.CDLL(p)
    vp, u32, u64, i32, i64 = ctypes.c_void_p, ctypes.c_uint32, ctypes.c_uint64, ctypes.c_int32, ctypes.c_int64
    PI, PO = ctypes.POINTER(Input), ctypes.POINTER(Output)
    L.nvfp4_workspace_bytes.argtypes = []
    L.nvfp4_workspace_bytes.restype = ctypes.c_size_t
    L.nvfp4_scale_bytes.argtypes = [i64, i64, u32]
    L.nvfp4_scale_bytes.restype = ctypes.c_size_t
    L.nvfp4_amax.argtypes = [PI, u32, ctypes.c_int, ctypes.c_uint16, PO, vp, vp]
    L.nvfp4_quantize_rne.argtypes = [PI, u32, PO, vp, vp]
    L.nvfp4_quantize_sr.argtypes = [PI, u32, u64, u64, PO, vp, vp]
    L.nvfp4_quantize_rht_sr.argtypes = [PI, u32, ctypes.c_uint16, u64, u64, PO, vp, vp]
    L.nvfp4_quantize_four_over_six.argtypes = [PI, u32, PO, vp, vp]
    L.nvfp4_quantize_rht_sr_static.argtypes = [PI, u32, ctypes.c_uint16, u64, u64, PO, vp]
    L.nvfp4_dequantize.argtypes = [vp, vp, vp, i64, i64, u32, vp, i32, vp]
    L.nvfp4_quantize_grouped.argtypes = [PI, u32, vp, i64, i32, ctypes.c_uint16, u64, u64, PO, vp]
    L.nvfp4_dequantize_rht.argtypes = [vp, vp, vp, i64, i64, u32, ctypes.c_uint16, vp, i32, vp]
    L.nvfp4_workspace_status.argtypes = [vp, vp]
    L.nvfp4_set_wait_limit.argtypes = [i64]
    for f in ("nvfp4_amax", "nvfp4_quantize_rne", "nvfp4_quantize_sr", "nvfp4_quantize_rht_sr",
              "nvfp4_quantize_four_over_six", "nvfp4_dequantize", "nvfp4_quantize_rht_sr_static",
              "nvfp4_quantize_grouped", "nvfp4_dequantize_rht", "nvfp4_workspace_status",
              "nvfp4_set_wait_limit"):
        getattr(L, f).restype = ctypes.c_int
    L.nvfp4_status_string.argtypes = [ctypes.c_int]
    L.nvfp4_status_string.restype = ctypes.c_char_p
    if path is None:
        _lib = L
    return L


def status_string(status: int) -> str:
    return load().nvfp4_status_string(status).decode()


# ----------------------------------------------------------- marshalling
def _ptr(t: torch.Tensor | None):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if isinstance(stream, torch.cuda.Stream) else int(stream))


def make_input(x: torch.Tensor, row0: int = 0, col0: int = 0) -> Input:
    """The C input descriptor of a 2-D tensor; (row0, col0) is its position in
    the full tensor when it is a shard (Philox block numbering only)."""
    if x.dim() != 2:
        raise ValueError("input must be 2-D")
    if x.dtype == torch.bfloat16:
        dt = IN_BF16
    elif x.dtype == torch.float32:
        dt = IN_FP32
    else:
        raise ValueError("input must be bfloat16 or float32")
    if x.numel() and x.stride(1) != 1:
        raise ValueError("input rows must be contiguous (stride(1) == 1)")
    per16 = 16 // x.element_size()
    # a single row has no meaningful pitch: report the row length rounded up
    ld = x.stride(0) if x.size(0) > 1 else (x.size(1) + per16 - 1) // per16 * per16
    return Input(x.data_ptr() if x.numel() else None, dt, x.size(0), x.size(1), ld, row0, col0)


def make_output(codes_row=None, scales_row=None, codes_col=None, scales_col=None, amax=None,
                global_scale=None) -> Output:
    return Output(*(_ptr(t) for t in (codes_row, scales_row, codes_col, scales_col, amax, global_scale)))


def _input(x) -> Input:
    return x if isinstance(x, Input) else make_input(x)


def _check(status: int, what: str) -> None:
    if status != OK:
        raise NVFP4Error(status, what)


# ------------------------------------------------ one-to-one entry points
def nvfp4_workspace_bytes() -> int:
    return int(load().nvfp4_workspace_bytes())


def nvfp4_scale_bytes(rows_out: int, cols_out: int, flags: int) -> int:
    return int(load().nvfp4_scale_bytes(rows_out, cols_out, flags))


def nvfp4_workspace_status(workspace, stream=None) -> int:
    """The workspace's failure record: OK, or ERR_TIMEOUT (then cleared) if a
    bounded device-side wait of an earlier call gave up.  Waits for the stream."""
    st = load().nvfp4_workspace_status(_ptr(workspace), _stream(stream))
    if st not in (OK, ERR_TIMEOUT):
        raise NVFP4Error(st, "nvfp4_workspace_status")
    return st


def nvfp4_set_wait_limit(polls: int) -> None:
    """Bound of the device-side waits on other CTAs for later calls (< 0: default)."""
    _check(load().nvfp4_set_wait_limit(polls), "nvfp4_set_wait_limit")


def nvfp4_amax(x, flags, use_rht, sign_mask, out: Output, workspace, stream=None) -> None:
    _check(load().nvfp4_amax(ctypes.byref(_input(x)), flags, int(use_rht), sign_mask & 0xFFFF,
                             ctypes.byref(out), _ptr(workspace), _stream(stream)), "nvfp4_amax")


def nvfp4_quantize_rne(x, flags, out: Output, workspace, stream=None) -> None:
    _check(load().nvfp4_quantize_rne(ctypes.byref(_input(x)), flags, ctypes.byref(out),
                                     _ptr(workspace), _stream(stream)), "nvfp4_quantize_rne")


def nvfp4_quantize_sr(x, flags, seed, offset, out: Output, workspace, stream=None) -> None:
    _check(load().nvfp4_quantize_sr(ctypes.byref(_input(x)), flags, seed, offset, ctypes.byref(out),
                                    _ptr(workspace), _stream(stream)), "nvfp4_quantize_sr")


def nvfp4_quantize_rht_sr(x, flags, sign_mask, seed, offset, out: Output, workspace, stream=None) -> None:
    _check(load().nvfp4_quantize_rht_sr(ctypes.byref(_input(x)), flags, sign_mask & 0xFFFF, seed, offset,
                                        ctypes.byref(out), _ptr(workspace), _stream(stream)),
           "nvfp4_quantize_rht_sr")


def nvfp4_quantize_rht_sr_static(x, flags, sign_mask, seed, offset, out: Output, stream=None) -> None:
    """RHT + SR quantize with the amax scratch held inside the library (for
    callers that cannot allocate device memory; see include/nvfp4.h)."""
    _check(load().nvfp4_quantize_rht_sr_static(ctypes.byref(_input(x)), flags, sign_mask & 0xFFFF, seed,
                                               offset, ctypes.byref(out), _stream(stream)),
           "nvfp4_quantize_rht_sr_static")


def nvfp4_quantize_four_over_six(x, flags, out: Output, workspace, stream=None) -> None:
    _check(load().nvfp4_quantize_four_over_six(ctypes.byref(_input(x)), flags, ctypes.byref(out),
                                               _ptr(workspace), _stream(stream)), "nvfp4_quantize_four_over_six")


def nvfp4_quantize_grouped(x, flags, group_offsets, n_groups, mode, sign_mask, seed, offset, out: Output,
                           stream=None) -> None:
    """Grouped rowwise quantize; group_offsets: int64 CUDA tensor of n_groups+1 row offsets."""
    _check(load().nvfp4_quantize_grouped(ctypes.byref(_input(x)), flags, _ptr(group_offsets), n_groups, mode,
                                         sign_mask & 0xFFFF, seed, offset, ctypes.byref(out), _stream(stream)),
           "nvfp4_quantize_grouped")


def _out_dtype(out) -> int:
    if out.dtype == torch.bfloat16:
        return IN_BF16
    if out.dtype == torch.float32:
        return IN_FP32
    raise ValueError("output must be bfloat16 or float32")


def nvfp4_dequantize(codes, scales, global_scale, rows, cols, flags, out, stream=None) -> None:
    _check(load().nvfp4_dequantize(_ptr(codes), _ptr(scales), _ptr(global_scale), rows, cols, flags, _ptr(out),
                                   _out_dtype(out), _stream(stream)), "nvfp4_dequantize")


def nvfp4_dequantize_rht(codes, scales, global_scale, rows, cols, flags, sign_mask, out, stream=None) -> None:
    _check(load().nvfp4_dequantize_rht(_ptr(codes), _ptr(scales), _ptr(global_scale), rows, cols, flags,
                                       sign_mask & 0xFFFF, _ptr(out), _out_dtype(out), _stream(stream)),
           "nvfp4_dequantize_rht")


# ------------------------------------------------------------ conveniences
@dataclass
class Quantized:
    codes_row: torch.Tensor | None
    scales_row: torch.Tensor | None
    codes_col: torch.Tensor | None
    scales_col: torch.Tensor | None
    amax: torch.Tensor
    global_scale: torch.Tensor
    flags: int


class Workspace:
    """A zeroed workspace per (device, stream): calls on one stream are ordered,
    calls on different streams get different workspaces and may overlap."""
    _cache: dict = {}

    @classmethod
    def get(cls, device, stream=None) -> torch.Tensor:
        dev = torch.device(device)
        if dev.index is None:
            dev = torch.device(dev.type, torch.cuda.current_device())
        if stream is None:
            stream = torch.cuda.current_stream(dev)
        key = (dev, stream.cuda_stream if isinstance(stream, torch.cuda.Stream) else int(stream))
        ws = cls._cache.get(key)
        if ws is None:
            ws = torch.zeros(nvfp4_workspace_bytes(), dtype=torch.uint8, device=dev)
            cls._cache[key] = ws
        return ws


def alloc_outputs(x: torch.Tensor, flags: int, rht: bool = False) -> Quantized:
    """Device outputs for `flags`; with the RHT in both orientations the amax
    and global scale hold two floats ([0] rowwise, [1] columnwise)."""
    R, C = x.shape
    dev = x.device
    cr = sr = cc = sc = None
    if flags & ROWWISE:
        cr = torch.empty(R, C // 2, dtype=torch.uint8, device=dev)
        sr = torch.empty(nvfp4_scale_bytes(R, C, flags), dtype=torch.uint8, device=dev)
    if flags & COLWISE:
        cc = torch.empty(C, R // 2, dtype=torch.uint8, device=dev)
        sc = torch.empty(nvfp4_scale_bytes(C, R, flags), dtype=torch.uint8, device=dev)
    n = R if flags & SCALE_PER_ROW else (2 if rht and flags & ROWWISE and flags & COLWISE else 1)
    amax = torch.empty(n, dtype=torch.float32, device=dev)
    gs = torch.empty(n, dtype=torch.float32, device=dev)
    return Quantized(cr, sr, cc, sc, amax, gs, flags)


def quantize(x: torch.Tensor, *, mode: str = "rne", rowwise: bool = True, colwise: bool = False,
             block2d: bool = False, per_row: bool = False, swizzled: bool = False, rht: bool = False,
             sign_mask: int = 0, seed: int = 0, offset: int = 0, amax: torch.Tensor | None = None,
             fast_math: bool = False, row0: int = 0, col0: int = 0, stream=None,
             out: Quantized | None = None) -> Quantized:
    flags = (ROWWISE if rowwise else 0) | (COLWISE if colwise else 0) | (BLOCK_2D if block2d else 0) | \
        (SCALE_PER_ROW if per_row else 0) | (SWIZZLED if swizzled else 0) | \
        (AMAX_GIVEN if amax is not None else 0) | (FAST_MATH if fast_math else 0)
    q = out if out is not None else alloc_outputs(x, flags, rht)
    if amax is not None:
        q.amax.copy_(amax)
    o = make_output(q.codes_row, q.scales_row, q.codes_col, q.scales_col, q.amax, q.global_scale)
    ws = Workspace.get(x.device, stream)
    xin = make_input(x, row0, col0)
    with torch.cuda.device(x.device):
        if rht:
            if mode != "sr":
                raise ValueError("the RHT entry point rounds stochastically (mode='sr')")
            nvfp4_quantize_rht_sr(xin, flags, sign_mask, seed, offset, o, ws, stream)
        elif mode == "rne":
            nvfp4_quantize_rne(xin, flags, o, ws, stream)
        elif mode == "sr":
            nvfp4_quantize_sr(xin, flags, seed, offset, o, ws, stream)
        elif mode == "4o6":
            nvfp4_quantize_four_over_six(xin, flags, o, ws, stream)
        else:
            raise ValueError(f"unknown mode {mode}")
    return q


def quantize_grouped(x: torch.Tensor, group_offsets: torch.Tensor, *, mode: str = "rne", swizzled: bool = False,
                     sign_mask: int = 0, seed: int = 0, offset: int = 0, amax: torch.Tensor | None = None,
                     stream=None) -> Quantized:
    """Rowwise quantize of the row groups [offs[g], offs[g+1]) of x, each with its
    own amax and global scale (n_groups of each)."""
    n = group_offsets.numel() - 1
    flags = ROWWISE | (SWIZZLED if swizzled else 0) | (AMAX_GIVEN if amax is not None else 0)
    R, C = x.shape
    q = Quantized(torch.empty(R, C // 2, dtype=torch.uint8, device=x.device),
                  torch.empty(nvfp4_scale_bytes(R, C, flags), dtype=torch.uint8, device=x.device), None, None,
                  torch.empty(n, dtype=torch.float32, device=x.device),
                  torch.empty(n, dtype=torch.float32, device=x.device), flags)
    if amax is not None:
        q.amax.copy_(amax)
    m = {"rne": MODE_RNE, "sr": MODE_SR, "rht_sr": MODE_RHT_SR, "4o6": MODE_FOUR_OVER_SIX}[mode]
    o = make_output(q.codes_row, q.scales_row, None, None, q.amax, q.global_scale)
    with torch.cuda.device(x.device):
        nvfp4_quantize_grouped(x, flags, group_offsets, n, m, sign_mask, seed, offset, o, stream)
    return q


def dequantize(codes: torch.Tensor, scales: torch.Tensor, global_scale: torch.Tensor, rows: int, cols: int, *,
               swizzled: bool = False, per_row: bool = False, out_dtype=torch.float32,
               rht_sign_mask: int | None = None, stream=None) -> torch.Tensor:
    """Standard decode; with rht_sign_mask, also the inverse RHT of every block."""
    out = torch.empty(rows, cols, dtype=out_dtype, device=codes.device)
    flags = (SWIZZLED if swizzled else 0) | (SCALE_PER_ROW if per_row else 0)
    with torch.cuda.device(codes.device):
        if rht_sign_mask is None:
            nvfp4_dequantize(codes, scales, global_scale, rows, cols, flags, out, stream)
        else:
            nvfp4_dequantize_rht(codes, scales, global_scale, rows, cols, flags, rht_sign_mask, out, stream)
    return out
