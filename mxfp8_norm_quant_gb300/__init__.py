"""Python binding of libmxgemm (MXFP8 Gemma-RMSNorm quantisation + block-scaled GEMM).

Argument marshalling only: every step of the computation runs in the CUDA
kernels behind the C ABI declared in include/mxgemm.h.  Functions named
``mx_*`` mirror the C entry points one to one; they accept torch tensors
(their device pointers are passed) or raw integer device addresses.  A torch
tensor is checked before its address is passed: it must be a contiguous CUDA
tensor on the current device holding at least the bytes the call reads or
writes (a ValueError otherwise), so that a wrong buffer is caught on the host
and never becomes an out-of-bounds access on the GPU.  Raw integer addresses
are passed as given.  The small helpers at the bottom only allocate outputs
with torch and call them.

There is no fallback: if libmxgemm.so has not been built, every call raises.
"""

from __future__ import annotations

import ctypes
import os

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libmxgemm.so")

MX_STATUS = {
    0: "MX_OK",
    1: "MX_ERR_NULL",
    2: "MX_ERR_ALIGN",
    3: "MX_ERR_SHAPE",
    4: "MX_ERR_ARCH",
    5: "MX_ERR_CUDA",
    6: "MX_ERR_DEVICE_TIMEOUT",
}

EXPORTED = (
    "mx_scale_bytes", "mx_rmsnorm_quant", "mx_rmsnorm_quant_ex", "mx_rmsnorm_bf16", "mx_swizzle_scales",
    "mx_unswizzle_scales", "mx_quant_weights", "mx_gemm", "mx_gemm_ex", "mx_gemm_quant", "mx_gemm_plan",
    "mx_e4m3_encode_f32", "mx_device_fault", "mx_last_cuda_error", "mx_status_string", "mx_version",
    "mx_gemm_selftest_stall", "mx_rmsnorm_plan", "mx_rmsnorm_selftest_stall", "mx_gemm_tile_for",
)

# scale layouts of mx_rmsnorm_quant_ex
MX_SCALES_F8_128X4 = 0
MX_SCALES_ROW_MAJOR = 1

# output forms of the norm, for mx_rmsnorm_plan
MX_NORM_SWIZZLED = 0
MX_NORM_ROW_MAJOR = 1
MX_NORM_BF16 = 2


class MxError(RuntimeError):
    def __init__(self, fn: str, status: int, cuda_error: int = 0):
        self.status = status
        self.status_name = MX_STATUS.get(status, str(status))
        self.cuda_error = cuda_error
        msg = f"{fn}: {self.status_name}"
        if status == 5:
            msg += f" (cudaError {cuda_error})"
        super().__init__(msg)


_lib = None


def lib() -> ctypes.CDLL:
    """The loaded libmxgemm.so (loaded on first use; raises if it is missing)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(
            f"libmxgemm.so is not built ({LIB_PATH} missing). Build it with "
            "`python -m mxfp8_norm_quant_gb300.build` or `__graft_entry__.build()`; there is no fallback.")
    L = ctypes.CDLL(LIB_PATH)
    i64, vp, u8p, i32 = ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int
    L.mx_scale_bytes.argtypes = [i64, i64]
    L.mx_scale_bytes.restype = ctypes.c_size_t
    L.mx_rmsnorm_quant.argtypes = [vp, vp, ctypes.c_float, u8p, u8p, i64, i64, vp]
    L.mx_rmsnorm_quant_ex.argtypes = [vp, vp, ctypes.c_float, u8p, u8p, i64, i64, i32, vp]
    L.mx_rmsnorm_bf16.argtypes = [vp, vp, ctypes.c_float, vp, i64, i64, vp]
    L.mx_swizzle_scales.argtypes = [u8p, u8p, i64, i64, vp]
    L.mx_unswizzle_scales.argtypes = [u8p, u8p, i64, i64, vp]
    L.mx_quant_weights.argtypes = [vp, u8p, u8p, i64, i64, vp]
    L.mx_gemm.argtypes = [u8p, u8p, u8p, u8p, vp, i64, i64, i64, vp]
    L.mx_gemm_ex.argtypes = [u8p, u8p, u8p, u8p, vp, i64, i64, i64, i32, i32, vp]
    L.mx_gemm_quant.argtypes = [u8p, u8p, u8p, u8p, u8p, u8p, i64, i64, i64, i32, i32, vp]
    L.mx_gemm_selftest_stall.argtypes = [u8p, u8p, u8p, u8p, vp, i64, i64, i64, i32, i32, ctypes.c_uint64, vp]
    L.mx_gemm_plan.argtypes = [i64, i64, i64] + [ctypes.POINTER(i32)] * 4
    L.mx_rmsnorm_plan.argtypes = [i64, i64, i32, i32, ctypes.POINTER(i32)]
    L.mx_gemm_tile_for.argtypes = [i64, i64, i64, i32, ctypes.POINTER(i32), ctypes.POINTER(i32)]
    L.mx_rmsnorm_selftest_stall.argtypes = [vp, vp, ctypes.c_float, u8p, u8p, i64, i64, ctypes.c_uint64, vp]
    L.mx_e4m3_encode_f32.argtypes = [vp, u8p, i64, vp]
    L.mx_device_fault.argtypes = [ctypes.POINTER(ctypes.c_uint32)]
    L.mx_last_cuda_error.argtypes = []
    L.mx_status_string.argtypes = [i32]
    L.mx_status_string.restype = ctypes.c_char_p
    L.mx_version.argtypes = []
    for name in ("mx_rmsnorm_quant", "mx_rmsnorm_quant_ex", "mx_rmsnorm_bf16", "mx_swizzle_scales",
                 "mx_unswizzle_scales", "mx_quant_weights", "mx_gemm", "mx_gemm_ex", "mx_gemm_quant", "mx_gemm_plan",
                 "mx_e4m3_encode_f32", "mx_device_fault", "mx_last_cuda_error", "mx_version",
                 "mx_gemm_selftest_stall", "mx_rmsnorm_plan", "mx_rmsnorm_selftest_stall", "mx_gemm_tile_for"):
        getattr(L, name).restype = ctypes.c_int
    _lib = L
    return L


def _ptr(t) -> int | None:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream, *tensors) -> int | None:
    if stream is None:
        import torch
        for t in tensors:
            if hasattr(t, "is_cuda") and t.is_cuda:
                return torch.cuda.current_stream(t.device).cuda_stream
        return None
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(fn: str, status: int):
    if status != 0:
        raise MxError(fn, status, lib().mx_last_cuda_error())


def _scale_bytes_py(rows: int, cols: int) -> int:
    return (-(-rows // 128) * 128) * (-(-(cols // 32) // 4) * 4)


def _need(fn: str, name: str, t, nbytes: int) -> None:
    """A torch tensor passed as a buffer must be a contiguous CUDA tensor on
    the current device with at least nbytes; ints and None pass unchecked
    (the C side rejects NULL)."""
    if t is None or isinstance(t, int) or nbytes <= 0:
        return
    import torch
    if not isinstance(t, torch.Tensor):
        raise ValueError(f"{fn}: {name} must be a torch tensor or an integer device address")
    if not t.is_cuda:
        raise ValueError(f"{fn}: {name} is on {t.device}, not on a CUDA device")
    if t.device.index != torch.cuda.current_device():
        raise ValueError(f"{fn}: {name} is on {t.device}, but cuda:{torch.cuda.current_device()} is current")
    if not t.is_contiguous():
        raise ValueError(f"{fn}: {name} is not contiguous")
    have = t.numel() * t.element_size()
    if have < nbytes:
        raise ValueError(f"{fn}: {name} holds {have} bytes, the call needs {nbytes}")


def _row_shape_ok(rows: int, cols: int) -> bool:
    return rows > 0 and cols >= 32 and cols % 32 == 0 and cols <= 16384


def _gemm_shape_ok(M: int, N: int, K: int) -> bool:
    return M > 0 and N >= 16 and N % 16 == 0 and K >= 32 and K % 32 == 0


# ------------------------------------------------------------- C entry points

def mx_scale_bytes(rows: int, cols: int) -> int:
    return int(lib().mx_scale_bytes(rows, cols))


def mx_rmsnorm_quant(x, w, eps: float, out_q, out_scales, M: int, H: int, stream=None) -> None:
    if _row_shape_ok(M, H):
        fn = "mx_rmsnorm_quant"
        _need(fn, "x", x, 2 * M * H)
        _need(fn, "w", w, 2 * H)
        _need(fn, "out_q", out_q, M * H)
        _need(fn, "out_scales", out_scales, _scale_bytes_py(M, H))
    _check("mx_rmsnorm_quant", lib().mx_rmsnorm_quant(_ptr(x), _ptr(w), float(eps), _ptr(out_q), _ptr(out_scales),
                                                      M, H, _stream(stream, x)))


def mx_rmsnorm_quant_ex(x, w, eps: float, out_q, out_scales, M: int, H: int, scale_layout: int,
                        stream=None) -> None:
    if _row_shape_ok(M, H) and scale_layout in (MX_SCALES_F8_128X4, MX_SCALES_ROW_MAJOR):
        fn = "mx_rmsnorm_quant_ex"
        _need(fn, "x", x, 2 * M * H)
        _need(fn, "w", w, 2 * H)
        _need(fn, "out_q", out_q, M * H)
        _need(fn, "out_scales", out_scales,
              M * (H // 32) if scale_layout == MX_SCALES_ROW_MAJOR else _scale_bytes_py(M, H))
    _check("mx_rmsnorm_quant_ex", lib().mx_rmsnorm_quant_ex(_ptr(x), _ptr(w), float(eps), _ptr(out_q),
                                                            _ptr(out_scales), M, H, scale_layout,
                                                            _stream(stream, x)))


def mx_rmsnorm_bf16(x, w, eps: float, out, M: int, H: int, stream=None) -> None:
    if _row_shape_ok(M, H):
        fn = "mx_rmsnorm_bf16"
        _need(fn, "x", x, 2 * M * H)
        _need(fn, "w", w, 2 * H)
        _need(fn, "out", out, 2 * M * H)
    _check("mx_rmsnorm_bf16", lib().mx_rmsnorm_bf16(_ptr(x), _ptr(w), float(eps), _ptr(out), M, H,
                                                    _stream(stream, x)))


def mx_swizzle_scales(in_row_major, out_swizzled, rows: int, cols: int, stream=None) -> None:
    if _row_shape_ok(rows, cols):
        _need("mx_swizzle_scales", "in_row_major", in_row_major, rows * (cols // 32))
        _need("mx_swizzle_scales", "out_swizzled", out_swizzled, _scale_bytes_py(rows, cols))
    _check("mx_swizzle_scales", lib().mx_swizzle_scales(_ptr(in_row_major), _ptr(out_swizzled), rows, cols,
                                                        _stream(stream, in_row_major)))


def mx_unswizzle_scales(in_swizzled, out_row_major, rows: int, cols: int, stream=None) -> None:
    if _row_shape_ok(rows, cols):
        _need("mx_unswizzle_scales", "in_swizzled", in_swizzled, _scale_bytes_py(rows, cols))
        _need("mx_unswizzle_scales", "out_row_major", out_row_major, rows * (cols // 32))
    _check("mx_unswizzle_scales", lib().mx_unswizzle_scales(_ptr(in_swizzled), _ptr(out_row_major), rows, cols,
                                                            _stream(stream, in_swizzled)))


def mx_quant_weights(x, out_q, out_scales, rows: int, cols: int, stream=None) -> None:
    if _row_shape_ok(rows, cols):
        fn = "mx_quant_weights"
        _need(fn, "x", x, 2 * rows * cols)
        _need(fn, "out_q", out_q, rows * cols)
        _need(fn, "out_scales", out_scales, _scale_bytes_py(rows, cols))
    _check("mx_quant_weights", lib().mx_quant_weights(_ptr(x), _ptr(out_q), _ptr(out_scales), rows, cols,
                                                      _stream(stream, x)))


def _need_gemm_inputs(fn, a_q, a_s, b_q, b_s, M, N, K):
    _need(fn, "a_q", a_q, M * K)
    _need(fn, "a_s", a_s, _scale_bytes_py(M, K))
    _need(fn, "b_q", b_q, N * K)
    _need(fn, "b_s", b_s, _scale_bytes_py(N, K))


def mx_gemm(a_q, a_s, b_q, b_s, out, M: int, N: int, K: int, stream=None) -> None:
    if _gemm_shape_ok(M, N, K):
        _need_gemm_inputs("mx_gemm", a_q, a_s, b_q, b_s, M, N, K)
        _need("mx_gemm", "out", out, 2 * M * N)
    _check("mx_gemm", lib().mx_gemm(_ptr(a_q), _ptr(a_s), _ptr(b_q), _ptr(b_s), _ptr(out), M, N, K,
                                    _stream(stream, a_q)))


def mx_gemm_ex(a_q, a_s, b_q, b_s, out, M: int, N: int, K: int, tile_m: int = 0, tile_n: int = 0,
               stream=None) -> None:
    if _gemm_shape_ok(M, N, K):
        _need_gemm_inputs("mx_gemm_ex", a_q, a_s, b_q, b_s, M, N, K)
        _need("mx_gemm_ex", "out", out, 2 * M * N)
    _check("mx_gemm_ex", lib().mx_gemm_ex(_ptr(a_q), _ptr(a_s), _ptr(b_q), _ptr(b_s), _ptr(out), M, N, K,
                                          tile_m, tile_n, _stream(stream, a_q)))


def mx_gemm_quant(a_q, a_s, b_q, b_s, out_q, out_scales, M: int, N: int, K: int, tile_m: int = 0,
                  tile_n: int = 0, stream=None) -> None:
    if _gemm_shape_ok(M, N, K) and N % 32 == 0:
        _need_gemm_inputs("mx_gemm_quant", a_q, a_s, b_q, b_s, M, N, K)
        _need("mx_gemm_quant", "out_q", out_q, M * N)
        _need("mx_gemm_quant", "out_scales", out_scales, _scale_bytes_py(M, N))
    _check("mx_gemm_quant", lib().mx_gemm_quant(_ptr(a_q), _ptr(a_s), _ptr(b_q), _ptr(b_s), _ptr(out_q),
                                                _ptr(out_scales), M, N, K, tile_m, tile_n, _stream(stream, a_q)))


def mx_gemm_selftest_stall(a_q, a_s, b_q, b_s, out, M: int, N: int, K: int, tile_m: int = 0, tile_n: int = 0,
                           wait_ns: int = 2_000_000, stream=None) -> None:
    if _gemm_shape_ok(M, N, K):
        _need_gemm_inputs("mx_gemm_selftest_stall", a_q, a_s, b_q, b_s, M, N, K)
        _need("mx_gemm_selftest_stall", "out", out, 2 * M * N)
    _check("mx_gemm_selftest_stall", lib().mx_gemm_selftest_stall(
        _ptr(a_q), _ptr(a_s), _ptr(b_q), _ptr(b_s), _ptr(out), M, N, K, tile_m, tile_n, int(wait_ns),
        _stream(stream, a_q)))


def mx_rmsnorm_selftest_stall(x, w, eps: float, out_q, out_scales, M: int, H: int, wait_ns: int = 2_000_000,
                              stream=None) -> None:
    if _row_shape_ok(M, H):
        fn = "mx_rmsnorm_selftest_stall"
        _need(fn, "x", x, 2 * M * H)
        _need(fn, "w", w, 2 * H)
        _need(fn, "out_q", out_q, M * H)
        _need(fn, "out_scales", out_scales, _scale_bytes_py(M, H))
    _check("mx_rmsnorm_selftest_stall", lib().mx_rmsnorm_selftest_stall(
        _ptr(x), _ptr(w), float(eps), _ptr(out_q), _ptr(out_scales), M, H, int(wait_ns), _stream(stream, x)))


def mx_gemm_tile_for(M: int, N: int, K: int, num_sms: int):
    """(tile_m, tile_n) mx_gemm chooses on a GPU of num_sms SMs; needs no GPU."""
    tm, tn = ctypes.c_int(0), ctypes.c_int(0)
    _check("mx_gemm_tile_for", lib().mx_gemm_tile_for(M, N, K, num_sms, ctypes.byref(tm), ctypes.byref(tn)))
    return tm.value, tn.value


def mx_gemm_plan(M: int, N: int, K: int):
    tm, tn, st, gr = (ctypes.c_int(0) for _ in range(4))
    _check("mx_gemm_plan", lib().mx_gemm_plan(M, N, K, ctypes.byref(tm), ctypes.byref(tn), ctypes.byref(st),
                                              ctypes.byref(gr)))
    return {"tile_m": tm.value, "tile_n": tn.value, "stages": st.value, "grid": gr.value}


def mx_rmsnorm_plan(M: int, H: int, form: int, num_sms: int):
    """(warps per row, chunks per warp, rows per CTA, row kept unpacked) of the
    lane-block kernel the norm launches, or (0, 0, 0, 0) for the chunked
    kernels; needs no GPU."""
    plan = (ctypes.c_int * 4)()
    _check("mx_rmsnorm_plan", lib().mx_rmsnorm_plan(M, H, form, num_sms, plan))
    return tuple(int(v) for v in plan)


def mx_e4m3_encode_f32(inp, out, n: int, stream=None) -> None:
    if n > 0:
        _need("mx_e4m3_encode_f32", "inp", inp, 4 * n)
        _need("mx_e4m3_encode_f32", "out", out, n)
    _check("mx_e4m3_encode_f32", lib().mx_e4m3_encode_f32(_ptr(inp), _ptr(out), n, _stream(stream, inp)))


def mx_device_fault() -> int:
    code = ctypes.c_uint32(0)
    st = lib().mx_device_fault(ctypes.byref(code))
    if st not in (0, 6):
        _check("mx_device_fault", st)
    return int(code.value)


def mx_status_string(status: int) -> str:
    return lib().mx_status_string(status).decode()


def mx_version() -> int:
    return int(lib().mx_version())


# ------------------------------------------------------------- conveniences

def rmsnorm_quant(x, w, eps: float = 1e-6, stream=None):
    """Allocates (q, scales) for an (M, H) bf16 CUDA tensor and runs mx_rmsnorm_quant."""
    import torch
    M, H = x.shape
    q = torch.empty((M, H), dtype=torch.uint8, device=x.device)
    s = torch.empty(mx_scale_bytes(M, H), dtype=torch.uint8, device=x.device)
    mx_rmsnorm_quant(x, w, eps, q, s, M, H, stream)
    return q, s


def rmsnorm_quant_rowmajor(x, w, eps: float = 1e-6, stream=None):
    """Allocates (q, [M][H/32] scales) and runs mx_rmsnorm_quant_ex with row-major scales."""
    import torch
    M, H = x.shape
    q = torch.empty((M, H), dtype=torch.uint8, device=x.device)
    s = torch.empty((M, H // 32), dtype=torch.uint8, device=x.device)
    mx_rmsnorm_quant_ex(x, w, eps, q, s, M, H, MX_SCALES_ROW_MAJOR, stream)
    return q, s


def rmsnorm_bf16(x, w, eps: float = 1e-6, stream=None):
    """Allocates the bf16 output for an (M, H) bf16 CUDA tensor and runs mx_rmsnorm_bf16."""
    out = x.new_empty(x.shape)
    mx_rmsnorm_bf16(x, w, eps, out, x.shape[0], x.shape[1], stream)
    return out


def swizzle_scales(s_row_major, cols: int, stream=None):
    """Allocates the F8_128x4 buffer for (rows, cols/32) row-major scales and runs mx_swizzle_scales."""
    import torch
    rows = s_row_major.shape[0]
    out = torch.empty(mx_scale_bytes(rows, cols), dtype=torch.uint8, device=s_row_major.device)
    mx_swizzle_scales(s_row_major, out, rows, cols, stream)
    return out


def quant(x, stream=None):
    """Allocates (q, scales) for an (R, C) bf16 CUDA tensor and runs mx_quant_weights."""
    import torch
    R, C = x.shape
    q = torch.empty((R, C), dtype=torch.uint8, device=x.device)
    s = torch.empty(mx_scale_bytes(R, C), dtype=torch.uint8, device=x.device)
    mx_quant_weights(x, q, s, R, C, stream)
    return q, s


def gemm_quant(a_q, a_s, b_q, b_s, tile=(0, 0), stream=None):
    """C = A . B^T leaving as MXFP8 (codes (M, N) uint8, F8_128x4 scales)."""
    import torch
    M, K = a_q.shape
    N = b_q.shape[0]
    q = torch.empty((M, N), dtype=torch.uint8, device=a_q.device)
    s = torch.empty(mx_scale_bytes(M, N), dtype=torch.uint8, device=a_q.device)
    mx_gemm_quant(a_q, a_s, b_q, b_s, q, s, M, N, K, tile[0], tile[1], stream)
    return q, s


def gemm(a_q, a_s, b_q, b_s, tile=(0, 0), stream=None):
    """C = A . B^T in bf16 for MXFP8 operands (A: M x K, B: N x K)."""
    import torch
    M, K = a_q.shape
    N = b_q.shape[0]
    out = torch.empty((M, N), dtype=torch.bfloat16, device=a_q.device)
    mx_gemm_ex(a_q, a_s, b_q, b_s, out, M, N, K, tile[0], tile[1], stream)
    return out
