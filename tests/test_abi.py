"""Host-side checks of the C ABI that need no GPU: the library loads, exports
every entry point the header declares, and rejects bad arguments before it
touches CUDA."""

import ctypes
import os
import re

import numpy as np
import pytest

import mxfp8_norm_quant_gb300 as mx
import oracle as O

HEADER = os.path.join(os.path.dirname(os.path.dirname(__file__)), "include", "mxgemm.h")


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(mx.LIB_PATH):
        from mxfp8_norm_quant_gb300 import build
        build.build()
    return mx.lib()


def _declared():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(mx_[a-z0-9_]+)\s*\(", src)))


def test_exports_every_declared_symbol(lib):
    names = _declared()
    assert len(names) >= 10
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) == set(mx.EXPORTED)


def test_header_is_plain_c_and_links(lib, tmp_path):
    # the boundary is a C ABI: the header compiles as C99 with no CUDA or C++
    # header, and a C caller links against the library and calls entry points
    # that need no GPU
    import shutil
    import subprocess
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("gcc not available")
    src = tmp_path / "caller.c"
    src.write_text(
        "#include <stdio.h>\n#include \"mxgemm.h\"\n"
        "int main(void) {\n"
        "  if (mx_scale_bytes(130, 6144) != 256u * 192u) return 1;\n"
        "  if (mx_rmsnorm_quant(0, 0, 1e-6f, 0, 0, 4, 48, 0) != MX_ERR_SHAPE) return 2;\n"
        "  if (mx_gemm(0, 0, 0, 0, 0, 0, 256, 256, 0) != MX_OK) return 3;\n"
        "  printf(\"%s %d\\n\", mx_status_string(MX_ERR_ALIGN), mx_version());\n"
        "  return 0;\n}\n")
    exe = tmp_path / "caller"
    libdir = os.path.dirname(mx.LIB_PATH)
    r = subprocess.run([gcc, "-std=c99", "-Wall", "-Werror", "-pedantic", "-I", os.path.dirname(HEADER), str(src),
                        "-o", str(exe), "-L", libdir, "-lmxgemm", f"-Wl,-rpath,{libdir}"],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([str(exe)], capture_output=True, text=True)
    assert r.returncode == 0, (r.returncode, r.stderr)
    assert r.stdout.startswith("MX_ERR_ALIGN")


def test_version_and_status_strings(lib):
    assert mx.mx_version() == 100
    for st, name in mx.MX_STATUS.items():
        assert mx.mx_status_string(st).startswith(name)


@pytest.mark.parametrize("rows,cols", [(0, 32), (1, 32), (127, 64), (128, 6144), (129, 96), (4096, 2048),
                                       (6144, 3072), (300, 160), (1, 16384)])
def test_scale_bytes_matches_oracle(lib, rows, cols):
    assert mx.mx_scale_bytes(rows, cols) == O.scale_bytes(rows, cols)


def test_scale_bytes_rejects(lib):
    assert mx.mx_scale_bytes(-1, 32) == 0
    assert mx.mx_scale_bytes(4, 33) == 0


def _status(fn, *args):
    return getattr(mx.lib(), fn)(*args)


GOOD = 1 << 20          # a 16-byte-aligned fake address; never dereferenced on these paths


@pytest.mark.parametrize("M,H,code", [(-1, 6144, 3), (4, 0, 3), (4, 48, 3), (4, 16, 3), (4, 16416, 3),
                                      (1 << 29, 64, 3)])
def test_rmsnorm_quant_rejects_shapes(lib, M, H, code):
    assert _status("mx_rmsnorm_quant", GOOD, GOOD, ctypes.c_float(1e-6), GOOD, GOOD, M, H, None) == code


def test_rmsnorm_quant_null_and_alignment(lib):
    f = ctypes.c_float(1e-6)
    assert _status("mx_rmsnorm_quant", None, GOOD, f, GOOD, GOOD, 4, 64, None) == 1
    assert _status("mx_rmsnorm_quant", GOOD, None, f, GOOD, GOOD, 4, 64, None) == 1
    assert _status("mx_rmsnorm_quant", GOOD, GOOD, f, None, GOOD, 4, 64, None) == 1
    assert _status("mx_rmsnorm_quant", GOOD, GOOD, f, GOOD, None, 4, 64, None) == 1
    assert _status("mx_rmsnorm_quant", GOOD + 8, GOOD, f, GOOD, GOOD, 4, 64, None) == 2
    assert _status("mx_rmsnorm_quant", GOOD, GOOD, f, GOOD, GOOD + 4, 4, 64, None) == 2
    # M == 0 is a no-op that touches nothing
    assert _status("mx_rmsnorm_quant", None, None, f, None, None, 0, 64, None) == 0


def test_quant_rejects(lib):
    assert _status("mx_quant_weights", GOOD, GOOD, GOOD, 4, 40, None) == 3
    assert _status("mx_quant_weights", GOOD, GOOD, GOOD, -3, 64, None) == 3
    assert _status("mx_quant_weights", None, GOOD, GOOD, 4, 64, None) == 1
    assert _status("mx_quant_weights", GOOD, GOOD + 1, GOOD, 4, 64, None) == 2
    assert _status("mx_quant_weights", None, None, None, 0, 64, None) == 0


def test_sp_entry_points_reject(lib):
    f = ctypes.c_float(1e-6)
    # unknown scale layout; the swizzled layout is mx_rmsnorm_quant itself
    assert _status("mx_rmsnorm_quant_ex", GOOD, GOOD, f, GOOD, GOOD, 4, 64, 2, None) == 3
    assert _status("mx_rmsnorm_quant_ex", GOOD, GOOD, f, GOOD, GOOD, 4, 48, 0, None) == 3
    assert _status("mx_rmsnorm_quant_ex", GOOD, GOOD, f, GOOD, GOOD, 4, 48, 1, None) == 3
    assert _status("mx_rmsnorm_quant_ex", GOOD, GOOD, f, GOOD, None, 4, 64, 1, None) == 1
    assert _status("mx_rmsnorm_quant_ex", GOOD, GOOD, f, GOOD + 8, GOOD, 4, 64, 1, None) == 2
    assert _status("mx_rmsnorm_quant_ex", GOOD, GOOD, f, GOOD, GOOD + 8, 4, 64, 0, None) == 2
    assert _status("mx_rmsnorm_quant_ex", None, None, f, None, None, 0, 64, 1, None) == 0
    assert _status("mx_rmsnorm_bf16", GOOD, GOOD, f, GOOD, 4, 16, None) == 3
    assert _status("mx_rmsnorm_bf16", GOOD, GOOD, f, None, 4, 64, None) == 1
    assert _status("mx_rmsnorm_bf16", GOOD, GOOD, f, GOOD + 2, 4, 64, None) == 2
    for fn in ("mx_swizzle_scales", "mx_unswizzle_scales"):
        assert _status(fn, GOOD, GOOD, 4, 40, None) == 3
        assert _status(fn, GOOD, GOOD, -1, 64, None) == 3
        assert _status(fn, None, GOOD, 4, 64, None) == 1
        assert _status(fn, GOOD, None, 4, 64, None) == 1
        assert _status(fn, None, None, 0, 64, None) == 0
    assert _status("mx_swizzle_scales", GOOD, GOOD + 4, 4, 64, None) == 2
    assert _status("mx_unswizzle_scales", GOOD + 4, GOOD, 4, 64, None) == 2


@pytest.mark.parametrize("M,N,K", [(-1, 6144, 2048), (128, 8, 2048), (128, 6150, 2048), (128, 6144, 48),
                                   (128, 6144, 0), ((1 << 20) + 1, 6144, 2048)])
def test_gemm_rejects_shapes(lib, M, N, K):
    assert _status("mx_gemm", GOOD, GOOD, GOOD, GOOD, GOOD, M, N, K, None) == 3


def test_gemm_null_alignment_and_block_n(lib):
    args = [GOOD] * 5
    for i in range(5):
        a = list(args)
        a[i] = None
        assert _status("mx_gemm", *a, 128, 256, 256, None) == 1
        a[i] = GOOD + 16 * 3 + 8
        assert _status("mx_gemm", *a, 128, 256, 256, None) == 2
    for tm, tn in ((128, 32), (128, 96), (128, 256), (256, 64), (256, 320), (64, 128), (0, 128), (128, 0)):
        assert _status("mx_gemm_ex", *args, 128, 256, 256, tm, tn, None) == 3
    assert _status("mx_gemm", None, None, None, None, None, 0, 256, 256, None) == 0


def test_gemm_quant_rejects(lib):
    args = [GOOD] * 6
    assert _status("mx_gemm_quant", *args, 128, 6144 + 16, 2048, 0, 0, None) == 3    # N % 32
    assert _status("mx_gemm_quant", *args, 128, 6144, 48, 0, 0, None) == 3
    assert _status("mx_gemm_quant", *args, -1, 6144, 2048, 0, 0, None) == 3
    assert _status("mx_gemm_quant", *args, 128, 6144, 2048, 256, 64, None) == 3
    for i in range(6):
        a = list(args)
        a[i] = None
        assert _status("mx_gemm_quant", *a, 128, 256, 256, 0, 0, None) == 1
        a[i] = GOOD + 8
        assert _status("mx_gemm_quant", *a, 128, 256, 256, 0, 0, None) == 2
    assert _status("mx_gemm_quant", None, None, None, None, None, None, 0, 256, 256, 0, 0, None) == 0


def test_gemm_selftest_stall_rejects(lib):
    args = [GOOD] * 5
    u64 = ctypes.c_uint64
    # the wait limit must lie in [100 us, 1 s]; M >= 1; shapes and tiles as for mx_gemm_ex
    assert _status("mx_gemm_selftest_stall", *args, 128, 256, 256, 0, 0, u64(99_999), None) == 3
    assert _status("mx_gemm_selftest_stall", *args, 128, 256, 256, 0, 0, u64(1_000_000_001), None) == 3
    assert _status("mx_gemm_selftest_stall", *args, 0, 256, 256, 0, 0, u64(2_000_000), None) == 3
    assert _status("mx_gemm_selftest_stall", *args, 128, 8, 256, 0, 0, u64(2_000_000), None) == 3
    assert _status("mx_gemm_selftest_stall", *args, 128, 256, 256, 256, 64, u64(2_000_000), None) == 3
    for i in range(5):
        a = list(args)
        a[i] = None
        assert _status("mx_gemm_selftest_stall", *a, 128, 256, 256, 0, 0, u64(2_000_000), None) == 1
        a[i] = GOOD + 8
        assert _status("mx_gemm_selftest_stall", *a, 128, 256, 256, 0, 0, u64(2_000_000), None) == 2


def test_rmsnorm_selftest_stall_rejects(lib):
    f, u64 = ctypes.c_float(1e-6), ctypes.c_uint64
    ok_wait = u64(2_000_000)
    # the wait limit must lie in [100 us, 1 s]; M >= 1; H a multiple of 64 (the
    # lane-block kernels) within the norm's limits
    assert _status("mx_rmsnorm_selftest_stall", GOOD, GOOD, f, GOOD, GOOD, 128, 6144, u64(99_999), None) == 3
    assert _status("mx_rmsnorm_selftest_stall", GOOD, GOOD, f, GOOD, GOOD, 128, 6144, u64(1_000_000_001), None) == 3
    assert _status("mx_rmsnorm_selftest_stall", GOOD, GOOD, f, GOOD, GOOD, 0, 6144, ok_wait, None) == 3
    assert _status("mx_rmsnorm_selftest_stall", GOOD, GOOD, f, GOOD, GOOD, 128, 6112, ok_wait, None) == 3
    assert _status("mx_rmsnorm_selftest_stall", GOOD, GOOD, f, GOOD, GOOD, 128, 16448, ok_wait, None) == 3
    for i in (0, 1, 3, 4):
        a = [GOOD, GOOD, f, GOOD, GOOD]
        a[i] = None
        assert _status("mx_rmsnorm_selftest_stall", *a, 128, 6144, ok_wait, None) == 1
        a[i] = GOOD + 8
        assert _status("mx_rmsnorm_selftest_stall", *a, 128, 6144, ok_wait, None) == 2


def test_binding_checks_tensor_buffers(lib):
    # a CPU tensor, or one too small for the call, is refused on the host
    # before its address reaches the library
    import torch
    small = torch.empty(16, dtype=torch.uint8)
    with pytest.raises(ValueError):
        mx.mx_quant_weights(small, GOOD, GOOD, 4, 64)
    with pytest.raises(ValueError):
        mx.mx_gemm(small, GOOD, GOOD, GOOD, GOOD, 128, 256, 256)


def test_e4m3_probe_and_fault_reject(lib):
    assert _status("mx_e4m3_encode_f32", GOOD, GOOD, -1, None) == 3
    assert _status("mx_e4m3_encode_f32", None, GOOD, 4, None) == 1
    assert _status("mx_e4m3_encode_f32", GOOD + 4, GOOD, 4, None) == 2
    assert _status("mx_device_fault", None) == 1


def test_binding_raises_loudly(lib):
    with pytest.raises(mx.MxError) as ei:
        mx.mx_gemm(GOOD, GOOD, GOOD, GOOD, GOOD, 128, 8, 2048)
    assert ei.value.status_name == "MX_ERR_SHAPE"


def test_e4m3_threshold_table_reproduces_oracle():
    # the step-function form of the oracle encoder used by the exhaustive GPU test
    from mxtest import e4m3_thresholds
    thr = e4m3_thresholds(O.e4m3_encode)
    assert np.all(np.diff(thr) > 0)
    rng = np.random.default_rng(0)
    bits = rng.integers(0, 0x7F800001, size=500_000, dtype=np.int64)
    expect = O.e4m3_encode(bits.astype(np.uint32).view(np.float32))
    got = np.searchsorted(thr, bits, side="right").astype(np.uint8)
    assert np.array_equal(got, expect)
    # sign symmetry of the oracle encoder
    neg = (bits.astype(np.uint32) | np.uint32(0x80000000)).view(np.float32)
    assert np.array_equal(O.e4m3_encode(neg), expect | 0x80)
