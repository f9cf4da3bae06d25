"""Failure handling of the GEMM and the norm on the GPU, without a broken device.

Every wait of the GEMM kernel on an mbarrier is bounded: a thread that waits
longer than the launch's limit sets a bit in the library's device fault word,
tells the other roles of its CTA to stop, and the kernel frees its tensor
memory and exits.  mx_gemm_selftest_stall launches the kernel with its
producer issuing no copies, so that the barriers the other roles wait on are
never armed and every wait runs out after a short limit.  Nothing faults,
traps or is left waiting: the test checks that the call returns within a few
limits, that the fault word names only stall bits, that C is untouched, and
that the next ordinary GEMM on the same context is correct."""

import time

import numpy as np
import pytest
import torch

import mxfp8_norm_quant_gb300 as mx
import oracle as O
from mxfp8_norm_quant_gb300 import workloads as W
from mxtest import bf16_bits, gemm_close, np_u8, to_dev

pytestmark = pytest.mark.gpu

# fault bits of the bounded waits (the device fault word)
FAULT_ROWQ_CONSUMER = 1 << 1
FAULT_GEMM_PRODUCER = 1 << 2
FAULT_GEMM_MMA = 1 << 3
FAULT_GEMM_EPILOGUE = 1 << 4
FAULT_DRAIN = 1 << 5
FAULT_GEMM_SCALES = 1 << 6
STALL_BITS = FAULT_GEMM_PRODUCER | FAULT_GEMM_MMA | FAULT_GEMM_EPILOGUE | FAULT_GEMM_SCALES


@pytest.mark.parametrize("M,N,K,tile", [(256, 384, 256, (128, 192)), (256, 384, 256, (128, 64)),
                                        (512, 768, 512, (256, 192)), (4096, 6144, 512, (256, 192)),
                                        (4096, 6144, 512, (128, 128)), (1024, 6144, 256, (256, 256))])
def test_gemm_stall_gives_up_and_recovers(cuda_dev, M, N, K, tile):
    a, wt = W.gemm_operands(M, K, seed=M + N + K, n=N)
    aq, as_ = O.quant(bf16_bits(a))
    bq, bs_ = O.quant(bf16_bits(wt))
    daq, das, dbq, dbs = (to_dev(t, cuda_dev) for t in (aq, as_, bq, bs_))
    torch.cuda.synchronize()
    assert mx.mx_device_fault() == 0
    out = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device=cuda_dev)
    wait_ns = 2_000_000
    t0 = time.time()
    mx.mx_gemm_selftest_stall(daq, das, dbq, dbs, out, M, N, K, *tile, wait_ns=wait_ns)
    torch.cuda.synchronize()
    elapsed = time.time() - t0
    code = mx.mx_device_fault()
    assert code != 0, "the stalled launch reported no fault"
    assert code & ~STALL_BITS == 0, f"unexpected fault bits {code:#x}"
    assert code & FAULT_DRAIN == 0
    assert elapsed < 2.0, f"the stalled launch took {elapsed:.3f} s"
    assert torch.isnan(out.float()).all(), "a stalled launch wrote C"
    # the word was read and cleared; the context is healthy: an ordinary GEMM is correct
    assert mx.mx_device_fault() == 0
    out2 = torch.empty((M, N), dtype=torch.bfloat16, device=cuda_dev)
    mx.mx_gemm_ex(daq, das, dbq, dbs, out2, M, N, K, *tile)
    torch.cuda.synchronize()
    assert mx.mx_device_fault() == 0
    rows = np.arange(0, M, max(1, M // 256))
    ok, worst = gemm_close(out2[torch.from_numpy(rows).to(cuda_dev)],
                           O.gemm_ref(aq[rows], O.swizzle_scales(O.unswizzle_scales(as_, M, K // 32)[rows]), bq, bs_))
    assert ok, f"worst err/tol = {worst:.3f}"


@pytest.mark.parametrize("M,H", [(128, 6144), (1024, 6144), (2000, 6144), (1000, 4160), (700, 2048), (5000, 8192),
                                 (300, 16384)])
def test_norm_stall_gives_up_and_recovers(cuda_dev, M, H):
    # mx_rmsnorm_selftest_stall withholds the lane-block kernel's row copies:
    # every warp's wait for its first row runs out, the warps of each row
    # group stop together, and the call ends within a few limits
    x, w = W.norm_inputs(M, H, seed=M + H)
    xd, wd = x.to(cuda_dev), w.to(cuda_dev)
    torch.cuda.synchronize()
    assert mx.mx_device_fault() == 0
    q = torch.full((M, H), 0xA5, dtype=torch.uint8, device=cuda_dev)
    s = torch.full((mx.mx_scale_bytes(M, H),), 0xA5, dtype=torch.uint8, device=cuda_dev)
    t0 = time.time()
    mx.mx_rmsnorm_selftest_stall(xd, wd, 1e-6, q, s, M, H, wait_ns=2_000_000)
    torch.cuda.synchronize()
    elapsed = time.time() - t0
    code = mx.mx_device_fault()
    assert code == FAULT_ROWQ_CONSUMER, f"fault bits {code:#x}"
    assert elapsed < 2.0, f"the stalled launch took {elapsed:.3f} s"
    assert bool((q == 0xA5).all()), "a stalled launch wrote codes"
    # the context is healthy: an ordinary launch is bit-exact
    mx.mx_rmsnorm_quant(xd, wd, 1e-6, q, s, M, H)
    torch.cuda.synchronize()
    assert mx.mx_device_fault() == 0
    rq, rs = O.rmsnorm_quant(bf16_bits(x), bf16_bits(w), 1e-6)
    assert np.array_equal(np_u8(q), rq) and np.array_equal(np_u8(s), rs)
