"""The allocation-free GEMV entry point (nwc_gemv_noalloc), called through the C ABI.

It is for callers that may not allocate device memory (a plugin whose host application's
allocator owns the device, a loop that cannot afford cudaMalloc's implicit synchronization): its
scratch is a fixed 4 MiB device array inside the library. The tests check its results against
nwc_gemv and the CPU oracle, and that its calls leave the device's free memory unchanged. This
file is collected last so that, if it fails, a run that stops at the first failure has already
run every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

import decode_gemv_nwc_gb300 as nwc
import oracle
from decode_gemv_nwc_gb300 import synth

TOL_REL, TOL_ABS = 2.0 ** -10, 1e-6


@pytest.fixture(scope="module", autouse=True)
def _built():
    from decode_gemv_nwc_gb300 import build
    build.build()


def _noalloc(mat, x_dev, y_dev):
    s = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return nwc.lib().nwc_gemv_noalloc(ctypes.byref(mat.m), ctypes.c_void_p(x_dev.data_ptr()),
                                      ctypes.c_void_p(y_dev.data_ptr()), s)


@pytest.mark.gpu
@pytest.mark.parametrize("table", [True, False])
def test_noalloc_matches_gemv_and_oracle_on_two_calls_in_a_row(table):
    """Two calls in a row on each matrix (the array keeps the previous call's contents): both
    within the GEMV tolerance of nwc_gemv's result and of the oracle's FP64 product; with and
    without a device copy of the decode table."""
    torch.cuda.init()
    cases = []
    # multi- and single-column-block, a last row block of 5 rows and a ragged last column block
    for shape, seed in (((520, 2600), 31), ((64, 512), 5), ((517, 1500), 7)):
        w = synth.normal_bf16(shape, 0.03, seed)
        x = synth.activations_bf16(shape[1], seed + 1)
        cases.append((nwc.encode(w), x))
    for blob, x in cases:
        mat = nwc.Matrix(blob, table=table)
        xd = torch.from_numpy(x.view(np.int16)).cuda()
        y_ref = mat.gemv(xd).cpu().numpy().astype(np.float64)
        ref = oracle.gemv(blob, x)
        bound = TOL_REL * oracle.abs_dot(blob, x) + TOL_ABS
        for _ in range(2):
            y = torch.full((mat.n,), float("nan"), dtype=torch.float32, device="cuda")
            assert _noalloc(mat, xd, y) == 0
            st, flags = nwc.check()
            assert st == 0, f"device error word {flags:#x}"
            got = y.cpu().numpy().astype(np.float64)
            assert (np.abs(got - y_ref) <= bound).all()
            assert (np.abs(got - ref) <= bound).all()


@pytest.mark.gpu
def test_noalloc_calls_leave_free_device_memory_unchanged():
    """After a first call (which resolves the array's address), further calls change neither
    the device's free memory nor torch's allocations."""
    torch.cuda.init()
    w = synth.normal_bf16((1024, 2048), 0.02, 3)
    mat = nwc.Matrix(nwc.encode(w))
    xd = torch.from_numpy(synth.activations_bf16(2048, 4).view(np.int16)).cuda()
    y = torch.empty(1024, dtype=torch.float32, device="cuda")
    assert _noalloc(mat, xd, y) == 0
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    alloc0 = torch.cuda.memory_allocated()
    for _ in range(5):
        assert _noalloc(mat, xd, y) == 0
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0 and torch.cuda.memory_allocated() == alloc0
    assert nwc.check()[0] == 0


def test_noalloc_rejects_matrices_beyond_its_scratch():
    """The size check comes before any device call, so a host-only struct suffices."""
    m = nwc.NwcMatrix()
    m.elem, m.n_ranked = 0, 12
    m.n, m.k = 1 << 22, 4096
    m.row_blocks, m.col_blocks = (1 << 22) // 8, 8
    m.block_tab = m.data = 0x10000
    x = ctypes.c_void_p(0x20000)
    y = ctypes.c_void_p(0x30000)
    assert nwc.lib().nwc_gemv_noalloc(ctypes.byref(m), x, y, None) == 1
