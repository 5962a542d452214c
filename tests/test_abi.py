"""The C ABI library loads, exports what include/nwc.h declares, and validates blobs on
the host (no GPU call)."""
import ctypes
import os
import re

import numpy as np
import pytest

import decode_gemv_nwc_gb300 as nwc
from decode_gemv_nwc_gb300 import synth

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "nwc.h")


@pytest.fixture(scope="module", autouse=True)
def _built():
    from decode_gemv_nwc_gb300 import build
    build.build()


def declared():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"\b(nwc_[a-z0-9_]+)\s*\(", text)))


def test_every_declared_symbol_is_exported():
    names = declared()
    assert len(names) >= 12
    L = nwc.lib()
    for n in names:
        assert hasattr(L, n), n


def test_status_strings_and_version():
    assert nwc.status_str(0) == "ok"
    assert nwc.status_str(2) == "malformed blob"
    assert b"sm_103a" in nwc.lib().nwc_version()


def bind_host(blob, dev_ptr=0x10000):
    """nwc_bind only parses the host copy; the device address is recorded, not touched."""
    m = nwc.NwcMatrix()
    b = np.frombuffer(blob, np.uint8)
    st = nwc.lib().nwc_bind(b.ctypes.data_as(ctypes.c_void_p), len(blob), ctypes.c_void_p(dev_ptr),
                            ctypes.byref(m))
    return st, m


def test_bind_geometry_and_workspace():
    w = synth.normal_bf16((4095, 4100), 0.02, seed=1)
    blob = nwc.encode(w)
    st, m = bind_host(blob)
    assert st == 0
    assert (m.n, m.k, m.row_blocks, m.col_blocks) == (4095, 4100, 512, 9)
    assert m.block_tab == 0x10000 + 80 and m.scales is None
    ws = nwc.lib().nwc_gemv_workspace_bytes(ctypes.byref(m))
    assert ws == 16384 + 4 * 9 * 4096 + 4 * 512
    assert bind_host(blob, dev_ptr=0x10008)[0] == 1  # misaligned device pointer


def test_validate_rejects_corruption():
    w = synth.normal_bf16((20, 1030), 0.02, seed=4)
    blob = bytearray(nwc.encode(w))
    assert nwc.validate(bytes(blob)) == 0
    def bad(mut):
        b = bytearray(blob)
        mut(b)
        return nwc.validate(bytes(b))
    assert bad(lambda b: b.__setitem__(0, 0)) == 2           # magic
    assert bad(lambda b: b.__setitem__(7, 12)) == 2          # n_ranked > 11
    assert bad(lambda b: b.__setitem__(64 + 1, b[64])) == 2  # duplicate ranked exponent
    assert nwc.validate(bytes(blob[:-16])) == 2              # truncated
    off_data = int(np.frombuffer(bytes(blob[48:56]), np.uint64)[0])
    assert bad(lambda b: b.__setitem__(off_data, b[off_data] + 4)) == 2  # lane word count (beyond padding)
    assert bad(lambda b: b.__setitem__(off_data + 3, 200)) == 2           # > 80 words
    assert nwc.validate(bytes(blob) + b"\0" * 16) == 2       # trailing bytes


def test_encode_argument_errors():
    L = nwc.lib()
    size = ctypes.c_size_t(0)
    assert L.nwc_encode(None, 2, 2, 2, 0, 1, None, ctypes.byref(size)) == 1
    w = np.zeros((2, 2), np.uint16)
    p = w.ctypes.data_as(ctypes.c_void_p)
    assert L.nwc_encode(p, 2, 2, 1, 0, 1, None, ctypes.byref(size)) == 1  # ld < k
    assert L.nwc_encode(p, 2, 2, 2, 7, 1, None, ctypes.byref(size)) == 1  # elem
    assert L.nwc_encode(p, 2, 2, 2, 0, 1, None, ctypes.byref(size)) == 0
    small = ctypes.c_size_t(size.value - 1)
    buf = np.zeros(size.value, np.uint8)
    assert L.nwc_encode(p, 2, 2, 2, 0, 1, buf.ctypes.data_as(ctypes.c_void_p), ctypes.byref(small)) == 1
