"""Blob files (nwc_file_* in include/nwc.h): compressed checkpoints saved once and loaded
straight into device memory, as the NWC page's usage block describes (save_pretrained /
load_pretrained, "straight to the GPU").

The CPU tests cover the file index and its error paths through the C ABI; the GPU test loads
BF16 and fp8 blobs with nwc_file_load and checks decode (bit-exact) and the GEMV (within the
parity tolerance) against the oracle.
"""
import ctypes
import os

import numpy as np
import pytest

import decode_gemv_nwc_gb300 as nwc
from decode_gemv_nwc_gb300 import synth

OK, INVALID, FORMAT, IO = 0, 1, 2, 7


@pytest.fixture(scope="module", autouse=True)
def _built():
    from decode_gemv_nwc_gb300 import build
    build.build()


def _blobs():
    w1 = synth.normal_bf16((9, 513), 0.02, 1)
    w2 = synth.normal_bf16((17, 100), 0.02, 2)
    q, s = nwc.quantize_fp8(synth.normal_bf16((24, 1030), 0.02, 3))
    return {"model.layers.0.self_attn.q_proj": nwc.encode(w1), "lm_head": nwc.encode(w2),
            "mlp.down_proj (fp8)": nwc.encode_fp8(q, s)}


def test_round_trip_entries_and_lookup(tmp_path):
    blobs = _blobs()
    path = str(tmp_path / "model.nwc")
    nwc.save(path, blobs)
    assert nwc.file_entries(path) == [(k, len(v)) for k, v in blobs.items()]
    assert nwc.load(path) == blobs
    raw = open(path, "rb").read()
    assert raw[:4] == b"NWCF" and int.from_bytes(raw[4:8], "little") == 3
    # every blob starts on a 16-byte file offset and the file ends with the last blob
    pos = 8
    for name, blob in blobs.items():
        ln = int.from_bytes(raw[pos:pos + 4], "little")
        assert raw[pos + 4:pos + 4 + ln].decode() == name
        size = int.from_bytes(raw[pos + 4 + ln:pos + 12 + ln], "little")
        start = (pos + 12 + ln + 15) // 16 * 16
        assert size == len(blob) and start % 16 == 0 and raw[start:start + size] == blob
        pos = start + size
    assert pos == len(raw)
    L = nwc.lib()
    idx = ctypes.c_int()
    assert L.nwc_file_find(path.encode(), b"lm_head", ctypes.byref(idx)) == OK and idx.value == 1
    assert L.nwc_file_find(path.encode(), b"absent", ctypes.byref(idx)) == INVALID
    size = ctypes.c_size_t()
    small = ctypes.create_string_buffer(4)
    assert L.nwc_file_entry(path.encode(), 0, small, 4, ctypes.byref(size)) == INVALID
    assert size.value == len(blobs["model.layers.0.self_attn.q_proj"])
    assert L.nwc_file_entry(path.encode(), 3, None, 0, None) == INVALID
    assert L.nwc_file_entry(path.encode(), -1, None, 0, None) == INVALID
    buf = np.empty(size.value - 1, np.uint8)
    assert L.nwc_file_read(path.encode(), 0, buf.ctypes.data_as(ctypes.c_void_p), buf.size,
                           ctypes.byref(size)) == INVALID


def test_empty_file_and_missing_file(tmp_path):
    path = str(tmp_path / "empty.nwc")
    nwc.save(path, {})
    assert open(path, "rb").read() == b"NWCF\0\0\0\0"
    assert nwc.load(path) == {}
    count = ctypes.c_int()
    assert nwc.lib().nwc_file_count(str(tmp_path / "none.nwc").encode(), ctypes.byref(count)) == IO


def _status_of_load(path):
    try:
        nwc.load(path)
    except nwc.NwcError as e:
        return e.status
    return OK


def test_damaged_files_are_format_errors(tmp_path):
    path = str(tmp_path / "m.nwc")
    blobs = _blobs()
    nwc.save(path, blobs)
    raw = open(path, "rb").read()
    first = (8 + 4 + len("model.layers.0.self_attn.q_proj") + 8 + 15) // 16 * 16

    def status_of(data):
        p = str(tmp_path / "bad.nwc")
        open(p, "wb").write(data)
        return _status_of_load(p)

    assert status_of(raw[:-1]) == FORMAT                       # truncated last blob
    assert status_of(raw + b"\0") == FORMAT                    # trailing byte
    assert status_of(b"NWCG" + raw[4:]) == FORMAT              # magic
    assert status_of(raw[:4] + (4).to_bytes(4, "little") + raw[8:]) == FORMAT  # count past the end
    assert status_of(raw[:8] + (0).to_bytes(4, "little") + raw[12:]) == FORMAT  # empty name
    assert status_of(raw[:8] + (1 << 30).to_bytes(4, "little") + raw[12:]) == FORMAT  # name past the end
    bad = bytearray(raw)
    bad[first + 28] ^= 0xFF                                    # the first blob's block count
    assert status_of(bytes(bad)) == FORMAT
    assert status_of(b"NW") == FORMAT


def test_save_checks_before_writing(tmp_path):
    path = str(tmp_path / "m.nwc")
    blobs = _blobs()
    nwc.save(path, blobs)
    before = open(path, "rb").read()
    broken = bytearray(blobs["lm_head"])
    broken[28] ^= 0xFF
    with pytest.raises(nwc.NwcError) as e:
        nwc.save(path, {"a": blobs["lm_head"], "b": bytes(broken)})
    assert e.value.status == FORMAT
    L = nwc.lib()
    b = np.frombuffer(blobs["lm_head"], np.uint8)
    names = (ctypes.c_char_p * 2)(b"same", b"same")
    ptrs = (ctypes.c_void_p * 2)(b.ctypes.data, b.ctypes.data)
    sizes = (ctypes.c_size_t * 2)(b.size, b.size)
    assert L.nwc_file_save(path.encode(), 2, names, ptrs, sizes) == INVALID  # duplicate names
    names = (ctypes.c_char_p * 1)(b"")
    assert L.nwc_file_save(path.encode(), 1, names, ptrs, sizes) == INVALID  # empty name
    assert open(path, "rb").read() == before
    assert not os.path.exists(path + ".partial")
    assert L.nwc_file_save(str(tmp_path / "no" / "dir.nwc").encode(), 0, None, None, None) == IO


@pytest.mark.gpu
def test_load_straight_to_device_then_decode_and_gemv(tmp_path):
    """Save BF16 and fp8 blobs, load each with nwc_file_load into device memory, then decode
    bit-exact and GEMV within tolerance against the oracle run on the original blob."""
    import torch
    import oracle
    torch.cuda.init()
    w = synth.normal_bf16((300, 1100), 0.02, 11)
    q, s = nwc.quantize_fp8(synth.normal_bf16((130, 2049), 0.02, 12))
    blobs = {"bf16": nwc.encode(w), "fp8": nwc.encode_fp8(q, s)}
    path = str(tmp_path / "ckpt.nwc")
    nwc.save(path, blobs)
    for name, blob in blobs.items():
        mat = nwc.Matrix.from_file(path, name)
        assert mat.blob_bytes == len(blob)
        assert bytes(mat.device_blob.cpu().numpy()) == blob
        dec = mat.decode()
        ref_dec = oracle.decode(blob)
        if name == "bf16":
            assert np.array_equal(dec.cpu().numpy().view(np.uint16), ref_dec[0])
        else:
            assert np.array_equal(dec[0].cpu().numpy(), ref_dec[0])
            assert np.array_equal(dec[1].cpu().numpy().view(np.uint32), ref_dec[1].view(np.uint32))
        x = synth.activations_bf16(mat.k, 40 + mat.k)
        y = mat.gemv(torch.from_numpy(x.view(np.int16)).cuda()).cpu().numpy().astype(np.float64)
        st, flags = nwc.check()
        assert st == 0, f"device error word {flags:#x}"
        ref = oracle.gemv(blob, x)
        bound = 2.0 ** -10 * oracle.abs_dot(blob, x) + 1e-6
        assert (np.abs(y - ref) <= bound).all()
