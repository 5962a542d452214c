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
    assert ws == 4 * 9 * 4096 + 4 * 512
    assert bind_host(blob, dev_ptr=0x10008)[0] == 1  # misaligned device pointer


def _esc_list(blob, i, n, k):
    """(byte offset, u32 words) of the escape list of block i (BF16, n x k matrix, one
    column block): after the code streams and the closed-form raw section (4096 bytes for a
    block of 512 real columns, else each lane's real columns at 8 bytes, padded to 16)."""
    b = np.frombuffer(bytes(blob), np.uint8)
    nb = int(b[24:32].view(np.uint64)[0])
    off_data = int(b[48:56].view(np.uint64)[0])
    tab = b[80:80 + 4 * (nb + 1)].view(np.uint32)
    start, end = off_data + 16 * int(tab[i]), off_data + 16 * int(tab[i + 1])
    at = start + -(-(32 + 4 * int(b[start:start + 32].astype(np.int64).sum())) // 16) * 16
    if k >= 512:
        at += 4096
    else:
        for lane in range(32):
            cols = max(0, min(16, k - 16 * lane))
            at += -(-8 * cols // 16) * 16
    return at, b[at:end].view(np.uint32)


def test_validate_rejects_corruption():
    # exponents 120..127 only: at most 8 distinct values, so no escapes and an empty list
    rng = np.random.default_rng(4)
    w = ((rng.integers(120, 128, (20, 1030)) << 7) | rng.integers(0, 128, (20, 1030))).astype(np.uint16)
    blob = bytearray(nwc.encode(w))
    assert nwc.validate(bytes(blob)) == 0
    def bad(mut, base=blob):
        b = bytearray(base)
        mut(b)
        return nwc.validate(bytes(b))
    assert bad(lambda b: b.__setitem__(0, 0)) == 2           # magic
    assert bad(lambda b: b.__setitem__(4, 1)) == 2           # format version
    assert bad(lambda b: b.__setitem__(7, 13)) == 2          # n_ranked > 12
    assert bad(lambda b: b.__setitem__(64 + 1, b[64])) == 2  # duplicate ranked exponent
    assert nwc.validate(bytes(blob[:-16])) == 2              # truncated
    off_data = int(np.frombuffer(bytes(blob[48:56]), np.uint64)[0])
    def all_lanes_26(b):  # code streams that no longer leave room for the raw section
        b[off_data:off_data + 32] = bytes([26] * 32)
    assert bad(all_lanes_26) == 2
    assert bad(lambda b: b.__setitem__(off_data + 3, 27)) == 2            # > 26 words (64 pairs x 13 bits)
    assert nwc.validate(bytes(blob) + b"\0" * 16) == 2       # trailing bytes
    # a header whose row blocks x column blocks wraps 64 bits (2^33 x 2^31 = 2^64 -> 0): rejected
    # before the product is formed, whatever block count it claims
    def huge(nb):
        def f(b):
            b[8:16] = np.array([1 << 36], "<u8").tobytes()
            b[16:24] = np.array([(1 << 40) - 1], "<u8").tobytes()
            b[24:32] = np.array([nb], "<u8").tobytes()
        return f
    assert bad(huge(0)) == 2
    assert bad(huge(1)) == 2
    assert bad(huge((1 << 33) * (1 << 31) % (1 << 64))) == 2


def test_validate_checks_escape_lists():
    w = synth.small_matrix_with_outliers(seed=0)  # 64 x 512, one block, escapes present
    blob = bytearray(nwc.encode(w))
    assert nwc.validate(bytes(blob)) == 0
    at, words = _esc_list(blob, 0, 64, 512)
    entries = [i for i in range(len(words)) if words[i] != 0xFFFFFFFF]
    assert len(entries) >= 2 and entries == list(range(len(entries)))
    n_pad = len(words) - len(entries)
    assert n_pad <= 3
    def with_word(off, value, base=blob):
        b = bytearray(base)
        b[off:off + 4] = int(value).to_bytes(4, "little")
        return nwc.validate(bytes(b))
    e0 = int(words[0])
    assert with_word(at, e0 | 0xFFF) == 2                      # lane 31, t 127: out of order
    assert with_word(at, 0xFFFFFFFF) == 2                      # padding before an entry
    assert with_word(at, (e0 & 0xFFF) | (256 << 12)) == 2      # exponent field wider than BF16's 8 bits
    assert with_word(at + 4, e0) == 2                          # repeated entry
    if n_pad > 0:  # an entry after the last one that is out of order
        assert with_word(at + 4 * len(entries), e0) == 2
    # a ragged block: an entry moved onto a filler position (row 5 of a 5-row block)
    blob2 = bytearray(nwc.encode(w[:5, :300]))
    at, words = _esc_list(blob2, 0, 5, 300)
    assert nwc.validate(bytes(blob2)) == 0 and words[0] != 0xFFFFFFFF
    assert with_word(at, (int(words[0]) & ~0x7) | 5, blob2) == 2
    # a column past K = 300 (lane 18, c 12 would be column 300)
    assert with_word(at, (int(words[0]) & ~0xFFF) | (18 << 7) | (12 << 3), blob2) == 2


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


def test_gpu_entry_points_reject_bad_arguments_before_any_launch():
    """Argument checks return NWC_ERR_INVALID_ARG before any CUDA call, so they run here with
    addresses that are never dereferenced."""
    w = synth.normal_bf16((40, 1100), 0.02, seed=3)
    st, m = bind_host(nwc.encode(w))
    assert st == 0
    L = nwc.lib()
    mp = ctypes.byref(m)
    P = ctypes.c_void_p
    ws = int(L.nwc_gemv_workspace_bytes(mp))
    assert ws == 512  # partials 3 column blocks x 40 rows x 4 B + 5 counters x 4 B, to 16 B
    assert L.nwc_gemv(mp, P(0x20002), P(0x30000), P(0x40000), ws, None) == 1   # x not 16-byte aligned
    assert L.nwc_gemv(mp, P(0x20000), P(0x30000), P(0x40008), ws, None) == 1   # workspace not aligned
    assert L.nwc_gemv(mp, P(0x20000), P(0x30000), P(0x40000), ws - 16, None) == 1  # workspace too small
    assert L.nwc_gemv(mp, P(0x20000), None, P(0x40000), ws, None) == 1
    assert L.nwc_gemv_prepare(mp, P(0x40000), ws - 16, None) == 1
    assert L.nwc_decode(mp, P(0x50000), 1099, None, None) == 1                  # ld_out < K
    assert L.nwc_gather(mp, P(0x60000), -1, P(0x50000), 1100, None) == 1
    assert L.nwc_gather(mp, P(0x60000), 0, P(0x50000), 1100, None) == 0        # nothing to do
    assert L.nwc_gather(mp, None, 3, P(0x50000), 1100, None) == 1
    assert L.nwc_gemv_noalloc(None, P(0x20000), P(0x30000), None) == 1
    r = ctypes.c_int(-1)
    assert L.nwc_gemv_route(None, ctypes.byref(r)) == 1
    assert L.nwc_gemv_route(mp, None) == 1


def test_batch_gemv_workspace_and_argument_checks():
    """nwc_gemv_batch's workspace size and its argument checks, all before any CUDA call."""
    w = synth.normal_bf16((40, 1100), 0.02, seed=3)
    st, m = bind_host(nwc.encode(w))
    assert st == 0
    L = nwc.lib()
    mp = ctypes.byref(m)
    P = ctypes.c_void_p
    # 5 counters (32 B with padding) + nb x 3 column blocks x 40 padded rows x 4 B
    for nb in range(1, 17):
        assert int(L.nwc_gemv_batch_workspace_bytes(mp, nb)) == 32 + nb * 3 * 40 * 4
    assert L.nwc_gemv_batch_workspace_bytes(mp, 0) == 0
    assert L.nwc_gemv_batch_workspace_bytes(mp, 17) == 0
    ws = int(L.nwc_gemv_batch_workspace_bytes(mp, 4))
    assert L.nwc_gemv_batch(mp, P(0x20000), 1104, 17, P(0x30000), 40, P(0x40000), 10 ** 6, None) == 1  # nb > 16
    assert L.nwc_gemv_batch(mp, P(0x20000), 1104, 0, P(0x30000), 40, P(0x40000), ws, None) == 1     # nb < 1
    assert L.nwc_gemv_batch(mp, P(0x20000), 1100, 4, P(0x30000), 40, P(0x40000), ws, None) == 1     # ld_x % 8
    assert L.nwc_gemv_batch(mp, P(0x20000), 1096, 4, P(0x30000), 40, P(0x40000), ws, None) == 1     # ld_x < K
    assert L.nwc_gemv_batch(mp, P(0x20000), 1104, 4, P(0x30000), 39, P(0x40000), ws, None) == 1     # ld_y < N
    assert L.nwc_gemv_batch(mp, P(0x20008), 1104, 4, P(0x30000), 40, P(0x40000), ws, None) == 1     # x alignment
    assert L.nwc_gemv_batch(mp, P(0x20000), 1104, 4, P(0x30000), 40, P(0x40008), ws, None) == 1     # ws alignment
    assert L.nwc_gemv_batch(mp, P(0x20000), 1104, 4, P(0x30000), 40, P(0x40000), ws - 16, None) == 1
    assert L.nwc_gemv_batch(mp, P(0x20000), 1104, 4, None, 40, P(0x40000), ws, None) == 1
    assert L.nwc_gemv_batch_prepare(mp, 4, P(0x40000), ws - 16, None) == 1
    assert L.nwc_gemv_batch_prepare(mp, 17, P(0x40000), 10 ** 6, None) == 1
    assert L.nwc_gemv_batch_prepare(mp, 4, P(0x40008), ws, None) == 1
    # one column block: no partials, no counters, 16 bytes
    st, m1 = bind_host(nwc.encode(synth.normal_bf16((9, 500), 0.02, seed=4)))
    assert st == 0 and L.nwc_gemv_batch_workspace_bytes(ctypes.byref(m1), 16) == 16
    assert nwc.BATCH_MAX == 16


def flip_code_bits(blob, seed, blocks=6, flips=3):
    """The blob with `flips` random bits flipped in the code streams of `blocks` random blocks:
    the structure (header, tables, region sizes, escape lists) is unchanged, so host validation
    still accepts it; only decoding can tell."""
    b = bytearray(blob)
    a = np.frombuffer(bytes(blob), np.uint8)
    nb = int(a[24:32].view(np.uint64)[0])
    off_data = int(a[48:56].view(np.uint64)[0])
    tab = a[80:80 + 4 * (nb + 1)].view(np.uint32)
    rng = np.random.default_rng(seed)
    for i in rng.choice(nb, min(blocks, nb), replace=False):
        start = off_data + 16 * int(tab[i])
        code_bytes = 4 * int(a[start:start + 32].astype(np.int64).sum())
        for bit in rng.choice(8 * code_bytes, min(flips, 8 * code_bytes), replace=False):
            b[start + 32 + bit // 8] ^= 1 << (bit % 8)
    return bytes(b)


@pytest.mark.parametrize("elem", [0, 1])
def test_code_bit_flips_pass_validation_and_the_oracle_never_crashes(elem):
    """Flipped code bits keep the blob structurally valid; the oracle decoder then either
    reports a malformed blob or decodes some other matrix of the same shape."""
    from oracle import decode as oracle_decode
    w = synth.normal_bf16((64, 1100), 0.02, seed=31)
    blob = nwc.encode(w, elem=elem)
    outcomes = set()
    for seed in range(12):
        bad = flip_code_bits(blob, seed)
        assert bad != blob
        assert nwc.lib().nwc_validate(np.frombuffer(bad, np.uint8).ctypes.data_as(ctypes.c_void_p), len(bad)) == 0
        try:
            q = oracle_decode(bad)[0]
            assert q.shape == w.shape
            outcomes.add("decoded")
        except ValueError:
            outcomes.add("rejected")
    assert "rejected" in outcomes  # most flips break a lane's bit count or escape pattern


def test_inflated_code_streams_pass_validation_and_the_oracle_rejects_them():
    """A block region whose lane streams are rewritten to the 26-word maximum (all ones, so every
    row pair is a 13-bit escape) with one short last lane: structurally valid, so host validation
    takes it and only decoding can tell; the oracle rejects it (escapes the list does not hold)."""
    import blob_edit
    from oracle import decode as oracle_decode
    w = synth.normal_bf16((64, 513), 0.02, seed=5)
    blob = nwc.encode(w)
    bad = blob_edit.replace_code_streams(blob, 3, [26] * 31 + [8])
    start, end = blob_edit.region_bounds(bad, 3)
    assert end - start <= 6144  # still fits a decoder's shared-memory stage
    assert nwc.validate(bad) == 0
    with pytest.raises(ValueError):
        oracle_decode(bad)


def test_validate_and_oracle_survive_random_byte_mutations():
    """Seeded fuzzing of the host validator: random byte edits anywhere in small blobs (header,
    tables, lane counts, code words, mantissas, escape lists) never crash it; it returns OK or
    NWC_ERR_FORMAT, and a blob it accepts is either rejected or decoded to the right shape by
    the oracle."""
    from oracle import decode as oracle_decode
    rng = np.random.default_rng(77)
    blobs = [nwc.encode(synth.small_matrix_with_outliers(0)),
             nwc.encode(synth.normal_bf16((13, 700), 0.02, seed=78)),
             nwc.encode(synth.normal_bf16((9, 1030), 0.02, seed=79), elem=nwc.FP8)]
    accepted = 0
    for blob in blobs:
        a = np.frombuffer(blob, np.uint8)
        for _ in range(100):
            b = a.copy()
            for pos in rng.integers(0, len(b), rng.integers(1, 4)):
                b[pos] = rng.integers(0, 256)
            st = nwc.lib().nwc_validate(b.ctypes.data_as(ctypes.c_void_p), len(b))
            assert st in (0, 2)
            if st == 0:
                accepted += 1
                try:
                    shape = oracle_decode(b.tobytes())[0].shape
                    assert shape == (int(a[8:16].view(np.int64)[0]), int(a[16:24].view(np.int64)[0]))
                except ValueError:
                    pass
    assert accepted > 0  # edits inside code words and mantissas keep the structure valid


def test_dequantize_fp8_argument_checks_before_any_launch():
    L = nwc.lib()
    P = ctypes.c_void_p
    assert L.nwc_dequantize_fp8(P(0x1000), 16, P(0x2000), 0, 16, P(0x3000), 16, None) == 0  # no rows: no-op
    assert L.nwc_dequantize_fp8(P(0x1000), 16, P(0x2000), 4, 0, P(0x3000), 16, None) == 0   # no columns
    assert L.nwc_dequantize_fp8(P(0x1000), 8, P(0x2000), 4, 16, P(0x3000), 16, None) == 1   # ld_q < K
    assert L.nwc_dequantize_fp8(P(0x1000), 16, P(0x2000), 4, 16, P(0x3000), 8, None) == 1   # ld_out < K
    assert L.nwc_dequantize_fp8(None, 16, P(0x2000), 4, 16, P(0x3000), 16, None) == 1
    assert L.nwc_dequantize_fp8(P(0x1000), 16, None, 4, 16, P(0x3000), 16, None) == 1
    assert L.nwc_dequantize_fp8(P(0x1000), 16, P(0x2000), 4, 16, None, 16, None) == 1
    assert L.nwc_dequantize_fp8(P(0x1000), 16, P(0x2000), -1, 16, P(0x3000), 16, None) == 1
