"""Pins of the CPU oracle to facts that do not come from the oracle itself.

The pages fix: lossless round trip ("bit-exact"), about 31% smaller than BF16
for LLM weights because that is the exponent entropy, a short code and no
mantissa per filler, a unary rank code with a raw sign bit and an escape for
rare exponents, a peek that yields up to two complete codes, and an fp8 variant
whose bytes come back bit for bit. Mathematics fixes the plain matrix-vector
product and the e4m3 rounding. Each test below would fail for a plausible
mistake in the oracle (dropped term, wrong sign, wrong bit order, transposed
operand, off-by-one rank, a pair cut at the wrong length).
"""
import math
import os

import numpy as np
import pytest
import torch

import oracle
from decode_gemv_nwc_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
PEEK, RMAX = 13, 12


# ----------------------------------------------------------------- helpers
def hdr(blob):
    b = np.frombuffer(blob, np.uint8)
    u64 = lambda o: int(b[o:o + 8].view(np.uint64)[0])
    return dict(elem=int(b[6]), nr=int(b[7]), N=u64(8), K=u64(16), nb=u64(24), off_blocks=u64(32),
                off_scales=u64(40), off_data=u64(48), total=u64(56), ranks=b[64:80].tolist())


def regions(blob):
    """Per block (start, end) byte offsets of its region, from the block table."""
    h = hdr(blob)
    b = np.frombuffer(blob, np.uint8)
    tab = b[h["off_blocks"]:h["off_blocks"] + 4 * (h["nb"] + 1)].view(np.uint32)
    return [(h["off_data"] + 16 * int(tab[i]), h["off_data"] + 16 * int(tab[i + 1])) for i in range(h["nb"])]


def lane_words(blob):
    """Per block, the 32 lane word counts read straight from the blob."""
    b = np.frombuffer(blob, np.uint8)
    return np.array([b[s:s + 32].astype(np.int64) for s, _ in regions(blob)])


def ranks_of(values, nvals):
    """Independent ranking: numpy histogram, (count desc, value asc), <= 12 ranks."""
    cnt = np.bincount(values.ravel(), minlength=nvals)
    order = sorted([v for v in range(nvals) if cnt[v] > 0], key=lambda v: (-cnt[v], v))
    return order[:RMAX]


def lane_cols(k, cb, lane):
    return int(np.clip(k - 512 * cb - 16 * lane, 0, 16))


def code_lengths(v, nvals):
    """Code length of every position of the padded matrix: rank + 1 for a ranked exponent,
    n_ranked for an unranked one, 1 for a filler. Returns (lengths (RB*8, CB*512), ranked)."""
    n, k = v.shape
    ranked = ranks_of(v, nvals)
    nr = len(ranked)
    length = np.full(nvals, nr, np.int64)
    for p, e in enumerate(ranked):
        length[e] = p + 1
    rb, cb = -(-n // 8), -(-k // 512)
    L = np.ones((rb * 8, cb * 512), np.int64)
    L[:n, :k] = length[v]
    return L, ranked


def pair_bits_per_lane(v, nvals):
    """Closed-form lane stream lengths: per pair of rows (2i, 2i+1) of a column, both codes
    when they fit 13 bits, else 13. Returns (RB*CB, 32) bits and the cut-pair mask of the
    padded matrix (True at the second element of a cut pair)."""
    L, _ = code_lengths(v, nvals)
    rb, cb = L.shape[0] // 8, L.shape[1] // 512
    la, lb = L[0::2], L[1::2]
    pair = np.where(la + lb <= PEEK, la + lb, PEEK)
    cut = np.zeros(L.shape, bool)
    cut[1::2] = la + lb > PEEK
    # (rb, 4 pairs, cb, lane, c) -> sum over pairs and columns
    bits = pair.reshape(rb, 4, cb, 32, 16).sum(axis=(1, 4))
    return bits.reshape(rb * cb, 32), cut


def raw_section_bytes(k, cb, col_bytes):
    if 512 * (cb + 1) <= k:
        return 32 * 16 * col_bytes
    return sum(-(-lane_cols(k, cb, l) * col_bytes // 16) * 16 for l in range(32))


def escape_lists(blob):
    """Per block, the escape-list entries read straight from the blob: the region's tail
    after the code streams and the closed-form raw section."""
    h = hdr(blob)
    b = np.frombuffer(blob, np.uint8)
    cb_n = -(-h["K"] // 512)
    col_bytes = 8 if h["elem"] == 0 else 4
    out = []
    for i, (start, end) in enumerate(regions(blob)):
        lw = b[start:start + 32].astype(np.int64)
        at = start + -(-(32 + 4 * int(lw.sum())) // 16) * 16 + raw_section_bytes(h["K"], i % cb_n, col_bytes)
        ent = b[at:end].view(np.uint32)
        out.append([int(e) for e in ent if e != 0xFFFFFFFF])
        assert all(e == 0xFFFFFFFF for e in ent[len(out[-1]):]), "padding must follow the entries"
        assert len(ent) - len(out[-1]) < 4
    return out


def expected_lists(v, listed_extra, nvals):
    """The escape lists the format prescribes, from numpy: unranked real elements, real second
    elements of cut pairs and the extra mask (fp8 subnormal and NaN codes), as
    t | lane << 7 | v << 12 in lane, then t order."""
    n, k = v.shape
    L, ranked = code_lengths(v, nvals)
    _, cut = pair_bits_per_lane(v, nvals)
    listed = cut[:n, :k] | ~np.isin(v, ranked) | listed_extra
    rb_n, cb_n = -(-n // 8), -(-k // 512)
    out = []
    for rb in range(rb_n):
        for cb in range(cb_n):
            ent = []
            for lane in range(32):
                for t in range(128):
                    r, c = 8 * rb + t % 8, 512 * cb + 16 * lane + t // 8
                    if r < n and c < k and listed[r, c]:
                        ent.append(t | lane << 7 | int(v[r, c]) << 12)
            out.append(ent)
    return out


def bf16_f64(bits):
    return synth.bf16_bits_to_f32(np.asarray(bits, np.uint16)).astype(np.float64)


def load_golden(name):
    want, checks = None, []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if not line:
                continue
            parts = line.split()
            if parts[0] == "total":
                want = int(parts[1])
            else:
                checks.append(parts)
    expected = np.zeros(want, np.uint8)
    for kind, off, *rest in checks:
        off = int(off)
        if kind == "u8s":
            val, count = int(rest[0], 0), int(rest[1])
            expected[off:off + count] = val
            continue
        width = {"u8": 1, "u16": 2, "u32": 4, "u64": 8}[kind]
        val = int(rest[0], 0)
        expected[off:off + width] = np.frombuffer(val.to_bytes(width, "little"), np.uint8)
    return expected


# ---------------------------------------------------------------- the pins
@pytest.mark.parametrize("name,w", [
    ("nwc_2x2_bf16.txt", [[0x3FC0, 0xC020], [0x3F20, 0x3F81]]),
    ("nwc_2x8_longpairs_bf16.txt", [[0xBF91, 0x3F80, 0x3680, 0x3780, 0x3280, 0x3380, 0x3500, 0x3600],
                                    [0x3F80, 0x3F80, 0x3400, 0x3200, 0x3300, 0x3480, 0x3580, 0xB700]]),
])
def test_golden_blobs_match_hand_derivation(name, w):
    w = np.array(w, np.uint16)
    blob = oracle.encode(w)
    expected = load_golden(name)
    assert len(blob) == len(expected)
    diff = np.nonzero(np.frombuffer(blob, np.uint8) != expected)[0]
    assert diff.size == 0, f"blob differs from the hand derivation at bytes {diff[:16]}"
    back, _ = oracle.decode(blob)
    assert np.array_equal(back, w)


def test_roundtrip_all_65536_bf16_patterns():
    """Every BF16 bit pattern once (+-0, subnormals, +-Inf, NaN payloads): 256 distinct
    exponents, all tied, rank the 12 smallest values and escape the other 244."""
    rng = np.random.default_rng(3)
    w = rng.permutation(np.arange(65536, dtype=np.uint32)).astype(np.uint16).reshape(128, 512)
    blob = oracle.encode(w)
    h = hdr(blob)
    assert h["nr"] == 12 and h["ranks"][:12] == list(range(12))
    back, _ = oracle.decode(blob)
    assert np.array_equal(back, w)
    bits, _ = pair_bits_per_lane((w >> 7) & 0xFF, 256)
    assert np.array_equal(lane_words(blob), -(-bits // 32))
    assert escape_lists(blob) == expected_lists((w.astype(np.int64) >> 7) & 0xFF, False, 256)


@pytest.mark.parametrize("shape", [(1, 1), (7, 9), (8, 512), (9, 513), (64, 512), (17, 1100)])
def test_roundtrip_random_shapes(shape):
    w = synth.normal_bf16(shape, 0.02, seed=sum(shape))
    blob = oracle.encode(w)
    back, _ = oracle.decode(blob)
    assert np.array_equal(back, w)
    bits, _ = pair_bits_per_lane((w >> 7) & 0xFF, 256)
    assert np.array_equal(lane_words(blob), -(-bits // 32))


@pytest.mark.parametrize("elem", [oracle.BF16, oracle.FP8])
def test_raw_section_layout(elem):
    """A full block (columns 0..511) keeps the raw bits interleaved across lanes in 16-byte
    units: BF16 columns 2u, 2u+1 of lane l at unit 32u + l, a byte per row; fp8 columns
    4u..4u+3, rows 2i and 2i+1 in the low and high nibble of a byte. The ragged block
    (columns 512..599, rows past N = 13 zero) keeps each lane's real columns in its own
    16-byte padded region. Reading the bits back that way gives every element's sign and
    mantissa."""
    K, N = 600, 13
    w = synth.normal_bf16((N, K), 0.02, seed=13)
    if elem == oracle.FP8:
        q, s = oracle.quantize_fp8(w)
        blob, vals = oracle.encode(q, oracle.FP8, s), q.astype(np.int64)
        raw_of = lambda e: ((e >> 7) << 3) | (e & 7)
        cbytes = 4
    else:
        blob, vals = oracle.encode(w), w.astype(np.int64)
        raw_of = lambda e: ((e >> 15) << 7) | (e & 0x7F)
        cbytes = 8
    b = np.frombuffer(blob, np.uint8)
    for i, (start, end) in enumerate(regions(blob)):
        rb, cb = divmod(i, 2)
        lw = b[start:start + 32].astype(np.int64)
        raw0 = start + -(-(32 + 4 * int(lw.sum())) // 16) * 16
        full = cb == 0
        lane_off = 0
        for l in range(32):
            cols = lane_cols(K, cb, l)
            for c in range(cols):
                for r in range(8):
                    row = 8 * rb + r
                    if cbytes == 8:
                        at = 16 * (32 * (c // 2) + l) + 8 * (c % 2) + r if full else lane_off + 8 * c + r
                        got = int(b[raw0 + at])
                    else:
                        at = 16 * (32 * (c // 4) + l) + 4 * (c % 4) + r // 2 if full else lane_off + 4 * c + r // 2
                        got = (int(b[raw0 + at]) >> (4 * (r % 2))) & 0xF
                    want = raw_of(int(vals[row, 512 * cb + 16 * l + c])) if row < N else 0
                    assert got == want, (i, l, c, r)
            lane_off += -(-cols * cbytes // 16) * 16
        if not full:
            assert raw0 + lane_off <= end


def test_filler_costs_one_bit_and_no_raw_bits_past_k():
    """A 1x1 matrix: every lane holds 64 pairs of one-bit codes = 128 bits = 4 words; the only
    raw region is lane 0's one column (8 bytes, rows past N zero) padded to 16."""
    w = np.array([[0x3F80]], np.uint16)
    blob = oracle.encode(w)
    lw = lane_words(blob)[0]
    assert (lw == 4).all()
    h = hdr(blob)
    assert h["total"] - h["off_data"] == -(-(32 + 4 * 128) // 16) * 16 + 16


def test_size_near_exponent_entropy_for_gaussian_weights():
    """N(0, 0.02), seed 0, 4096x4096: exponent code bits per weight (stream and escape
    lists) within 0.35 of the exponent entropy H; whole blob 65.9%..69.5% of BF16 (the
    pages: about 31% smaller); the entropy bound (8 + H) / 16 below it."""
    w = synth.normal_bf16((4096, 4096), 0.02, seed=0)
    e = (w >> 7) & 0xFF
    p = np.bincount(e.ravel(), minlength=256) / e.size
    H = -(p[p > 0] * np.log2(p[p > 0])).sum()
    bits, _ = pair_bits_per_lane(e, 256)
    blob = oracle.encode(w)
    assert np.array_equal(lane_words(blob), -(-bits // 32))
    n_list = sum(len(x) for x in escape_lists(blob))
    coded = (bits.sum() + 32 * n_list) / w.size
    assert 0.0 <= coded - H <= 0.35, (coded, H)
    frac = len(blob) / (2 * w.size)
    assert 0.659 <= frac <= 0.695, frac
    assert (8 + H) / 16 < frac


def test_outlier_matrix_escapes_and_zeros():
    w = synth.small_matrix_with_outliers(seed=0)
    e = (w >> 7) & 0xFF
    ranked = ranks_of(e, 256)
    escaped = ~np.isin(e, ranked)
    assert len(ranked) == 12 and escaped.sum() > 0
    assert (w == 0).sum() >= 8
    blob = oracle.encode(w)
    back, _ = oracle.decode(blob)
    assert np.array_equal(back, w)
    bits, _ = pair_bits_per_lane(e, 256)
    assert np.array_equal(lane_words(blob), -(-bits // 32))


def test_escape_list_holds_unranked_and_cut_elements_in_lane_t_order():
    """Each listed element appears once, as t | lane << 7 | v << 12, lanes in order and t
    increasing: the unranked real elements and the real second elements of pairs longer
    than 13 bits, no other."""
    rng = np.random.default_rng(3)
    perm = rng.permutation(np.arange(65536, dtype=np.uint32)).astype(np.uint16).reshape(128, 512)
    for w in [synth.small_matrix_with_outliers(seed=0), perm[:13, :512 - 188],
              synth.normal_bf16((40, 1100), 0.02, seed=8)]:
        e = (w.astype(np.int64) >> 7) & 0xFF
        lists = escape_lists(oracle.encode(w))
        assert lists == expected_lists(e, False, 256)
        assert sum(len(x) for x in lists) > 0


def test_fp8_subnormal_and_nan_codes_are_listed():
    """fp8 codes with exponent field 0 and a nonzero mantissa (subnormals) and S.1111.111
    (NaN) are listed whatever their rank; zeros (exponent 0, mantissa 0) are not."""
    rng = np.random.default_rng(5)
    q = rng.integers(0x30, 0x48, size=(16, 600)).astype(np.uint8)     # normal codes near 1.0
    q[0, :40] = np.arange(40) % 8                                      # subnormals and +0
    q[1, 5] = 0x7F
    q[2, 7] = 0xFF                                                     # NaN codes
    q[3, :20] = 0x80                                                   # -0
    s = np.linspace(0.5, 2.0, 16).astype(np.float32)
    blob = oracle.encode(q, oracle.FP8, s)
    back, s2 = oracle.decode(blob)
    assert np.array_equal(back, q) and np.array_equal(s2, s)
    v = (q.astype(np.int64) >> 3) & 0xF
    m = q.astype(np.int64) & 7
    special = ((v == 0) & (m != 0)) | ((v == 15) & (m == 7))
    lists = escape_lists(blob)
    assert lists == expected_lists(v, special, 16)
    flat = {(e & 127, (e >> 7) & 31) for x in lists for e in x}
    # (t, lane) with t = 8 * column + row: q[0, 0] = 0 and q[0, 8] = 0 are zeros, not listed;
    # q[0, 1] = 0x01 is a subnormal, listed
    assert (0, 0) not in flat and (64, 0) not in flat
    assert (8, 0) in flat


def test_encoding_is_deterministic():
    w = synth.normal_bf16((33, 700), 0.02, seed=5)
    assert oracle.encode(w) == oracle.encode(w.copy())


def test_gemv_equals_exact_sum_of_products():
    """Tiny shapes: the oracle's FP64 y equals math.fsum of the exact products
    (BF16 x BF16 is exact in FP64) within FP64 summation error."""
    for n, k, seed in [(3, 5, 1), (9, 513, 2), (16, 1030, 3)]:
        w = synth.normal_bf16((n, k), 0.02, seed)
        x = synth.activations_bf16(k, seed + 100)
        blob = oracle.encode(w)
        y = oracle.gemv(blob, x)
        wf, xf = bf16_f64(w), bf16_f64(x)
        for i in range(n):
            prods = [wf[i, j] * xf[j] for j in range(k)]
            exact = math.fsum(prods)
            bound = k * 2.0 ** -52 * math.fsum(abs(p) for p in prods)
            assert abs(y[i] - exact) <= bound
    # a sampled-row query agrees with the full product
    rows = [8, 0, 15, 8]
    assert np.array_equal(oracle.gemv(blob, x, rows), y[rows])
    ad = oracle.abs_dot(blob, x, rows)
    assert np.allclose(ad, np.abs(wf[rows] * xf).sum(axis=1), rtol=1e-12)


def test_e4m3_rounding_special_cases():
    f = oracle.e4m3_from_f32
    assert f(448.0) == 0x7E and f(1e30) == 0x7E and f(-500.0) == 0xFE  # saturate
    assert f(0.0) == 0x00 and f(-0.0) == 0x80
    assert f(2.0 ** -9) == 0x01            # smallest subnormal
    assert f(2.0 ** -10) == 0x00           # halfway to 0: ties to even
    assert f(3 * 2.0 ** -10) == 0x02       # halfway between codes 1 and 2
    assert f(1.0625) == 0x38               # halfway 1.0 / 1.125 -> even (1.0)
    assert f(1.1875) == 0x3A               # halfway 1.125 / 1.25 -> even (1.25)
    assert f(2.0 ** -6) == 0x08            # smallest normal


def test_e4m3_matches_torch_conversion_in_range():
    """Inside +-448 the e4m3 conversion is round-to-nearest-even, which is
    what torch's float8_e4m3fn cast implements."""
    rng = np.random.default_rng(11)
    xs = np.concatenate([
        rng.uniform(-448, 448, 3000),
        rng.standard_normal(3000) * 2.0 ** rng.integers(-12, 8, 3000),
    ]).astype(np.float32)
    ref = torch.from_numpy(xs).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([oracle.e4m3_from_f32(float(v)) for v in xs], np.uint8)
    assert np.array_equal(got, ref)


def test_fp8_quantization_and_lossless_bytes():
    w = synth.normal_bf16((40, 2560), 0.02, seed=21)
    q, s = oracle.quantize_fp8(w)
    wf = bf16_f64(w)
    absmax = np.abs(wf).max(axis=1).astype(np.float32)
    assert np.array_equal(s, absmax / np.float32(448.0))
    # the largest-magnitude element of each row lands on +-448
    top = np.abs(wf).argmax(axis=1)
    assert np.all((q[np.arange(40), top] & 0x7F) == 0x7E)
    # element-wise: the nearest e4m3 to fp32(w)/s, checked against torch
    quot = (wf.astype(np.float32) / s[:, None]).astype(np.float32)
    ref = torch.from_numpy(quot).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(q, ref)
    blob = oracle.encode(q, oracle.FP8, s)
    back, s2 = oracle.decode(blob)
    assert np.array_equal(back, q) and np.array_equal(s2, s)
    bits, _ = pair_bits_per_lane((q >> 3) & 0xF, 16)
    assert np.array_equal(lane_words(blob), -(-bits // 32))
    # fp8 bytes compress to well under 1 byte (pages: 0.87 on real weights)
    assert 0.78 <= len(blob) / q.size <= 0.90


def test_fp8_gemv_applies_row_scale():
    w = synth.normal_bf16((8, 600), 0.02, seed=4)
    q, s = oracle.quantize_fp8(w)
    blob = oracle.encode(q, oracle.FP8, s)
    x = synth.activations_bf16(600, 9)
    y = oracle.gemv(blob, x)
    qv = torch.from_numpy(q).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    ref = s.astype(np.float64) * (qv @ bf16_f64(x))
    assert np.allclose(y, ref, rtol=1e-12, atol=0)


def test_zero_row_fp8_scale_is_one():
    w = np.zeros((2, 16), np.uint16)
    w[1, 3] = 0x3F80
    q, s = oracle.quantize_fp8(w)
    assert s[0] == 1.0 and (q[0] == 0).all()
    assert q[1, 3] == 0x7E


def test_fp8_dequantize_pins():
    """Dequantization for prefill: BF16 nearest (ties to even) to the FP32 product e4m3(q) * s_n.
    Power-of-two scales make every product exact (an e4m3 value has at most 4 significant bits),
    so the BF16 equals torch's e4m3 value times the scale; hand-worked products pin the rounding."""
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], np.uint8)  # no NaN codes
    for j in (-3, 0, 5):
        s = np.float32(2.0 ** j)
        got = oracle.dequantize_fp8(codes[None, :], np.array([s], np.float32))[0]
        exact = (torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float32) * float(s)).numpy()
        bits = exact.view(np.uint32)
        assert (bits & 0xFFFF == 0).all()
        assert np.array_equal(got, (bits >> 16).astype(np.uint16))
    q = np.array([[0x7E, 0x38, 0x39, 0x38, 0x7F, 0xFF, 0x00, 0x80, 0x01]], np.uint8)
    third = np.float32(1.0 / 3.0)  # 0x3EAAAAAB
    # 448 * fp32(1/3): the FP32 product is 0x43155556, whose low half 0x5556 rounds down -> 0x4315
    assert oracle.dequantize_fp8(q[:, :1], np.array([third], np.float32))[0, 0] == 0x4315
    # 1.0 * (1 + 2^-8) = 0x3F808000: a tie, high half even -> 0x3F80
    # 1.125 * (1 + 2^-8) = 0x3F909000: above the tie -> 0x3F91
    assert list(oracle.dequantize_fp8(q[:, 1:3], np.array([1 + 2.0 ** -8], np.float32))[0]) == [0x3F80, 0x3F91]
    # 1.0 * (1 + 2^-7 + 2^-8) = 0x3F818000: a tie, high half odd -> 0x3F82
    assert oracle.dequantize_fp8(q[:, 3:4], np.array([1 + 2.0 ** -7 + 2.0 ** -8], np.float32))[0, 0] == 0x3F82
    # NaN codes -> 0x7FC0; +0 and -0 keep their sign; the smallest subnormal 2^-9 -> 0x3B00
    assert list(oracle.dequantize_fp8(q[:, 4:], np.array([1.0], np.float32))[0]) == [0x7FC0, 0x7FC0, 0x0000,
                                                                                      0x8000, 0x3B00]
