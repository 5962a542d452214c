"""Pins of the CPU oracle to facts that do not come from the oracle itself.

The pages fix: lossless round trip ("bit-exact"), about 31% smaller than BF16
for LLM weights because that is the exponent entropy, 2 bits per filler with
no mantissa, a unary rank code with a raw sign bit and an escape for rare
exponents, and an fp8 variant whose bytes come back bit for bit. Mathematics
fixes the plain matrix-vector product and the e4m3 rounding. Each test below
would fail for a plausible mistake in the oracle (dropped term, wrong sign,
wrong bit order, transposed operand, off-by-one rank).
"""
import math
import os

import numpy as np
import pytest
import torch

import oracle
from decode_gemv_nwc_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ----------------------------------------------------------------- helpers
def hdr(blob):
    b = np.frombuffer(blob, np.uint8)
    u64 = lambda o: int(b[o:o + 8].view(np.uint64)[0])
    return dict(nr=int(b[7]), N=u64(8), K=u64(16), nb=u64(24), off_blocks=u64(32),
                off_scales=u64(40), off_data=u64(48), total=u64(56), ranks=b[64:80].tolist())


def lane_words(blob):
    """Per block, the 32 lane word counts read straight from the blob."""
    h = hdr(blob)
    b = np.frombuffer(blob, np.uint8)
    tab = b[h["off_blocks"]:h["off_blocks"] + 4 * (h["nb"] + 1)].view(np.uint32)
    out = []
    for i in range(h["nb"]):
        start = h["off_data"] + 16 * int(tab[i])
        out.append(b[start:start + 32].astype(np.int64))
    return np.array(out)


def ranks_of(values, nvals):
    """Independent ranking: numpy histogram, (count desc, value asc), <= 11 ranks."""
    cnt = np.bincount(values.ravel(), minlength=nvals)
    order = sorted([v for v in range(nvals) if cnt[v] > 0], key=lambda v: (-cnt[v], v))
    return order[:11]


def code_bits_per_lane(v, nvals, exp_bits):
    """Closed-form lane stream lengths: rank+2 bits per ranked element,
    n_ranked + 1 per escaped one (its exponent lives in the escape list), 2 per
    filler. Returns (RB*CB, 32)."""
    n, k = v.shape
    ranked = ranks_of(v, nvals)
    nr = len(ranked)
    length = np.full(nvals, nr + 1, np.int64)
    for p, e in enumerate(ranked):
        length[e] = p + 2
    rb, cb = -(-n // 8), -(-k // 512)
    L = np.full((rb * 8, cb * 512), 2, np.int64)
    L[:n, :k] = length[v]
    # (rb, r, cb, lane, c) -> sum over r, c
    L = L.reshape(rb, 8, cb, 32, 16).sum(axis=(1, 4))
    return L.reshape(rb * cb, 32), nr


def bf16_f64(bits):
    return synth.bf16_bits_to_f32(np.asarray(bits, np.uint16)).astype(np.float64)


# ---------------------------------------------------------------- the pins
def test_golden_tiny_blob_matches_hand_derivation():
    w = np.array([[0x3FC0, 0xC020], [0x3F20, 0x3F81]], np.uint16)
    blob = oracle.encode(w)
    want = None
    checks = []
    with open(os.path.join(GOLDEN, "nwc_2x2_bf16.txt")) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if not line:
                continue
            parts = line.split()
            if parts[0] == "total":
                want = int(parts[1])
            else:
                checks.append(parts)
    assert len(blob) == want
    b = np.frombuffer(blob, np.uint8)
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
    diff = np.nonzero(b != expected)[0]
    assert diff.size == 0, f"blob differs from the hand derivation at bytes {diff[:16]}"
    back, _ = oracle.decode(blob)
    assert np.array_equal(back, w)


def test_roundtrip_all_65536_bf16_patterns():
    """Every BF16 bit pattern once (+-0, subnormals, +-Inf, NaN payloads):
    256 distinct exponents force 245 escaped exponent values."""
    rng = np.random.default_rng(3)
    w = rng.permutation(np.arange(65536, dtype=np.uint32)).astype(np.uint16).reshape(128, 512)
    blob = oracle.encode(w)
    h = hdr(blob)
    assert h["nr"] == 11
    # all exponents tie (256 each): ranks are the 11 smallest exponent values
    assert h["ranks"][:11] == list(range(11))
    back, _ = oracle.decode(blob)
    assert np.array_equal(back, w)
    bits, nr = code_bits_per_lane((w >> 7) & 0xFF, 256, 8)
    assert nr == 11
    assert np.array_equal(lane_words(blob), -(-bits // 32))


@pytest.mark.parametrize("shape", [(1, 1), (7, 9), (8, 512), (9, 513), (64, 512), (17, 1100)])
def test_roundtrip_random_shapes(shape):
    w = synth.normal_bf16(shape, 0.02, seed=sum(shape))
    blob = oracle.encode(w)
    back, _ = oracle.decode(blob)
    assert np.array_equal(back, w)
    bits, _ = code_bits_per_lane((w >> 7) & 0xFF, 256, 8)
    assert np.array_equal(lane_words(blob), -(-bits // 32))


def test_mantissas_interleaved_when_lanes_agree():
    """A full block (every lane 28 words): word k of lane l is word 32k + l of the mantissa
    section. The ragged block (columns 512..599) keeps the lanes' regions one after another.
    Reading the fields back that way gives every element's raw 7-bit mantissa."""
    K = 600
    w = synth.normal_bf16((8, K), 0.02, seed=13)
    blob = oracle.encode(w)
    h = hdr(blob)
    b = np.frombuffer(blob, np.uint8)
    tab = b[h["off_blocks"]:h["off_blocks"] + 4 * (h["nb"] + 1)].view(np.uint32)
    for cb in range(2):
        start = h["off_data"] + 16 * int(tab[cb])
        lw = b[start:start + 32].astype(np.int64)
        man0 = start + -(-(32 + 4 * int(lw.sum())) // 16) * 16
        cols = [min(16, max(0, K - 512 * cb - 16 * l)) for l in range(32)]
        mw = [-(-(-(-7 * c * 4 // 16)) // 4) * 4 for c in cols]
        uniform = len(set(mw)) == 1
        assert uniform == (cb == 0)
        words = b[man0:man0 + 4 * sum(mw)].view(np.uint32)
        off = 0
        for l in range(32):
            lane_words = [int(words[32 * j + l]) if uniform else int(words[off + j]) for j in range(mw[l])]
            off += mw[l]
            for half, rows in ((0, (0, 2, 4, 6)), (1, (1, 3, 5, 7))):
                stream = 0
                for j, wd in enumerate(lane_words):
                    stream |= ((wd >> (16 * half)) & 0xFFFF) << (16 * j)
                jfield = 0
                for c in range(cols[l]):
                    for r in rows:
                        m = (stream >> (7 * jfield)) & 0x7F
                        assert m == int(w[r, 512 * cb + 16 * l + c]) & 0x7F
                        jfield += 1


def test_filler_costs_two_bits_and_no_mantissa():
    """A 1x1 matrix: lanes 1..31 hold 128 fillers = 256 bits = 8 words; the
    only mantissa region is lane 0's 16 bytes."""
    w = np.array([[0x3F80]], np.uint16)
    blob = oracle.encode(w)
    lw = lane_words(blob)[0]
    assert lw[0] == -(-(2 + 127 * 2) // 32) and (lw[1:] == 8).all()
    h = hdr(blob)
    code_region = -(-(32 + 4 * int(lw.sum())) // 16) * 16
    assert h["total"] - h["off_data"] == code_region + 16


def test_size_near_exponent_entropy_for_gaussian_weights():
    """N(0, 0.02), seed 0, 4096x4096: coded bits per weight within 0.25 of
    1 + H(exponent) (sign + entropy); whole blob 65.9%..69.5% of BF16 (the
    pages: about 31% smaller)."""
    w = synth.normal_bf16((4096, 4096), 0.02, seed=0)
    e = (w >> 7) & 0xFF
    p = np.bincount(e.ravel(), minlength=256) / e.size
    H = -(p[p > 0] * np.log2(p[p > 0])).sum()
    bits, nr = code_bits_per_lane(e, 256, 8)
    coded_per_weight = bits.sum() / w.size
    assert 0.0 <= coded_per_weight - (1 + H) <= 0.25
    blob = oracle.encode(w)
    assert np.array_equal(lane_words(blob), -(-bits // 32))
    frac = len(blob) / (2 * w.size)
    assert 0.659 <= frac <= 0.695, frac
    # and the entropy bound itself (7 raw + 1 sign + H) / 16 is below it
    assert (8 + H) / 16 < frac


def test_outlier_matrix_escapes_and_zeros():
    w = synth.small_matrix_with_outliers(seed=0)
    e = (w >> 7) & 0xFF
    ranked = ranks_of(e, 256)
    escaped = ~np.isin(e, ranked)
    assert len(ranked) == 11 and escaped.sum() > 0
    assert (w == 0).sum() >= 8
    blob = oracle.encode(w)
    back, _ = oracle.decode(blob)
    assert np.array_equal(back, w)
    bits, _ = code_bits_per_lane(e, 256, 8)
    assert np.array_equal(lane_words(blob), -(-bits // 32))


def escape_lists(blob, elem_bits_F):
    """Per block, the escape-list entries read straight from the blob: the
    region's tail after the code streams and the closed-form mantissa regions."""
    h = hdr(blob)
    b = np.frombuffer(blob, np.uint8)
    tab = b[h["off_blocks"]:h["off_blocks"] + 4 * (h["nb"] + 1)].view(np.uint32)
    N, K = h["N"], h["K"]
    cb_n = -(-K // 512)
    out = []
    for i in range(h["nb"]):
        start, end = h["off_data"] + 16 * int(tab[i]), h["off_data"] + 16 * int(tab[i + 1])
        lw = b[start:start + 32].astype(np.int64)
        at = start + -(-(32 + 4 * int(lw.sum())) // 16) * 16
        rb, cb = divmod(i, cb_n)
        rows = min(8, N - 8 * rb)
        for lane in range(32):
            cols = int(np.clip(K - 512 * cb - 16 * lane, 0, 16))
            n_even = cols * ((rows + 1) // 2)
            words = -(-(-(-elem_bits_F * n_even // 16)) // 4) * 4
            at += 4 * words
        ent = b[at:end].view(np.uint32)
        out.append([int(e) for e in ent if e != 0xFFFFFFFF])
        assert all(e == 0xFFFFFFFF for e in ent[len(out[-1]):]), "padding must follow the entries"
    return out


def test_escape_list_holds_every_unranked_element_in_lane_t_order():
    """Each escaped element appears once, as t | lane << 7 | bits << 12, lanes in
    order and t increasing; no ranked element appears."""
    for w, elem, F, nvals, ebits in [
        (synth.small_matrix_with_outliers(seed=0), oracle.BF16, 7, 256, 8),
        (np.random.default_rng(3).permutation(np.arange(65536, dtype=np.uint32)).astype(np.uint16)
         .reshape(128, 512)[:13, :700 - 188], oracle.BF16, 7, 256, 8),
    ]:
        e = (w.astype(np.int64) >> 7) & 0xFF
        ranked = ranks_of(e, nvals)
        blob = oracle.encode(w)
        lists = escape_lists(blob, F)
        n, k = w.shape
        cb_n = -(-k // 512)
        total = 0
        for i, ent in enumerate(lists):
            rb, cb = divmod(i, cb_n)
            want = []
            for lane in range(32):
                for t in range(128):
                    r, c = 8 * rb + t % 8, 512 * cb + 16 * lane + t // 8
                    if r < n and c < k and e[r, c] not in ranked:
                        want.append(t | lane << 7 | int(w[r, c]) << 12)
            assert ent == want
            total += len(ent)
        assert total == int((~np.isin(e, ranked)).sum()) > 0


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
    bits, _ = code_bits_per_lane((q >> 3) & 0xF, 16, 4)
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
