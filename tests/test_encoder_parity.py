"""Library host encoder (C++) against the CPU oracle, byte for byte (no GPU needed)."""
import numpy as np
import pytest

import decode_gemv_nwc_gb300 as nwc
import oracle
from decode_gemv_nwc_gb300 import synth


@pytest.fixture(scope="module", autouse=True)
def _built():
    from decode_gemv_nwc_gb300 import build
    build.build()


SHAPES = [(1, 1), (1, 513), (7, 9), (8, 512), (9, 513), (64, 512), (17, 1100), (130, 2049)]


@pytest.mark.parametrize("shape", SHAPES)
def test_bf16_bytes_equal_oracle(shape):
    w = synth.normal_bf16(shape, 0.02, seed=shape[0] * 7 + shape[1])
    assert nwc.encode(w) == oracle.encode(w)


def test_all_bf16_patterns_equal_oracle():
    rng = np.random.default_rng(3)
    w = rng.permutation(np.arange(65536, dtype=np.uint32)).astype(np.uint16).reshape(128, 512)
    assert nwc.encode(w) == oracle.encode(w)


def test_outlier_matrix_equal_oracle():
    w = synth.small_matrix_with_outliers(0)
    assert nwc.encode(w) == oracle.encode(w)


def test_few_distinct_exponents():
    # fewer than 11 distinct exponents: no escape code exists
    w = np.tile(np.array([0x3F80, 0xBF80, 0x4000, 0x3F00, 0x0000], np.uint16), (9, 200))[:, :997]
    assert nwc.encode(w) == oracle.encode(w)
    assert oracle.info(oracle.encode(w))["n_ranked"] == 4


def test_strided_input():
    base = synth.normal_bf16((40, 1200), 0.02, seed=9)
    view = base[:, 100:1123]
    assert nwc.encode(view) == oracle.encode(np.ascontiguousarray(view))


def test_thread_count_does_not_change_bytes():
    w = synth.normal_bf16((300, 3000), 0.05, seed=2)
    one = nwc.encode(w, threads=1)
    assert one == nwc.encode(w, threads=0) == nwc.encode(w, threads=5)


@pytest.mark.slow
def test_square_4096_equal_oracle():
    w = synth.normal_bf16((4096, 4096), 0.02, seed=0)
    assert nwc.encode(w) == oracle.encode(w)


def test_fp8_quantizer_equals_oracle():
    w = synth.normal_bf16((64, 2560), 0.02, seed=21)
    q1, s1 = nwc.quantize_fp8(w)
    q2, s2 = oracle.quantize_fp8(w)
    assert np.array_equal(q1, q2) and np.array_equal(s1, s2)
    # exhaustive-ish: many magnitudes through the library quantizer vs the oracle search
    rng = np.random.default_rng(5)
    vals = (rng.standard_normal(4096) * 2.0 ** rng.integers(-14, 6, 4096)).astype(np.float32)
    vals[:3] = [0.0, -0.0, 1e-30]
    w2 = (vals.view(np.uint32) >> 16).astype(np.uint16).reshape(4, 1024)
    q1, s1 = nwc.quantize_fp8(w2)
    q2, s2 = oracle.quantize_fp8(w2)
    assert np.array_equal(q1, q2) and np.array_equal(s1, s2)


@pytest.mark.parametrize("shape", [(8, 512), (9, 2600), (2560, 700)])
def test_fp8_bytes_equal_oracle(shape):
    w = synth.normal_bf16(shape, 0.02, seed=shape[1])
    q, s = oracle.quantize_fp8(w)
    assert nwc.encode_fp8(q, s) == oracle.encode(q, oracle.FP8, s)
    assert nwc.encode(w, elem=nwc.FP8) == oracle.encode(q, oracle.FP8, s)


def test_fp8_rejects_non_finite():
    w = synth.normal_bf16((2, 16), 0.02, seed=1)
    w[1, 3] = 0x7F80  # +Inf
    with pytest.raises(nwc.NwcError):
        nwc.encode(w, elem=nwc.FP8)


def test_encode_fused_stacks_rows():
    """Fused projections: one blob of the row-stacked matrices (equal to encoding the stack),
    with the row offsets of each part; a mismatched column count is refused."""
    ws = [synth.normal_bf16((n, 700), 0.02, seed=n) for n in (24, 5, 5)]
    blob, off = nwc.encode_fused(ws)
    assert blob == oracle.encode(np.concatenate(ws))
    assert list(off) == [0, 24, 29, 34]
    with pytest.raises(ValueError):
        nwc.encode_fused([ws[0], synth.normal_bf16((4, 600), 0.02, seed=1)])
