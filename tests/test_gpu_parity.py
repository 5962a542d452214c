"""GPU parity against the CPU oracle, through the C ABI (needs a CUDA GPU).

Decode and gather must be bit-exact. The matrix-vector product must satisfy, per row,
|y - y_ref| <= 2^-10 * sum_k |w x| + 1e-6 (FP32 output against the oracle's FP64 sum).
"""
import numpy as np
import pytest
import torch

import decode_gemv_nwc_gb300 as nwc
import oracle
from decode_gemv_nwc_gb300 import synth

pytestmark = pytest.mark.gpu
TOL_REL, TOL_ABS = 2.0 ** -10, 1e-6


@pytest.fixture(scope="module", autouse=True)
def _built():
    from decode_gemv_nwc_gb300 import build
    from oracle import parallel
    build.build()
    torch.cuda.init()
    yield
    parallel.shutdown()


def dev_bits(a: np.ndarray):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda()


def assert_clean():
    st, flags = nwc.check()
    assert st == 0, f"device error word {flags:#x}"


def gemv_check(blob, x_bits, rows=None, mat=None):
    mat = mat or nwc.Matrix(blob)
    y = mat.gemv(dev_bits(x_bits)).cpu().numpy().astype(np.float64)
    assert_clean()
    if rows is None:
        rows = np.arange(mat.n)
    ref = oracle.gemv(blob, x_bits, rows)
    scale = oracle.abs_dot(blob, x_bits, rows)
    err = np.abs(y[rows] - ref)
    bound = TOL_REL * scale + TOL_ABS
    worst = int(np.argmax(err - bound))
    assert (err <= bound).all(), f"row {rows[worst]}: |{y[rows][worst]} - {ref[worst]}| > {bound[worst]}"
    return y


def gemv_check_all(blob, x_bits, mat):
    """gemv_check on every row of a large matrix: the oracle's rows split by 8-row blocks over
    the host's cores (oracle.parallel, bit-identical to one process)."""
    from oracle import parallel
    y = mat.gemv(dev_bits(x_bits)).cpu().numpy().astype(np.float64)
    assert_clean()
    with parallel.Oracle(blob) as po:
        ref = po.gemv(x_bits)
        scale = po.abs_dot(x_bits)
    assert ref.shape == y.shape
    err = np.abs(y - ref)
    bound = TOL_REL * scale + TOL_ABS
    worst = int(np.argmax(err - bound))
    assert (err <= bound).all(), f"row {worst}: |{y[worst]} - {ref[worst]}| > {bound[worst]}"
    return y


# --------------------------------------------------------------------- decode
@pytest.mark.parametrize("shape", [(1, 1), (7, 9), (9, 513), (17, 1100), (64, 512), (130, 2049)])
def test_decode_bit_exact_shapes(shape):
    w = synth.normal_bf16(shape, 0.02, seed=sum(shape))
    blob = nwc.encode(w)
    out = nwc.Matrix(blob).decode().cpu().numpy().view(np.uint16)
    assert_clean()
    assert np.array_equal(out, oracle.decode(blob)[0])
    assert np.array_equal(out, w)


def test_decode_all_bf16_patterns():
    rng = np.random.default_rng(3)
    w = rng.permutation(np.arange(65536, dtype=np.uint32)).astype(np.uint16).reshape(128, 512)
    blob = nwc.encode(w)
    out = nwc.Matrix(blob).decode().cpu().numpy().view(np.uint16)
    assert_clean()
    assert np.array_equal(out, w)


def test_decode_outlier_matrix_then_gemv():
    w = synth.small_matrix_with_outliers(0)
    x = synth.activations_bf16(512, 1000)
    blob = nwc.encode(w)
    assert blob == oracle.encode(w)
    mat = nwc.Matrix(blob)
    out = mat.decode().cpu().numpy().view(np.uint16)
    assert np.array_equal(out, w)
    gemv_check(blob, x, mat=mat)


@pytest.mark.parametrize("shape", [(4096, 4096), (4095, 4100)])
def test_square_and_odd_decode_and_gemv(shape):
    w = synth.normal_bf16(shape, 0.02, seed=0 if shape[0] == 4096 else 1)
    x = synth.activations_bf16(shape[1], 1001)
    blob = nwc.encode(w)
    mat = nwc.Matrix(blob)
    out = mat.decode().cpu().numpy().view(np.uint16)
    assert_clean()
    assert np.array_equal(out, w)
    gemv_check(blob, x, mat=mat)


# ----------------------------------------------------------------------- gemv
@pytest.mark.parametrize("shape", [(1, 1), (8, 512), (9, 513), (17, 1100), (33, 4000), (1000, 512), (40, 9728)])
def test_gemv_shapes(shape):
    w = synth.normal_bf16(shape, 0.02, seed=shape[0] + 3 * shape[1])
    x = synth.activations_bf16(shape[1], 7)
    gemv_check(nwc.encode(w), x)


def test_gemv_special_values():
    """Zeros, subnormals, large finite values and +-0 in one matrix (finite only)."""
    rng = np.random.default_rng(17)
    pats = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    finite = pats[((pats >> 7) & 0xFF) != 0xFF]
    # keep magnitudes below 2^40 so the FP32 sum stays finite
    finite = finite[((finite >> 7) & 0xFF) < 127 + 40]
    w = rng.choice(finite, size=(24, 2048)).astype(np.uint16)
    x = synth.activations_bf16(2048, 5)
    gemv_check(nwc.encode(w), x)


def test_gemv_escape_heavy_staged_blocks():
    """About 3% of the elements get exponents far from the bulk (escaped): the regions
    still fit the shared-memory stage, so the fast path's placeholder products and the
    escape-list corrections carry them."""
    rng = np.random.default_rng(23)
    w = synth.normal_bf16((256, 4096), 0.02, seed=23)
    hit = rng.random(w.shape) < 0.03
    odd = (rng.integers(0, 2, w.shape) << 15) | (rng.integers(100, 150, w.shape) << 7) | rng.integers(0, 128, w.shape)
    w = np.where(hit, odd, w).astype(np.uint16)
    blob = nwc.encode(w)
    assert blob == oracle.encode(w)
    mat = nwc.Matrix(blob)
    assert np.array_equal(mat.decode().cpu().numpy().view(np.uint16), w)
    assert_clean()
    gemv_check(blob, synth.activations_bf16(4096, 24), mat=mat)


def test_escape_list_mismatch_is_flagged_not_faulted():
    """An escape list one entry short (still a valid list on the host) leaves a lane
    stream's escape without its entry: decode and the check word report it."""
    w = synth.small_matrix_with_outliers(seed=0)  # 64 x 512: 8 full blocks
    blob = bytearray(nwc.encode(w))
    b = np.frombuffer(bytes(blob), np.uint8)
    off_data = int(b[48:56].view(np.uint64)[0])
    tab = b[80:80 + 4 * 9].view(np.uint32)
    for i in range(8):
        start, end = off_data + 16 * int(tab[i]), off_data + 16 * int(tab[i + 1])
        # escape list: after the code streams and the 4096-byte raw section of a full block
        at = start + -(-(32 + 4 * int(b[start:start + 32].astype(np.int64).sum())) // 16) * 16 + 4096
        words = b[at:end].view(np.uint32)
        n_entries = int((words != 0xFFFFFFFF).sum())
        if n_entries >= 1 and len(words) - n_entries < 3:
            blob[at + 4 * (n_entries - 1):at + 4 * n_entries] = b"\xff\xff\xff\xff"
            break
    else:
        pytest.skip("no block with room for one more padding word")
    assert nwc.validate(bytes(blob)) == 0
    nwc.Matrix(bytes(blob)).decode()
    st, flags = nwc.check()
    assert st == 5 and flags & 1


@pytest.mark.parametrize("elem", [0, 1])
def test_table_built_in_kernel_equals_copied_table(elem):
    """A bound matrix without a device decode table (every kernel builds it in shared memory)
    gives bit for bit the same decode and GEMV as one whose table was copied in."""
    w = synth.normal_bf16((200, 1300), 0.02, seed=17 + elem)
    blob = nwc.encode(w, elem=elem)
    a, b = nwc.Matrix(blob), nwc.Matrix(blob, table=False)
    assert a.table is not None and b.table is None
    da, db = a.decode(), b.decode()
    if elem == 1:
        assert torch.equal(da[0], db[0]) and torch.equal(da[1], db[1])
    else:
        assert torch.equal(da, db)
    x = dev_bits(synth.activations_bf16(1300, 18))
    assert torch.equal(a.gemv(x), b.gemv(x))
    assert_clean()
    gemv_check(blob, synth.activations_bf16(1300, 18), mat=b)


def test_gemv_next_equals_gemv_bitwise():
    """nwc_gemv_next (the same product, with the next matrix's bytes prefetched into L2) gives
    nwc_gemv's result bit for bit, for a chain of three matrices of different shapes."""
    shapes = [(4096, 1024), (1000, 4096), (300, 700)]
    mats, xs = [], []
    for i, (n, k) in enumerate(shapes):
        mats.append(nwc.Matrix(nwc.encode(synth.normal_bf16((n, k), 0.02, seed=60 + i))))
        xs.append(dev_bits(synth.activations_bf16(k, 70 + i)))
    for i, m in enumerate(mats):
        a = m.gemv(xs[i])
        b = m.gemv(xs[i], next=mats[(i + 1) % 3])
        assert torch.equal(a, b)
    assert_clean()


def test_matmul_batch_via_decode_and_cublas():
    """Batch > 1 (prefill): decode to BF16, then cuBLAS. Output BF16, so each entry is checked
    against the FP64 product with BF16 rounding added to the GEMV bound."""
    w = synth.normal_bf16((300, 1100), 0.02, seed=41)
    blob = nwc.encode(w)
    mat = nwc.Matrix(blob)
    xs = np.stack([synth.activations_bf16(1100, 50 + i) for i in range(5)])
    y = mat.matmul(dev_bits(xs)).float().cpu().numpy().astype(np.float64)
    assert_clean()
    for i in range(5):
        ref = oracle.gemv(blob, xs[i])
        scale = oracle.abs_dot(blob, xs[i], np.arange(300))
        assert (np.abs(y[i] - ref) <= TOL_REL * scale + 2.0 ** -8 * np.abs(ref) + TOL_ABS).all()


def test_gemv_repeat_graph_and_stream():
    w = synth.normal_bf16((520, 2600), 0.03, seed=31)
    x = synth.activations_bf16(2600, 32)
    blob = nwc.encode(w)
    mat = nwc.Matrix(blob)
    xd = dev_bits(x)
    y0 = mat.gemv(xd).clone()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        y1 = mat.gemv(xd, stream=s)
    s.synchronize()
    assert torch.equal(y0, y1)  # fixed reduction order: bitwise reproducible
    yg = torch.empty_like(y0)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        mat.gemv(xd, y=yg)
    for _ in range(3):
        yg.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(yg, y0)
    assert_clean()
    gemv_check(blob, x, mat=mat)


# ------------------------------------------------------------------------ fp8
@pytest.mark.parametrize("shape", [(9728, 2560), (2560, 9728), (9, 700)])
def test_fp8_decode_and_gemv(shape):
    w = synth.normal_bf16(shape, 0.02, seed=50 + shape[0])
    q, s = oracle.quantize_fp8(w)
    blob = nwc.encode(w, elem=nwc.FP8)
    assert blob == oracle.encode(q, oracle.FP8, s)
    mat = nwc.Matrix(blob)
    qd, sd = mat.decode()
    assert_clean()
    assert np.array_equal(qd.cpu().numpy(), q) and np.array_equal(sd.cpu().numpy(), s)
    x = synth.activations_bf16(shape[1], 77)
    gemv_check_all(blob, x, mat)


@pytest.mark.parametrize("layer", [0, 17, 35])
@pytest.mark.parametrize("name", [s[0] for s in synth.LAYER_SHAPES])
def test_decoder_stack_matrices_full_size(name, layer):
    """Matrices of the 36-layer stack at full size (BF16; each layer has its own sigma and so its
    own exponent ranking): the first, a middle and the last layer, decode bit-exact and the GEMV
    within tolerance on every row (the shapes the benchmark times)."""
    w = synth.layer_matrix(layer, name)  # BF16 bits, numpy uint16
    n, k = w.shape
    blob = nwc.encode(w)
    mat = nwc.Matrix(blob)
    out = mat.decode().cpu().numpy().view(np.uint16)
    assert_clean()
    assert np.array_equal(out, w)
    x = synth.activations_bf16(k, 2000 + k)
    gemv_check_all(blob, x, mat)


@pytest.mark.parametrize("layer", [0, 35])
@pytest.mark.parametrize("group", [("q", "k", "v"), ("gate", "up")])
def test_fused_projection_blobs(group, layer):
    """Fused projections (the NWC page's fuse step): q|k|v and gate|up of one layer stacked
    row-wise and coded as one blob. The blob decodes to the parts one after another (bit-exact,
    at the offsets encode_fused returns) and its GEMV is within tolerance on every row; each
    part's rows also agree with the GEMV of that part's own blob within the same bound."""
    parts = [synth.layer_matrix(layer, g) for g in group]
    k = parts[0].shape[1]
    blob, offsets = nwc.encode_fused(parts)
    assert offsets.tolist() == np.cumsum([0] + [p.shape[0] for p in parts]).tolist()
    mat = nwc.Matrix(blob)
    out = mat.decode().cpu().numpy().view(np.uint16)
    assert_clean()
    assert np.array_equal(out, np.concatenate(parts))
    x = synth.activations_bf16(k, 2000 + k)
    y = gemv_check_all(blob, x, mat)
    for i, p in enumerate(parts):
        pb = nwc.encode(p)
        yp = nwc.Matrix(pb).gemv(dev_bits(x)).cpu().numpy().astype(np.float64)
        assert_clean()
        bound = 2 * (TOL_REL * oracle.abs_dot(pb, x) + TOL_ABS)
        assert (np.abs(y[offsets[i]:offsets[i + 1]] - yp) <= bound).all()


def test_fp8_subnormal_and_zero_codes():
    rng = np.random.default_rng(8)
    q = rng.integers(0, 256, size=(16, 1024)).astype(np.uint8)
    q[(q & 0x7F) == 0x7F] = 0x01  # no NaN codes in a GEMV test
    s = rng.uniform(0.5, 2.0, 16).astype(np.float32)
    blob = nwc.encode_fp8(q, s)
    mat = nwc.Matrix(blob)
    qd, _ = mat.decode()
    assert np.array_equal(qd.cpu().numpy(), q)
    gemv_check(blob, synth.activations_bf16(1024, 3), mat=mat)


# --------------------------------------------------------------------- gather
def test_gather_bit_exact_and_bad_id():
    w = synth.normal_bf16((1000, 2560), 0.02, seed=7)
    blob = nwc.encode(w)
    mat = nwc.Matrix(blob)
    ids = synth.token_ids(300, 1000, seed=8)
    out = mat.gather(torch.from_numpy(ids).cuda()).cpu().numpy().view(np.uint16)
    assert_clean()
    assert np.array_equal(out, w[ids])
    bad = torch.tensor([3, 1000, -1, 999], dtype=torch.int32, device="cuda")
    out = mat.gather(bad).cpu().numpy().view(np.uint16)
    st, flags = nwc.check()
    assert st == 5 and flags & 2
    assert np.array_equal(out[0], w[3]) and np.array_equal(out[3], w[999])
    assert (out[1] == 0).all() and (out[2] == 0).all()
    assert_clean()  # cleared by the previous check


def test_gather_ragged_width_fp8():
    w = synth.normal_bf16((77, 1300), 0.02, seed=70)
    q, s = oracle.quantize_fp8(w)
    blob = nwc.encode_fp8(q, s)
    mat = nwc.Matrix(blob)
    ids = np.array([0, 76, 8, 8, 15, 64], np.int32)
    out = mat.gather(torch.from_numpy(ids).cuda()).cpu().numpy()
    assert_clean()
    assert np.array_equal(out, q[ids])


def _escape_heavy(shape, seed):
    rng = np.random.default_rng(seed)
    w = synth.normal_bf16(shape, 0.02, seed=seed)
    hit = rng.random(w.shape) < 0.03
    odd = (rng.integers(0, 2, w.shape) << 15) | (rng.integers(100, 150, w.shape) << 7) | rng.integers(0, 128, w.shape)
    return np.where(hit, odd, w).astype(np.uint16)


def test_decode_and_gather_strided_unaligned_outputs():
    """Row strides that are not multiples of 4 and an output start off 8-byte alignment take
    the element-wise store path; untouched columns keep their sentinel."""
    n, k = 40, 2600
    w = _escape_heavy((n, k), 31)
    mat = nwc.Matrix(nwc.encode(w))
    big = torch.full((n, k + 3), -7, dtype=torch.int16, device="cuda")
    view = big[:, 1:k + 1]
    mat.decode(out=view)
    assert_clean()
    got = big.cpu().numpy().view(np.uint16)
    assert np.array_equal(got[:, 1:k + 1], w)
    assert (got[:, 0] == np.uint16(0xFFF9)).all() and (got[:, k + 1:] == np.uint16(0xFFF9)).all()
    ids = np.array([39, 0, 17, 17, 8, 33], np.int32)
    gbig = torch.full((len(ids), k + 1), -7, dtype=torch.int16, device="cuda")
    mat.gather(torch.from_numpy(ids).cuda(), out=gbig[:, :k])
    assert_clean()
    g = gbig.cpu().numpy().view(np.uint16)
    assert np.array_equal(g[:, :k], w[ids]) and (g[:, k] == np.uint16(0xFFF9)).all()
    # fp8 bytes, stride k + 1
    q, sc = oracle.quantize_fp8(w)
    m8 = nwc.Matrix(nwc.encode_fp8(q, sc))
    out8 = torch.zeros((n, k + 1), dtype=torch.uint8, device="cuda")
    o8, s8 = m8.decode(out=out8[:, :k])
    assert_clean()
    assert np.array_equal(out8.cpu().numpy()[:, :k], q) and np.array_equal(s8.cpu().numpy(), sc)


def test_gather_escape_heavy_rows():
    w = _escape_heavy((512, 4096), 32)
    mat = nwc.Matrix(nwc.encode(w))
    ids = synth.token_ids(700, 512, seed=33)
    out = mat.gather(torch.from_numpy(ids).cuda()).cpu().numpy().view(np.uint16)
    assert_clean()
    assert np.array_equal(out, w[ids])


@pytest.mark.slow
def test_embedding_table_gather_and_lm_head_every_row():
    """151936 x 2560 tied table: 4096 random ids bit-exact, then the lm_head GEMV on every
    row (full size, the launch configuration the benchmark times)."""
    w = synth.normal_bf16((synth.VOCAB, synth.HIDDEN), 0.02, seed=7)
    blob = nwc.encode(w)
    mat = nwc.Matrix(blob)
    ids = synth.token_ids(4096, synth.VOCAB, seed=8)
    out = mat.gather(torch.from_numpy(ids).cuda()).cpu().numpy().view(np.uint16)
    assert_clean()
    assert np.array_equal(out, w[ids])
    x = synth.activations_bf16(synth.HIDDEN, 9)
    gemv_check_all(blob, x, mat)


# --------------------------------------------------------------------- small-batch GEMV
def batch_check(blob, xs, rows=None, mat=None, ld_x=None, ld_y=None, repeat=1):
    """nwc_gemv_batch on the vectors xs (list of BF16 bit arrays) against the oracle, per vector;
    x rows ld_x apart and y rows ld_y apart (defaults: K rounded up to 8, N)."""
    mat = mat or nwc.Matrix(blob)
    nb, k, n = len(xs), mat.k, mat.n
    ld_x = ld_x or (k + 7) // 8 * 8
    ld_y = ld_y or n
    xb = np.zeros((nb, ld_x), np.uint16)
    for v, x in enumerate(xs):
        xb[v, :k] = x
    xd = dev_bits(xb)[:, :k]
    yd = torch.full((nb, ld_y), float("nan"), dtype=torch.float32, device="cuda")[:, :n]
    for _ in range(repeat):
        mat.gemv_batch(xd, yd)
    y = yd.cpu().numpy().astype(np.float64)
    assert_clean()
    if rows is None:
        rows = np.arange(n)
    for v, x in enumerate(xs):
        ref = oracle.gemv(blob, x, rows)
        bound = TOL_REL * oracle.abs_dot(blob, x, rows) + TOL_ABS
        err = np.abs(y[v, rows] - ref)
        worst = int(np.argmax(err - bound))
        assert (err <= bound).all(), f"vector {v} row {rows[worst]}: |{y[v, rows][worst]} - {ref[worst]}| > {bound[worst]}"
    return y


@pytest.mark.parametrize("nb", [1, 2, 3, 5, 8, 9, 16])
@pytest.mark.parametrize("shape", [(1, 1), (9, 513), (33, 4000), (40, 9728), (257, 1100)])
def test_gemv_batch_shapes(shape, nb):
    w = synth.normal_bf16(shape, 0.02, seed=shape[0] + 5 * shape[1])
    xs = [synth.activations_bf16(shape[1], 100 + v) for v in range(nb)]
    batch_check(nwc.encode(w), xs)


@pytest.mark.parametrize("nb", [2, 7, 13])
def test_gemv_batch_fp8(nb):
    w = synth.normal_bf16((300, 2600), 0.02, seed=61)
    blob = nwc.encode(w, elem=nwc.FP8)
    xs = [synth.activations_bf16(2600, 200 + v) for v in range(nb)]
    batch_check(blob, xs)


def test_gemv_batch_escape_heavy_and_strided():
    """Escape-list corrections applied to every vector; x and y with padded row strides and a
    second call on the same workspace (counters left at zero by the first)."""
    w = _escape_heavy((256, 4096), 29)
    blob = nwc.encode(w)
    for nb in (6, 11):
        xs = [synth.activations_bf16(4096, 300 + v) for v in range(nb)]
        batch_check(blob, xs, ld_x=4096 + 24, ld_y=256 + 5, repeat=2)


def test_gemv_batch_matches_single_vector_calls_in_tolerance_full_size():
    """The gate projection of the stack at full size, 16 vectors, sampled rows; the same vectors
    through nwc_gemv one at a time agree with the batch within twice the tolerance."""
    w = synth.layer_matrix(0, "gate")
    n, k = w.shape
    blob = nwc.encode(w)
    mat = nwc.Matrix(blob)
    xs = [synth.activations_bf16(k, 400 + v) for v in range(16)]
    rows = np.sort(np.random.default_rng(5).choice(n, 256, False))
    y = batch_check(blob, xs, rows=rows, mat=mat)
    for v in (0, 7, 8, 15):
        y1 = mat.gemv(dev_bits(xs[v])).cpu().numpy().astype(np.float64)
        bound = 2 * (TOL_REL * oracle.abs_dot(blob, xs[v], rows) + TOL_ABS)
        assert (np.abs(y1[rows] - y[v, rows]) <= bound).all()


def test_gemv_batch_fp8_full_size_sampled():
    """fp8 gate projection at full size, 16 vectors: sampled rows of every vector against the
    oracle (row scales applied at the end)."""
    w = synth.normal_bf16((9728, 2560), 0.02, seed=150)
    blob = nwc.encode(w, elem=nwc.FP8)
    xs = [synth.activations_bf16(2560, 500 + v) for v in range(16)]
    rows = np.sort(np.random.default_rng(9).choice(9728, 256, False))
    batch_check(blob, xs, rows=rows)


def test_gemv_batch_one_vector_equals_gemv_bitwise():
    """nwc_gemv_batch with one vector runs the single-vector kernel on the batch workspace."""
    w = synth.normal_bf16((300, 2600), 0.02, seed=88)
    mat = nwc.Matrix(nwc.encode(w))
    x = synth.activations_bf16(2600, 89)
    xb = np.zeros((1, 2608), np.uint16)
    xb[0, :2600] = x
    yb = mat.gemv_batch(dev_bits(xb)[:, :2600]).cpu().numpy()
    y1 = mat.gemv(dev_bits(x)).cpu().numpy()
    assert_clean()
    assert np.array_equal(yb[0].view(np.uint32), y1.view(np.uint32))


def _flip_code_bits(blob, seed, blocks=6, flips=3):
    """Flips random bits in the code streams of random blocks (structure unchanged, so host
    validation accepts the blob)."""
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
@pytest.mark.parametrize("shape", [(64, 1100), (256, 4096)])
def test_corrupted_code_streams_are_flagged_or_decoded_never_faulted(shape, elem):
    """Blobs with flipped code bits (valid structure) through decode, GEMV, batch GEMV and
    gather: every call completes with the device error word clear or set (never a CUDA
    error); where the oracle accepts the corrupted blob and the device word stays clear, the
    decode equals the oracle's bit for bit. A clean matrix afterwards is still exact."""
    w = synth.normal_bf16(shape, 0.02, seed=shape[0] + elem)
    blob = nwc.encode(w, elem=elem)
    n, k = shape
    x = synth.activations_bf16(k, 3)
    for seed in range(4):
        bad = _flip_code_bits(blob, 100 + seed)
        mat = nwc.Matrix(bad)
        out = mat.decode()
        out = (out if elem == 0 else out[0]).cpu().numpy()
        st, _ = nwc.check()
        assert st in (0, 5)
        try:
            ref = oracle.decode(bad)[0]
        except ValueError:
            ref = None
        if ref is not None and st == 0:
            assert np.array_equal(out.view(ref.dtype), ref)
        mat.gemv(dev_bits(x))
        assert nwc.check()[0] in (0, 5)
        xb = np.zeros((3, (k + 7) // 8 * 8), np.uint16)
        xb[:, :k] = x
        mat.gemv_batch(dev_bits(xb)[:, :k])
        assert nwc.check()[0] in (0, 5)
        mat.gather(torch.tensor([0, n - 1, n // 2], dtype=torch.int32, device="cuda"))
        assert nwc.check()[0] in (0, 5)
    gemv_check(blob, x)


def test_tiny_shape_sweep_decode_gemv_batch():
    """Every N, K in {1, 7, 8, 9, 511, 512, 513}: decode bit-exact, GEMV and a 3-vector batch
    GEMV within tolerance (partial row blocks, partial column blocks and single elements)."""
    sizes = [1, 7, 8, 9, 511, 512, 513]
    for n in sizes:
        for k in sizes:
            w = synth.normal_bf16((n, k), 0.02, seed=7 * n + k)
            blob = nwc.encode(w)
            mat = nwc.Matrix(blob)
            assert np.array_equal(mat.decode().cpu().numpy().view(np.uint16), w), (n, k)
            gemv_check(blob, synth.activations_bf16(k, n + k), mat=mat)
            batch_check(blob, [synth.activations_bf16(k, n + k + v) for v in range(3)], mat=mat)


def test_decode_and_gather_8_byte_aligned_rows():
    """Row strides that keep 8-byte but not 16-byte alignment (BF16 K + 4, fp8 K + 8) take the
    8-byte store path; the padding columns keep their sentinel."""
    n, k = 40, 2600
    w = _escape_heavy((n, k), 41)
    mat = nwc.Matrix(nwc.encode(w))
    big = torch.full((n, k + 4), -7, dtype=torch.int16, device="cuda")
    mat.decode(out=big[:, :k])
    assert_clean()
    got = big.cpu().numpy().view(np.uint16)
    assert np.array_equal(got[:, :k], w) and (got[:, k:] == np.uint16(0xFFF9)).all()
    ids = np.array([39, 0, 17, 17, 8, 33], np.int32)
    gbig = torch.full((len(ids), k + 4), -7, dtype=torch.int16, device="cuda")
    mat.gather(torch.from_numpy(ids).cuda(), out=gbig[:, :k])
    assert_clean()
    g = gbig.cpu().numpy().view(np.uint16)
    assert np.array_equal(g[:, :k], w[ids]) and (g[:, k:] == np.uint16(0xFFF9)).all()
    q, sc = oracle.quantize_fp8(w)
    m8 = nwc.Matrix(nwc.encode_fp8(q, sc))
    out8 = torch.full((n, k + 8), 0xAB, dtype=torch.uint8, device="cuda")
    m8.decode(out=out8[:, :k])
    assert_clean()
    o = out8.cpu().numpy()
    assert np.array_equal(o[:, :k], q) and (o[:, k:] == 0xAB).all()


def test_decode_and_gather_4_byte_aligned_rows():
    """Row strides that keep 4-byte but not 8-byte alignment (BF16 K + 2, fp8 K + 4) take the
    4-byte store path; the padding columns keep their sentinel."""
    n, k = 40, 2600
    w = _escape_heavy((n, k), 43)
    mat = nwc.Matrix(nwc.encode(w))
    big = torch.full((n, k + 2), -7, dtype=torch.int16, device="cuda")
    mat.decode(out=big[:, :k])
    assert_clean()
    got = big.cpu().numpy().view(np.uint16)
    assert np.array_equal(got[:, :k], w) and (got[:, k:] == np.uint16(0xFFF9)).all()
    ids = np.array([39, 0, 17, 17, 8, 33], np.int32)
    gbig = torch.full((len(ids), k + 2), -7, dtype=torch.int16, device="cuda")
    mat.gather(torch.from_numpy(ids).cuda(), out=gbig[:, :k])
    assert_clean()
    g = gbig.cpu().numpy().view(np.uint16)
    assert np.array_equal(g[:, :k], w[ids]) and (g[:, k:] == np.uint16(0xFFF9)).all()
    q, sc = oracle.quantize_fp8(w)
    m8 = nwc.Matrix(nwc.encode_fp8(q, sc))
    out8 = torch.full((n, k + 4), 0xAB, dtype=torch.uint8, device="cuda")
    m8.decode(out=out8[:, :k])
    assert_clean()
    o = out8.cpu().numpy()
    assert np.array_equal(o[:, :k], q) and (o[:, k:] == 0xAB).all()
    g8 = torch.full((len(ids), k + 4), 0xAB, dtype=torch.uint8, device="cuda")
    m8.gather(torch.from_numpy(ids).cuda(), out=g8[:, :k])
    assert_clean()
    o = g8.cpu().numpy()
    assert np.array_equal(o[:, :k], q[ids]) and (o[:, k:] == 0xAB).all()


def test_ragged_k_11008_gemv_batch_and_decode():
    """K = 11008 (21.5 column blocks): the ragged last column block of every row block takes the
    fast decoders (single vector, two vectors, 16 vectors on the tensor cores, decode)."""
    n, k = 512, 11008
    w = synth.normal_bf16((n, k), 0.02, seed=110)
    blob = nwc.encode(w)
    mat = nwc.Matrix(blob)
    assert np.array_equal(mat.decode().cpu().numpy().view(np.uint16), w)
    assert_clean()
    rows = np.sort(np.random.default_rng(11).choice(n, 192, False))
    gemv_check(blob, synth.activations_bf16(k, 12), rows=rows, mat=mat)
    for nb in (2, 16):
        batch_check(blob, [synth.activations_bf16(k, 20 + v) for v in range(nb)], rows=rows, mat=mat)


def test_row_ragged_last_row_block_every_height():
    """N = 8 q + r for r = 1..7 (the last row block has r real rows), K full and ragged:
    decode bit-exact; GEMV for one and two vectors and the batch GEMV for 3 and 16 vectors
    within tolerance; BF16 with escapes in the ragged rows, and fp8."""
    for r in range(1, 8):
        for k in (1024, 1000):
            n = 24 + r
            w = _escape_heavy((n, k), 60 + 8 * r + k % 7)
            blob = nwc.encode(w)
            mat = nwc.Matrix(blob)
            assert np.array_equal(mat.decode().cpu().numpy().view(np.uint16), w), (r, k)
            assert_clean()
            gemv_check(blob, synth.activations_bf16(k, 300 + r), mat=mat)
            for nb in (2, 3, 16):
                batch_check(blob, [synth.activations_bf16(k, 310 + r + v) for v in range(nb)], mat=mat)
            q, sc = oracle.quantize_fp8(w)
            b8 = nwc.encode_fp8(q, sc)
            m8 = nwc.Matrix(b8)
            qd, sd = m8.decode()
            assert_clean()
            assert np.array_equal(qd.cpu().numpy(), q) and np.array_equal(sd.cpu().numpy(), sc), (r, k)
            gemv_check(b8, synth.activations_bf16(k, 320 + r), mat=m8)
            for nb in (2, 5):
                batch_check(b8, [synth.activations_bf16(k, 330 + r + v) for v in range(nb)], mat=m8)


def test_infinite_rank0_exponent_keeps_fillers_out_of_real_rows():
    """The most frequent exponent is 0xFF (most elements +-Inf), so filler codes would decode to
    Inf and Inf * 0 would put NaN into real rows: blocks past K or N must skip their fillers.
    Row 0 is finite and must match the oracle; the other rows are non-finite on both sides."""
    rng = np.random.default_rng(91)
    n, k = 13, 1100
    w = np.where(rng.random((n, k)) < 0.5, 0x7F80, 0xFF80).astype(np.uint16)
    w[0] = synth.normal_bf16((1, k), 0.02, seed=92)[0]
    blob = nwc.encode(w)
    mat = nwc.Matrix(blob)
    assert np.array_equal(mat.decode().cpu().numpy().view(np.uint16), w)
    x = synth.activations_bf16(k, 93)
    y = mat.gemv(dev_bits(x)).cpu().numpy().astype(np.float64)
    assert_clean()
    ref = oracle.gemv(blob, x, np.array([0]))
    assert abs(y[0] - ref[0]) <= TOL_REL * oracle.abs_dot(blob, x, np.array([0]))[0] + TOL_ABS
    assert not np.isfinite(y[1:]).any()
    xs = [synth.activations_bf16(k, 94 + v) for v in range(3)]
    xb = np.zeros((3, (k + 7) // 8 * 8), np.uint16)
    for v in range(3):
        xb[v, :k] = xs[v]
    yb = mat.gemv_batch(dev_bits(xb)[:, :k]).cpu().numpy().astype(np.float64)
    assert_clean()
    for v in range(3):
        rv = oracle.gemv(blob, xs[v], np.array([0]))
        assert abs(yb[v, 0] - rv[0]) <= TOL_REL * oracle.abs_dot(blob, xs[v], np.array([0]))[0] + TOL_ABS
        assert not np.isfinite(yb[v, 1:]).any()


def test_inflated_code_streams_in_the_last_stage_are_flagged_not_faulted():
    """Blocks of a ragged K whose lane streams are rewritten to the 26-word maximum with a short
    last lane (valid to the host, every row pair a 13-bit escape), placed where the last warp of
    each CTA stages them (GEMV: warp 31, decode: warp 15): the lanes' decoders read their longest
    possible streams and the last lane reads past its words. Every kernel finishes, the device
    error word reports the malformed blocks, and the context stays usable."""
    import blob_edit
    sms = nwc.sm_count()
    n, k = 8 * 2400, 513  # two column blocks; block 2 rb + 1 is the ragged one
    w = synth.normal_bf16((n, k), 0.02, seed=150)
    blob = nwc.encode(w)
    targets = sorted({(31 * sms) | 1, (15 * sms) | 1})
    bad = blob
    for b in targets:
        assert b < 2 * (n // 8) and b % 2 == 1
        bad = blob_edit.replace_code_streams(bad, b, [26] * 31 + [8])
        start, end = blob_edit.region_bounds(bad, b)
        assert end - start <= 6144
    assert nwc.validate(bad) == 0
    mat = nwc.Matrix(bad)
    x = synth.activations_bf16(k, 151)
    mat.gemv(dev_bits(x))
    st, flags = nwc.check()
    assert st == 5 and flags & 1, (st, flags)
    xb = np.zeros((3, 520), np.uint16)
    for v in range(3):
        xb[v, :k] = synth.activations_bf16(k, 152 + v)
    mat.gemv_batch(dev_bits(xb)[:, :k])
    st, flags = nwc.check()
    assert st == 5 and flags & 1, (st, flags)
    mat.decode()
    st, flags = nwc.check()
    assert st == 5 and flags & 1, (st, flags)
    assert_clean()
    # the rest of the matrix is untouched: rows outside the two rewritten row blocks still match
    good_rows = np.array([r for r in range(0, n, 97) if r // 8 not in {b // 2 for b in targets}])
    gemv_check(blob, x, rows=good_rows, mat=nwc.Matrix(blob))


def test_fp8_dequantize_bit_exact_and_prefill():
    """fp8 prefill: nwc_dequantize_fp8 equals the oracle bit for bit (every byte value, NaN codes
    included; aligned rows on the vector path, ragged and strided rows element by element), and
    Matrix.matmul on an fp8 matrix meets the BF16 GEMM bound against FP64 products of the oracle's
    BF16 weights."""
    import ctypes
    rng = np.random.default_rng(404)
    # every byte value, random row scales; 8-aligned rows (vector path) and a ragged width
    for n, k in ((64, 512), (33, 1001)):
        q = rng.integers(0, 256, (n, k)).astype(np.uint8)
        s = rng.uniform(1e-3, 2.0, n).astype(np.float32)
        qd, sd = torch.from_numpy(q).cuda(), torch.from_numpy(s).cuda()
        out = torch.full((n, k), -7, dtype=torch.int16, device="cuda")
        assert nwc.lib().nwc_dequantize_fp8(ctypes.c_void_p(qd.data_ptr()), k, ctypes.c_void_p(sd.data_ptr()), n, k,
                                            ctypes.c_void_p(out.data_ptr()), k, None) == 0
        torch.cuda.synchronize()
        assert np.array_equal(out.cpu().numpy().view(np.uint16), oracle.dequantize_fp8(q, s)), (n, k)
    # strided output rows with sentinels past K
    q = rng.integers(0, 256, (20, 1000)).astype(np.uint8)
    s = rng.uniform(0.01, 1.0, 20).astype(np.float32)
    qpad = torch.zeros((20, 1008), dtype=torch.uint8, device="cuda")
    qpad[:, :1000] = torch.from_numpy(q).cuda()
    big = torch.full((20, 1016), -7, dtype=torch.int16, device="cuda")
    assert nwc.lib().nwc_dequantize_fp8(ctypes.c_void_p(qpad.data_ptr()), 1008,
                                        ctypes.c_void_p(torch.from_numpy(s).cuda().data_ptr()), 20, 1000,
                                        ctypes.c_void_p(big.data_ptr()), 1016, None) == 0
    torch.cuda.synchronize()
    got = big.cpu().numpy().view(np.uint16)
    assert np.array_equal(got[:, :1000], oracle.dequantize_fp8(q, s)) and (got[:, 1000:] == 0xFFF9).all()
    # through the matrix: decode + dequantize, then prefill on cuBLAS
    w = synth.normal_bf16((300, 2600), 0.02, seed=405)
    qm, sm = oracle.quantize_fp8(w)
    mat = nwc.Matrix(nwc.encode_fp8(qm, sm))
    wq = oracle.dequantize_fp8(qm, sm)
    assert np.array_equal(mat.dequantize().cpu().numpy().view(np.uint16), wq)
    X = np.stack([synth.activations_bf16(2600, 406 + b) for b in range(6)])
    Y = mat.matmul(torch.from_numpy(X.view(np.int16)).cuda()).float().cpu().numpy().astype(np.float64)
    assert_clean()
    Wf = synth.bf16_bits_to_f32(wq).astype(np.float64)
    Xf = synth.bf16_bits_to_f32(X).astype(np.float64)
    ref = Xf @ Wf.T
    bound = 2.0 ** -7 * (np.abs(Xf) @ np.abs(Wf).T) + 1e-6
    assert (np.abs(Y - ref) <= bound).all()


# --------------------------------------------------------------------- GEMV list (one launch)
def _list_run(items, stream=None):
    """nwc_gemv_list over (blob, x_bits) pairs; returns the matrices, the outputs and the inputs."""
    mats = [nwc.Matrix(b) for b, _ in items]
    xs = [dev_bits(x) for _, x in items]
    ys = [torch.full((m.n,), float("nan"), dtype=torch.float32, device="cuda") for m in mats]
    nwc.gemv_list(list(zip(mats, xs, ys)), stream=stream)
    return mats, xs, ys


def test_gemv_list_full_layer_every_row():
    """One decoder layer's products (q|k|v and gate|up fused, o, down, and the seven unfused
    matrices) as one list launch: every y equals that matrix's own nwc_gemv bit for bit and is
    within tolerance of the oracle on every row."""
    ws = {name: synth.layer_matrix(17, name) for name, _, _ in synth.LAYER_SHAPES}
    blobs = [nwc.encode_fused([ws["q"], ws["k"], ws["v"]])[0], nwc.encode(ws["o"]),
             nwc.encode_fused([ws["gate"], ws["up"]])[0], nwc.encode(ws["down"])]
    blobs += [nwc.encode(ws[name]) for name, _, _ in synth.LAYER_SHAPES]
    items = []
    for b in blobs:
        k = oracle.info(b)["K"]
        items.append((b, synth.activations_bf16(k, 5000 + k + len(items))))
    mats, xs, ys = _list_run(items)
    torch.cuda.synchronize()
    assert_clean()
    from oracle import parallel
    for (blob, x), mat, xd, y in zip(items, mats, xs, ys):
        y_one = mat.gemv(xd)
        torch.cuda.synchronize()
        assert torch.equal(y.view(torch.int32), y_one.view(torch.int32))
        with parallel.Oracle(blob) as po:
            ref, scale = po.gemv(x), po.abs_dot(x)
        yy = y.cpu().numpy().astype(np.float64)
        assert (np.abs(yy - ref) <= TOL_REL * scale + TOL_ABS).all()
    assert_clean()


@pytest.mark.parametrize("elem", [nwc.BF16, nwc.FP8])
def test_gemv_list_mixed_shapes_and_many_items(elem):
    """Ragged rows and columns, single-block and one-column-block items, and 200 small items, so
    that CTA ranges cross many item boundaries (a table copy each): every y equals nwc_gemv's bit
    for bit and the oracle's within tolerance."""
    rng = np.random.default_rng(3 + elem)
    shapes = [(1, 1), (7, 9), (9, 513), (17, 1100), (64, 512), (130, 2049), (4095, 4100), (300, 1030)]
    shapes += [(int(rng.integers(1, 40)), int(rng.integers(1, 1600))) for _ in range(192)]
    items = []
    for i, s in enumerate(shapes):
        w = synth.normal_bf16(s, 0.02, seed=900 + i)
        items.append((nwc.encode(w, elem=elem), synth.activations_bf16(s[1], 901 + i)))
    mats, xs, ys = _list_run(items)
    torch.cuda.synchronize()
    assert_clean()
    for (blob, x), mat, xd, y in zip(items, mats, xs, ys):
        assert torch.equal(y.view(torch.int32), mat.gemv(xd).view(torch.int32))
        ref, scale = oracle.gemv(blob, x), oracle.abs_dot(blob, x)
        yy = y.cpu().numpy().astype(np.float64)
        assert (np.abs(yy - ref) <= TOL_REL * scale + TOL_ABS).all()
    assert_clean()


def test_gemv_list_repeats_in_a_graph_and_checks_arguments():
    """The list launch leaves every workspace prepared: graph replays give the same bits. Bad
    lists are rejected before any launch."""
    items = [(nwc.encode(synth.normal_bf16((520, 1500), 0.02, seed=i)), synth.activations_bf16(1500, i))
             for i in range(3)]
    mats, xs, ys = _list_run(items)
    torch.cuda.synchronize()
    first = [y.clone() for y in ys]
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        nwc.gemv_list(list(zip(mats, xs, ys)), stream=s)
    for _ in range(3):
        for y in ys:
            y.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert all(torch.equal(a.view(torch.int32), b.view(torch.int32)) for a, b in zip(ys, first))
    assert_clean()
    import ctypes
    L = nwc.lib()
    arr = (nwc.NwcGemvItem * 2)()
    for i in range(2):
        arr[i].m = ctypes.pointer(mats[i].m)
        arr[i].x = xs[i].data_ptr()
        arr[i].y = ys[i].data_ptr()
        arr[i].ws = mats[0].workspace.data_ptr()  # both items on one workspace
        arr[i].ws_bytes = mats[0].ws_bytes
    st = torch.cuda.current_stream().cuda_stream
    assert L.nwc_gemv_list(arr, 2, ctypes.c_void_p(st)) == 1
    assert L.nwc_gemv_list(arr, 0, ctypes.c_void_p(st)) == 1
    assert L.nwc_gemv_list(arr, 257, ctypes.c_void_p(st)) == 1
    fp8 = nwc.Matrix(nwc.encode(synth.normal_bf16((16, 600), 0.02, seed=5), elem=nwc.FP8))
    arr[1].m = ctypes.pointer(fp8.m)  # mixed element types
    arr[1].ws = fp8.workspace.data_ptr()
    arr[1].ws_bytes = fp8.ws_bytes
    assert L.nwc_gemv_list(arr, 2, ctypes.c_void_p(st)) == 1
    notable = nwc.Matrix(items[0][0], table=False)  # no device decode table
    arr[0].m = ctypes.pointer(notable.m)
    arr[0].ws = notable.workspace.data_ptr()
    assert L.nwc_gemv_list(arr, 1, ctypes.c_void_p(st)) == 1


@pytest.mark.parametrize("elem", [nwc.BF16, nwc.FP8])
def test_tall_matrix_through_the_list_kernel_equals_the_single_kernel(elem):
    """A matrix tall enough that every SM's share holds 32 whole row blocks (41000 x 1030: ragged
    K, three column blocks) runs nwc_gemv through the list kernel, whose whole row blocks are
    summed by one warp each: y equals the single-matrix kernel's (the path taken without a device
    decode table) bit for bit, and the oracle's within tolerance on every row."""
    w = synth.normal_bf16((41000, 1030), 0.02, seed=77)
    blob = nwc.encode(w, elem=elem)
    x = synth.activations_bf16(1030, 78)
    routed = nwc.Matrix(blob)
    single = nwc.Matrix(blob, table=False)
    y = gemv_check_all(blob, x, routed)
    y_single = single.gemv(dev_bits(x)).cpu().numpy().astype(np.float64)
    assert_clean()
    assert np.array_equal(y.view(np.uint64), y_single.view(np.uint64))


# every shape below runs the round-robin kernel on a 152-SM GB300 except 41000x1030 (the list
# kernel)
ROUTES_152 = {(13, 700): nwc.ROUTE_GEMV, (72, 1500): nwc.ROUTE_GEMV, (1000, 1030): nwc.ROUTE_GEMV,
              (1024, 2560): nwc.ROUTE_GEMV, (4096, 4096): nwc.ROUTE_GEMV, (41000, 1030): nwc.ROUTE_LIST}


@pytest.mark.parametrize("elem", [nwc.BF16, nwc.FP8])
@pytest.mark.parametrize("shape", list(ROUTES_152))
def test_every_route_equals_the_list_kernel_bitwise(shape, elem):
    """nwc_gemv through the kernel nwc_gemv_route names equals nwc_gemv_list with the matrix as
    its only item bit for bit (one fixed order of the column blocks' sums in every kernel), and
    the oracle within tolerance on every row; ragged K (700, 1030) takes the edge layout. Twice
    in a row, so the workspace is back in its prepared state after each call."""
    n, k = shape
    w = synth.normal_bf16((n, k), 0.02, seed=n + k)
    blob = nwc.encode(w, elem=elem)
    x = synth.activations_bf16(k, 7)
    m = nwc.Matrix(blob)
    if nwc.sm_count() == 152:
        assert m.route() == ROUTES_152[shape]
    y = gemv_check_all(blob, x, m) if n * k > 4_000_000 else gemv_check(blob, x, mat=m)
    y2 = m.gemv(dev_bits(x)).cpu().numpy().astype(np.float64)
    yl = torch.empty(n, dtype=torch.float32, device="cuda")
    nwc.gemv_list([(m, dev_bits(x), yl)])
    torch.cuda.synchronize()
    assert_clean()
    yl = yl.cpu().numpy().astype(np.float64)
    assert np.array_equal(y.view(np.uint64), y2.view(np.uint64))
    assert np.array_equal(y.view(np.uint64), yl.view(np.uint64))
