"""Python binding of the NWC C ABI (``include/nwc.h``, ``_build/libnwc.so``).

Argument marshalling only: every step of encode, decode, gather and the fused
decode-GEMV runs in the library (host encoder in C++, sm_103a kernels). PyTorch
supplies device memory and streams. There is no fallback: if the library is
missing or fails to load, every call raises.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

__all__ = [
    "BF16", "FP8", "NwcError", "lib", "encode", "encode_fp8", "quantize_fp8", "validate",
    "Matrix", "check", "sm_count", "status_str", "save", "load", "file_entries", "decode_table", "gemv_list",
]

BF16, FP8 = 0, 1
BATCH_MAX = 16  # NWC_GEMV_BATCH_MAX: vectors per nwc_gemv_batch call
_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "_build", "libnwc.so")


class NwcError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: {status_str(status) if _lib else status} ({status})")
        self.status = status


LIST_MAX = 256  # NWC_GEMV_LIST_MAX: products per nwc_gemv_list call
ROUTE_GEMV, ROUTE_LIST = 0, 2  # NWC_ROUTE_*: the kernel nwc_gemv launches


class NwcMatrix(ctypes.Structure):
    """Mirror of struct nwc_matrix."""
    _fields_ = [
        ("elem", ctypes.c_int32), ("n_ranked", ctypes.c_int32),
        ("n", ctypes.c_int64), ("k", ctypes.c_int64),
        ("row_blocks", ctypes.c_int64), ("col_blocks", ctypes.c_int64),
        ("rank_exp", ctypes.c_uint8 * 16),
        ("block_tab", ctypes.c_void_p), ("data", ctypes.c_void_p), ("scales", ctypes.c_void_p),
        ("blob_bytes", ctypes.c_uint64), ("max_block_bytes", ctypes.c_uint64),
        ("data_bytes", ctypes.c_uint64), ("table", ctypes.c_void_p),
    ]


class NwcGemvItem(ctypes.Structure):
    """Mirror of struct nwc_gemv_item."""
    _fields_ = [("m", ctypes.POINTER(NwcMatrix)), ("x", ctypes.c_void_p), ("y", ctypes.c_void_p),
                ("ws", ctypes.c_void_p), ("ws_bytes", ctypes.c_size_t)]


_lib = None


def lib():
    """The loaded libnwc.so (built by ``__graft_entry__.build()`` / ``build.build()``)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"libnwc.so not built ({LIB_PATH}); run decode_gemv_nwc_gb300.build.build()")
    L = ctypes.CDLL(LIB_PATH)
    p, i64, u64, i32, sz = ctypes.c_void_p, ctypes.c_int64, ctypes.c_uint64, ctypes.c_int, ctypes.c_size_t
    L.nwc_status_str.argtypes = [i32]
    L.nwc_status_str.restype = ctypes.c_char_p
    L.nwc_version.restype = ctypes.c_char_p
    L.nwc_encode.argtypes = [p, i64, i64, i64, i32, i32, p, ctypes.POINTER(sz)]
    L.nwc_encode_fp8.argtypes = [p, p, i64, i64, i64, i32, p, ctypes.POINTER(sz)]
    L.nwc_quantize_fp8.argtypes = [p, i64, i64, i64, p, i64, p]
    L.nwc_validate.argtypes = [p, sz]
    L.nwc_bind.argtypes = [p, sz, p, ctypes.POINTER(NwcMatrix)]
    L.nwc_decode.argtypes = [ctypes.POINTER(NwcMatrix), p, i64, p, p]
    L.nwc_dequantize_fp8.argtypes = [p, i64, p, i64, i64, p, i64, p]
    L.nwc_gemv_workspace_bytes.argtypes = [ctypes.POINTER(NwcMatrix)]
    L.nwc_gemv_workspace_bytes.restype = sz
    L.nwc_gemv_prepare.argtypes = [ctypes.POINTER(NwcMatrix), p, sz, p]
    L.nwc_gemv.argtypes = [ctypes.POINTER(NwcMatrix), p, p, p, sz, p]
    L.nwc_gemv_next.argtypes = [ctypes.POINTER(NwcMatrix), p, p, p, sz, ctypes.POINTER(NwcMatrix), p]
    L.nwc_gemv_noalloc.argtypes = [ctypes.POINTER(NwcMatrix), p, p, p]
    L.nwc_gemv_batch_workspace_bytes.argtypes = [ctypes.POINTER(NwcMatrix), i32]
    L.nwc_gemv_batch_workspace_bytes.restype = sz
    L.nwc_gemv_batch_prepare.argtypes = [ctypes.POINTER(NwcMatrix), i32, p, sz, p]
    L.nwc_gemv_batch.argtypes = [ctypes.POINTER(NwcMatrix), p, i64, i32, p, i64, p, sz, p]
    L.nwc_gather.argtypes = [ctypes.POINTER(NwcMatrix), p, i64, p, i64, p]
    L.nwc_check.argtypes = [p, ctypes.POINTER(ctypes.c_uint32)]
    L.nwc_decode_table.argtypes = [ctypes.POINTER(NwcMatrix), p]
    L.nwc_sm_count.restype = i32
    cp = ctypes.c_char_p
    L.nwc_file_save.argtypes = [cp, i32, ctypes.POINTER(cp), ctypes.POINTER(p), ctypes.POINTER(sz)]
    L.nwc_file_count.argtypes = [cp, ctypes.POINTER(i32)]
    L.nwc_file_entry.argtypes = [cp, i32, p, sz, ctypes.POINTER(sz)]
    L.nwc_file_find.argtypes = [cp, cp, ctypes.POINTER(i32)]
    L.nwc_file_read.argtypes = [cp, i32, p, sz, ctypes.POINTER(sz)]
    L.nwc_file_load.argtypes = [cp, i32, p, sz, p, sz, ctypes.POINTER(NwcMatrix), p]
    L.nwc_gemv_list.argtypes = [ctypes.POINTER(NwcGemvItem), i32, p]
    L.nwc_gemv_route.argtypes = [ctypes.POINTER(NwcMatrix), ctypes.POINTER(i32)]
    for name in ("nwc_encode", "nwc_encode_fp8", "nwc_quantize_fp8", "nwc_validate", "nwc_bind",
                 "nwc_decode", "nwc_gemv_prepare", "nwc_gemv", "nwc_gemv_noalloc", "nwc_gemv_batch_prepare",
                 "nwc_gemv_batch", "nwc_gather", "nwc_check", "nwc_decode_table", "nwc_gemv_next",
                 "nwc_dequantize_fp8", "nwc_file_save", "nwc_file_count", "nwc_file_entry", "nwc_file_find",
                 "nwc_file_read", "nwc_file_load", "nwc_gemv_list", "nwc_gemv_route"):
        getattr(L, name).restype = i32
    _lib = L
    return L


def status_str(status: int) -> str:
    return lib().nwc_status_str(int(status)).decode()


def _ok(status: int, what: str):
    if status != 0:
        raise NwcError(status, what)


def _np_ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _stream_ptr(stream):
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def encode(w_bits: np.ndarray, elem: int = BF16, threads: int = 0) -> bytes:
    """Host encoder: (N, K) BF16 bit patterns (uint16, any row stride) -> blob."""
    w = np.asarray(w_bits)
    if w.dtype != np.uint16 or w.ndim != 2 or w.strides[1] != 2:
        w = np.ascontiguousarray(w, dtype=np.uint16)
    n, k = w.shape
    ld = w.strides[0] // 2
    size = ctypes.c_size_t(0)
    _ok(lib().nwc_encode(_np_ptr(w), n, k, ld, elem, threads, None, ctypes.byref(size)), "nwc_encode")
    out = np.empty(size.value, np.uint8)
    _ok(lib().nwc_encode(_np_ptr(w), n, k, ld, elem, threads, _np_ptr(out), ctypes.byref(size)), "nwc_encode")
    return out.tobytes()


def encode_fused(ws, elem: int = BF16, threads: int = 0):
    """Fused projections (the NWC page's fuse step): matrices that read the same input (q, k, v;
    gate, up) stacked row-wise and encoded as one blob, so that one GEMV serves them all.
    ws: (N_i, K) BF16 bit arrays with a common K. Returns (blob, offsets), where rows
    offsets[i] .. offsets[i + 1] of the fused output belong to ws[i]."""
    ws = [np.asarray(w) for w in ws]
    if not ws or any(w.ndim != 2 or w.shape[1] != ws[0].shape[1] for w in ws):
        raise ValueError("encode_fused: 2-D matrices with a common column count")
    offsets = np.concatenate([[0], np.cumsum([w.shape[0] for w in ws])]).astype(np.int64)
    return encode(np.concatenate(ws, axis=0), elem=elem, threads=threads), offsets


def encode_fp8(q: np.ndarray, scales: np.ndarray, threads: int = 0) -> bytes:
    q = np.ascontiguousarray(q, dtype=np.uint8)
    s = np.ascontiguousarray(scales, dtype=np.float32)
    n, k = q.shape
    size = ctypes.c_size_t(0)
    _ok(lib().nwc_encode_fp8(_np_ptr(q), _np_ptr(s), n, k, k, threads, None, ctypes.byref(size)), "nwc_encode_fp8")
    out = np.empty(size.value, np.uint8)
    _ok(lib().nwc_encode_fp8(_np_ptr(q), _np_ptr(s), n, k, k, threads, _np_ptr(out), ctypes.byref(size)),
        "nwc_encode_fp8")
    return out.tobytes()


def quantize_fp8(w_bits: np.ndarray):
    w = np.ascontiguousarray(w_bits, dtype=np.uint16)
    n, k = w.shape
    q = np.empty((n, k), np.uint8)
    s = np.empty(n, np.float32)
    _ok(lib().nwc_quantize_fp8(_np_ptr(w), n, k, k, _np_ptr(q), k, _np_ptr(s)), "nwc_quantize_fp8")
    return q, s


def validate(blob: bytes) -> int:
    b = np.frombuffer(blob, np.uint8)
    return int(lib().nwc_validate(_np_ptr(b), len(blob)))


def sm_count() -> int:
    return int(lib().nwc_sm_count())


def check(stream=None):
    """(status, flags) of the device error word; synchronizes the stream."""
    flags = ctypes.c_uint32(0)
    st = lib().nwc_check(_stream_ptr(stream), ctypes.byref(flags))
    return int(st), int(flags.value)


def decode_table(m: NwcMatrix) -> np.ndarray:
    """The matrix's decode table (uint32[8192]) built on the host by nwc_decode_table."""
    t = np.empty(8192, np.uint32)
    _ok(lib().nwc_decode_table(ctypes.byref(m), _np_ptr(t)), "nwc_decode_table")
    return t


class Matrix:
    """A blob resident in device memory and bound through nwc_bind.

    ``device_blob`` is a torch uint8 CUDA tensor holding the blob (caller-visible so that
    benchmarks can keep several copies); the decode table is built on the host, copied to the
    device once and named in the bound matrix (``table=False`` leaves it out: every kernel then
    builds it in shared memory); the GEMV workspace is allocated once, put in its starting state
    by nwc_gemv_prepare, and reused by every call.
    """

    def __init__(self, blob: bytes, device="cuda", device_blob=None, table: bool = True):
        import torch
        host = np.frombuffer(blob, np.uint8)
        if device_blob is None:
            device_blob = torch.from_numpy(host.copy()).to(device)
        m = NwcMatrix()
        _ok(lib().nwc_bind(_np_ptr(host), len(blob), ctypes.c_void_p(device_blob.data_ptr()), ctypes.byref(m)),
            "nwc_bind")
        self._set_up(m, device_blob, table, None)

    @classmethod
    def from_file(cls, path: str, name: str, device="cuda", table: bool = True, stream=None):
        """The blob called ``name`` in a file written by save(), loaded straight into device memory
        by nwc_file_load (read into a page-locked host buffer, validated, bound, one copy)."""
        import torch
        idx, size = ctypes.c_int(), ctypes.c_size_t()
        path_b = os.fsencode(path)
        _ok(lib().nwc_file_find(path_b, name.encode(), ctypes.byref(idx)), f"nwc_file_find {name}")
        _ok(lib().nwc_file_entry(path_b, idx.value, None, 0, ctypes.byref(size)), "nwc_file_entry")
        host = torch.empty(size.value, dtype=torch.uint8, pin_memory=True)
        device_blob = torch.empty(size.value, dtype=torch.uint8, device=device)
        m = NwcMatrix()
        _ok(lib().nwc_file_load(path_b, idx.value, ctypes.c_void_p(host.data_ptr()), size.value,
                                ctypes.c_void_p(device_blob.data_ptr()), size.value, ctypes.byref(m),
                                _stream_ptr(stream)), f"nwc_file_load {name}")
        self = cls.__new__(cls)
        self._set_up(m, device_blob, table, stream)
        (stream or torch.cuda.current_stream()).synchronize()  # the host buffer may go now
        return self

    def _set_up(self, m: NwcMatrix, device_blob, table: bool, stream):
        import torch
        self.device_blob = device_blob
        self.m = m
        self.table = None
        if table:
            self.table = torch.from_numpy(decode_table(self.m).view(np.int32)).to(device_blob.device)
            self.m.table = ctypes.c_void_p(self.table.data_ptr())
        self.elem, self.n, self.k = self.m.elem, self.m.n, self.m.k
        self.blob_bytes = int(m.blob_bytes)
        ws = int(lib().nwc_gemv_workspace_bytes(ctypes.byref(self.m)))
        self.workspace = torch.empty(ws, dtype=torch.uint8, device=device_blob.device)
        self.ws_bytes = ws
        _ok(lib().nwc_gemv_prepare(ctypes.byref(self.m), ctypes.c_void_p(self.workspace.data_ptr()), ws,
                                   _stream_ptr(stream)), "nwc_gemv_prepare")

    def gemv(self, x, y=None, stream=None, next=None):
        """y (float32[N]) = W x for x a BF16 vector given as an int16/bfloat16 CUDA tensor. next: the
        Matrix multiplied after this one, whose weights this call brings into L2 (nwc_gemv_next)."""
        import torch
        assert x.numel() == self.k and x.is_cuda and x.is_contiguous()
        if y is None:
            y = torch.empty(self.n, dtype=torch.float32, device=x.device)
        if next is None:
            _ok(lib().nwc_gemv(ctypes.byref(self.m), ctypes.c_void_p(x.data_ptr()), ctypes.c_void_p(y.data_ptr()),
                               ctypes.c_void_p(self.workspace.data_ptr()), self.ws_bytes,
                               _stream_ptr(stream)), "nwc_gemv")
        else:
            _ok(lib().nwc_gemv_next(ctypes.byref(self.m), ctypes.c_void_p(x.data_ptr()), ctypes.c_void_p(y.data_ptr()),
                                    ctypes.c_void_p(self.workspace.data_ptr()), self.ws_bytes, ctypes.byref(next.m),
                                    _stream_ptr(stream)), "nwc_gemv_next")
        return y

    def route(self) -> int:
        """The kernel gemv() launches for this matrix on the current device (nwc_gemv_route):
        ROUTE_GEMV or ROUTE_LIST."""
        r = ctypes.c_int(-1)
        _ok(lib().nwc_gemv_route(ctypes.byref(self.m), ctypes.byref(r)), "nwc_gemv_route")
        return r.value

    def gemv_batch(self, x, y=None, stream=None):
        """Y (float32[nb, N]) = W x[v] for the nb <= 16 rows of x (BF16 [nb, K] as an int16/bfloat16
        CUDA tensor, row stride a multiple of 8): one fused pass that decodes every weight once
        (one vector: the single-vector kernel).
        The batch workspace (sized for 16 vectors) is allocated and prepared on first use."""
        import torch
        assert x.dim() == 2 and x.shape[1] == self.k and x.is_cuda and x.stride(1) == 1
        nb = x.shape[0]
        if y is None:
            y = torch.empty((nb, self.n), dtype=torch.float32, device=x.device)
        if getattr(self, "_bws", None) is None:
            bws = int(lib().nwc_gemv_batch_workspace_bytes(ctypes.byref(self.m), BATCH_MAX))
            self._bws = torch.empty(bws, dtype=torch.uint8, device=self.device_blob.device)
            _ok(lib().nwc_gemv_batch_prepare(ctypes.byref(self.m), BATCH_MAX, ctypes.c_void_p(self._bws.data_ptr()), bws,
                                             _stream_ptr(stream)), "nwc_gemv_batch_prepare")
        _ok(lib().nwc_gemv_batch(ctypes.byref(self.m), ctypes.c_void_p(x.data_ptr()), x.stride(0), nb,
                                 ctypes.c_void_p(y.data_ptr()), y.stride(0), ctypes.c_void_p(self._bws.data_ptr()),
                                 self._bws.numel(), _stream_ptr(stream)), "nwc_gemv_batch")
        return y

    def decode(self, out=None, stream=None):
        """Stored elements: int16 (BF16 bits) [N, K], or (uint8 e4m3 [N, K], float32 scales [N])."""
        import torch
        dev = self.device_blob.device
        if self.elem == BF16:
            out = out if out is not None else torch.empty((self.n, self.k), dtype=torch.int16, device=dev)
            _ok(lib().nwc_decode(ctypes.byref(self.m), ctypes.c_void_p(out.data_ptr()), out.stride(0), None,
                                 _stream_ptr(stream)), "nwc_decode")
            return out
        out = out if out is not None else torch.empty((self.n, self.k), dtype=torch.uint8, device=dev)
        scales = torch.empty(self.n, dtype=torch.float32, device=dev)
        _ok(lib().nwc_decode(ctypes.byref(self.m), ctypes.c_void_p(out.data_ptr()), out.stride(0),
                             ctypes.c_void_p(scales.data_ptr()), _stream_ptr(stream)), "nwc_decode")
        return out, scales

    def dequantize(self, out=None, stream=None):
        """fp8 matrices: BF16 weights [N, K] (int16 bits), each the BF16 nearest to e4m3(q) * s_n
        (nwc_decode to e4m3 bytes and scales, then nwc_dequantize_fp8). The e4m3 bytes and scales
        pass through one scratch pair kept by this Matrix, so calls on the same Matrix must be
        ordered on one stream (calls on different streams that overlap would overwrite it)."""
        import torch
        assert self.elem == FP8, "dequantize serves fp8 matrices"
        dev = self.device_blob.device
        if getattr(self, "_q8", None) is None:  # kept: the kernels may still read it after return
            self._q8 = torch.empty((self.n, self.k), dtype=torch.uint8, device=dev)
            self._s8 = torch.empty(self.n, dtype=torch.float32, device=dev)
        q, scales = self._q8, self._s8
        _ok(lib().nwc_decode(ctypes.byref(self.m), ctypes.c_void_p(q.data_ptr()), q.stride(0),
                             ctypes.c_void_p(scales.data_ptr()), _stream_ptr(stream)), "nwc_decode")
        out = out if out is not None else torch.empty((self.n, self.k), dtype=torch.int16, device=dev)
        _ok(lib().nwc_dequantize_fp8(ctypes.c_void_p(q.data_ptr()), q.stride(0), ctypes.c_void_p(scales.data_ptr()),
                                     self.n, self.k, ctypes.c_void_p(out.data_ptr()), out.stride(0),
                                     _stream_ptr(stream)), "nwc_dequantize_fp8")
        return out

    def matmul(self, x, scratch=None, stream=None):
        """Batch > 1 (prefill): Y[B, N] = X[B, K] W^T in BF16. The matrix is decoded into a BF16
        scratch (allocated once and kept unless given; fp8 matrices are dequantized into it) and
        multiplied by cuBLAS through torch: the pages' prefill (weights back to BF16, then a BF16
        GEMM). The kept scratch is shared by every call on this Matrix: order such calls on one
        stream, or pass each stream its own scratch."""
        import torch
        if scratch is None:
            scratch = getattr(self, "_scratch", None)
            if scratch is None:
                scratch = torch.empty((self.n, self.k), dtype=torch.int16, device=self.device_blob.device)
                self._scratch = scratch
        if self.elem == BF16:
            self.decode(out=scratch, stream=stream)
        else:
            self.dequantize(out=scratch, stream=stream)
        s = stream if stream is not None else torch.cuda.current_stream()
        with torch.cuda.stream(s):
            return torch.nn.functional.linear(x.view(torch.bfloat16), scratch.view(torch.bfloat16))

    def gather(self, ids, out=None, stream=None):
        """Rows ids (int32 CUDA tensor) of the stored matrix, bit-exact."""
        import torch
        assert ids.dtype == torch.int32 and ids.is_cuda and ids.is_contiguous()
        dt = torch.int16 if self.elem == BF16 else torch.uint8
        out = out if out is not None else torch.empty((ids.numel(), self.k), dtype=dt, device=ids.device)
        _ok(lib().nwc_gather(ctypes.byref(self.m), ctypes.c_void_p(ids.data_ptr()), ids.numel(),
                             ctypes.c_void_p(out.data_ptr()), out.stride(0), _stream_ptr(stream)), "nwc_gather")
        return out


def gemv_list(items, stream=None):
    """y_i = W_i x_i for independent products in one launch (nwc_gemv_list). items: (Matrix, x,
    y) triples (x BF16 [K] as an int16/bfloat16 CUDA tensor, y float32 [N]), each matrix with
    its device decode table and using its own workspace; every x must be ready (no item reads
    another's y). Each y equals Matrix.gemv's result bit for bit."""
    arr = (NwcGemvItem * len(items))()
    for i, (mat, x, y) in enumerate(items):
        assert x.numel() == mat.k and x.is_cuda and x.is_contiguous() and y.numel() == mat.n and y.is_contiguous()
        arr[i].m = ctypes.pointer(mat.m)
        arr[i].x = x.data_ptr()
        arr[i].y = y.data_ptr()
        arr[i].ws = mat.workspace.data_ptr()
        arr[i].ws_bytes = mat.ws_bytes
    _ok(lib().nwc_gemv_list(arr, len(items), _stream_ptr(stream)), "nwc_gemv_list")


# ------------------------------------------------------------------ blob files
def save(path: str, blobs: dict) -> None:
    """Writes named blobs (name -> blob bytes) to one file with nwc_file_save (every blob
    validated; the file is replaced whole or left as it was)."""
    names = list(blobs)
    n = len(names)
    c_names = (ctypes.c_char_p * n)(*[k.encode() for k in names])
    bufs = [np.frombuffer(blobs[k], np.uint8) for k in names]
    c_blobs = (ctypes.c_void_p * n)(*[b.ctypes.data for b in bufs])
    c_sizes = (ctypes.c_size_t * n)(*[b.size for b in bufs])
    _ok(lib().nwc_file_save(os.fsencode(path), n, c_names, c_blobs, c_sizes), f"nwc_file_save {path}")


def file_entries(path: str) -> list:
    """(name, blob length) of every entry of a blob file, in file order."""
    path_b = os.fsencode(path)
    count = ctypes.c_int()
    _ok(lib().nwc_file_count(path_b, ctypes.byref(count)), f"nwc_file_count {path}")
    out, name, size = [], ctypes.create_string_buffer(4097), ctypes.c_size_t()
    for i in range(count.value):
        _ok(lib().nwc_file_entry(path_b, i, name, len(name), ctypes.byref(size)), "nwc_file_entry")
        out.append((name.value.decode(), size.value))
    return out


def load(path: str) -> dict:
    """Every blob of a file written by save(), read and validated by nwc_file_read."""
    path_b = os.fsencode(path)
    out = {}
    for i, (name, size) in enumerate(file_entries(path)):
        buf = np.empty(size, np.uint8)
        _ok(lib().nwc_file_read(path_b, i, _np_ptr(buf), size, None), f"nwc_file_read {name}")
        out[name] = buf.tobytes()
    return out
