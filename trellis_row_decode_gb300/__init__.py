"""Python binding of libcp, the GB300 (sm_103a) CP lookup-decode.

Argument marshalling only: every step of the decode runs in the CUDA kernels of
libcp.so (built in-tree by ``trellis_row_decode_gb300.build_ext``).  PyTorch is
used for device memory and streams.  There is no CPU fallback: if libcp.so is
missing or fails to load, every call raises.

The operations (pages cited by title, [P4] "2비트 코드와 공유 트렐리스로 n-gram
룩업 테이블을 4~8배 압축한다"): a table row is an independently addressable
record (code c_i, bf16 scale alpha_i); looking up ids r_j returns
e_hat_j = alpha_{r_j} * f(c_{r_j}) as bf16 rows in lookup order [P4 sections
어떻게 동작하나 and 무엇과 다른가].  The C ABI is declared in include/cp.h.
"""
from __future__ import annotations

import ctypes as C
from pathlib import Path

import numpy as np
import torch

__all__ = [
    "CPError", "Table", "load_table", "lookup_decode", "lookup_decode_host", "get_status",
    "record_bytes", "soa_bytes", "default_lut", "lib", "LIB_PATH", "lookup_decode_host_noalloc",
    "lookup_decode_reduce", "set_cache", "load_mixed_table", "encode_rows",
    "measure_stream_read", "measure_record_read", "encode_workspace", "encode_rows_ws",
    "CP_LAYOUT_AOS", "CP_LAYOUT_SOA", "CP_RESIDENT_DEVICE", "CP_RESIDENT_HOST",
]

_PKG = Path(__file__).resolve().parent
LIB_PATH = _PKG / "_build" / "libcp.so"
LUT_PATH = _PKG / "data" / "cp_lut_v2_l16_512.bin"

CP_OK, CP_ERR_INVALID_ARG, CP_ERR_INDEX_OOB, CP_ERR_CUDA, CP_ERR_NO_MEMORY, CP_ERR_FORMAT = range(6)
CP_LAYOUT_AOS, CP_LAYOUT_SOA = 0, 1
CP_RESIDENT_DEVICE, CP_RESIDENT_HOST = 0, 1

_lib = None


class CPError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        msg = _lib.cp_status_string(status).decode() if _lib else str(status)
        detail = _lib.cp_last_error().decode() if _lib else ""
        super().__init__(f"{what}: {msg}" + (f" ({detail})" if detail else ""))


def lib():
    """The loaded libcp.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not LIB_PATH.exists():
            raise RuntimeError(f"libcp.so not built at {LIB_PATH}; run "
                               "`python -c 'import __graft_entry__ as g; g.build()'`")
        L = C.CDLL(str(LIB_PATH))
        vp, u64, u32, i32 = C.c_void_p, C.c_uint64, C.c_uint32, C.c_int
        L.cp_record_bytes.restype = u64
        L.cp_record_bytes.argtypes = [u32, u32]
        L.cp_soa_bytes.restype = u64
        L.cp_soa_bytes.argtypes = [u64, u32, u32]
        L.cp_table_load.restype = i32
        L.cp_table_load.argtypes = [C.POINTER(vp), vp, u64, u32, u32, vp, i32, i32, vp, vp]
        L.cp_lookup_decode.restype = i32
        L.cp_lookup_decode.argtypes = [vp, vp, u64, vp, vp]
        L.cp_lookup_decode_host.restype = i32
        L.cp_lookup_decode_host.argtypes = [vp, vp, u64, vp, vp]
        L.cp_get_status.restype = i32
        L.cp_get_status.argtypes = [vp, vp]
        L.cp_table_free.restype = None
        L.cp_table_free.argtypes = [vp]
        L.cp_status_string.restype = C.c_char_p
        L.cp_status_string.argtypes = [i32]
        L.cp_last_error.restype = C.c_char_p
        L.cp_last_error.argtypes = []
        L.cp_test_inject_failure.restype = i32
        L.cp_test_inject_failure.argtypes = [i32, i32]
        L.cp_encode_rows.restype = i32
        L.cp_encode_rows.argtypes = [vp, u64, u32, u32, vp, vp, vp, vp]
        L.cp_table_load_mixed.restype = i32
        L.cp_table_load_mixed.argtypes = [C.POINTER(vp), vp, vp, u64, u32, vp, vp]
        L.cp_table_set_cache.restype = i32
        L.cp_table_set_cache.argtypes = [vp, vp, u64, vp, vp]
        L.cp_lookup_decode_reduce.restype = i32
        L.cp_lookup_decode_reduce.argtypes = [vp, vp, u64, u32, vp, vp, vp]
        L.cp_lookup_decode_host_noalloc.restype = i32
        L.cp_lookup_decode_host_noalloc.argtypes = [vp, u64, u32, u32, vp, vp, u64, vp, vp, vp]
        L.cp_encode_workspace_bytes.restype = u64
        L.cp_encode_workspace_bytes.argtypes = [u64, u32, u32]
        L.cp_encode_rows_ws.restype = i32
        L.cp_encode_rows_ws.argtypes = [vp, u64, u32, u32, vp, vp, vp, vp, u64, vp]
        L.cp_measure_stream_read.restype = i32
        L.cp_measure_stream_read.argtypes = [vp, u64, vp]
        L.cp_measure_record_read.restype = i32
        L.cp_measure_record_read.argtypes = [vp, u64, u32, vp, u64, vp]
        _lib = L
    return _lib


def _check(status: int, what: str) -> None:
    if status != CP_OK:
        raise CPError(status, what)


def _stream_ptr(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream)


def record_bytes(d: int, k: int) -> int:
    return int(lib().cp_record_bytes(d, k))


def soa_bytes(n_rows: int, d: int, k: int) -> int:
    return int(lib().cp_soa_bytes(n_rows, d, k))


def default_lut() -> np.ndarray:
    """The shared fp16 LUT (512 x (y0, y1) bit patterns) of this format."""
    return np.fromfile(LUT_PATH, dtype="<u2").reshape(512, 2)


class Table:
    """A loaded compressed table.  Borrows `records` (and `soa`); keeps them alive."""

    def __init__(self, handle: int, n_rows: int, d: int, k: int, residency: int, layout: int,
                 keepalive: tuple):
        self.handle = handle
        self.n_rows, self.d, self.k = n_rows, d, k
        self.residency, self.layout = residency, layout
        self._keepalive = keepalive

    def close(self) -> None:
        if self.handle:
            lib().cp_table_free(self.handle)
            self.handle = 0

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def _check_span(records: torch.Tensor, n_rows: int, d: int, k: int) -> None:
    """The kernels read up to n_rows * R bytes of `records` (R = record_bytes(d, k)),
    which the C ABI cannot check: refuse a shorter buffer before anything is queued."""
    R = record_bytes(d, k)
    if R and n_rows > 0 and records.numel() < n_rows * R:
        raise ValueError(f"records holds {records.numel()} bytes, fewer than n_rows * R = "
                         f"{n_rows} * {R}")


def load_table(records: torch.Tensor, n_rows: int, d: int, k: int, lut: np.ndarray | None = None,
               layout: int = CP_LAYOUT_AOS, soa: torch.Tensor | None = None,
               stream=None) -> Table:
    """Bind AoS records (uint8, device tensor or pinned host tensor) to a handle.

    Residency follows the tensor: CUDA -> CP_RESIDENT_DEVICE, CPU -> CP_RESIDENT_HOST.
    For layout=CP_LAYOUT_SOA pass `soa` (uint8, soa_bytes(n_rows, d, k) bytes) to
    receive the on-device repack.
    """
    L = lib()
    if records.dtype != torch.uint8 or not records.is_contiguous():
        raise ValueError("records must be a contiguous uint8 tensor")
    residency = CP_RESIDENT_DEVICE if records.is_cuda else CP_RESIDENT_HOST
    _check_span(records, n_rows, d, k)
    if lut is None:
        lut = default_lut()
    lut = np.ascontiguousarray(lut, dtype=np.uint16).reshape(512, 2)
    h = C.c_void_p(0)
    soa_ptr = None
    if layout == CP_LAYOUT_SOA:
        if soa is None:
            raise ValueError("CP_LAYOUT_SOA needs the soa buffer")
        if soa.dtype != torch.uint8 or not soa.is_contiguous() or soa.is_cuda != records.is_cuda \
                or soa.numel() < soa_bytes(n_rows, d, k):
            raise ValueError("soa must be a contiguous uint8 tensor of soa_bytes(n_rows, d, k) "
                             "bytes on the records' side (device or pinned host)")
        soa_ptr = soa.data_ptr()
    st = L.cp_table_load(C.byref(h), records.data_ptr(), n_rows, d, k,
                         lut.ctypes.data, residency, layout, soa_ptr, _stream_ptr(stream))
    _check(st, "cp_table_load")
    return Table(h.value, n_rows, d, k, residency, layout, (records, soa, lut))


def load_mixed_table(records: torch.Tensor, offsets: torch.Tensor, d: int,
                     lut: np.ndarray | None = None, stream=None) -> Table:
    """Bind a mixed-rate table: record r at records[offsets[r]:offsets[r+1]] (device
    uint8 / int64 tensors); each row's rate follows from its record length."""
    if not (records.is_cuda and offsets.is_cuda) or records.dtype != torch.uint8 \
            or offsets.dtype != torch.int64:
        raise ValueError("records (uint8) and offsets (int64) must be CUDA tensors")
    if lut is None:
        lut = default_lut()
    lut = np.ascontiguousarray(lut, dtype=np.uint16).reshape(512, 2)
    if not offsets.is_contiguous() or not records.is_contiguous() or offsets.numel() < 2:
        raise ValueError("records and offsets must be contiguous, offsets of n_rows + 1 entries")
    if int(offsets[-1].item()) > records.numel():
        raise ValueError("offsets[n_rows] exceeds the bytes held by records")
    h = C.c_void_p(0)
    n_rows = offsets.numel() - 1
    st = lib().cp_table_load_mixed(C.byref(h), records.data_ptr(), offsets.data_ptr(), n_rows, d,
                                   lut.ctypes.data, _stream_ptr(stream))
    _check(st, "cp_table_load_mixed")
    return Table(h.value, n_rows, d, 0, CP_RESIDENT_DEVICE, CP_LAYOUT_AOS, (records, offsets, lut))


def _decode(fn, table: Table, idx: torch.Tensor, out: torch.Tensor | None, stream, what: str):
    if idx.dtype != torch.int64 or not idx.is_cuda or not idx.is_contiguous():
        raise ValueError("idx must be a contiguous int64 CUDA tensor")
    n = idx.numel()
    if out is None:
        out = torch.empty((n, table.d), dtype=torch.bfloat16, device=idx.device)
    elif out.dtype != torch.bfloat16 or out.shape != (n, table.d) or not out.is_contiguous():
        raise ValueError("out must be a contiguous bf16 tensor of shape (n, d)")
    _check(fn(table.handle, idx.data_ptr(), n, out.data_ptr(), _stream_ptr(stream)), what)
    return out


def lookup_decode(table: Table, idx: torch.Tensor, out: torch.Tensor | None = None,
                  stream=None) -> torch.Tensor:
    """bf16 [n, d] rows alpha_r * f(c_r) for r = idx[j], in lookup order (HBM-resident table).

    `out` may be a CUDA tensor or a pinned host tensor (the kernel then writes the
    rows over the host link).  Only kernels are queued, so the call can be
    captured into a CUDA graph."""
    return _decode(lib().cp_lookup_decode, table, idx, out, stream, "cp_lookup_decode")


def lookup_decode_host(table: Table, idx: torch.Tensor, out: torch.Tensor | None = None,
                       stream=None) -> torch.Tensor:
    """Same as lookup_decode for a table resident in pinned host memory (zero-copy reads)."""
    return _decode(lib().cp_lookup_decode_host, table, idx, out, stream,
                   "cp_lookup_decode_host")


def lookup_decode_reduce(table: Table, idx: torch.Tensor, group: int,
                         weights: torch.Tensor | None = None, out: torch.Tensor | None = None,
                         stream=None) -> torch.Tensor:
    """Decode fused with a weighted group readout: bf16 [n // group, d], row g =
    bf16(sum_i w_i * row_i) over lookups g*group .. g*group+group-1 (fp32 fmaf in order)."""
    if idx.dtype != torch.int64 or not idx.is_cuda or not idx.is_contiguous():
        raise ValueError("idx must be a contiguous int64 CUDA tensor")
    if group <= 0 or idx.numel() % group:
        raise ValueError("the number of ids must be a multiple of group")
    n_groups = idx.numel() // group
    if out is None:
        out = torch.empty((n_groups, table.d), dtype=torch.bfloat16, device=idx.device)
    elif out.dtype != torch.bfloat16 or out.shape != (n_groups, table.d) or not out.is_contiguous():
        raise ValueError("out must be a contiguous bf16 tensor of shape (n_groups, d)")
    wp = None
    if weights is not None:
        if weights.dtype != torch.float32 or not weights.is_cuda or weights.numel() != idx.numel():
            raise ValueError("weights must be float32 CUDA with one weight per id")
        wp = weights.contiguous().data_ptr()
    _check(lib().cp_lookup_decode_reduce(table.handle, idx.data_ptr(), n_groups, group, wp,
                                         out.data_ptr(), _stream_ptr(stream)),
           "cp_lookup_decode_reduce")
    return out


def set_cache(table: Table, hot_rows, cache: torch.Tensor | None = None, stream=None) -> None:
    """Keep device copies of the records of `hot_rows` (distinct ids) for a host-resident
    table; `cache` is a uint8 CUDA tensor of len(hot_rows) * R bytes (allocated if None).
    An empty list removes the cache."""
    rows = np.ascontiguousarray(np.asarray(hot_rows, dtype=np.int64))
    m = rows.size
    if m and cache is None:
        cache = torch.empty(m * record_bytes(table.d, table.k), dtype=torch.uint8, device="cuda")
    if m and (not cache.is_cuda or cache.dtype != torch.uint8 or not cache.is_contiguous()
              or cache.numel() < m * record_bytes(table.d, table.k)):
        raise ValueError("cache must be a contiguous uint8 CUDA tensor of len(hot_rows) * R bytes")
    ptr = cache.data_ptr() if m else None
    _check(lib().cp_table_set_cache(table.handle, rows.ctypes.data if m else None, m, ptr,
                                    _stream_ptr(stream)), "cp_table_set_cache")
    table._cache = cache if m else None


def encode_rows(e: torch.Tensor, k: int, lut: np.ndarray | None = None, stream=None):
    """GPU compression of fp32 rows e [rows, d] into AoS records (uint8 [rows, R]) and the
    fp32 search costs; tail-biting two-pass Viterbi, norm-restoring bf16 alpha."""
    if not e.is_cuda or e.dtype != torch.float32 or e.dim() != 2 or not e.is_contiguous():
        raise ValueError("e must be a contiguous 2-D float32 CUDA tensor")
    rows, d = e.shape
    if lut is None:
        lut = default_lut()
    lut = np.ascontiguousarray(lut, dtype=np.uint16).reshape(512, 2)
    rec = torch.empty((rows, record_bytes(d, k)), dtype=torch.uint8, device=e.device)
    cost = torch.empty(rows, dtype=torch.float32, device=e.device)
    _check(lib().cp_encode_rows(e.data_ptr(), rows, d, k, lut.ctypes.data, rec.data_ptr(),
                                cost.data_ptr(), _stream_ptr(stream)), "cp_encode_rows")
    return rec, cost


def measure_stream_read(buf: torch.Tensor, stream=None) -> None:
    """Queue one streaming read of all of `buf` (device memory, or pinned host memory
    read zero-copy over the host link); time it with events on `stream`."""
    if not buf.is_contiguous() or (buf.numel() * buf.element_size()) % 16:
        raise ValueError("buf must be contiguous with a size that is a multiple of 16 bytes")
    _check(lib().cp_measure_stream_read(buf.data_ptr(), buf.numel() * buf.element_size(),
                                        _stream_ptr(stream)), "cp_measure_stream_read")


def measure_record_read(table: torch.Tensor, record_bytes: int, rows: torch.Tensor,
                        stream=None) -> None:
    """Queue one read of the records `rows` (device int64) of `table` (a record
    table in device memory or pinned host memory, R = record_bytes per row), each
    as the 16-byte pieces that cover it; time it with events on `stream`."""
    if not table.is_contiguous() or not rows.is_contiguous() or rows.dtype != torch.int64:
        raise ValueError("table must be contiguous and rows a contiguous int64 tensor")
    if not rows.is_cuda:
        raise ValueError("rows must be in device memory")
    _check(lib().cp_measure_record_read(table.data_ptr(), table.numel() * table.element_size(),
                                        record_bytes, rows.data_ptr(), rows.numel(),
                                        _stream_ptr(stream)), "cp_measure_record_read")


def encode_workspace(rows: int, d: int, k: int) -> torch.Tensor:
    """A device workspace for encode_rows_ws (uint8, cp_encode_workspace_bytes bytes)."""
    nb = int(lib().cp_encode_workspace_bytes(rows, d, k))
    if nb == 0:
        raise CPError(CP_ERR_INVALID_ARG, "cp_encode_workspace_bytes")
    return torch.empty(nb, dtype=torch.uint8, device="cuda")


def encode_rows_ws(e: torch.Tensor, k: int, workspace: torch.Tensor, records: torch.Tensor,
                   cost: torch.Tensor | None = None, lut: np.ndarray | None = None,
                   stream=None) -> None:
    """encode_rows into caller buffers with a caller-owned workspace; only queues work
    on `stream` (no synchronisation, no allocation)."""
    if not e.is_cuda or e.dtype != torch.float32 or e.dim() != 2 or not e.is_contiguous():
        raise ValueError("e must be a contiguous 2-D float32 CUDA tensor")
    rows, d = e.shape
    if records.dtype != torch.uint8 or not records.is_cuda or not records.is_contiguous() \
            or records.numel() < rows * record_bytes(d, k):
        raise ValueError("records must be a contiguous uint8 CUDA tensor of rows * R bytes")
    if cost is not None and (cost.dtype != torch.float32 or not cost.is_cuda
                             or cost.numel() < rows):
        raise ValueError("cost must be a float32 CUDA tensor of one value per row")
    if lut is None:
        lut = default_lut()
    lut = np.ascontiguousarray(lut, dtype=np.uint16).reshape(512, 2)
    _check(lib().cp_encode_rows_ws(e.data_ptr(), rows, d, k, lut.ctypes.data, records.data_ptr(),
                                   cost.data_ptr() if cost is not None else None,
                                   workspace.data_ptr(), workspace.numel(), _stream_ptr(stream)),
           "cp_encode_rows_ws")


def get_status(table: Table, stream=None) -> int:
    """Synchronise the stream; CP_ERR_INDEX_OOB if an id was out of range since the last call."""
    return int(lib().cp_get_status(table.handle, _stream_ptr(stream)))


def lookup_decode_host_noalloc(records: torch.Tensor, n_rows: int, d: int, k: int,
                               idx: torch.Tensor, out: torch.Tensor, status: torch.Tensor,
                               lut: np.ndarray | None = None, stream=None) -> torch.Tensor:
    """Host-resident decode that allocates no device memory in the library.

    For callers that cannot allocate device memory themselves at decode time:
    `records` (pinned host uint8), `out` (bf16 [n, d]) and `status` (one int32 on
    the device, bit 0 set for out-of-range ids) are all provided by the caller;
    at most 65,536 lookups per call.  Calls that overlap on the GPU race on the
    library's static scratch: order them on one stream.
    """
    if records.is_cuda or records.dtype != torch.uint8 or not records.is_contiguous():
        raise ValueError("records must be a contiguous pinned uint8 host tensor")
    _check_span(records, n_rows, d, k)
    if idx.dtype != torch.int64 or not idx.is_cuda or not idx.is_contiguous():
        raise ValueError("idx must be a contiguous int64 CUDA tensor")
    if out.dtype != torch.bfloat16 or out.shape != (idx.numel(), d) or not out.is_contiguous():
        raise ValueError("out must be a contiguous bf16 tensor of shape (n, d)")
    if status.dtype != torch.int32 or not status.is_cuda:
        raise ValueError("status must be an int32 CUDA tensor")
    if lut is None:
        lut = default_lut()
    lut = np.ascontiguousarray(lut, dtype=np.uint16).reshape(512, 2)
    st = lib().cp_lookup_decode_host_noalloc(records.data_ptr(), n_rows, d, k, lut.ctypes.data,
                                             idx.data_ptr(), idx.numel(), out.data_ptr(),
                                             status.data_ptr(), _stream_ptr(stream))
    _check(st, "cp_lookup_decode_host_noalloc")
    return out
