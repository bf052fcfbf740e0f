"""Host-side checks of libcp: it loads, exports every symbol include/cp.h declares,
and rejects bad arguments on the host (no kernel launch, no GPU needed)."""
import ctypes as C
import re
import subprocess
from pathlib import Path

import pytest

ROOT = Path(__file__).resolve().parent.parent
HEADER = ROOT / "include" / "cp.h"


@pytest.fixture(scope="module")
def cplib():
    import trellis_row_decode_gb300 as cp
    from trellis_row_decode_gb300 import build_ext
    if not cp.LIB_PATH.exists():
        build_ext.build()
    return cp.lib()


def declared_functions():
    text = HEADER.read_text()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(cp_[a-z_0-9]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for must in ["cp_table_load", "cp_lookup_decode", "cp_lookup_decode_host", "cp_get_status",
                 "cp_table_free", "cp_status_string", "cp_record_bytes", "cp_soa_bytes"]:
        assert must in names


def test_library_exports_every_declared_symbol(cplib):
    import trellis_row_decode_gb300 as cp
    out = subprocess.run(["nm", "-D", "--defined-only", str(cp.LIB_PATH)], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r"\bT (cp_[a-z_0-9]+)$", out, flags=re.M))
    missing = [n for n in declared_functions() if n not in exported]
    assert not missing, missing
    for n in declared_functions():
        getattr(cplib, n)


def test_record_and_soa_sizes(cplib):
    import trellis_row_decode_gb300 as cp
    assert cp.record_bytes(1024, 4) == 258
    assert cp.record_bytes(512, 4) == 130
    assert cp.record_bytes(1024, 3) == 194
    assert cp.record_bytes(1024, 6) == 386
    assert cp.record_bytes(256, 4) == 66
    assert cp.record_bytes(1004, 4) == 0          # d % 8 != 0
    assert cp.record_bytes(8, 6) == 0             # odd number of code bytes
    assert cp.record_bytes(1024, 7) == 0
    assert cp.soa_bytes(10, 1024, 4) == 10 * 256 + 32
    assert cp.soa_bytes(3, 512, 6) == 3 * 192 + 16


def test_status_strings(cplib):
    for s, name in enumerate(["CP_OK", "CP_ERR_INVALID_ARG", "CP_ERR_INDEX_OOB", "CP_ERR_CUDA",
                              "CP_ERR_NO_MEMORY", "CP_ERR_FORMAT"]):
        assert cplib.cp_status_string(s).decode() == name


def test_bad_arguments_rejected_on_host(cplib):
    import numpy as np
    import trellis_row_decode_gb300 as cp
    h = C.c_void_p(0)
    lut = cp.default_lut()
    buf = (C.c_uint8 * 4096)()
    base = C.addressof(buf)
    aligned = (base + 15) & ~15
    # null handle out-pointer, null records, zero rows, bad k, bad d, misaligned records
    assert cplib.cp_table_load(None, aligned, 4, 256, 4, lut.ctypes.data, 0, 0, None, None) == 1
    assert cplib.cp_table_load(C.byref(h), None, 4, 256, 4, lut.ctypes.data, 0, 0, None, None) == 1
    assert cplib.cp_table_load(C.byref(h), aligned, 0, 256, 4, lut.ctypes.data, 0, 0, None, None) == 1
    assert cplib.cp_table_load(C.byref(h), aligned, 4, 256, 7, lut.ctypes.data, 0, 0, None, None) == 1
    assert cplib.cp_table_load(C.byref(h), aligned, 4, 260, 4, lut.ctypes.data, 0, 0, None, None) == 1
    assert cplib.cp_table_load(C.byref(h), aligned + 2, 4, 256, 4, lut.ctypes.data, 0, 0, None,
                               None) == 1
    # SoA without a destination, AoS with one
    assert cplib.cp_table_load(C.byref(h), aligned, 4, 256, 4, lut.ctypes.data, 0, 1, None, None) == 1
    assert cplib.cp_table_load(C.byref(h), aligned, 4, 256, 4, lut.ctypes.data, 0, 0, aligned,
                               None) == 1
    # non-finite LUT entry -> CP_ERR_FORMAT
    bad = lut.copy()
    bad[7, 1] = 0x7C00
    assert cplib.cp_table_load(C.byref(h), aligned, 4, 256, 4, bad.ctypes.data, 0, 0, None,
                               None) == 5
    assert h.value is None
    # decode on a null handle
    assert cplib.cp_lookup_decode(None, aligned, 1, aligned, None) == 1
    assert cplib.cp_get_status(None, None) == 1
    cplib.cp_table_free(None)
    assert cplib.cp_test_inject_failure(9, 1) == 1
    assert np.isfinite(lut.view(np.float16).astype(float)).all()


def test_wrappers_reject_short_record_buffers(cplib):
    """A records buffer shorter than n_rows * R would let the kernels read past its
    end (the C ABI only sees a pointer), so the binding refuses it before any call
    into the library; the same for a short SoA destination."""
    import torch
    import trellis_row_decode_gb300 as cp
    d, k, n_rows = 256, 4, 100
    R = cp.record_bytes(d, k)
    short = torch.zeros(n_rows * R - 2, dtype=torch.uint8)
    with pytest.raises(ValueError):
        cp.load_table(short, n_rows, d, k)
    with pytest.raises(ValueError):
        cp.lookup_decode_host_noalloc(short, n_rows, d, k, torch.zeros(1, dtype=torch.int64),
                                      torch.empty((1, d), dtype=torch.bfloat16),
                                      torch.zeros(1, dtype=torch.int32))
    full = torch.zeros(n_rows * R, dtype=torch.uint8)
    with pytest.raises(ValueError):
        cp.load_table(full, n_rows, d, k, layout=cp.CP_LAYOUT_SOA,
                      soa=torch.zeros(cp.soa_bytes(n_rows, d, k) - 16, dtype=torch.uint8))


def test_stream_read_argument_checks_on_host(cplib):
    """Null, misaligned or ragged buffers are refused before any CUDA call."""
    import ctypes
    buf = (ctypes.c_uint8 * 64)()
    base = (ctypes.addressof(buf) + 15) & ~15
    assert cplib.cp_measure_stream_read(None, 16, None) == 1
    assert cplib.cp_measure_stream_read(base + 4, 16, None) == 1
    assert cplib.cp_measure_stream_read(base, 0, None) == 1
    assert cplib.cp_measure_stream_read(base, 24, None) == 1


def test_record_read_argument_checks_on_host(cplib):
    """Null or misaligned buffers, no rows, a zero or oversized record are refused
    before any CUDA call."""
    import ctypes
    f = cplib.cp_measure_record_read
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.c_void_p, ctypes.c_uint64, ctypes.c_uint32, ctypes.c_void_p,
                  ctypes.c_uint64, ctypes.c_void_p]
    buf = (ctypes.c_uint8 * 1024)()
    base = (ctypes.addressof(buf) + 15) & ~15
    rows = (ctypes.c_int64 * 4)()
    r = ctypes.addressof(rows)
    assert f(None, 512, 258, r, 1, None) == 1
    assert f(base, 512, 258, None, 1, None) == 1
    assert f(base, 512, 0, r, 1, None) == 1
    assert f(base, 512, 258, r, 0, None) == 1
    assert f(base, 100, 258, r, 1, None) == 1
    assert f(base + 4, 512, 258, r, 1, None) == 1
    assert f(base, 512, 258, r + 4, 1, None) == 1
    assert f(base, 512, 258, r, 1 << 48, None) == 1
