"""GPU parity of the CUDA lookup-decode against the CPU oracle (through the C ABI).

The bar: bit-exact bf16 outputs.  Each output is one fp32 product of a bf16
scale and an fp16 LUT value (exact) rounded once to bf16 on both sides, so no
tolerance applies; a failure reports the count of deviating elements and the
largest ulp distance.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import trellis_row_decode_gb300 as cp
from trellis_row_decode_gb300 import synth

from gpu_util import bits, compare, compare_all_rows, device_table, oracle_decode, NT

pytestmark = pytest.mark.gpu

SEED = 11


@pytest.fixture(scope="module")
def lut():
    return cp.default_lut()


def _run(table, idx_np, layout_host=False):
    idx = torch.from_numpy(np.ascontiguousarray(idx_np, dtype=np.int64)).cuda()
    fn = cp.lookup_decode_host if layout_host else cp.lookup_decode
    out = fn(table, idx)
    torch.cuda.synchronize()
    return bits(out)


def _assert_exact(got, ref, what=""):
    n, ulp = compare(got, ref)
    assert n == 0, f"{what}: {n} of {got.size} elements differ (max {ulp} ulp)"


# ---------------------------------------------------------------------------
# Full element-by-element parity at oracle-sized cases.
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("n", [4099, 10007])   # ragged against warps and batches of 32
@pytest.mark.parametrize("layout", [cp.CP_LAYOUT_AOS, cp.CP_LAYOUT_SOA])
@pytest.mark.parametrize("k", [3, 4, 5, 6])
@pytest.mark.parametrize("d", [256, 512, 1024])
def test_full_parity(lut, d, k, layout, n):
    n_rows = 3001                      # odd: the table's end is not 16-byte aligned
    rec = device_table(SEED, n_rows, d, k)
    soa = None
    if layout == cp.CP_LAYOUT_SOA:
        soa = torch.empty(cp.soa_bytes(n_rows, d, k), dtype=torch.uint8, device="cuda")
    table = cp.load_table(rec, n_rows, d, k, lut, layout=layout, soa=soa)
    idx = synth.zipf_indices(5, n, n_rows)
    idx[:3] = [n_rows - 1, 0, n_rows - 1]          # last record (table-end clamp) and first
    got = _run(table, idx)
    assert cp.get_status(table) == cp.CP_OK
    ref = oracle_decode(SEED, d, k, idx, n_rows, lut)
    _assert_exact(got.reshape(n, d), ref, f"d={d} k={k} layout={layout}")


@pytest.mark.parametrize("layout", [cp.CP_LAYOUT_AOS, cp.CP_LAYOUT_SOA])
@pytest.mark.parametrize("d,k", [(8, 4), (16, 6), (32, 3), (32, 5), (64, 4), (2048, 5),
                                 (4096, 6), (4096, 3)])
def test_parity_small_and_large_rows(lut, d, k, layout):
    n_rows, n = 777, 2049
    rec = device_table(SEED + 1, n_rows, d, k)
    soa = None
    if layout == cp.CP_LAYOUT_SOA:
        soa = torch.empty(cp.soa_bytes(n_rows, d, k), dtype=torch.uint8, device="cuda")
    table = cp.load_table(rec, n_rows, d, k, lut, layout=layout, soa=soa)
    idx = synth.uniform_indices(7, n, n_rows)
    got = _run(table, idx)
    _assert_exact(got.reshape(n, d), oracle_decode(SEED + 1, d, k, idx, n_rows, lut), f"d={d}")


def test_tiny_workload_with_encoded_rows(lut):
    """Tiny: 4096 rows d=256 b=2, 4096 uniform lookups; rows 0..63 are oracle-encoded N(0,1) rows."""
    import importlib.util
    from pathlib import Path
    import oracle
    w = synth.WORKLOADS["tiny"]
    p = Path(__file__).resolve().parent / "golden" / "make_golden.py"
    spec = importlib.util.spec_from_file_location("make_golden", p)
    mg = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mg)
    enc, alpha_exact, _ = mg.load()
    rec_cpu = synth.gen_records(synth.SEED_TABLE, torch.arange(w.n_rows), w.d, w.k).numpy()
    rec_cpu[:64] = enc
    rec = torch.from_numpy(rec_cpu.reshape(-1).copy()).cuda()
    table = cp.load_table(rec, w.n_rows, w.d, w.k, lut)
    idx = np.concatenate([w.indices(), np.arange(64)])
    got = _run(table, idx).reshape(-1, w.d)
    ref, bad = oracle.lookup_decode(rec_cpu, w.n_rows, w.d, w.k, rec_cpu.shape[1], lut, idx,
                                    n_threads=NT)
    assert bad == 0
    _assert_exact(got, ref, "tiny")
    # round trip of the encoded rows: norm restored within bf16 rounding, error below RTN
    e = synth.normal_rows(synth.SEED_ENCODER_ROWS, 64, w.d)
    ehat = (got[-64:].astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    rel = np.abs(np.linalg.norm(ehat, axis=1) / np.linalg.norm(e, axis=1) - 1)
    assert rel.max() <= 2.0 ** -8 + 1e-3
    mse = np.mean(np.sum((e - ehat) ** 2, 1) / np.sum(e * e, 1))
    rtn = np.mean([np.sum((r - oracle.rtn2(r, 0)) ** 2) / np.sum(r * r) for r in e])
    assert mse < rtn


# ---------------------------------------------------------------------------
# Edge cases and the error contract.
# ---------------------------------------------------------------------------

def test_empty_and_single(lut):
    d, k, n_rows = 256, 4, 100
    table = cp.load_table(device_table(SEED, n_rows, d, k), n_rows, d, k, lut)
    out = torch.full((0, d), 7, dtype=torch.bfloat16, device="cuda")
    cp.lookup_decode(table, torch.empty(0, dtype=torch.int64, device="cuda"), out)
    got = _run(table, np.array([42]))
    _assert_exact(got.reshape(1, d), oracle_decode(SEED, d, k, [42], n_rows, lut))


def test_out_of_range_ids(lut):
    d, k, n_rows = 512, 4, 1000
    table = cp.load_table(device_table(SEED, n_rows, d, k), n_rows, d, k, lut)
    idx = np.array([5, -1, n_rows, 999, 1 << 40, -(1 << 62), 0] * 9, dtype=np.int64)
    got = _run(table, idx).reshape(-1, d)
    bad = (idx < 0) | (idx >= n_rows)
    assert not got[bad].any()
    _assert_exact(got[~bad], oracle_decode(SEED, d, k, idx[~bad], n_rows, lut))
    assert cp.get_status(table) == cp.CP_ERR_INDEX_OOB
    assert cp.get_status(table) == cp.CP_OK          # cleared by the read
    _run(table, np.array([1, 2, 3]))
    assert cp.get_status(table) == cp.CP_OK


def test_special_alphas(lut):
    d, k = 256, 4
    specials = np.array([0x0000, 0x8000, 0x7F80, 0xFF80, 0x7FC0, 0xFFC1, 0x0001, 0x8001, 0x007F,
                         0x7F7F, 0xFF7F, 0x3F80, 0x0080], dtype=np.uint16)
    n_rows = len(specials)
    rec = synth.gen_records(SEED, torch.arange(n_rows), d, k).numpy()
    cb = d * k // 16
    rec[:, cb] = specials & 0xFF
    rec[:, cb + 1] = specials >> 8
    table = cp.load_table(torch.from_numpy(rec.reshape(-1).copy()).cuda(), n_rows, d, k, lut)
    import oracle
    idx = np.arange(n_rows)
    got = _run(table, idx).reshape(-1, d)
    ref, _ = oracle.lookup_decode(rec, n_rows, d, k, rec.shape[1], lut, idx)
    _assert_exact(got, ref, "special alphas")
    assert np.all((got[4] & 0x7FFF) > 0x7F80)                    # NaN stays NaN


def test_duplicates_and_order(lut):
    d, k, n_rows = 1024, 4, 500
    table = cp.load_table(device_table(SEED, n_rows, d, k), n_rows, d, k, lut)
    idx = np.array([7] * 100 + [3, 7, 3, 499, 0] * 50)
    got = _run(table, idx).reshape(-1, d)
    for j in range(1, len(idx)):
        if idx[j] == idx[0]:
            assert np.array_equal(got[j], got[0])
    single = [_run(table, idx[j:j + 1]).reshape(d) for j in [100, 101, 103, 104]]
    for j, s in zip([100, 101, 103, 104], single):
        assert np.array_equal(got[j], s)
    _assert_exact(got, oracle_decode(SEED, d, k, idx, n_rows, lut))


def test_argument_errors(lut):
    d, k, n_rows = 256, 4, 64
    table = cp.load_table(device_table(SEED, n_rows, d, k), n_rows, d, k, lut)
    idx = torch.arange(8, dtype=torch.int64, device="cuda")
    raw = torch.empty(8 * d * 2 + 16, dtype=torch.uint8, device="cuda")
    L = cp.lib()
    # misaligned output pointer
    assert L.cp_lookup_decode(table.handle, idx.data_ptr(), 8, raw.data_ptr() + 2, None) == 1
    # host entry point on a device table
    with pytest.raises(cp.CPError):
        cp.lookup_decode_host(table, idx)
    with pytest.raises(ValueError):
        cp.lookup_decode(table, idx.to(torch.int32))


def test_non_default_stream(lut):
    d, k, n_rows = 512, 6, 2000
    table = cp.load_table(device_table(SEED, n_rows, d, k), n_rows, d, k, lut)
    idx_np = synth.uniform_indices(3, 5000, n_rows)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        idx = torch.from_numpy(idx_np).cuda(non_blocking=False)
        out = cp.lookup_decode(table, idx, stream=s)
    s.synchronize()
    _assert_exact(bits(out).reshape(-1, d), oracle_decode(SEED, d, k, idx_np, n_rows, lut))


def test_output_in_pinned_host_memory(lut):
    """cp_lookup_decode writing straight into page-locked host memory (over the
    host link) gives the oracle's rows, including a ragged tail and bad ids."""
    d, k, n_rows = 1024, 4, 3000
    table = cp.load_table(device_table(SEED, n_rows, d, k), n_rows, d, k, lut)
    idx_np = synth.uniform_indices(11, 4099, n_rows)
    idx_np[7] = n_rows                                  # out of range -> zero row
    out_h = torch.empty((idx_np.size, d), dtype=torch.bfloat16, pin_memory=True)
    cp.lookup_decode(table, torch.from_numpy(idx_np).cuda(), out_h)
    torch.cuda.synchronize()
    _assert_exact(bits(out_h).reshape(-1, d), oracle_decode(SEED, d, k, idx_np, n_rows, lut))
    assert cp.get_status(table) == cp.CP_ERR_INDEX_OOB


def test_injected_failures(lut):
    d, k, n_rows = 256, 4, 16
    rec = device_table(SEED, n_rows, d, k)
    L = cp.lib()
    L.cp_test_inject_failure(1, 1)
    with pytest.raises(cp.CPError) as ei:
        cp.load_table(rec, n_rows, d, k, lut)
    assert ei.value.status == cp.CP_ERR_NO_MEMORY
    cp.load_table(rec, n_rows, d, k, lut).close()            # the next load succeeds
    host = torch.empty(n_rows * synth.record_bytes(d, k), dtype=torch.uint8).pin_memory()
    L.cp_test_inject_failure(2, 1)
    with pytest.raises(cp.CPError) as ei:
        cp.load_table(host, n_rows, d, k, lut)
    assert ei.value.status == cp.CP_ERR_CUDA
    L.cp_test_inject_failure(2, 0)


# ---------------------------------------------------------------------------
# Host-resident tables (zero-copy reads over the host link).
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("pinned", [True, False])
@pytest.mark.parametrize("layout", [cp.CP_LAYOUT_AOS, cp.CP_LAYOUT_SOA])
def test_host_resident_parity(lut, pinned, layout):
    d, k, n_rows, n = 1024, 4, 20011, 30000
    rec_cpu = synth.gen_records(SEED, torch.arange(n_rows), d, k).reshape(-1).contiguous()
    host = rec_cpu.pin_memory() if pinned else rec_cpu
    soa = None
    if layout == cp.CP_LAYOUT_SOA:
        soa = torch.empty(cp.soa_bytes(n_rows, d, k), dtype=torch.uint8, pin_memory=True)
    table = cp.load_table(host, n_rows, d, k, lut, layout=layout, soa=soa)
    idx = synth.zipf_indices(9, n, n_rows)
    idx[-1] = n_rows - 1
    idx[5:9] = [-1, n_rows, 1 << 45, -(1 << 40)]          # out of range: zero rows
    got = _run(table, idx, layout_host=True).reshape(n, d)
    assert cp.get_status(table) == cp.CP_ERR_INDEX_OOB
    assert not got[5:9].any()
    dev_table = cp.load_table(rec_cpu.cuda(), n_rows, d, k, lut)
    assert np.array_equal(got, _run(dev_table, idx).reshape(n, d))
    _assert_exact(got, oracle_decode(SEED, d, k, idx, n_rows, lut), "host-resident")
    table.close()


def test_host_resident_multi_pass(lut):
    """More lookups than one pass (2^20), most of them repeated ids: passes chain on the stream."""
    d, k, n_rows = 8, 4, 100003
    n = (1 << 20) * 2 + 12345
    rec_cpu = synth.gen_records(SEED, torch.arange(n_rows), d, k).reshape(-1).contiguous()
    table = cp.load_table(rec_cpu.pin_memory(), n_rows, d, k, lut)
    idx = synth.uniform_indices(4, n, n_rows)
    got = _run(table, idx, layout_host=True).reshape(n, d)
    dev = cp.load_table(rec_cpu.cuda(), n_rows, d, k, lut)
    assert np.array_equal(got, _run(dev, idx).reshape(n, d))
    ref = np.concatenate([oracle_decode(SEED, d, k, idx[j:j + (1 << 18)], n_rows, lut)
                          for j in range(0, n, 1 << 18)])
    _assert_exact(got, ref, "multi-pass")


# ---------------------------------------------------------------------------
# Full-size workloads, in the launch configuration the benchmark times: every
# output row compared with the oracle, element by element.
# ---------------------------------------------------------------------------

def _full_check(table, w, lut, host=False):
    idx_np = w.indices()
    idx = torch.from_numpy(idx_np).cuda()
    fn = cp.lookup_decode_host if host else cp.lookup_decode
    out = fn(table, idx)
    torch.cuda.synchronize()
    assert cp.get_status(table) == cp.CP_OK
    n_bad, ulp = compare_all_rows(out, idx_np, synth.SEED_TABLE, w.d, w.k, w.n_rows, lut)
    assert n_bad == 0, f"{w.name}: {n_bad} of {out.numel()} elements differ (max {ulp} ulp)"


@pytest.mark.parametrize("name", ["mid", "sweep_b1.5", "sweep_b2", "sweep_b2.5", "sweep_b3"])
def test_full_size_workloads(lut, name):
    w = synth.WORKLOADS[name]
    rec = device_table(synth.SEED_TABLE, w.n_rows, w.d, w.k)
    table = cp.load_table(rec, w.n_rows, w.d, w.k, lut)
    _full_check(table, w, lut)
    table.close()
    del rec
    torch.cuda.empty_cache()


def test_deepseek_scale_resident(lut):
    """1.98e8 rows x d=1024 at b=2 (51 GB) in HBM: prefill replay and a decode step."""
    w = synth.WORKLOADS["deepseek_prefill"]
    rec = device_table(synth.SEED_TABLE, w.n_rows, w.d, w.k)
    table = cp.load_table(rec, w.n_rows, w.d, w.k, lut)
    _full_check(table, w, lut)
    _full_check(table, synth.WORKLOADS["deepseek_decode"], lut)
    table.close()
    del rec
    torch.cuda.empty_cache()


def test_deepseek_scale_host_resident(lut):
    """The same 51 GB table in pinned host DRAM, read zero-copy by cp_lookup_decode_host."""
    w = synth.WORKLOADS["host_prefill"]
    R = w.rec_bytes
    host = torch.empty(w.n_rows * R, dtype=torch.uint8, pin_memory=True)
    chunk = 1 << 22
    stage = torch.empty(chunk * R, dtype=torch.uint8, device="cuda")
    for r0 in range(0, w.n_rows, chunk):
        r1 = min(w.n_rows, r0 + chunk)
        rows = torch.arange(r0, r1, dtype=torch.int64, device="cuda")
        stage[: (r1 - r0) * R].view(r1 - r0, R).copy_(synth.gen_records(synth.SEED_TABLE, rows,
                                                                        w.d, w.k))
        host[r0 * R: r1 * R].copy_(stage[: (r1 - r0) * R])
    del stage
    table = cp.load_table(host, w.n_rows, w.d, w.k, lut)
    _full_check(table, w, lut, host=True)
    table.close()


def test_device_generator_matches_host():
    """The seeded generators give identical bytes on the device and on the host."""
    rows = torch.tensor([0, 1, 12345, 197_999_999], dtype=torch.int64)
    a = synth.gen_records(3, rows.cuda(), 1024, 5).cpu()
    b = synth.gen_records(3, rows, 1024, 5)
    assert torch.equal(a, b)


def test_cuda_graph_capture_and_replay(lut):
    """cp_lookup_decode and cp_lookup_decode_host queue only kernels (no host
    synchronisation, no allocation), so both can be captured into a CUDA graph;
    replays with new ids in the captured buffers give the oracle's rows."""
    d, k, n_rows, n = 512, 4, 5000, 3000
    rec = device_table(SEED, n_rows, d, k)
    table = cp.load_table(rec, n_rows, d, k, lut)
    host_rec = rec.cpu().pin_memory()
    htable = cp.load_table(host_rec, n_rows, d, k, lut)
    idx = torch.empty(n, dtype=torch.int64, device="cuda")
    out = torch.empty((n, d), dtype=torch.bfloat16, device="cuda")
    out_h = torch.empty((n, d), dtype=torch.bfloat16, device="cuda")
    idx.copy_(torch.from_numpy(synth.uniform_indices(1, n, n_rows)))
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):                          # first calls outside the capture
        cp.lookup_decode(table, idx, out, s)
        cp.lookup_decode_host(htable, idx, out_h, s)
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        cp.lookup_decode(table, idx, out, s)
        cp.lookup_decode_host(htable, idx, out_h, s)
    for seed in (21, 22):
        idx_np = synth.uniform_indices(seed, n, n_rows)
        idx.copy_(torch.from_numpy(idx_np))
        out.zero_()
        out_h.zero_()
        torch.cuda.synchronize()
        g.replay()
        torch.cuda.synchronize()
        ref = oracle_decode(SEED, d, k, idx_np, n_rows, lut)
        _assert_exact(bits(out).reshape(-1, d), ref, f"graph replay, seed {seed}")
        _assert_exact(bits(out_h).reshape(-1, d), ref, f"graph replay (host table), seed {seed}")
    assert cp.get_status(table) == cp.CP_OK and cp.get_status(htable) == cp.CP_OK
    table.close()
    htable.close()


@pytest.mark.parametrize("n_rows", [1, 2, 5, 4097])
def test_host_resident_tiny_tables(lut, n_rows):
    """Host-resident tables with one or a few row ranges (the partition's edge cases)."""
    d, k, n = 512, 4, 3001
    rec_cpu = synth.gen_records(SEED, torch.arange(n_rows), d, k).reshape(-1).contiguous()
    table = cp.load_table(rec_cpu.pin_memory(), n_rows, d, k, lut)
    idx = synth.uniform_indices(n_rows, n, n_rows)
    idx[::97] = n_rows                                    # out of range: zero rows
    got = _run(table, idx, layout_host=True).reshape(n, d)
    assert cp.get_status(table) == cp.CP_ERR_INDEX_OOB
    _assert_exact(got, oracle_decode(SEED, d, k, idx, n_rows, lut), f"host n_rows={n_rows}")
    table.close()


@pytest.mark.parametrize("pattern", ["one_id", "dominant_id", "sorted", "reversed"])
def test_host_resident_skewed_ids(lut, pattern):
    """Lookup streams that load the partition unevenly, over many partition CTAs
    (2,048 lookups each): every lookup on one id (one range takes every rank), a
    dominant id mixed with uniform ids, and ids in ascending or descending order
    (each CTA's lookups in one or two ranges).  Every element against the oracle."""
    d, k, n_rows, n = 256, 4, 70001, 100003
    rec_cpu = synth.gen_records(SEED, torch.arange(n_rows), d, k).reshape(-1).contiguous()
    table = cp.load_table(rec_cpu.pin_memory(), n_rows, d, k, lut)
    idx = synth.uniform_indices(21, n, n_rows)
    if pattern == "one_id":
        idx[:] = 4321
    elif pattern == "dominant_id":
        idx[::2] = n_rows - 1                           # the last record, half the lookups
    elif pattern == "sorted":
        idx.sort()
    else:
        idx[::-1].sort()
    got = _run(table, idx, layout_host=True).reshape(n, d)
    assert cp.get_status(table) == cp.CP_OK
    _assert_exact(got, oracle_decode(SEED, d, k, idx, n_rows, lut), f"host {pattern}")
    table.close()


@pytest.mark.parametrize("layout", [cp.CP_LAYOUT_AOS, cp.CP_LAYOUT_SOA])
@pytest.mark.parametrize("d,k", [(16, 6), (64, 4), (256, 3), (512, 5), (2048, 5), (4096, 6),
                                 (4096, 3)])
def test_host_resident_small_and_large_rows(lut, d, k, layout):
    """Host-resident tables outside d = 1024: the register-ring kernel at d = 256
    and 512, the staged kernel (cp.async ring) for every other d, both layouts; the
    table's last record is looked up (its reads end at the table's end)."""
    n_rows, n = 777, 2049
    rec_cpu = synth.gen_records(SEED + 2, torch.arange(n_rows), d, k).reshape(-1).contiguous()
    soa = None
    if layout == cp.CP_LAYOUT_SOA:
        soa = torch.empty(cp.soa_bytes(n_rows, d, k), dtype=torch.uint8, pin_memory=True)
    table = cp.load_table(rec_cpu.pin_memory(), n_rows, d, k, lut, layout=layout, soa=soa)
    idx = synth.uniform_indices(8, n, n_rows)
    idx[-1] = n_rows - 1
    got = _run(table, idx, layout_host=True).reshape(n, d)
    assert cp.get_status(table) == cp.CP_OK
    _assert_exact(got, oracle_decode(SEED + 2, d, k, idx, n_rows, lut), f"host d={d} k={k}")
    table.close()
