"""GPU tail-biting TCQ encoder (cp_encode_rows) against the oracle's fp32 encoder:
records (codes and bf16 alphas) bit for bit, costs bit for bit."""
import numpy as np
import pytest
import torch

import oracle
import trellis_row_decode_gb300 as cp
from trellis_row_decode_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("d,k", [(256, 4), (64, 3), (64, 5), (32, 6), (128, 4), (512, 4)])
def test_encoder_matches_oracle_f32(d, k):
    rows = 24 if d <= 256 else 8
    e = synth.normal_rows(100 + d + k, rows, d).astype(np.float32)
    e[3] *= 37.5                                     # scale does not change the code
    e[5] = 0.0                                       # zero row -> zero record
    rec, cost = cp.encode_rows(torch.from_numpy(e).cuda(), k)
    torch.cuda.synchronize()
    ref, ref_cost = oracle.encode_rows_f32(e, d, k, cp.default_lut())
    got = rec.cpu().numpy()
    bad = [i for i in range(rows) if not np.array_equal(got[i], ref[i])]
    assert not bad, f"rows {bad} differ"
    assert np.array_equal(cost.cpu().numpy().view(np.uint32), ref_cost.view(np.uint32))


def test_encoder_round_trip_through_decode():
    """Encode 64 N(0,1) rows on the GPU, decode them on the GPU: norm restored, error < RTN."""
    d, k, rows = 256, 4, 64
    e = synth.normal_rows(synth.SEED_ENCODER_ROWS, rows, d).astype(np.float32)
    rec, cost = cp.encode_rows(torch.from_numpy(e).cuda(), k)
    table = cp.load_table(rec.reshape(-1).contiguous(), rows, d, k)
    out = cp.lookup_decode(table, torch.arange(rows, device="cuda"))
    ehat = out.float().cpu().numpy().astype(np.float64)
    e64 = e.astype(np.float64)
    rel = np.abs(np.linalg.norm(ehat, axis=1) / np.linalg.norm(e64, axis=1) - 1)
    assert rel.max() <= 2.0 ** -8 + 1e-3
    mse = np.mean(np.sum((e64 - ehat) ** 2, 1) / np.sum(e64 ** 2, 1))
    rtn = np.mean([np.sum((r - oracle.rtn2(r, 0)) ** 2) / np.sum(r * r) for r in e64])
    assert mse < rtn and mse < 0.1175


@pytest.mark.parametrize("d,k", [(16, 4), (16, 6), (32, 3), (1024, 4), (1024, 3), (1024, 5),
                                 (1024, 6), (4096, 3), (4096, 6)])
def test_encoder_edge_and_large_rows(d, k):
    """Smallest rows (T = 8 steps), the d = 1024 tables at every k, and the largest
    rows (k = 3 has the largest group-minimum buffers): records and costs bit for bit."""
    rows = 40 if d <= 16 else 6
    e = synth.normal_rows(7 + d + k, rows, d).astype(np.float32)
    e[1] = 0.0
    rec, cost = cp.encode_rows(torch.from_numpy(e).cuda(), k)
    torch.cuda.synchronize()
    ref, ref_cost = oracle.encode_rows_f32(e, d, k, cp.default_lut())
    got = rec.cpu().numpy()
    bad = [i for i in range(rows) if not np.array_equal(got[i], ref[i])]
    assert not bad, f"rows {bad} differ"
    assert np.array_equal(cost.cpu().numpy().view(np.uint32), ref_cost.view(np.uint32))


@pytest.mark.parametrize("k", [3, 4, 6])
def test_encoder_more_rows_than_clusters(k):
    """Several rows per cluster (the persistent loop), d = 64."""
    d, rows = 64, 300
    e = synth.normal_rows(77, rows, d).astype(np.float32)
    rec, cost = cp.encode_rows(torch.from_numpy(e).cuda(), k)
    torch.cuda.synchronize()
    ref, ref_cost = oracle.encode_rows_f32(e, d, k, cp.default_lut())
    assert np.array_equal(rec.cpu().numpy(), ref)
    assert np.array_equal(cost.cpu().numpy().view(np.uint32), ref_cost.view(np.uint32))


def test_encoder_rejects_bad_geometry():
    with pytest.raises(cp.CPError):
        cp.encode_rows(torch.zeros((2, 8), device="cuda"), 4)      # d < 16


def test_encoder_with_caller_workspace_matches():
    """cp_encode_rows_ws (caller-owned workspace, queue-only) gives the records and
    costs of cp_encode_rows, reuses one workspace across calls, and rejects a
    workspace smaller than cp_encode_workspace_bytes."""
    d, k, rows = 128, 5, 20
    e = torch.from_numpy(synth.normal_rows(71, rows, d).astype(np.float32)).cuda()
    ref, ref_cost = cp.encode_rows(e, k)
    ws = cp.encode_workspace(rows, d, k)
    for _ in range(2):
        rec = torch.empty_like(ref)
        cost = torch.empty_like(ref_cost)
        cp.encode_rows_ws(e, k, ws, rec, cost)
        torch.cuda.synchronize()
        assert torch.equal(rec, ref)
        assert torch.equal(cost.view(torch.int32), ref_cost.view(torch.int32))
    L = cp.lib()
    lut = cp.default_lut()
    small = ws[: ws.numel() - 256]
    rc = L.cp_encode_rows_ws(e.data_ptr(), rows, d, k, lut.ctypes.data, rec.data_ptr(), None,
                             small.data_ptr(), small.numel(), None)
    assert rc == cp.CP_ERR_INVALID_ARG
