"""Benchmark of the CP lookup-decode on GB300: rows/s and achieved HBM GB/s.

A step is one cp_lookup_decode over the whole replay batch (default: the
DeepSeek-scale table, 1.98e8 rows x d=1024 at b=2 = 51 GB of records in HBM,
4096 tokens x 48 rows = 196,608 Zipf(1.0) lookups).  W untimed warm-up steps,
then K timed steps; each step is bracketed by CUDA events on the launching
stream and followed (outside the timed interval) by a 512 MB write and a 512 MB
read that flush the 129 MB L2, so no step reuses the previous step's records
from L2 and no dirty flush lines are written back inside the next step.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                  [--impl ours|reference] [--layout aos|soa] [--no-host-path]

At N = 1 the same run also times cp_lookup_decode_host on the same table placed
in pinned host DRAM ("host_path" in the JSON line, against the measured
host-to-device copy bandwidth; unless --no-host-path), the fused readout, the
mixed-rate table, the encoder, the other table configs and the CPU oracle.
Under torchrun these single-GPU legs are skipped; the e2e figure is then the
whole job's (all ranks' lookups over the slowest rank's time).

Under torchrun (N > 1) every rank holds its own replica of the table and
decodes its own replay (seed + rank); no collective touches the data path
(weak scaling).  Rank 0 prints one JSON line.

--impl reference times the CPU oracle (the plain C++ restatement of the
method, test infrastructure) on this machine's host cores over bounded samples
of the same workload.
"""
from __future__ import annotations

import argparse
import csv
import hashlib
import io
import json
import os
import subprocess
import sys
import time
from pathlib import Path

import numpy as np

ROOT = Path(__file__).resolve().parent
sys.path.insert(0, str(ROOT))

FALLBACK_HBM_GBS = 6800.0       # earlier GB300 copy measurement, used when no measured file
PAGES_LATENCY_S = 0.190e-3      # pages' HBM-resident replay latency on one H200
L2_FLUSH_BYTES = 1024 << 20     # 512 MB written + 512 MB read between steps
METRIC = "CP lookup-decode rows/s & achieved HBM GB/s, 4096-tok×48-row replay"
REFERENCE_SECONDS = 60.0        # oracle time of a whole --impl reference run


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--workload", default="deepseek_prefill")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--layout", default="aos", choices=["aos", "soa"])
    ap.add_argument("--no-host-path", action="store_true",
                    help="skip timing cp_lookup_decode_host on the table in pinned host DRAM")
    ap.add_argument("--e2e-steps", type=int, default=30)
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--only", choices=["encoder", "decode", "host", "mixed", "reduce"],
                    default=None,
                    help="run one leg alone on --workload and print its JSON (profiling)")
    ap.add_argument("--mixed-rows", type=int, default=1 << 24,
                    help="rows of the mixed-rate table (mixed leg)")
    ap.add_argument("--encoder-rows", type=int, default=0,
                    help="rows per encoder call (default 4 x SM count)")
    ap.add_argument("--sustained-calls", type=int, default=50,
                    help="back-to-back calls in the sustained window (0: skip)")
    ap.add_argument("--no-other-configs", action="store_true",
                    help="skip timing the other table configs (mid, bit-rate sweep, decode step)")
    return ap.parse_args()


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def measured_peaks():
    p = ROOT / "MEASURED_PEAKS.json"
    if p.exists():
        try:
            j = json.loads(p.read_text())
            for key in ("hbm_gbs", "hbm_GBs", "hbm"):
                if key in j and isinstance(j[key], (int, float)):
                    return float(j[key]), "measured"
        except Exception:
            pass
    return FALLBACK_HBM_GBS, "fallback"


def kernel_source_sha() -> str:
    """Hash of the HBM-path kernel's source (its header holds the kernel, its helpers
    and its launch constants), used to tell whether committed ncu counters still apply."""
    h = hashlib.sha256()
    f = ROOT / "trellis_row_decode_gb300" / "csrc" / "cp_kernels.cuh"
    h.update(f.name.encode())
    h.update(f.read_bytes())
    return h.hexdigest()


ISSUE_PEAK_WARP_INST_S = 152 * 4 * 2.07e9   # SMs x schedulers x 1 warp-instruction/clock x max SM clock


def header_sha(name: str) -> str:
    h = hashlib.sha256()
    f = ROOT / "trellis_row_decode_gb300" / "csrc" / name
    h.update(f.name.encode())
    h.update(f.read_bytes())
    return h.hexdigest()


def ncu_inst(kernel: str, n: int, d: int, k: int, group: int):
    """Committed warp-instruction count per launch, or None (header changed / no entry)."""
    try:
        data = json.loads((ROOT / "profiles" / "ncu_inst.json").read_text())
    except (OSError, ValueError):
        return None
    for e in data.get("entries", []):
        if (e.get("kernel"), e.get("n"), e.get("d"), e.get("k"), e.get("group")) == \
                (kernel, n, d, k, group) and e.get("header_sha256") == header_sha(e["header"]):
            return int(e["warp_instructions"])
    return None


def ncu_encoder_inst_per_row(d: int, k: int):
    """Committed encoder warp instructions per row at (d, k), or None."""
    try:
        data = json.loads((ROOT / "profiles" / "ncu_inst.json").read_text())
    except (OSError, ValueError):
        return None
    for e in data.get("entries", []):
        if (e.get("kernel"), e.get("d"), e.get("k")) == ("tcq_encode_kernel", d, k) and \
                e.get("header_sha256") == header_sha(e["header"]):
            return float(e["warp_instructions_per_row"])
    return None


def ncu_traffic(workload: str, layout: str):
    """DRAM bytes per launch from the committed ncu summary, if it matches this kernel source."""
    p = ROOT / "profiles" / "ncu_traffic.json"
    if not p.exists():
        return None
    try:
        j = json.loads(p.read_text())
    except Exception:
        return None
    for e in j.get("entries", []):
        if e.get("workload") == workload and e.get("layout") == layout and \
                e.get("kernel_source_sha256") == kernel_source_sha():
            return e.get("dram_bytes_per_launch")
    return None


class ClockSampler:
    """nvidia-smi clock/throttle samples during the timed region."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *a):
        time.sleep(0.2)
        self.out = ""
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        rows = []
        for r in csv.reader(io.StringIO(self.out or "")):
            if len(r) >= 9:
                rows.append([x.strip() for x in r])
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i] == "Active"})
        loaded = [s for s in sm if s > 0.5 * max(sm)] if sm else []
        return {"sm_mhz": float(np.median(loaded)) if loaded else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(rows)}


def cpu_model() -> str:
    """Host CPU model name (lscpu, else /proc/cpuinfo, else the machine type)."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    try:
        for line in Path("/proc/cpuinfo").read_text().splitlines():
            if line.lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except OSError:
        pass
    import platform
    return platform.machine()


def workload_config(w, layout: str, world: int, idx_np: np.ndarray, index_seed: int) -> dict:
    """The `config` object of both arms' JSON lines (identical keys and values)."""
    from trellis_row_decode_gb300 import synth
    return {"workload": w.name, "n_rows": w.n_rows, "d": w.d, "b": w.k / 2,
            "record_bytes": w.rec_bytes, "lookups": int(idx_np.size), "tokens": w.tokens,
            "rows_per_token": w.rows_per_token, "index_dist": f"{w.dist}({w.zipf_s})",
            "unique_ids": int(np.unique(idx_np).size), "layout": layout,
            "table_gb": w.table_bytes / 1e9,
            "seeds": {"table": synth.SEED_TABLE, "index": index_seed},
            "l2": "flushed between steps (512 MB write then 512 MB read, outside the timed interval)",
            "parallelism": f"replicas x{world}", "cpu_model": cpu_model()}


def oracle_parity(w, idx_np: np.ndarray, out_host, lut, chunk: int = 1 << 16) -> dict:
    """Every element of a timed step's output (bf16 [n, d] on the host) against the
    oracle's decode of the same lookups (records regenerated on the host).  Part of
    the CPU-baseline leg: the only place besides --impl reference where the bench
    runs the oracle."""
    import torch
    import oracle
    from trellis_row_decode_gb300 import synth
    got_all = out_host.view(torch.int16).numpy().view(np.uint16)
    n_bad, max_ulp = 0, 0
    nt = max(1, os.cpu_count() or 1)
    for j0 in range(0, idx_np.size, chunk):
        ids = idx_np[j0:j0 + chunk]
        valid = (ids >= 0) & (ids < w.n_rows)
        uniq, inv = np.unique(np.where(valid, ids, 0), return_inverse=True)
        rec = synth.gen_records(synth.SEED_TABLE, torch.from_numpy(uniq), w.d, w.k).numpy()
        local = np.where(valid, inv, -1).astype(np.int64)
        ref, _ = oracle.lookup_decode(rec, len(uniq), w.d, w.k, rec.shape[1], lut, local,
                                      n_threads=nt)
        got = got_all[j0:j0 + chunk].reshape(ref.shape)
        if np.array_equal(got, ref):
            continue
        g, r = got.astype(np.int32), ref.astype(np.int32)
        nan = ((g & 0x7FFF) > 0x7F80) & ((r & 0x7FFF) > 0x7F80)
        diff = (g != r) & ~nan
        line = lambda x: np.where(x & 0x8000, -(x & 0x7FFF), x & 0x7FFF)  # noqa: E731
        n_bad += int(diff.sum())
        if diff.any():
            max_ulp = max(max_ulp, int(np.abs(line(g) - line(r))[diff].max()))
    return {"checked_elements": int(idx_np.size) * w.d, "deviating": n_bad, "max_ulp": max_ulp,
            "against": "oracle (every row of the last timed step)"}


# ---------------------------------------------------------------------------
# Reference arm: the CPU oracle on the host cores.
# ---------------------------------------------------------------------------

def oracle_runner(w, idx: np.ndarray, lut, threads: int = 0):
    """run(m) -> seconds the oracle takes to decode the first m lookups of the
    replay (records regenerated on the host first, outside the timing)."""
    import torch
    import oracle
    from trellis_row_decode_gb300 import synth
    nt = threads or max(1, os.cpu_count() or 1)

    cache = {}

    def run(m):
        if m not in cache:                       # records of the prefix, built once per m
            uniq, inv = np.unique(idx[:m], return_inverse=True)
            rec = synth.gen_records(synth.SEED_TABLE, torch.from_numpy(uniq), w.d, w.k).numpy()
            cache.clear()
            cache[m] = (rec, len(uniq), inv.astype(np.int64))
        rec, nu, inv = cache[m]
        t0 = time.perf_counter()
        oracle.lookup_decode(rec, nu, w.d, w.k, rec.shape[1], lut, inv, n_threads=nt)
        return time.perf_counter() - t0
    return run, nt


def oracle_sample_size(run, n: int, seconds: float, m0: int) -> int:
    """Prefix length whose decode takes about `seconds` (calibrated on m0 lookups)."""
    m0 = min(n, m0)
    dt0 = run(m0)
    return int(min(n, max(m0, m0 * seconds / max(dt0, 1e-6))))


def oracle_sample_rate(w, idx: np.ndarray, seconds: float, lut, threads: int = 0):
    """Oracle lookup-decode rows/s on a bounded prefix of the replay (all host
    cores unless `threads`)."""
    run, nt = oracle_runner(w, idx, lut, threads)
    m = oracle_sample_size(run, idx.size, seconds, 2048 if nt > 1 else 256)
    return m / run(m), m, nt


def reference_arm(args, w, rank):
    if rank != 0:
        return
    import trellis_row_decode_gb300 as cp
    from trellis_row_decode_gb300 import synth
    lut = cp.default_lut()
    idx = w.indices(synth.SEED_INDEX)
    # the whole run stays near args.cpu_seconds: each step times a prefix sized
    # for its share (at least the 2048-lookup calibration prefix)
    # one calibration, then every step times the same prefix, sized so that the
    # whole run takes about REFERENCE_SECONDS of oracle time
    run, nt = oracle_runner(w, idx, lut)
    per_step = REFERENCE_SECONDS / max(1, args.steps + args.warmup)
    run(2048)                                    # first call: thread pool and pages warm
    m = oracle_sample_size(run, idx.size, min(max(per_step, 0.002), 10.0), 2048)
    rates, sizes = [], []
    for s in range(args.warmup + args.steps):
        dt = run(m)
        if s >= args.warmup:
            rates.append(m / dt)
            sizes.append(m)
    value = float(np.median(rates))
    bpl = w.algorithmic_bytes_per_lookup()
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "rows/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * w.n_lookups / value, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "fp32", "data": "synthetic",
        "config": workload_config(w, args.layout, args.gpus, idx, synth.SEED_INDEX),
        "cpu_baseline": {"value": value, "unit": "rows/s", "cores": nt, "kind": "oracle",
                         "sample": f"first {sizes[0]} lookups of the replay per step (records "
                                   f"regenerated on the host once), {nt} threads"},
        "e2e": {"value": value, "unit": "rows/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "achieved_gbs_algorithmic": value * bpl / 1e9,
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
# Our arm.
# ---------------------------------------------------------------------------

def build_table(w, layout: str, seed: int):
    import torch
    import trellis_row_decode_gb300 as cp
    from trellis_row_decode_gb300 import synth
    rec = torch.empty(w.table_bytes, dtype=torch.uint8, device="cuda")
    synth.fill_records(rec, seed, w.n_rows, w.d, w.k)
    soa = None
    lay = cp.CP_LAYOUT_AOS
    if layout == "soa":
        soa = torch.empty(cp.soa_bytes(w.n_rows, w.d, w.k), dtype=torch.uint8, device="cuda")
        lay = cp.CP_LAYOUT_SOA
    table = cp.load_table(rec, w.n_rows, w.d, w.k, cp.default_lut(), layout=lay, soa=soa)
    torch.cuda.synchronize()
    return table, rec, soa


def flush_l2(flush):
    """Write the first half of `flush` (> L2), then read the second half so the
    written lines leave L2 before the next timed step (outside the timed interval)."""
    half = flush.numel() // 2
    flush[:half].zero_()
    flush[half:].view(torch_int64()).amax()


def torch_int64():
    import torch
    return torch.int64


def time_steps(fn, steps, warmup, flush, stream, nvtx: str = "timed"):
    """Per-step device times (s) of fn() with an L2 flush between steps.  Each timed
    call is wrapped in an NVTX range `nvtx`, so a profiler filtered on "timed" sees
    exactly the launches the CUDA events time (not the flushes)."""
    import torch
    for _ in range(warmup):
        fn()
        flush_l2(flush)
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(steps)]
    for a, b in ev:
        a.record(stream)
        torch.cuda.nvtx.range_push(nvtx)
        fn()
        torch.cuda.nvtx.range_pop()
        b.record(stream)
        flush_l2(flush)
    torch.cuda.synchronize()
    return np.array([a.elapsed_time(b) * 1e-3 for a, b in ev])


def hbm_same_run(flush, stream, steps: int = 20):
    """Context for the HBM roofline, taken on this GPU in this run with a library
    kernel: a 1 GiB device-to-device copy, read + write bytes counted."""
    import torch
    src = torch.ones(1 << 30, dtype=torch.uint8, device="cuda")
    dst = torch.empty_like(src)
    tc = time_steps(lambda: dst.copy_(src), steps, 3, flush, stream, "copy")
    del src, dst
    return {"copy_gbs": 2 * (1 << 30) / float(np.median(tc)) / 1e9,
            "copy": "torch copy_ of a 1 GiB device buffer, read + write bytes, median of "
                    f"{steps}, L2 flushed between"}


def d2h_link_gbs(flush, stream) -> float:
    """Device-to-host link rate in this run: 1 GB copies to pinned memory (the bound of
    the e2e step, which moves every row to the host)."""
    import torch
    src = torch.ones(1 << 30, dtype=torch.uint8, device="cuda")
    dst = torch.empty(1 << 30, dtype=torch.uint8, pin_memory=True)
    t = time_steps(lambda: dst.copy_(src, non_blocking=True), 10, 2, flush, stream, "link")
    del src, dst
    return (1 << 30) / float(np.median(t)) / 1e9


def aggregate(local_time_s: float, local_units: int, world: int, dist, device):
    """Max of the ranks' timed totals and the whole-job throughput.

    Every rank processes `local_units` in `local_time_s`; the job takes as long as
    its slowest rank, so value = local_units * world / max_rank(time).
    """
    total = local_time_s
    if dist is not None and world > 1:
        import torch
        tt = torch.tensor([total], dtype=torch.float64, device=device)
        dist.all_reduce(tt, op=dist.ReduceOp.MAX)
        total = float(tt.item())
    return total, local_units * world / total


def our_arm(args, w, rank, world, local):
    import torch
    import trellis_row_decode_gb300 as cp
    from trellis_row_decode_gb300 import synth
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))

    table, rec, soa = build_table(w, args.layout, synth.SEED_TABLE)
    idx_np = w.indices(synth.SEED_INDEX + rank)
    idx = torch.from_numpy(idx_np).cuda()
    n = idx_np.size
    out = torch.empty((n, w.d), dtype=torch.bfloat16, device="cuda")
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream()
    step = lambda: cp.lookup_decode(table, idx, out, stream)  # noqa: E731

    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clocks:
        t = time_steps(step, args.steps, args.warmup, flush, stream, "step")
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    status = cp.get_status(table)
    assert status == cp.CP_OK, status
    out_host = out.cpu()                       # the last timed step's rows, for the parity check
    total, value = aggregate(float(t.sum()), n * args.steps, world, dist, "cuda")
    mean_t = total / args.steps
    bpl = w.algorithmic_bytes_per_lookup()
    achieved = n * bpl / float(t.mean()) / 1e9
    peak, peak_kind = measured_peaks()

    others = None
    # single-GPU characterisation legs run at N = 1 only (they would hold every
    # GPU of a multi-rank job while rank 0 alone works)
    solo = world == 1
    sustained = None
    if solo and args.sustained_calls > 0:
        sustained = sustained_measure(args, w, table, out, flush, stream, bpl=w.algorithmic_bytes_per_lookup())
    ctx = hbm_same_run(flush, stream) if solo else None
    if ctx is not None:
        ctx["decode_frac_of_copy"] = achieved / ctx["copy_gbs"]
    if solo and not args.no_other_configs:
        others = other_configs(args, w, table, idx, out, flush, stream)

    # Decode fused with a weighted readout over each token's 24 rows of a layer.
    fused = fused_measure(args, w, table, idx, flush, stream) if solo else None

    # Mixed per-row bit rates (frequency-based allocation): 2^24 rows x the same d,
    # rates uniform over b = 1.5 .. 3, the same replay shape.
    mixed = mixed_measure(args, w, n, flush, stream) if solo else None

    # Offline compression on the GPU (the step before the hot path).
    enc = encoder_measure(args, w) if solo and w.d >= 16 else None

    # End to end through the public API: ids from pinned host memory, rows back
    # to pinned host memory, both copies inside the timed region.
    idx_h = torch.from_numpy(idx_np).pin_memory()
    out_h = torch.empty((n, w.d), dtype=torch.bfloat16, pin_memory=True)
    idx_d = torch.empty_like(idx)

    def e2e_step():                 # rows written by the kernel straight into pinned host memory
        idx_d.copy_(idx_h, non_blocking=True)
        cp.lookup_decode(table, idx_d, out_h, stream)

    te = time_steps(e2e_step, args.e2e_steps, 3, flush, stream, "e2e")
    _, e2e_value = aggregate(float(te.sum()), n * args.e2e_steps, world, dist, "cuda")
    d2h = d2h_link_gbs(flush, stream) if solo else None

    host_obj = None
    if not args.no_host_path and solo and w.residency in ("device", "host") \
            and w.d >= 256:
        del rec, soa
        table.close()
        torch.cuda.empty_cache()
        host_obj = host_path_measure(args, w, idx, flush, stream)

    cpu = None
    parity = None
    if solo and not args.no_cpu_baseline:
        parity = oracle_parity(w, idx_np, out_host, cp.default_lut())
        rate, m, nt = oracle_sample_rate(w, idx_np, args.cpu_seconds, cp.default_lut())
        rate1, m1, _ = oracle_sample_rate(w, idx_np, args.cpu_seconds / 4, cp.default_lut(), 1)
        cpu = {"value": rate, "unit": "rows/s", "cores": nt, "kind": "oracle",
               "sample": f"first {m} lookups of the replay, records regenerated on the host, "
                         f"{nt} threads",
               "single_thread": {"value": rate1, "unit": "rows/s", "cores": 1,
                                 "sample": f"first {m1} lookups of the replay"}}

    if rank == 0:
        clk = clocks.summary()
        line = {
            "metric": METRIC, "value": value, "unit": "rows/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": mean_t * 1e3,
            "higher_is_better": True, "scaling": "weak",
            "vs_baseline": value / world / (w.n_lookups / PAGES_LATENCY_S)
            if w.name == "deepseek_prefill" else None,
            "dtype": "fp32", "data": "synthetic",
            "config": workload_config(w, args.layout, world, idx_np, synth.SEED_INDEX + rank),
            "achieved_gbs_algorithmic": achieved,
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak, "peak_kind": peak_kind,
                         "traffic": ncu_traffic(w.name, args.layout),
                         "bytes_per_lookup": bpl, "kernel": "lookup_decode_block_kernel"},
            "e2e": {"value": e2e_value, "unit": "rows/s", "h2d_bytes_per_step": n * 8,
                    "path": "ids copied from pinned host memory; rows written by the decode kernel into pinned host memory",
                    "d2h_bytes_per_step": n * w.d * 2,
                    **({"d2h_link_gbs": d2h,
                        "frac_of_d2h_link": n * w.d * 2 * e2e_value / n / 1e9 / d2h,
                        "d2h_link_kind": "measured: cudaMemcpyAsync device->pinned, 1 GB"}
                       if d2h else {})},
            "gpu_launches": args.steps,
            "clocks": clk,
            "step_ms": {"min": float(t.min() * 1e3), "median": float(np.median(t) * 1e3),
                        "max": float(t.max() * 1e3)},
        }
        if parity is not None:
            line["parity"] = parity
        if sustained is not None:
            line["sustained"] = sustained
        if cpu is not None:
            line["cpu_baseline"] = cpu
        if ctx is not None:
            line["hbm_same_run"] = ctx
        if host_obj is not None:
            line["host_path"] = host_obj
        if fused is not None:
            line["fused_readout"] = fused
        if mixed is not None:
            line["mixed_rate"] = mixed
        if enc is not None:
            line["encoder"] = enc
        if others is not None:
            line["other_configs"] = others
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()


def fused_measure(args, w, table, idx, flush, stream):
    """cp_lookup_decode_reduce over each token's 24 rows of a layer, random gates."""
    import torch
    import trellis_row_decode_gb300 as cp
    n = idx.numel()
    if w.d not in (256, 512, 1024) or w.rows_per_token % 24 != 0:
        return None
    group = 24
    gates = torch.rand(n, dtype=torch.float32, device="cuda",
                       generator=torch.Generator(device="cuda").manual_seed(5))
    red_out = torch.empty((n // group, w.d), dtype=torch.bfloat16, device="cuda")
    tr = time_steps(lambda: cp.lookup_decode_reduce(table, idx, group, gates, red_out, stream),
                    min(args.steps, 500), args.warmup, flush, stream, "reduce")
    tm = float(np.median(tr))
    fbytes = n * (w.rec_bytes + 8 + 4) + (n // group) * 2 * w.d
    fused = {"entry_point": "cp_lookup_decode_reduce", "group": group,
             "ms_per_step": tm * 1e3, "lookups_per_s": n / tm,
             "algorithmic_gbs": fbytes / tm / 1e9, "bytes_per_step": fbytes,
             "frac_of_hbm_peak": fbytes / tm / 1e9 / measured_peaks()[0]}
    inst = ncu_inst("lookup_decode_reduce_kernel", n, w.d, w.k, group)
    if inst is not None:
        fused["roofline"] = {"bound": "alu", "achieved": inst / tm,
                             "peak": ISSUE_PEAK_WARP_INST_S, "unit": "warp-inst/s",
                             "frac": inst / tm / ISSUE_PEAK_WARP_INST_S,
                             "peak_kind": "derived: 152 SMs x 4 schedulers x 2.07 GHz",
                             "inst_per_launch": inst}
    return fused


def mixed_measure(args, w, n, flush, stream, mrows: int = 1 << 24):
    """cp_lookup_decode on a mixed-rate table of mrows rows x the workload's d, rates
    uniform over b = 1.5 .. 3, a Zipf(1.0) replay of n lookups."""
    import torch
    import trellis_row_decode_gb300 as cp
    from trellis_row_decode_gb300 import synth
    if w.d % 32 != 0 or w.d > 4096:
        return None
    ks = synth.mixed_rates(synth.SEED_TABLE, torch.arange(mrows, device="cuda"))
    moffs = synth.mixed_offsets(ks, w.d)
    mbuf = torch.empty(int(moffs[-1].item()), dtype=torch.uint8, device="cuda")
    synth.fill_mixed_records(mbuf, synth.SEED_TABLE, ks, moffs, w.d)
    mtable = cp.load_mixed_table(mbuf, moffs, w.d)
    midx = torch.from_numpy(synth.zipf_indices(synth.SEED_INDEX, n, mrows)).cuda()
    mout = torch.empty((n, w.d), dtype=torch.bfloat16, device="cuda")
    mrec = (moffs[1:] - moffs[:-1])[midx].sum().item()
    tmx = time_steps(lambda: cp.lookup_decode(mtable, midx, mout, stream), min(args.steps, 500),
                     args.warmup, flush, stream, "mixed")
    assert cp.get_status(mtable) == cp.CP_OK
    tmm = float(np.median(tmx))
    mbytes = mrec + n * (2 * w.d + 8 + 16)
    res = {"entry_point": "cp_lookup_decode (mixed-rate table)", "n_rows": mrows,
           "mean_bits_per_param": float(mbuf.numel() * 8 / (mrows * w.d)),
           "ms_per_step": tmm * 1e3, "rows_per_s": n / tmm,
           "algorithmic_gbs": mbytes / tmm / 1e9,
           "frac_of_hbm_peak": mbytes / tmm / 1e9 / measured_peaks()[0]}
    mtable.close()
    return res


def sustained_measure(args, w, table, out, flush, stream, bpl: int):
    """Back-to-back decode calls with no flush between them, each over its own replay
    (index seeds SEED_INDEX + i), after one L2 flush: every call pays the write-back
    of the rows the previous calls left dirty in L2, as in a serving loop.  The rows
    alternate between two output buffers (each larger than L2)."""
    import torch
    import trellis_row_decode_gb300 as cp
    from trellis_row_decode_gb300 import synth
    K = args.sustained_calls
    ids = [torch.from_numpy(w.indices(synth.SEED_INDEX + i)).cuda() for i in range(K)]
    outs = [out, torch.empty_like(out)]
    for i in range(min(K, 3)):                                    # warm-up
        cp.lookup_decode(table, ids[i], outs[i & 1], stream)
    flush_l2(flush)
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for i in range(K):
        cp.lookup_decode(table, ids[i], outs[i & 1], stream)
    b.record(stream)
    torch.cuda.synchronize()
    assert cp.get_status(table) == cp.CP_OK
    per = a.elapsed_time(b) * 1e-3 / K
    n = ids[0].numel()
    peak = measured_peaks()[0]
    del outs[1]
    return {"calls": K, "ms_per_step": per * 1e3, "rows_per_s": n / per,
            "achieved_gbs": n * bpl / per / 1e9, "frac": n * bpl / per / 1e9 / peak,
            "replays": f"index seeds {synth.SEED_INDEX}..{synth.SEED_INDEX + K - 1}, one per call",
            "l2": "flushed once before the window; no flush between calls"}


def encoder_measure(args, w):
    """cp_encode_rows_ws on N(0,1) rows of the workload's d and rate: the workspace
    is allocated once outside the timing; one warm-up call on half the rows, then
    one call timed with CUDA events on the launching stream (LUT copy + kernel)."""
    import torch
    import trellis_row_decode_gb300 as cp
    from trellis_row_decode_gb300 import synth
    erows = args.encoder_rows or 4 * torch.cuda.get_device_properties(0).multi_processor_count
    e_in = torch.from_numpy(synth.normal_rows(synth.SEED_ENCODER_ROWS, erows, w.d)
                            .astype(np.float32)).cuda()
    ws = cp.encode_workspace(erows, w.d, w.k)
    rec = torch.empty((erows, w.rec_bytes), dtype=torch.uint8, device="cuda")
    ecost = torch.empty(erows, dtype=torch.float32, device="cuda")
    stream = torch.cuda.current_stream()
    half = max(1, erows // 2)
    cp.encode_rows_ws(e_in[:half], w.k, ws, rec[:half], ecost[:half], stream=stream)
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    cp.encode_rows_ws(e_in, w.k, ws, rec, ecost, stream=stream)
    b.record(stream)
    torch.cuda.synchronize()
    et = a.elapsed_time(b) * 1e-3
    res = {"entry_point": "cp_encode_rows_ws", "rows": erows, "d": w.d, "b": w.k / 2,
           "seconds": et, "rows_per_s": erows / et,
           "mean_cost_per_coord": float(ecost.mean()) / w.d,
           "timing": "CUDA events on the launching stream around the queued LUT copy and "
                     "kernel; workspace allocated once before"}
    ipr = ncu_encoder_inst_per_row(w.d, w.k)
    if ipr is not None:
        res["roofline"] = {"bound": "alu", "achieved": ipr * erows / et,
                           "peak": ISSUE_PEAK_WARP_INST_S, "unit": "warp-inst/s",
                           "frac": ipr * erows / et / ISSUE_PEAK_WARP_INST_S,
                           "peak_kind": "derived: 152 SMs x 4 schedulers x 2.07 GHz",
                           "inst_per_row": ipr}
    return res


OTHER_CONFIGS = ("mid", "sweep_b1.5", "sweep_b2", "sweep_b2.5", "sweep_b3", "deepseek_decode")


def other_configs(args, w, table, idx, out, flush, stream):
    """Median step of cp_lookup_decode on the other table configs (HBM, AoS):
    the 2^24-row d=512 table, the d=1024 bit-rate sweep, the decode step of 2048
    sequences x 48 rows on the main table, and the prefill replay issued as one
    call per layer (token-major ids [token][layer][24])."""
    import torch
    import trellis_row_decode_gb300 as cp
    from trellis_row_decode_gb300 import synth
    steps = min(args.steps, 300)
    peak = measured_peaks()[0]
    res = {}

    def entry(ow, n, tm):
        bpl = ow.algorithmic_bytes_per_lookup()
        return {"lookups": n, "d": ow.d, "b": ow.k / 2, "n_rows": ow.n_rows,
                "ms_per_step": tm * 1e3, "rows_per_s": n / tm,
                "algorithmic_gbs": n * bpl / tm / 1e9, "frac_of_hbm_peak": n * bpl / tm / 1e9 / peak}

    for name in OTHER_CONFIGS:
        ow = synth.WORKLOADS[name]
        if name == w.name:
            continue
        same_table = (ow.n_rows, ow.d, ow.k) == (w.n_rows, w.d, w.k)
        if not same_table and ow.table_bytes > (16 << 30):
            continue
        tab, rec, _ = (table, None, None) if same_table else build_table(ow, "aos", synth.SEED_TABLE)
        oidx = torch.from_numpy(ow.indices()).cuda()
        oout = torch.empty((oidx.numel(), ow.d), dtype=torch.bfloat16, device="cuda")
        t = time_steps(lambda: cp.lookup_decode(tab, oidx, oout, stream), steps, args.warmup,
                       flush, stream, "configs")
        assert cp.get_status(tab) == cp.CP_OK
        res[name] = entry(ow, oidx.numel(), float(np.median(t)))
        if not same_table:
            tab.close()
        del rec, oidx, oout
        torch.cuda.empty_cache()

    # the SoA layout (codes and scales in separate arrays) on the 2^24-row b = 2 table
    ow = synth.WORKLOADS["sweep_b2"]
    if ow.table_bytes <= (16 << 30):
        tab, rec, soa = build_table(ow, "soa", synth.SEED_TABLE)
        oidx = torch.from_numpy(ow.indices()).cuda()
        oout = torch.empty((oidx.numel(), ow.d), dtype=torch.bfloat16, device="cuda")
        t = time_steps(lambda: cp.lookup_decode(tab, oidx, oout, stream), steps, args.warmup,
                       flush, stream, "configs")
        assert cp.get_status(tab) == cp.CP_OK
        res["sweep_b2 (SoA layout)"] = entry(ow, oidx.numel(), float(np.median(t)))
        tab.close()
        del rec, soa, oidx, oout
        torch.cuda.empty_cache()

    # the same replay as two calls, one per layer of 24 rows per token
    if w.rows_per_token == 48:
        lay = idx.view(w.tokens, 2, 24)
        parts = [lay[:, l, :].contiguous().view(-1) for l in range(2)]
        outs = [out[: p.numel()] for p in parts]
        outs[1] = out[parts[0].numel():]

        def two():
            cp.lookup_decode(table, parts[0], outs[0], stream)
            cp.lookup_decode(table, parts[1], outs[1], stream)
        t = time_steps(two, steps, args.warmup, flush, stream, "configs")
        assert cp.get_status(table) == cp.CP_OK
        e = entry(w, idx.numel(), float(np.median(t)))
        e["calls_per_step"] = 2
        res[w.name + " (one call per layer)"] = e
    return res


def host_path_measure(args, w, idx, flush, stream):
    """cp_lookup_decode_host on the same table in pinned host DRAM, against measured H2D."""
    import torch
    import trellis_row_decode_gb300 as cp
    from trellis_row_decode_gb300 import synth
    R = w.rec_bytes
    host = torch.empty(w.table_bytes, dtype=torch.uint8, pin_memory=True)
    chunk = 1 << 22
    stage = torch.empty(chunk * R, dtype=torch.uint8, device="cuda")
    for r0 in range(0, w.n_rows, chunk):
        r1 = min(w.n_rows, r0 + chunk)
        rows = torch.arange(r0, r1, dtype=torch.int64, device="cuda")
        stage[: (r1 - r0) * R].view(r1 - r0, R).copy_(
            synth.gen_records(synth.SEED_TABLE, rows, w.d, w.k))
        host[r0 * R: r1 * R].copy_(stage[: (r1 - r0) * R])
    torch.cuda.synchronize()
    # measured host link: 1 GB copies from pinned memory (copy engines), and the
    # same 1 GB read zero-copy by a streaming kernel on the SMs (the decode's own
    # access path); the larger of the two is the roofline
    dst = stage[: 1 << 30]
    src = host[: 1 << 30]
    th = time_steps(lambda: dst.copy_(src, non_blocking=True), 10, 2, flush, stream, "link")
    h2d = (1 << 30) / float(np.median(th)) / 1e9
    tz = time_steps(lambda: cp.measure_stream_read(src, stream), 10, 2, flush, stream, "link")
    zero_copy = (1 << 30) / float(np.median(tz)) / 1e9
    link = max(h2d, zero_copy)
    link_kind = ("zero-copy streaming read of 1 GB pinned (cp_measure_stream_read)"
                 if zero_copy >= h2d else "cudaMemcpyAsync pinned->device, 1 GB")
    del stage, dst
    # the access pattern's own roofline: the replay's distinct records, sorted, read
    # once each over the link as the 16-byte pieces that cover them (no decode)
    uq_rows = torch.unique(idx)
    tr = time_steps(lambda: cp.measure_record_read(host, R, uq_rows, stream), 10, 2, flush, stream,
                    "link")
    record_read = int(uq_rows.numel()) * R / float(np.median(tr)) / 1e9
    table = cp.load_table(host, w.n_rows, w.d, w.k, cp.default_lut())
    n = idx.numel()
    out = torch.empty((n, w.d), dtype=torch.bfloat16, device="cuda")
    hsteps = min(args.steps, 50) if args.only == "host" else 50
    t = time_steps(lambda: cp.lookup_decode_host(table, idx, out, stream), hsteps, 3, flush, stream,
                   "host")
    assert cp.get_status(table) == cp.CP_OK
    tm = float(np.median(t))
    link_gbs = n * R / tm / 1e9
    uniq = int(torch.unique(idx).numel())
    cached = None
    if w.d in (256, 512, 1024) and w.dist == "zipf":
        # frequency-based cache: the 2^20 most frequent rows of the Zipf law in HBM
        hot = synth.feistel_bijection(np.arange(1 << 20), w.n_rows, synth.SEED_INDEX)
        cp.set_cache(table, hot)
        tc = time_steps(lambda: cp.lookup_decode_host(table, idx, out, stream), hsteps, 3, flush,
                        stream, "host_cached")
        assert cp.get_status(table) == cp.CP_OK
        tcm = float(np.median(tc))
        cached = {"hot_rows": 1 << 20, "cache_bytes": (1 << 20) * R, "ms_per_step": tcm * 1e3,
                  "rows_per_s": n / tcm,
                  "lookup_record_gbs": n * R / tcm / 1e9,
                  "note": "cached ids are read from HBM, so no link fraction applies"}
    table.close()
    return {"entry_point": "cp_lookup_decode_host", "table": "pinned host DRAM",
            "with_hot_row_cache": cached,
            "ms_per_step": tm * 1e3, "rows_per_s": n / tm,
            "bound": "host link", "unit": "GB/s",
            "link_peak": link, "link_peak_kind": f"measured: {link_kind}",
            "h2d_memcpy_gbs": h2d, "zero_copy_read_gbs": zero_copy,
            "unique_ids": uniq, "bytes_per_lookup": R,
            "achieved_unique": uniq * R / tm / 1e9,
            "link_frac_unique": uniq * R / tm / 1e9 / link,
            "record_read_gbs": record_read,
            "record_read_kind": "measured: cp_measure_record_read of the replay's distinct ids, "
                                "sorted, no decode (record bytes / time)",
            "frac_of_record_read": uniq * R / tm / 1e9 / record_read,
            "achieved_lookup_bytes": link_gbs,
            "frac_lookup_bytes": link_gbs / link,
            "note": "link_frac_unique counts the records that cross the link (one per distinct "
                    "id); frac_lookup_bytes counts n * R, every lookup's record with repeats"}


def only_leg(args, w):
    """One leg of the bench on its own (the workload's table built only when the leg
    needs it); steps / warm-up from the command line."""
    import torch
    import trellis_row_decode_gb300 as cp
    from trellis_row_decode_gb300 import synth
    if args.only == "encoder":
        return encoder_measure(args, w)
    stream = torch.cuda.current_stream()
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device="cuda")
    idx = torch.from_numpy(w.indices(synth.SEED_INDEX)).cuda()
    n = idx.numel()
    if args.only == "mixed":
        return mixed_measure(args, w, n, flush, stream, mrows=args.mixed_rows)
    if args.only == "host":
        return host_path_measure(args, w, idx, flush, stream)
    table, rec, soa = build_table(w, args.layout, synth.SEED_TABLE)
    if args.only == "reduce":
        return fused_measure(args, w, table, idx, flush, stream)
    out = torch.empty((n, w.d), dtype=torch.bfloat16, device="cuda")
    t = time_steps(lambda: cp.lookup_decode(table, idx, out, stream), args.steps, args.warmup,
                   flush, stream)
    assert cp.get_status(table) == cp.CP_OK
    bpl = w.algorithmic_bytes_per_lookup()
    tm = float(np.median(t))
    return {"entry_point": "cp_lookup_decode", "workload": w.name, "layout": args.layout,
            "ms_per_step": tm * 1e3, "rows_per_s": n / tm, "achieved_gbs": n * bpl / tm / 1e9,
            "frac_of_hbm_peak": n * bpl / tm / 1e9 / measured_peaks()[0]}


def main():
    args = parse()
    from trellis_row_decode_gb300 import synth
    w = synth.WORKLOADS[args.workload]
    rank, world, local = dist_env()
    if args.gpus != world and world > 1:
        print(f"warning: --gpus {args.gpus} but WORLD_SIZE {world}", file=sys.stderr)
    if args.impl == "reference":
        reference_arm(args, w, rank)
        return
    if args.only is not None:
        import torch
        torch.cuda.set_device(local)
        res = only_leg(args, w)
        if rank == 0:
            print(json.dumps({args.only: res}), flush=True)
        return
    our_arm(args, w, rank, world, local)


if __name__ == "__main__":
    main()
