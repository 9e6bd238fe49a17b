#!/usr/bin/env python
"""Throughput of the sparse / lazy optimizer step on GB300.

Workload: a 10,000,000 x 128 fp32 embedding table (p, m, v: 15.4 GB; last_step
int64 per row); every step is a raw COO gradient of 262,144 row lookups drawn
Zipf(1.05) (unsorted, with duplicates), values N(0, 0.01^2).  One step =
canonicalise (range check, radix sort, run detection, segmented sum of
duplicates) + lazy Adam (DormancyDecay by default, --mode lazy for Lazy) on the
touched rows, through the C-ABI entry point sparse_adam_table_step.

Metric: updated coordinates per second (touched rows x 128), whole job.  The
JSON line also carries the achieved algorithmic HBM bandwidth, a roofline object
for the dominant kernel (timed live with the library's per-kernel CUDA events on
the launch stream), an end-to-end number with host<->device copies, and the CPU
oracle timed on the host cores.

Launch: python bench.py [--gpus 1 --steps K --warmup W]; for N > 1 under
torchrun, every rank runs an independent replica of the workload on its own GPU
(no collective on the data path: weak scaling).  --impl reference times the CPU
oracle instead (rank 0 only).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from lazy_optimizers_embedding_gb300 import workloads as wl  # noqa: E402

METRIC = "sparse Adam step: updated coords/s and achieved HBM GB/s vs ~8 TB/s peak"
W_CFG = wl.CFG_ZIPF_10M_128  # replaced by a smaller table with --rows (profiling captures only)


# ---------------------------------------------------------------------------- distributed plumbing
def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def aggregate(elapsed_s: float, units: float, world: int, device=None):
    """Whole-job numbers: max elapsed over ranks, total units over ranks."""
    if world == 1:
        return elapsed_s, units
    import torch
    import torch.distributed as dist
    t = torch.tensor([elapsed_s], dtype=torch.float64, device=device)
    u = torch.tensor([units], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.all_reduce(u, op=dist.ReduceOp.SUM)
    return float(t.item()), float(u.item())


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ---------------------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi sampling of SM clock and throttle reasons while the GPU is under load."""
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, interval_ms: int = 50):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        self.proc = None
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={gpu_index}", f"--query-gpu={self.QUERY}",
                                          "--format=csv,noheader,nounits", f"-lms={interval_ms}"],
                                         stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        for line in open(self.path):
            f = [x.strip() for x in line.split(",")]
            if len(f) >= 9:
                rows.append(f)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [v for v in (num(r[1]) for r in rows) if v is not None]
        mx = [v for v in (num(r[2]) for r in rows) if v is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


# The device-timed regions start behind a bounded GPU clock spin (about 10 ms): the host
# enqueues all K steps while the GPU waits, so host-side launch jitter (a descheduled
# thread, a driver query of the clock sampler) cannot leave the GPU idle inside the
# region.  The spin lies before the first timed event.
GATE_CYCLES = 20_000_000
GATE_NOTE = ("the K steps are enqueued while the GPU waits in a bounded clock spin placed before the first "
             "timed event, so host launch jitter does not enter the device-timed region")


def launch_gate():
    import torch
    torch.cuda._sleep(GATE_CYCLES)


# ---------------------------------------------------------------------------- peaks and bytes
def hbm_peak():
    try:
        pk = json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))
        if pk.get("hbm_gbs"):
            return float(pk["hbm_gbs"]), "measured (MEASURED_PEAKS.json hbm_gbs, STREAM-style copy)"
    except (OSError, ValueError):
        pass
    return 6800.0, "fallback 6.8 TB/s (no MEASURED_PEAKS.json)"


TRAFFIC_RECORD = os.path.join(ROOT, "profiles", "row_kernel_traffic.json")
ROW_KERNEL_SOURCES = ("fused.cuh", "common.cuh", "fused_adam.cu")


def row_kernel_digest():
    import hashlib
    csrc = os.path.join(ROOT, "lazy_optimizers_embedding_gb300", "csrc")
    inner = "".join(hashlib.sha256(open(os.path.join(csrc, f), "rb").read()).hexdigest() for f in ROW_KERNEL_SOURCES)
    return hashlib.sha256(inner.encode()).hexdigest()[:16]


def recorded_traffic():
    """DRAM bytes (read + write) per launch of the row kernel from the committed ncu record
    (profiles/row_kernel_traffic.json), or None once the kernel sources differ from the captured ones."""
    try:
        rec = json.load(open(TRAFFIC_RECORD))
        if rec.get("kernel_source_digest") != row_kernel_digest():
            return None
        return int(rec["traffic_bytes_per_launch"])
    except (OSError, KeyError, ValueError):
        return None


def step_bytes(u_rows, c, n, dd):
    """Algorithmic bytes of one raw row-COO lazy Adam step: touched state rows (p, m, v) read and
    written, last_step (read in DormancyDecay, written always), gradient values and indices read."""
    return u_rows * c * 4 * 3 * 2 + u_rows * 8 * (2 if dd else 1) + n * c * 4 + n * 8


# Segments of more than this many lookups are summed in pieces by the row kernel and
# finished (merged and applied) by the two combine kernels.
SPLIT_LEN = 32


def fused_kernel_bytes(u_rows, split_rows, c, n, dd):
    """Bytes the row kernel moves by definition: the state rows and last_step of the rows it
    updates (all but those of split segments) and every gradient value."""
    rows = u_rows - split_rows
    return rows * c * 4 * 3 * 2 + rows * 8 * (2 if dd else 1) + n * c * 4


def host_inputs(n_batches, threads):
    batches = wl.coo_steps_parallel(W_CFG, range(n_batches), threads=threads)
    u_rows, split_rows = [], []
    for idx, _ in batches:
        _, cnt = np.unique(idx, return_counts=True)
        u_rows.append(int(cnt.shape[0]))
        split_rows.append(int((cnt > SPLIT_LEN).sum()))
    return batches, u_rows, split_rows


def oracle_steps(p, m, v, ls, batches, u_rows, first_t, steps, dd, budget_s=None):
    """Runs the CPU oracle over `steps` steps; returns (updated coords, seconds spent in the oracle)."""
    import oracle
    w = W_CFG
    mode = oracle.MODE_DORMANCY_DECAY if dd else oracle.MODE_LAZY
    spent, units, done = 0.0, 0, 0
    for k in range(steps):
        b = (first_t - 1 + k) % len(batches)
        idx, vals = batches[b]
        t0 = time.perf_counter()
        rc = oracle.adam_table_step(p, m, v, ls, first_t + k, rows=idx, vals=vals, mode=mode, lr=w.lr,
                                    beta1=w.beta1, beta2=w.beta2, eps=w.eps)
        spent += time.perf_counter() - t0
        assert rc == 0, rc
        units += u_rows[b] * w.cols
        done += 1
        if budget_s is not None and spent >= budget_s:
            break
    return units, spent, done


def config_dict(dd, n_batches, world):
    w = W_CFG
    return {"workload": f"table {w.rows:,} x {w.cols} fp32, raw COO {w.lookups:,} lookups/step Zipf({w.zipf_s}) "
                        f"with duplicates, canonicalise + lazy Adam ({'DormancyDecay' if dd else 'Lazy'})",
            "rows": w.rows, "cols": w.cols, "lookups_per_step": w.lookups, "zipf_s": w.zipf_s,
            "mode": "dormancy_decay" if dd else "lazy", "last_step": "int64 per row",
            "lr": w.lr, "beta1": w.beta1, "beta2": w.beta2, "eps": w.eps,
            "parallelism": f"independent replicas x{world}" if world > 1 else "single GPU",
            "l2": "inputs larger than L2: each step reads a fresh 134 MB gradient batch and ~260 MB of touched "
                  "state (L2 is 129 MB); Zipf-hot rows may stay L2-resident across steps",
            "distinct_batches": n_batches}


# ---------------------------------------------------------------------------- our arm
def run_ours(args):
    import torch
    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=device)
    from lazy_optimizers_embedding_gb300 import binding as so
    K, W = args.steps, args.warmup
    dd = args.mode == "dd"
    w = W_CFG
    threads = os.cpu_count() or 8
    n_batches = min(K + W, args.distinct)
    batches, u_rows, split_rows = host_inputs(n_batches, threads)
    p0 = wl.table_init(w, threads=threads)

    p = torch.from_numpy(p0).to(device)
    m = torch.zeros_like(p)
    v = torch.zeros_like(p)
    ls = torch.zeros(w.rows, dtype=torch.int64, device=device)
    d_in = [(torch.from_numpy(i).to(device), torch.from_numpy(x).to(device)) for i, x in batches]
    grads = [so.row_coo(i, x, False) for i, x in d_in]
    ws = so.workspace(w.lookups, w.cols, w.rows, device)
    err = so.error_word(device)
    cfg = so.AdamConfig(lr=w.lr, beta1=w.beta1, beta2=w.beta2, eps=w.eps)
    mode = so.DORMANCY_DECAY if dd else so.LAZY
    stream = torch.cuda.current_stream(device)
    state = {"t": 0}

    def step(b, grad=None, s=None):
        state["t"] += 1
        rc = so.sparse_adam_table_step(p, m, v, ls, so.LAST_STEP_PER_ROW, w.rows, w.cols,
                                       grad if grad is not None else grads[b], state["t"], cfg, mode, ws, err,
                                       s if s is not None else stream)
        if rc:
            raise RuntimeError(so.status_string(rc))

    def check_err():
        e = int(err.item())
        if e:
            raise RuntimeError(f"device error word {e}: {so.status_string(e)}")

    batch_of = [i % n_batches for i in range(W + K)]
    for i in range(W):
        step(batch_of[i])
    torch.cuda.synchronize()
    check_err()

    # ---- device-resident timed region
    sampler = ClockSampler(local) if rank == 0 else None
    time.sleep(0.2)
    barrier(world)
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    launch_gate()
    ev0.record(stream)
    for i in range(W, W + K):
        step(batch_of[i])
    ev1.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    elapsed = ev0.elapsed_time(ev1) / 1e3
    # the same step loop keeps running ~1 s so the clock sampler sees this load
    t_busy, j = time.time(), 0
    while time.time() - t_busy < 1.0:
        for _ in range(20):
            step(j % n_batches)
            j += 1
        torch.cuda.synchronize()
    clocks = sampler.stop() if sampler else None
    check_err()
    timed = batch_of[W:W + K]
    units_local = float(sum(u_rows[b] * w.cols for b in timed))
    bytes_local = float(sum(step_bytes(u_rows[b], w.cols, w.lookups, dd) for b in timed))
    elapsed_max, units_all = aggregate(elapsed, units_local, world, device)

    # ---- per-kernel times of the same step loop (library CUDA events on the launch stream)
    so.sparse_profile_reset()
    so.sparse_profile_enable(True)
    for b in timed:
        step(b)
    torch.cuda.synchronize()
    prof = so.sparse_profile_read()
    so.sparse_profile_enable(False)
    total_prof = sum(ms for _, ms in prof.values())
    dom = "fused_rows_adam"
    dom_launches, dom_ms = prof.get(dom, (0, 0.0))
    dom_bytes = sum(fused_kernel_bytes(u_rows[b], split_rows[b], w.cols, w.lookups, dd) for b in timed) / K
    peak, peak_src = hbm_peak()
    dom_avg_s = (dom_ms / 1e3) / max(1, dom_launches)
    achieved = dom_bytes / dom_avg_s / 1e9 if dom_avg_s > 0 else None
    our_kernels = sum(l for l, _ in prof.values())
    check_err()

    # ---- per-step distribution of the same steps (events around every step), and the same
    # steps again with L2 flushed before each (a buffer of twice the L2 size written first)
    def timed_steps(before=None):
        evs = []
        for b in timed:
            if before is not None:
                before()
            a, z = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            step(b)
            z.record(stream)
            evs.append((a, z))
        torch.cuda.synchronize()
        return [a.elapsed_time(z) for a, z in evs]

    per_step = timed_steps()
    l2_bytes = int(getattr(torch.cuda.get_device_properties(device), "L2_cache_size", 0) or 129 * 2 ** 20)
    flush = torch.empty(2 * l2_bytes // 4, dtype=torch.float32, device=device)
    cold = timed_steps(lambda: flush.fill_(float(len(flush) % 7)))
    del flush
    check_err()

    def pct(xs):
        return {"median": float(np.median(xs)), "p10": float(np.percentile(xs, 10)),
                "p90": float(np.percentile(xs, 90))}

    # ---- end to end: each step's inputs copied from pinned host memory (copy stream,
    # double-buffered), the C-ABI step, the error word read back to pinned host memory
    h_in = [(torch.from_numpy(i).pin_memory(), torch.from_numpy(x).pin_memory()) for i, x in batches]
    stage = [(torch.empty_like(d_in[0][0]), torch.empty_like(d_in[0][1])) for _ in range(2)]
    stage_grads = [so.row_coo(i, x, False) for i, x in stage]
    h_err = torch.zeros(1, dtype=torch.int32).pin_memory()
    copy_stream = torch.cuda.Stream(device)
    free_ev = [torch.cuda.Event() for _ in range(2)]
    ready_ev = [torch.cuda.Event() for _ in range(2)]
    for e in free_ev:
        e.record(stream)

    def e2e_step(b, slot):
        hi, hv = h_in[b]
        di, dv = stage[slot]
        copy_stream.wait_event(free_ev[slot])
        with torch.cuda.stream(copy_stream):
            di.copy_(hi, non_blocking=True)
            dv.copy_(hv, non_blocking=True)
        ready_ev[slot].record(copy_stream)
        stream.wait_event(ready_ev[slot])
        step(b, stage_grads[slot])
        free_ev[slot].record(stream)
        h_err.copy_(err, non_blocking=True)

    for i in range(2):
        e2e_step(batch_of[i], i % 2)
    torch.cuda.synchronize()
    barrier(world)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    copy_stream.wait_event(e0)
    for k, i in enumerate(range(W, W + K)):
        e2e_step(batch_of[i], k % 2)
    e1.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    e2e_elapsed, e2e_units = aggregate(e0.elapsed_time(e1) / 1e3, units_local, world, device)
    check_err()
    assert int(h_err.item()) == 0
    bi = w.lookups * 8 + w.lookups * w.cols * 4
    bo = 4

    # ---- the oracle on the host cores, bounded sample of the same workload
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        hp = p0  # the device holds its own copy
        hm, hv = np.zeros_like(hp), np.zeros_like(hp)
        hls = np.zeros(w.rows, np.int64)
        units, spent, done = oracle_steps(hp, hm, hv, hls, batches, u_rows, 1, K + W, dd, args.cpu_seconds)
        cpu = {"value": units / spent, "unit": "coords/s", "cores": 1, "host_cores": os.cpu_count(), "kind": "oracle",
               "sample": f"first {done} steps of the same workload (full-size table, same seeded inputs); "
                         f"{spent:.1f} s of single-threaded oracle time (canonicalise + update in fp64)"}

    if rank == 0:
        achieved_gbs = bytes_local * world / elapsed_max / 1e9
        line = {
            "metric": METRIC,
            "value": units_all / elapsed_max,
            "unit": "coords/s",
            "n_gpus": world,
            "steps": K,
            "warmup": W,
            "ms_per_step": elapsed_max / K * 1e3,
            "higher_is_better": True,
            "scaling": "weak",
            "vs_baseline": None,
            "dtype": "f32",
            "data": "synthetic (seeded numpy PCG64: Zipf row indices, normal values; random-init table)",
            "config": config_dict(dd, n_batches, world),
            "achieved_hbm_gbs": achieved_gbs,
            "hbm_frac_of_peak": achieved_gbs / peak,
            "algorithmic_bytes_per_step": bytes_local / K,
            "updated_coords_per_step": units_local / K,
            "gpu_launches": int(our_kernels),
            "timed_region": GATE_NOTE,
            "roofline": {"bound": "hbm", "kernel": dom, "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": (achieved / peak) if achieved else None,
                         "traffic": recorded_traffic() if (w is wl.CFG_ZIPF_10M_128 and dd) else None,
                         "traffic_source": "ncu dram__bytes_read.sum + dram__bytes_write.sum per launch, "
                                           "profiles/row_kernel_traffic.json (a 2M-row capture scaled to the "
                                           "full launch; null once the kernel sources change)",
                         "peak_source": peak_src, "bytes_per_launch": dom_bytes,
                         "avg_launch_us": dom_avg_s * 1e6},
            "kernel_share": {k: {"launches": l, "ms": ms, "share": ms / total_prof if total_prof else None}
                             for k, (l, ms) in sorted(prof.items(), key=lambda kv: -kv[1][1])},
            "per_step_ms": dict(pct(per_step), steps=len(per_step),
                                method="CUDA events around each of the K steps, a pass after the timed one; the "
                                       "event between two steps also costs their overlap"),
            "cold_l2_ms": dict(pct(cold), flush_bytes=2 * l2_bytes,
                               method="the same steps, each after writing a buffer of twice the L2 size"),
            "clocks": dict(clocks or {}, window="timed region plus 1 s of the same step loop"),
            "e2e": {"value": e2e_units / e2e_elapsed, "unit": "coords/s", "h2d_bytes_per_step": bi,
                    "d2h_bytes_per_step": bo},
            "cpu_baseline": cpu,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


# ---------------------------------------------------------------------------- other workloads
# The other specified workloads, measured one GPU at a time with --workload (not the headline
# line): a 1-D parameter with 1,000 unique ascending coordinates per step (Adam Lazy / DD, SGD),
# a 1,000,000 x 64 table fed a CSR of summed Zipf(1.1) lookups, a 4,000,000 x 256 table fed an
# element-granular CSR with per-coordinate state, and a 50,000,000 x 32 table fed raw uniform
# lookups with lazy-momentum SGD.  Bytes per step as algorithmic traffic: state read + written
# for every touched coordinate, last_step read (DormancyDecay) and written, gradient values,
# indices / offsets / columns read.
WORKLOADS = {
    "d1_lazy": (wl.CFG_1D, "lazy"), "d1_dd": (wl.CFG_1D, "dd"), "d1_sgd": (wl.CFG_1D_SGD, None),
    "zipf1m_csr": (wl.CFG_ZIPF_1M_64, "dd"), "csr4m": (wl.CFG_CSR_4M_256, "dd"),
    "sgd50m": (wl.CFG_SGD_50M_32, None),
    # the forward-side row gather (read_rows) of the 10M x 128 table at the Zipf lookups
    "gather10m": (wl.CFG_ZIPF_10M_128, "gather"),
}


def run_workload(args):
    import torch
    from lazy_optimizers_embedding_gb300 import binding as so
    import oracle
    w, mode = WORKLOADS[args.workload]
    if args.rows is not None and args.rows != w.rows:   # a smaller table, for ncu captures only
        w = w.scaled(name=f"{w.name}_rows{args.rows}", rows=args.rows)
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    K, W = args.steps, args.warmup
    nb = min(K + W, 8)
    threads = os.cpu_count() or 8
    c = w.cols
    sgd = w.optimizer == "sgd"
    dd = mode == "dd"
    # host inputs: per batch the step's gradient, touched coordinates and algorithmic bytes
    host, units, nbytes = [], [], []
    for b in range(nb):
        if w.index_dist == "csr_elem":
            row_off, cols, vals = wl.csr_elem_step(w, b)
            nnz = cols.shape[0]
            host.append(("csr", row_off, cols, vals))
            units.append(nnz)
            nbytes.append(nnz * (24 + 16 if dd else 24 + 8) + nnz * 8 + (w.rows + 1) * 8)
        elif args.workload == "zipf1m_csr":
            idx, vals = wl.coo_step(w, b)
            uidx, inv = np.unique(idx, return_inverse=True)
            summed = np.zeros((uidx.shape[0], c), np.float64)
            np.add.at(summed, inv, vals.astype(np.float64))
            row_off = np.zeros(w.rows + 1, np.int64)
            cnt = np.zeros(w.rows, np.int64)
            cnt[uidx] = c
            np.cumsum(cnt, out=row_off[1:])
            cols = np.tile(np.arange(c, dtype=np.int32), uidx.shape[0])
            host.append(("csr", row_off, cols, summed.astype(np.float32).reshape(-1)))
            u = uidx.shape[0]
            units.append(u * c)
            nbytes.append(u * c * 24 + u * 16 + u * c * 8 + (w.rows + 1) * 8)
        elif mode == "gather":
            idx = wl.step_indices(w, b)
            host.append(("gather", idx))
            units.append(idx.shape[0] * c)
            # distinct table rows read once (repeats are L2 hits), every output row written, indices read
            nbytes.append(int(np.unique(idx).shape[0]) * c * 4 + idx.shape[0] * (c * 4 + 8))
        else:
            idx, vals = wl.coo_step(w, b)
            host.append(("coo", idx, vals))
            u = int(np.unique(idx).shape[0])
            units.append(u * c)
            per = (16 if sgd else (24 + (16 if dd else 8)))   # state (+ last_step) bytes per coordinate
            nbytes.append(u * c * per + idx.shape[0] * (8 + c * 4) if c > 1 else u * per + idx.shape[0] * 12)
    p0 = wl.table_init(w, threads=threads)
    p = torch.from_numpy(p0).to(dev).reshape(-1)
    err = so.error_word(dev)
    m = v = ls = buf = None
    if mode == "gather":
        pass
    elif sgd:
        buf = torch.zeros_like(p)
    else:
        m, v = torch.zeros_like(p), torch.zeros_like(p)
        ls = torch.zeros(p.numel() if (c == 1 or w.index_dist == "csr_elem") else w.rows, dtype=torch.int64,
                         device=dev)
    dev_in, grads, ws = [], [], None
    gather_out = None
    for h in host:
        if h[0] == "gather":
            dev_in.append((torch.from_numpy(h[1]).to(dev),))
            grads.append(None)
            if gather_out is None:
                gather_out = torch.empty((h[1].shape[0], c), dtype=torch.float32, device=dev)
        elif h[0] == "csr":
            t3 = tuple(torch.from_numpy(a).to(dev) for a in h[1:])
            dev_in.append(t3)
            grads.append(so.csr(*t3))
        else:
            t2 = (torch.from_numpy(h[1]).to(dev), torch.from_numpy(h[2]).to(dev).reshape(h[1].shape[0], -1))
            dev_in.append(t2)
            grads.append(so.row_coo(t2[0], t2[1], w.index_dist == "unique_sorted"))
    if any(h[0] == "coo" for h in host) and w.index_dist != "unique_sorted":
        ws = so.workspace(w.lookups, c, w.rows, dev)
    elif any(h[0] == "csr" for h in host) and w.index_dist != "csr_elem":
        # full-row CSR with a per-row last_step: room for the list of listed rows (<= lookups)
        ws = so.workspace(w.lookups + 1, 1, w.rows, dev)
    elif any(h[0] == "csr" for h in host):
        # element CSR with a per-coordinate last_step: room for every entry's row and gap
        ws = so.workspace(max(int(h[2].shape[0]) for h in host) + 64, 1, w.rows, dev)
    acfg = so.AdamConfig(lr=w.lr, beta1=w.beta1, beta2=w.beta2, eps=w.eps)
    scfg = so.SgdConfig(lr=w.lr, momentum=w.momentum, weight_decay=w.weight_decay)
    amode = so.DORMANCY_DECAY if dd else so.LAZY
    stream = torch.cuda.current_stream(dev)
    state = {"t": 0}
    per_coord = so.LAST_STEP_PER_COORD if (c == 1 or w.index_dist == "csr_elem") else so.LAST_STEP_PER_ROW

    def step(b):
        state["t"] += 1
        if mode == "gather":
            i = dev_in[b][0]
            rc = so.sparse_read_rows(p, w.rows, c, i, i.numel(), gather_out, err, stream)
        elif c == 1:
            i, g = dev_in[b]
            if sgd:
                rc = so.sparse_sgd_step(p, buf, w.rows, i, g, i.numel(), 1, scfg, None, err, stream)
            else:
                rc = so.sparse_adam_step(p, m, v, ls, w.rows, i, g, i.numel(), 1, state["t"], acfg, amode, None,
                                         err, stream)
        elif sgd:
            rc = so.sparse_sgd_table_step(p, buf, w.rows, c, grads[b], scfg, ws, err, stream)
        else:
            rc = so.sparse_adam_table_step(p, m, v, ls, per_coord, w.rows, c, grads[b], state["t"], acfg, amode,
                                           ws, err, stream)
        if rc:
            raise RuntimeError(so.status_string(rc))

    order = [i % nb for i in range(W + K)]
    for i in range(W):
        step(order[i])
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    launch_gate()
    e0.record(stream)
    for i in range(W, W + K):
        step(order[i])
    e1.record(stream)
    torch.cuda.synchronize()
    el = e0.elapsed_time(e1) / 1e3
    if int(err.item()):
        raise RuntimeError(so.status_string(int(err.item())))
    timed = order[W:]
    u_tot = float(sum(units[b] for b in timed))
    by_tot = float(sum(nbytes[b] for b in timed))
    so.sparse_profile_reset()
    so.sparse_profile_enable(True)
    for b in timed:
        step(b)
    torch.cuda.synchronize()
    prof = so.sparse_profile_read()
    so.sparse_profile_enable(False)
    dom, (dl, dms) = max(prof.items(), key=lambda kv: kv[1][1])
    peak, peak_src = hbm_peak()
    # the dominant kernel carries the step's state and gradient traffic (the CSR and row kernels)
    dom_bytes = by_tot / K
    dom_s = dms / 1e3 / max(1, dl)
    # the oracle on the host: a bounded sample of the same steps
    cpu = None
    if not args.no_cpu_baseline:
        hp = p0.reshape(-1).copy() if c == 1 else p0.copy()
        hm = hv = hls = hbuf = None
        if mode == "gather":
            pass
        elif sgd:
            hbuf = np.zeros_like(hp)
        else:
            hm, hv = np.zeros_like(hp), np.zeros_like(hp)
            hls = np.zeros(hp.size if per_coord == so.LAST_STEP_PER_COORD else w.rows, np.int64)
        spent, done, cu = 0.0, 0, 0
        for k in range(K + W):
            h = host[order[k]]
            t0 = time.perf_counter()
            if mode == "gather":
                oracle.read_rows(hp, h[1])
                rc = 0
            elif sgd and c == 1:
                rc = oracle.sgd_step(hp, hbuf, h[1], h[2].reshape(-1), lr=w.lr, momentum=w.momentum,
                                     weight_decay=w.weight_decay)
            elif sgd:
                rc = oracle.sgd_table_step(hp, hbuf, lr=w.lr, momentum=w.momentum, weight_decay=w.weight_decay,
                                           rows=h[1], vals=h[2])
            elif c == 1:
                rc = oracle.adam_step(hp, hm, hv, hls, h[1], h[2].reshape(-1), k + 1, lr=w.lr, beta1=w.beta1,
                                      beta2=w.beta2, eps=w.eps,
                                      mode=oracle.MODE_DORMANCY_DECAY if dd else oracle.MODE_LAZY)
            else:
                kw = dict(row_off=h[1], cols=h[2], vals=h[3]) if h[0] == "csr" else dict(rows=h[1], vals=h[2])
                rc = oracle.adam_table_step(hp, hm, hv, hls, k + 1, lr=w.lr, beta1=w.beta1, beta2=w.beta2,
                                            eps=w.eps, mode=oracle.MODE_DORMANCY_DECAY if dd else oracle.MODE_LAZY,
                                            ls_per_coord=per_coord == so.LAST_STEP_PER_COORD, **kw)
            spent += time.perf_counter() - t0
            assert rc == 0, rc
            cu += units[order[k]]
            done += 1
            if spent >= args.cpu_seconds:
                break
        cpu = {"value": cu / spent, "unit": "coords/s", "cores": 1, "host_cores": os.cpu_count(), "kind": "oracle",
               "sample": f"first {done} steps of the same workload; {spent:.1f} s of single-threaded oracle time"}
    line = {"metric": METRIC, "value": u_tot / el, "unit": "coords/s", "n_gpus": 1, "steps": K, "warmup": W,
            "ms_per_step": el / K * 1e3, "higher_is_better": True, "dtype": "f32", "data": "synthetic",
            "config": {"workload": w.name.replace("_coo", "_read_rows") if mode == "gather" else w.name,
                       "mode": mode or "sgd", "rows": w.rows, "cols": c,
                       "lookups_per_step": w.lookups, "distinct_batches": nb},
            "achieved_hbm_gbs": by_tot / el / 1e9, "hbm_frac_of_peak": by_tot / el / 1e9 / peak,
            "algorithmic_bytes_per_step": by_tot / K, "updated_coords_per_step": u_tot / K,
            "roofline": {"bound": "hbm", "kernel": dom, "achieved": dom_bytes / dom_s / 1e9 if dom_s else None,
                         "peak": peak, "unit": "GB/s",
                         "frac": dom_bytes / dom_s / 1e9 / peak if dom_s else None, "traffic": None,
                         "peak_source": peak_src, "avg_launch_us": dom_s * 1e6,
                         "bytes_note": "the step's algorithmic bytes, all moved by this kernel"},
            "kernel_share": {k: {"launches": l, "ms": ms} for k, (l, ms) in
                             sorted(prof.items(), key=lambda kv: -kv[1][1])},
            "timed_region": GATE_NOTE, "cpu_baseline": cpu}
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------- reference arm
def run_reference(args):
    """The CPU oracle as the reference arm: same workload, metric and unit (rank 0 only)."""
    world, rank, _ = dist_env()
    if rank != 0:
        return
    K, W = args.steps, args.warmup
    dd = args.mode == "dd"
    w = W_CFG
    threads = os.cpu_count() or 8
    n_batches = min(K + W, args.distinct)
    batches, u_rows, split_rows = host_inputs(n_batches, threads)
    p = wl.table_init(w, threads=threads)
    m, v = np.zeros_like(p), np.zeros_like(p)
    ls = np.zeros(w.rows, np.int64)
    oracle_steps(p, m, v, ls, batches, u_rows, 1, W, dd)
    t0 = time.perf_counter()
    units, _, _ = oracle_steps(p, m, v, ls, batches, u_rows, W + 1, K, dd)
    el = time.perf_counter() - t0
    val = units / el
    line = {"impl": "reference", "metric": METRIC, "value": val, "unit": "coords/s", "n_gpus": world,
            "steps": K, "warmup": W, "ms_per_step": el / K * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded numpy PCG64: Zipf row indices, normal values; random-init table)",
            "config": dict(config_dict(dd, n_batches, 1), parallelism="host CPU oracle, 1 thread"),
            "cpu_baseline": {"value": val, "unit": "coords/s", "cores": 1, "host_cores": os.cpu_count(), "kind": "oracle",
                             "sample": f"{K} timed steps after {W} warm-up steps of the full workload"},
            "e2e": {"value": val, "unit": "coords/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--mode", choices=["dd", "lazy"], default="dd")
    ap.add_argument("--distinct", type=int, default=64, help="at most this many distinct input batches")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--workload", choices=["zipf10m"] + sorted(WORKLOADS), default="zipf10m",
                    help="another specified workload instead of the headline one (1 GPU, one JSON line)")
    ap.add_argument("--rows", type=int, default=None,
                    help="table rows (default: the workload's); smaller tables are for ncu captures, not bench lines")
    args = ap.parse_args(argv)
    if args.rows is not None and args.rows != W_CFG.rows and args.workload == "zipf10m":
        globals()["W_CFG"] = W_CFG.scaled(name=f"{W_CFG.name}_rows{args.rows}", rows=args.rows)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.workload != "zipf10m":
        run_workload(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
