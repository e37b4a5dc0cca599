#!/usr/bin/env python3
"""Sparse MLA decode throughput on GB300: query-rows/s and gathered-KV GB/s.

One step = one smla_decode call over one batch of the workload: the decode
kernel (gather, QK, softmax, PV, epilogue), the merge kernel when rows are
shared between CTAs, and the row-trim pass before them when the workload has
-1 padding (has_invalid); the KV cache, queries and index stream are resident
in HBM.  L2 is flushed between timed steps (a 256 MB write, then a 256 MB
read: the read leaves the L2 holding clean lines, so the flush's own
write-back does not land inside the timed step).  Prints ONE JSON line
(rank 0).

  python bench.py [--gpus N --steps K --warmup W] [--workload decode]
  python bench.py --impl reference ...   # the fp64 CPU oracle on host cores

Multi-GPU (torchrun, one process per GPU): every rank decodes its own batch
of the workload (rows are independent: no data-path collective), so scaling is
weak; only the timing uses a barrier and a max over ranks.
"""

from __future__ import annotations

import argparse
import hashlib
import re
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import smla_workloads as W  # noqa: E402

METRIC = "sparse MLA decode query-rows/s and gathered-KV GB/s (% of GB300 HBM peak)"
FALLBACK_HBM_GBS = 6800.0


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="smla", choices=["smla", "reference"])
    ap.add_argument("--workload", default="decode", choices=sorted(W.WORKLOADS))
    ap.add_argument("--also", default="wide,ragged,long",
                    help="comma list of extra workloads to time ('' for none)")
    ap.add_argument("--cpu-seconds", type=float, default=12.0, help="oracle CPU-baseline budget")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--kernel", default="tc", choices=["tc", "fp8", "bf16", "simt"],
                    help="tc: the default tensor-core choice (native fp8 up to 16 heads, else bf16); "
                         "fp8 / bf16: force one tcgen05 kernel; simt: the CUDA-core cross-check kernel")
    return ap.parse_args()


def dist_env():
    return (int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)),
            int(os.environ.get("LOCAL_RANK", 0)))


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def source_digest() -> str:
    """Digest of the kernel sources' code: comments and runs of white space
    are left out, so that a recorded ncu traffic figure stays tied to the code
    it was measured on, not to its comments."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "sparse_mla_decode_csr_gb300", "csrc")
    for name in sorted(os.listdir(csrc)):
        if not name.endswith((".cu", ".cuh", ".h")):
            continue
        with open(os.path.join(csrc, name), encoding="utf-8") as f:
            text = f.read()
        text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
        text = re.sub(r"//[^\n]*", " ", text)
        h.update(name.encode() + re.sub(r"\s+", " ", text).strip().encode())
    return h.hexdigest()[:16]


def ncu_traffic(workload: str):
    """DRAM bytes per decode launch from the committed ncu summary, if it was
    taken on the current kernel sources (else None)."""
    path = os.path.join(ROOT, "profiles", "decode_traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
        entry = d.get(workload)
        if entry and entry.get("source_digest") == source_digest():
            return float(entry["dram_bytes_per_launch"])
    except Exception:
        pass
    return None


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.file = None

    def __enter__(self):
        try:
            self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=self.file, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.2)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        if self.proc is None or self.file is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.file.flush()
        rows = []
        with open(self.file.name) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.file.name)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


class Problem:
    """A workload resident on one device: records, queries, index stream, outputs."""

    def __init__(self, w: W.Workload, dev, kernel: str = "tc"):
        import sparse_mla_decode_csr_gb300 as smla

        self.smla = smla
        self.w = w
        self.dev = dev
        self.kernel = {"tc": smla.KERNEL_TENSOR_CORE, "fp8": smla.KERNEL_TENSOR_CORE_FP8,
                       "bf16": smla.KERNEL_TENSOR_CORE_BF16, "simt": smla.KERNEL_CUDA_CORE}[kernel]
        self.kv = torch.empty(w.n_kv_rows, 656, dtype=torch.uint8, device=dev)
        for s in range(W.n_slabs(w)):
            lat, rope = W.latent_slab(w, s, dev)
            start = s * W.SLAB_ROWS
            smla.smla_pack_records(lat, rope, self.kv[start:start + lat.shape[0]])
            del lat, rope
        self.q = W.queries(w, dev)
        self.indices, self.indptr = W.index_stream(w, dev)
        self.sink = W.sinks(w, dev)
        self.out = torch.empty(w.n_q, w.heads, 512, dtype=torch.bfloat16, device=dev)
        self.lse = torch.empty(w.n_q, w.heads, dtype=torch.float32, device=dev)
        self.plan = smla.smla_plan(w.n_q, w.heads, w.max_row_len, self.indices.numel(), 0,
                                   has_invalid=w.has_invalid, kernel=self.kernel)
        # a workspace of this problem's own (zeroed): its ticket counters stay valid
        nbytes = int(self.plan.workspace_bytes)
        self.ws = torch.zeros(nbytes, dtype=torch.uint8, device=dev) if nbytes else None
        ind = self.indices
        self.valid_keys = int(((ind >= 0) & (ind < w.n_kv_rows)).sum().item())
        torch.cuda.synchronize(dev)

    def bytes_per_step(self):
        w = self.w
        return self.valid_keys * 656 + w.n_q * w.heads * (576 + 512) * 2

    def step(self, q=None, indices=None, indptr=None, out=None, lse=None, stream=None):
        w = self.w
        self.smla.smla_decode(self.q if q is None else q, self.kv, w.n_kv_rows,
                              self.indices if indices is None else indices,
                              self.indptr if indptr is None else indptr, None, w.sm_scale, self.sink,
                              self.out if out is None else out, self.lse if lse is None else lse,
                              stream, max_row_len=w.max_row_len, has_invalid=w.has_invalid,
                              workspace_tensor=self.ws, kernel=self.kernel)


def reduce_max(x: float, dev) -> float:
    """Max of a per-rank number over all ranks (identity on one process)."""
    dist = torch.distributed
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def weak_scaling_rows_per_s(world: int, rows_per_rank: int, steps: int, max_total_ms: float) -> float:
    """Whole-job rows/s: every rank decodes its own batch of rows each step;
    the job takes as long as its slowest rank."""
    return world * rows_per_rank * steps / (max_total_ms * 1e-3)


def l2_flusher(dev):
    """Evicts the workload from L2 between timed steps: writes a buffer of at
    least twice the L2 size, then reads another of the same size, so that the
    L2 is left holding clean lines.  A write-only flush leaves up to an L2 of
    dirty lines whose write-back then lands inside the next timed step (8-12 us
    per launch on a 688 MB gather, measured with a gather-only kernel)."""
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    n = max(2 * l2, 256 << 20)
    wbuf = torch.empty(n, dtype=torch.uint8, device=dev)
    rbuf = torch.ones(n // 4, dtype=torch.float32, device=dev)
    sink = torch.empty((), dtype=torch.float32, device=dev)

    def flush():
        wbuf.fill_(1)
        torch.sum(rbuf, dim=0, out=sink)

    return flush


NOMINAL_HBM_GBS = 7900.0  # GB300 HBM3e, nominal
KERNEL_NAMES = {1: "CUDA-core", 2: "bf16 tcgen05", 3: "native-fp8 tcgen05"}
# the type each kernel multiplies in (all accumulate in f32)
KERNEL_DTYPES = {1: "f32", 2: "bf16", 3: "e4m3"}


def scale_histogram(kv: torch.Tensor) -> dict:
    """log2 of the records' block scales (bytes [512, 528) as f32): how many
    blocks have each power of two."""
    sc = kv[:, 512:528].contiguous().view(torch.float32).flatten()
    e = torch.log2(sc).round().to(torch.int64)
    lo = int(e.min().item())
    counts = torch.bincount(e - lo)
    return {str(lo + i): int(c) for i, c in enumerate(counts.tolist()) if c}


def time_writer(dev, n: int = 1 << 20, reps: int = 10) -> dict:
    """The record writer (smla_pack_records) on n records of bf16 latent and
    rope already in HBM: 1152 B read and 656 B written per record, L2 flushed
    before each call."""
    import sparse_mla_decode_csr_gb300 as smla

    g = torch.Generator(device=dev)
    g.manual_seed(0x5EED)
    lat = torch.randn(n, 512, generator=g, device=dev).to(torch.bfloat16)
    rope = torch.randn(n, 64, generator=g, device=dev).to(torch.bfloat16)
    kv = torch.empty(n, 656, dtype=torch.uint8, device=dev)
    flush = l2_flusher(dev)
    stream = torch.cuda.current_stream(dev)
    for _ in range(3):
        smla.smla_pack_records(lat, rope, kv, stream)
    ms = []
    for _ in range(reps):
        flush()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        smla.smla_pack_records(lat, rope, kv, stream)
        b.record(stream)
        b.synchronize()
        ms.append(a.elapsed_time(b))
    t = statistics.mean(ms)
    gbs = n * (1152 + 656) / (t * 1e-3) / 1e9
    peak, _ = measured_peaks()
    return {"records": n, "ms_per_call": t, "gbs": gbs, "hbm_frac": gbs / peak,
            "bytes_per_record": 1152 + 656}


def time_device(prob: Problem, steps: int, warmup: int, flush, dist_ok: bool):
    stream = torch.cuda.current_stream(prob.dev)
    for _ in range(warmup):
        flush()
        prob.step(stream=stream)
    torch.cuda.synchronize(prob.dev)
    if dist_ok:
        torch.distributed.barrier()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    torch.cuda.nvtx.range_push("timed")
    for a, b in evs:
        flush()
        a.record(stream)
        prob.step(stream=stream)
        b.record(stream)
    torch.cuda.synchronize(prob.dev)
    torch.cuda.nvtx.range_pop()
    if dist_ok:
        torch.distributed.barrier()
    return [a.elapsed_time(b) for a, b in evs]


def _staging(tensors, dev):
    """One pinned host buffer and one device buffer holding the given tensors
    back to back (256-byte aligned), and views of both in their shapes."""
    offs, n = [], 0
    for t in tensors:
        offs.append(n)
        n += (t.numel() * t.element_size() + 255) // 256 * 256
    host = torch.empty(n, dtype=torch.uint8).pin_memory()
    devb = torch.empty(n, dtype=torch.uint8, device=dev)

    def views(buf):
        return [buf[o:o + t.numel() * t.element_size()].view(t.dtype).view(t.shape) for o, t in zip(offs, tensors)]

    return host, devb, views(host), views(devb)


def time_e2e(prob: Problem, steps: int, flush):
    """Per step: one pinned-host -> device copy of the step's inputs (q,
    indices and indptr staged back to back), the decode on views of that
    buffer, and one device -> pinned-host copy of its outputs (out and lse
    back to back); all inside the events."""
    stream = torch.cuda.current_stream(prob.dev)
    h_in, d_in, (h_q, h_i, h_p), (d_q, d_i, d_p) = _staging([prob.q, prob.indices, prob.indptr], prob.dev)
    h_q.copy_(prob.q.cpu())
    h_i.copy_(prob.indices.cpu())
    h_p.copy_(prob.indptr.cpu())
    h_out, d_out, _, (d_o, d_l) = _staging([prob.out, prob.lse], prob.dev)
    h2d, d2h = h_in.numel(), h_out.numel()  # bytes copied, alignment gaps included
    total = 0.0
    for i in range(steps + 2):
        flush()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        d_in.copy_(h_in, non_blocking=True)
        prob.step(q=d_q, indices=d_i, indptr=d_p, out=d_o, lse=d_l, stream=stream)
        h_out.copy_(d_out, non_blocking=True)
        b.record(stream)
        b.synchronize()
        if i >= 2:
            total += a.elapsed_time(b)
    return total, h2d, d2h


class OracleSample:
    """The workload's rows prepared for the oracle: records of every key the
    rows gather, packed by the oracle's own writer, and the CSR remapped onto
    them (done once, outside any timing)."""

    def __init__(self, w: W.Workload, max_rows: int = 256):
        import oracle

        self.oracle = oracle
        self.w = w
        indices, indptr = W.index_stream(w, "cpu")
        self.rows = list(range(min(w.n_q, max_rows)))
        self.q = W.queries(w, "cpu").double().numpy()
        sink = W.sinks(w, "cpu")
        self.sink = None if sink is None else sink.double().numpy()
        ind, ptr = indices.numpy(), indptr.numpy()
        sl = [ind[ptr[r]:ptr[r + 1]] for r in self.rows]
        cat = np.concatenate(sl)
        ok = (cat >= 0) & (cat < w.n_kv_rows)
        ids = np.unique(cat[ok])
        lat, rope = W.latent_rows(w, torch.from_numpy(ids), "cpu")
        self.rec = oracle.pack_records(lat.view(torch.int16).numpy().view(np.uint16),
                                       rope.view(torch.int16).numpy().view(np.uint16))
        self.idx = np.where(ok, np.searchsorted(ids, np.where(ok, cat, 0)), -1).astype(np.int32)
        self.ptr = np.concatenate([[0], np.cumsum([len(x) for x in sl])]).astype(np.int64)

    def decode_row(self, i: int):
        r = self.rows[i % len(self.rows)]
        a, b = self.ptr[i % len(self.rows)], self.ptr[i % len(self.rows) + 1]
        self.oracle.sparse_mla_decode(self.q[r:r + 1], self.rec, self.idx[a:b],
                                      np.array([0, b - a], np.int32), None, self.w.sm_scale,
                                      self.sink, n_kv_rows=len(self.rec))

    def time(self, budget_s: float, start: int = 0):
        done, spent = 0, 0.0
        while done == 0 or spent < budget_s:
            t0 = time.perf_counter()
            self.decode_row(start + done)
            spent += time.perf_counter() - t0
            done += 1
        return done, spent


def blas_threads() -> int:
    t = os.environ.get("OPENBLAS_NUM_THREADS") or os.environ.get("OMP_NUM_THREADS")
    return int(t) if t else (os.cpu_count() or 1)


def cpu_baseline(w: W.Workload, budget_s: float):
    """The oracle as it stands, on this host's cores, over a bounded sample of
    the workload's rows."""
    smp = OracleSample(w)
    done, spent = smp.time(budget_s)
    cores = blas_threads()
    return {"value": done / spent, "unit": "rows/s", "cores": cores, "kind": "oracle",
            "sample": f"{done} query rows of {w.name} in {spent:.1f} s of oracle time "
                      f"(numpy fp64; BLAS threads up to {cores})"}


def run_reference(args, rank, world):
    """The reference arm: the fp64 oracle on the host cores, each step a
    bounded sample of the workload's rows (rank 0 only)."""
    if rank != 0:
        return
    w = W.WORKLOADS[args.workload]
    smp = OracleSample(w)
    for i in range(args.warmup):
        smp.decode_row(i)
    budget = max(0.5, min(args.cpu_seconds, 120.0 / max(args.steps, 1)))
    done, spent = 0, 0.0
    for _ in range(args.steps):
        d, s_ = smp.time(budget, start=done)
        done += d
        spent += s_
    value = done / spent
    cores = blas_threads()
    line = {"metric": METRIC, "value": value, "unit": "rows/s", "impl": "reference", "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1000.0 * spent / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic",
            "config": {"workload": w.name, "n_q": w.n_q, "heads": w.heads, "topk": w.topk,
                       "n_kv_rows": w.n_kv_rows},
            "cpu_baseline": {"value": value, "unit": "rows/s", "cores": cores, "kind": "oracle",
                             "sample": f"{done} query rows of {w.name} over {args.steps} steps "
                                       f"({spent:.1f} s of oracle time)"},
            "e2e": {"value": value, "unit": "rows/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    args = parse_args()
    rank, world, local_rank = dist_env()
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    assert args.warmup >= 3, "at least 3 warm-up steps"
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    dist_ok = world > 1
    if dist_ok:
        torch.distributed.init_process_group("nccl", device_id=dev)
    w = W.WORKLOADS[args.workload]
    prob = Problem(w, dev, args.kernel)
    flush = l2_flusher(dev)
    with ClockSampler(local_rank) as clk:
        times = time_device(prob, args.steps, args.warmup, flush, dist_ok)
    total_ms = reduce_max(sum(times), dev)
    e2e_ms, h2d, d2h = time_e2e(prob, args.steps, flush)
    e2e_ms = reduce_max(e2e_ms, dev)
    # the same steps without the L2 flush (records gathered by several rows,
    # and with caches under the L2's size the whole cache, stay in L2)
    warm_ms = statistics.mean(time_device(prob, max(10, args.steps // 2), args.warmup, lambda: None, False))

    extra = {}
    writer = time_writer(dev) if rank == 0 else None
    for name in [x for x in args.also.split(",") if x and x != args.workload]:
        wx = W.WORKLOADS[name]
        px = Problem(wx, dev, args.kernel)
        tx = time_device(px, max(10, args.steps // 2), args.warmup, flush, False)
        mean_ms = statistics.mean(tx)
        peak, _ = measured_peaks()
        gbs = px.bytes_per_step() / (mean_ms * 1e-3) / 1e9
        extra[wx.name] = {"rows_per_s": wx.n_q / (mean_ms * 1e-3), "ms_per_step": mean_ms,
                          "gathered_kv_gbs": gbs, "hbm_frac": gbs / peak,
                          "roofline": {"bound": "hbm", "achieved": gbs, "peak": peak, "unit": "GB/s",
                                       "frac": gbs / peak, "traffic": ncu_traffic(wx.name),
                                       "algorithmic_bytes_per_launch": px.bytes_per_step()},
                          "kernel": KERNEL_NAMES[px.plan.kernel],
                          "gpu_launches_per_step": 1 + int(px.plan.merge_kernel) + int(px.plan.trim_kernel),
                          "num_splits": px.plan.num_splits, "grid": px.plan.grid}
        if wx.latent != "normal":
            extra[wx.name]["log2_scale_histogram"] = scale_histogram(px.kv)
        del px
        torch.cuda.empty_cache()

    if rank != 0:
        if dist_ok:
            torch.distributed.destroy_process_group()
        return
    steps = args.steps
    sec = total_ms * 1e-3
    value = weak_scaling_rows_per_s(world, w.n_q, steps, total_ms)
    mean_ms = total_ms / steps
    bytes_step = prob.bytes_per_step()
    achieved = bytes_step / (mean_ms * 1e-3) / 1e9
    peak, peak_src = measured_peaks()
    cpu = None
    if not args.no_cpu_baseline:
        cpu = cpu_baseline(w, args.cpu_seconds)
    line = {
        "metric": METRIC, "value": value, "unit": "rows/s", "n_gpus": world, "steps": steps,
        "warmup": args.warmup, "ms_per_step": mean_ms, "ms_per_step_median": statistics.median(times),
        "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": KERNEL_DTYPES[prob.plan.kernel], "data": "synthetic",
        "config": {"workload": w.name, "n_q": w.n_q, "heads": w.heads, "topk": w.topk,
                   "n_kv_rows": w.n_kv_rows, "rows_per_gpu": w.n_q,
                   "l2": "flushed between steps (256 MB written, then 256 MB read)",
                   "num_splits": prob.plan.num_splits, "grid": prob.plan.grid},
        "gathered_kv_gbs": achieved * world,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": ncu_traffic(w.name),
                     "peak_source": peak_src,
                     "kernel": (f"one smla_decode call ({KERNEL_NAMES[prob.plan.kernel]} decode kernel"
                                + (" + merge kernel" if prob.plan.merge_kernel else "")
                                + (" + row-trim pass" if prob.plan.trim_kernel else "") + "), CUDA events"),
                     "algorithmic_bytes_per_launch": bytes_step,
                     "frac_of_nominal": achieved / NOMINAL_HBM_GBS, "nominal_gbs": NOMINAL_HBM_GBS},
        "warm_l2": {"ms_per_step": warm_ms, "gathered_kv_gbs": bytes_step / (warm_ms * 1e-3) / 1e9,
                    "note": "no L2 flush between steps; not an HBM figure"},
        "e2e": {"value": weak_scaling_rows_per_s(world, w.n_q, steps, e2e_ms), "unit": "rows/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches": steps * (1 + int(prob.plan.merge_kernel) + int(prob.plan.trim_kernel)),
        "clocks": clk.summary(),
        "cpu_baseline": cpu,
        "also": extra,
        "writer": writer,
    }
    print(json.dumps(line), flush=True)
    if dist_ok:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
