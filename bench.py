#!/usr/bin/env python
"""Throughput of the packed-training hot path on GB300.

One step = the whole path over one batch of synthetic input already resident
in HBM: spd_pack_tokens (documents -> packed rows, cu_seqlens), then
spd_varlen_attn_fwd and spd_varlen_attn_bwd over the packed rows.

metric: unmasked attention FLOPs (fwd + bwd) per second. Only the entries of
the per-document causal mask count: pairs = sum over segments L (L + 1) / 2,
fwd = 4 d Hq pairs, bwd = 2.5 x fwd (five GEMMs including the S recompute);
the strict count (bwd = 2 x fwd) is printed beside it.

Default workload: the load-balance stress case, the largest one that the
library is measured on: one packed row of 1,048,576 tokens (micro_bsz 1,
SEQ_LEN 1048576), document lengths 95% uniform [16, 512] and 5% uniform
[32768, 131072], 4 q / 4 kv heads, head_dim 128, bf16. Inputs (1 GiB per
tensor) exceed the 129 MB L2, so no flush runs between steps. The three other
packed workloads (4 x 8192 lognormal, 32K GQA, the 131K sequence-parallel rank
shape) are timed after it and reported under "per_config".

  python bench.py [--gpus N --steps K --warmup W] [--workload c5|c2|c3|c4|tiny]
  python bench.py --impl reference ...     # the CPU oracle as the reference arm
  python bench.py --cpu-table tiny,c2      # the fp64 oracle over whole workloads (host cores)

Several GPUs (torchrun): each rank runs an independent replica of the same
step (the path has no exchange step); rank 0 prints the aggregate.
"""
import argparse
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "packed varlen causal attn fwd+bwd TFLOP/s (unmasked FLOPs), % bf16 peak"
UNIT = "TFLOP/s"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return p, "measured"
    except OSError:
        return dict(FALLBACK_PEAKS), "fallback"


# Sources the main backward kernel is compiled from: a recorded DRAM-traffic
# figure is reported only while their hash matches the one the capture recorded.
BWD_SOURCES = ("attn_bwd.cu", "ptx.cuh", "internal.h", "sched.cu")   # the schedule shapes the traffic too
TRAFFIC_RECORD = os.path.join(ROOT, "profiles", "attn_bwd_traffic.json")


def kernel_source_hash(files):
    import hashlib
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, "sample_packing_document_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def recorded_traffic(path, files, w):
    """DRAM bytes per launch of a kernel from a one-pass ncu record (JSON:
    source hash of the kernel at capture time, the captured workload's
    documents, q heads, group and head_dim, and dram__bytes_read.sum +
    dram__bytes_write.sum of one launch). The capture runs the same documents
    with fewer heads; the heads are independent, so traffic scales with the
    head count. None when the record is missing, is for other documents or
    another shape, or the kernel's sources have changed since."""
    try:
        with open(path) as f:
            rec = json.load(f)
        if (rec["source"] != kernel_source_hash(files) or rec["docs"] != w.docs_name
                or int(rec["group"]) != w.Hq // w.Hkv or int(rec["d"]) != w.head_dim):
            return None
        return int(rec["dram_bytes"]) * w.Hq // int(rec["hq"])
    except (OSError, KeyError, ValueError):
        return None


def workload_docs(name):
    from sample_packing_document_gb300 import workloads as W
    w = W.WORKLOADS[name]
    lens, toks = W.documents(w)
    return w, lens, toks


def segment_lengths(lens, w):
    """Segment lengths of the packed rows (host arithmetic for the FLOP count
    only; the kernels compute cu_seqlens themselves every step)."""
    plen = w.micro_bsz * w.seq_len
    if w.use_packed_dataset:
        starts = np.concatenate([[0], np.cumsum(lens)[:-1]])
        total = int(lens.sum())
        rows = -(-total // plen)
        b = set(starts.tolist()) | set(range(0, rows * plen + 1, plen)) | {total}
        b = np.array(sorted(b))
        return np.diff(b)
    segs = []
    for r in range(0, len(lens), w.micro_bsz):
        kept = np.minimum(lens[r:r + w.micro_bsz], w.seq_len)
        segs += kept.tolist()
        if kept.sum() < plen:
            segs.append(plen - int(kept.sum()))
    return np.array(segs)


def flops(seg_lens, Hq, d):
    pairs = float(np.sum(seg_lens.astype(np.float64) * (seg_lens + 1) / 2))
    fwd = 4.0 * d * Hq * pairs
    return {"pairs": pairs, "fwd": fwd, "bwd": 2.5 * fwd, "total": 3.5 * fwd, "strict_total": 3.0 * fwd}


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms; summary()
    keeps the samples taken inside a host-time window."""
    Q = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = os.path.join("/tmp", "spd_clocks_%d_%d.csv" % (os.getpid(), gpu_index))

    def __enter__(self):
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.Q,
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=self.fh, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.fh.close()

    def summary(self, t0, t1):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        import datetime
        mhz, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        try:
            for line in open(self.path):
                f = [x.strip() for x in line.split(",")]
                if len(f) < 10:
                    continue
                try:
                    ts = datetime.datetime.strptime(f[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                    sm, smax = float(f[2]), float(f[3])
                except ValueError:
                    continue
                if not (t0 <= ts <= t1):
                    continue
                mhz.append(sm)
                mx = smax
                for n, v in zip(names, f[6:10]):
                    if v.lower().startswith("active"):
                        reasons.add(n)
        finally:
            try:
                os.remove(self.path)
            except OSError:
                pass
        return {"sm_mhz": statistics.median(mhz) if mhz else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(mhz)}


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def dist_max(value, ws):
    """Max of a host float over ranks (gloo on host tensors; timing only)."""
    if ws == 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def dist_barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def replica_value(ws, flops_per_rank, ms_max):
    """Whole-job TFLOP/s of ws independent replicas: every rank does
    flops_per_rank per step, the job's step time is the slowest rank's."""
    return ws * flops_per_rank / (ms_max * 1e-3) / 1e12


# ----------------------------------------------------------------------------- CPU oracle timing

def oracle_sample(w, seg_lens, cu, budget_pairs):
    """Whole segments, in a fixed shuffled order, until the unmasked pair count
    reaches budget_pairs (all heads of each segment are computed)."""
    rng = np.random.default_rng(2024)
    order = rng.permutation(len(seg_lens))
    chosen, pairs = [], 0.0
    for s in order:
        L = float(seg_lens[s])
        if chosen and pairs + L * (L + 1) / 2 > budget_pairs:
            continue
        chosen.append(int(s))
        pairs += L * (L + 1) / 2
        if pairs >= budget_pairs:
            break
    return sorted(chosen), pairs


def run_oracle_once(q16, k16, v16, do16, cu, segs, scale, nthreads):
    """fwd + bwd of the oracle over the chosen segments; returns seconds."""
    from oracle import attention as OA
    T = q16.shape[0]
    Hq = q16.shape[1]
    items = np.concatenate([np.arange(cu[s], cu[s + 1]) for s in segs])
    items = (np.arange(Hq)[:, None] * T + items[None, :]).reshape(-1)
    t0 = time.perf_counter()
    OA.attn_fwd(q16, k16, v16, cu, scale=scale, items=items, nthreads=nthreads)
    OA.attn_bwd(q16, k16, v16, do16, cu, segs=segs, scale=scale, nthreads=nthreads)
    return time.perf_counter() - t0


def cpu_inputs(w, T):
    import torch
    from sample_packing_document_gb300 import workloads as W
    q, k, v, do = W.qkv(T, w.Hq, w.Hkv, w.head_dim, w.seed, device="cpu", q_scale=w.q_scale)
    u = lambda t: t.view(torch.int16).numpy().view(np.uint16)
    return u(q), u(k), u(v), u(do)


def oracle_inputs_for(w, seg_lens):
    cu = np.concatenate([[0], np.cumsum(seg_lens)]).astype(np.int32)
    return cu


def cpu_baseline(w, seg_lens, target_s=12.0):
    """The oracle as it stands, on this host's cores, on a bounded sample."""
    from oracle import build as OB
    OB.build()
    cores = len(os.sched_getaffinity(0))
    cu = oracle_inputs_for(w, seg_lens)
    q16, k16, v16, do16 = cpu_inputs(w, int(cu[-1]))
    scale = 1.0 / np.sqrt(w.head_dim)
    # calibrate on a small sample, then size the sample to ~target_s
    segs, pairs = oracle_sample(w, seg_lens, cu, 2.0e5)
    t = run_oracle_once(q16, k16, v16, do16, cu, segs, scale, cores)
    rate = pairs / max(t, 1e-3)
    segs, pairs = oracle_sample(w, seg_lens, cu, rate * target_s)
    t = run_oracle_once(q16, k16, v16, do16, cu, segs, scale, cores)
    # Every whole segment that fits the budget may still run short of it (the
    # next ones are too long for the budget): repeat the same sample.
    reps = 1
    while t < 0.75 * target_s and reps < 64:
        t += run_oracle_once(q16, k16, v16, do16, cu, segs, scale, cores)
        reps += 1
    f = 14.0 * w.head_dim * w.Hq * pairs * reps
    return {"value": f / t / 1e12, "unit": UNIT, "cores": cores, "kind": "oracle", "cpu_model": cpu_model(),
            "sample": "fp64 oracle fwd+bwd over %d whole segments of the %s documents (%.3g of %.3g unmasked pairs, "
                      "all %d heads), %d pass(es), %.1f s"
                      % (len(segs), w.name, pairs, float(np.sum(seg_lens * (seg_lens + 1.0) / 2)), w.Hq, reps, t),
            "pack": cpu_pack_baseline()}


def cpu_pack_baseline(name="c5", reps=5):
    """The pack oracle's C twin (sequential, one core) on the workload the GPU
    pack is measured on, in the same algorithmic bytes."""
    from oracle import attention as OA
    w, lens, toks = workload_docs(name)
    times = []
    for _ in range(reps):
        t0 = time.perf_counter()
        r = OA.pack(toks, lens, w.micro_bsz, w.seq_len, w.use_packed_dataset)
        times.append(time.perf_counter() - t0)
    npos = r["rows"] * w.micro_bsz * w.seq_len
    nbytes = 4 * len(toks) + 4 * len(lens) + 12 * npos + 4 * (r["num_segs"] + 1) + 4 * (2 * r["rows"] + 2)
    s = statistics.median(times)
    # all cores: one independent pack of the same documents per core at once
    # (the C call releases the interpreter lock)
    import concurrent.futures as cf
    cores = len(os.sched_getaffinity(0))
    with cf.ThreadPoolExecutor(cores) as ex:
        list(ex.map(lambda _: OA.pack(toks, lens, w.micro_bsz, w.seq_len, w.use_packed_dataset), range(cores)))
        t0 = time.perf_counter()
        list(ex.map(lambda _: OA.pack(toks, lens, w.micro_bsz, w.seq_len, w.use_packed_dataset), range(2 * cores)))
        s_all = time.perf_counter() - t0
    return {"GB/s": nbytes / s / 1e9, "ms": s * 1e3, "bytes": nbytes, "cores": 1, "kind": "oracle (C twin of the rules)",
            "sample": "%s documents: %d tokens, %d documents, median of %d calls" % (name, len(toks), len(lens), reps),
            "all_cores": {"GB/s": 2 * cores * nbytes / s_all / 1e9, "cores": cores,
                          "sample": "%d independent packs of the same documents, %d at a time" % (2 * cores, cores)}}


def cpu_model():
    """The host CPU's model name as lscpu prints it (None if unavailable)."""
    try:
        outp = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
    except (OSError, subprocess.TimeoutExpired):
        return None
    for line in outp.splitlines():
        if line.strip().lower().startswith("model name"):
            return line.split(":", 1)[1].strip()
    return None


def cpu_table(names):
    """The fp64 oracle over whole workloads, forward (every row of every head)
    and backward (every segment) timed separately on all host cores; one JSON
    line per workload. Same FLOP convention as the GPU metric (fwd 4 d Hq
    pairs, bwd 10 d Hq pairs)."""
    from oracle import attention as OA
    from oracle import build as OB
    OB.build()
    cores = len(os.sched_getaffinity(0))
    model = cpu_model()
    for name in names:
        w, lens, toks = workload_docs(name)
        seg_lens = segment_lengths(lens, w)
        fl = flops(seg_lens, w.Hq, w.head_dim)
        cu = oracle_inputs_for(w, seg_lens)
        q16, k16, v16, do16 = cpu_inputs(w, int(cu[-1]))
        t0 = time.perf_counter()
        packed = OA.pack(toks, lens, w.micro_bsz, w.seq_len, w.use_packed_dataset)
        t_pack = time.perf_counter() - t0
        t0 = time.perf_counter()
        OA.attn_fwd(q16, k16, v16, cu, nthreads=cores)
        t_fwd = time.perf_counter() - t0
        t0 = time.perf_counter()
        OA.attn_bwd(q16, k16, v16, do16, cu, nthreads=cores)
        t_bwd = time.perf_counter() - t0
        print(json.dumps({"workload": workload_config(w, seg_lens)["workload"], "kind": "oracle", "cores": cores,
                          "cpu_model": model, "pack_s_one_core": t_pack, "rows": int(packed["rows"]),
                          "fwd_s": t_fwd, "bwd_s": t_bwd, "fwd_tflops": fl["fwd"] / t_fwd / 1e12,
                          "fwd_bwd_tflops": fl["total"] / (t_fwd + t_bwd) / 1e12,
                          "sample": "whole workload, all %d heads" % w.Hq}), flush=True)
    return 0


def run_reference(args):
    """--impl reference: the CPU oracle timed as the reference arm."""
    ws, rank, _ = dist_env()
    if rank != 0:
        return 0
    w, lens, toks = workload_docs(args.workload)
    seg_lens = segment_lengths(lens, w)
    from oracle import build as OB
    OB.build()
    cores = len(os.sched_getaffinity(0))
    cu = oracle_inputs_for(w, seg_lens)
    q16, k16, v16, do16 = cpu_inputs(w, int(cu[-1]))
    scale = 1.0 / np.sqrt(w.head_dim)
    # each step: a bounded sample sized so the whole run stays within minutes
    n_total = args.steps + args.warmup
    per_step = max(0.5, min(6.0, 150.0 / max(n_total, 1)))
    segs, pairs = oracle_sample(w, seg_lens, cu, 2.0e5)
    t = run_oracle_once(q16, k16, v16, do16, cu, segs, scale, cores)
    segs, pairs = oracle_sample(w, seg_lens, cu, pairs / max(t, 1e-3) * per_step)
    for _ in range(args.warmup):
        run_oracle_once(q16, k16, v16, do16, cu, segs, scale, cores)
    times = [run_oracle_once(q16, k16, v16, do16, cu, segs, scale, cores) for _ in range(args.steps)]
    total = sum(times)
    f = 14.0 * w.head_dim * w.Hq * pairs
    value = f * args.steps / total / 1e12
    sample = "fp64 oracle fwd+bwd over %d whole segments per step (%.3g unmasked pairs, all %d heads)" % (
        len(segs), pairs, w.Hq)
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": workload_config(w, seg_lens),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "gpu_launches": 0}
    print(json.dumps(line))
    return 0


def workload_config(w, seg_lens):
    return {"workload": "%s: %d tokens in %d packed row(s) (micro_bsz %d, SEQ_LEN %d, use_packed_dataset=%s), "
                        "%d segments, Hq %d / Hkv %d, head_dim %d" % (
                            w.name, int(seg_lens.sum()), -(-int(seg_lens.sum()) // (w.micro_bsz * w.seq_len)),
                            w.micro_bsz, w.seq_len, w.use_packed_dataset, len(seg_lens), w.Hq, w.Hkv,
                            w.head_dim),
            "tokens": int(seg_lens.sum()), "segments": int(len(seg_lens)), "max_segment": int(seg_lens.max()),
            "Hq": w.Hq, "Hkv": w.Hkv, "head_dim": w.head_dim,
            "l2": "inputs larger than L2 (no flush)" if int(seg_lens.sum()) * w.Hq * w.head_dim * 2 > 129e6
            else "L2 flushed between steps"}


# ----------------------------------------------------------------------------- GPU arm

def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1,
                    help="GPUs of the job (one process each under torchrun; independent replicas)")
    ap.add_argument("--steps", type=int, default=10, help="timed steps")
    ap.add_argument("--warmup", type=int, default=3, help="untimed warm-up steps before them")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"],
                    help="ours: the library on the GPU; reference: the fp64 oracle on this host's cores")
    ap.add_argument("--workload", default="c5",
                    help="the step's workload (default: the 1,048,576-token stress row)")
    ap.add_argument("--no-cpu-baseline", action="store_true", help="skip the oracle's CPU timing")
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer end-to-end measurement")
    ap.add_argument("--no-per-config", action="store_true", help="skip the three other workloads' step timings")
    ap.add_argument("--only", choices=["pack", "data"], default=None,
                    help="run only the pack (c5 documents) or the data-step measurements and print their JSON "
                         "(for profiling those kernels without the attention step)")
    ap.add_argument("--cpu-table", default=None,
                    help="comma-separated workloads: time the fp64 oracle (fwd and bwd) over each whole workload "
                         "on this host's cores and print one JSON line per workload; no GPU is used")
    args = ap.parse_args()
    if args.cpu_table:
        return cpu_table(args.cpu_table.split(","))
    if args.impl == "reference":
        return run_reference(args)

    import torch
    ws_n, rank, local = dist_env()
    if ws_n > 1:
        import torch.distributed as dist
        dist.init_process_group("gloo")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    import __graft_entry__
    __graft_entry__.build()
    from sample_packing_document_gb300 import ops
    if args.only:
        if rank == 0:
            print(json.dumps(pack_measure(ops, dev) if args.only == "pack" else data_measure(ops, dev)))
        return 0

    w, lens, toks = workload_docs(args.workload)
    seg_lens = segment_lengths(lens, w)
    fl = flops(seg_lens, w.Hq, w.head_dim)
    pk_, how = peaks()
    burst = pk_.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"])
    sustained = pk_.get("bf16_tflops_sustained", FALLBACK_PEAKS["bf16_tflops_sustained"])

    with ClockSampler(local) as clk:
        r = attn_step_measure(ops, dev, w, lens, toks, args.steps, args.warmup, ws_n, keep_running_s=2.0)
    clocks = clk.summary(r["host_t0"], r["host_t2"])
    clocks["window"] = "timed region" + (" + %d identical untimed steps" % r["extra"] if r["extra"] else "")
    ms = dist_max(r["ms"], ws_n)
    fwd_ms, bwd_ms = r["fwd_ms"], r["bwd_ms"]
    value = replica_value(ws_n, fl["total"], ms)

    bwd_tf = fl["bwd"] / (bwd_ms * 1e-3) / 1e12
    fwd_tf = fl["fwd"] / (fwd_ms * 1e-3) / 1e12
    roofline = {"kernel": "attn_bwd_kernel (main backward kernel, %d%% of step time)" % round(100 * bwd_ms / ms),
                "bound": "tensor", "achieved": bwd_tf, "peak": burst, "unit": "TFLOP/s",
                "frac": bwd_tf / burst, "traffic": recorded_traffic(TRAFFIC_RECORD, BWD_SOURCES, w),
                "traffic_source": "dram__bytes_read.sum + dram__bytes_write.sum per launch from a one-pass ncu "
                                  "capture of the same documents with one head (profiles/attn_bwd_traffic.json), "
                                  "scaled by the head count; null once the kernel's sources change",
                "peak_source": "%s bf16_tflops (burst): the kernel is timed in a loop of a few seconds" % how,
                "frac_of_sustained": bwd_tf / sustained,
                "flops_per_launch": fl["bwd"], "ms_per_launch": bwd_ms,
                "algorithmic": "10 d Hq pairs per launch (pairs = sum over segments L (L + 1) / 2)"}

    # end to end through the public API with host buffers, right after the
    # device-resident measurement of the same workload
    e2e = None
    if not args.no_e2e:
        e2e = e2e_measure(args, ops, w, toks, lens, dev, step_ms=ms)
        torch.cuda.empty_cache()

    per_config = None
    if rank == 0 and not args.no_per_config:
        per_config = {}
        for name in ("c2", "c3", "c4"):
            if name == args.workload:
                continue
            wc, lc, tc = workload_docs(name)
            sc = segment_lengths(lc, wc)
            fc = flops(sc, wc.Hq, wc.head_dim)
            rc = attn_step_measure(ops, dev, wc, lc, tc, 10, 3, 1)
            per_config[name] = {
                "workload": workload_config(wc, sc)["workload"], "value": fc["total"] / (rc["ms"] * 1e-3) / 1e12,
                "unit": UNIT, "ms_per_step": rc["ms"], "pct_burst": 100 * fc["total"] / (rc["ms"] * 1e-3) / 1e12 / burst,
                "kernels_ms": {"attn_fwd": rc["fwd_ms"], "attn_bwd": rc["bwd_ms"]},
                "kernels_tflops": {"attn_fwd": fc["fwd"] / (rc["fwd_ms"] * 1e-3) / 1e12,
                                   "attn_bwd": fc["bwd"] / (rc["bwd_ms"] * 1e-3) / 1e12},
                "kernels_pct_burst": {"attn_fwd": 100 * fc["fwd"] / (rc["fwd_ms"] * 1e-3) / 1e12 / burst,
                                      "attn_bwd": 100 * fc["bwd"] / (rc["bwd_ms"] * 1e-3) / 1e12 / burst},
                "grad_dtype": "bf16", "steps": 10, "warmup": 3}
            torch.cuda.empty_cache()

    pack = pack_measure(ops, dev) if rank == 0 else None
    data_steps = data_measure(ops, dev) if rank == 0 else None
    torch.cuda.empty_cache()

    cpu = None
    if rank == 0 and ws_n == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(w, seg_lens)

    if rank == 0:
        line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws_n, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
                "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded documents and N(0,1) q/k/v/dO)",
                "config": workload_config(w, seg_lens),
                "pct_bf16_peak": {"burst": 100 * value / ws_n / burst, "sustained": 100 * value / ws_n / sustained},
                "flops_per_step": fl["total"], "strict_flops_value": ws_n * fl["strict_total"] / (ms * 1e-3) / 1e12,
                "grad_dtype": "bf16",
                "kernels_ms": {"attn_fwd": fwd_ms, "attn_bwd": bwd_ms},
                "kernels_tflops": {"attn_fwd": fwd_tf, "attn_bwd": bwd_tf},
                "kernels_pct_burst": {"attn_fwd": 100 * fwd_tf / burst, "attn_bwd": 100 * bwd_tf / burst},
                "roofline": roofline, "per_config": per_config, "pack_tokens": pack, "data_steps": data_steps,
                "clocks": clocks, "e2e": e2e, "gpu_launches": r["launches_per_step"] * args.steps,
                "cpu_baseline": cpu}
        print(json.dumps(line))
    if ws_n > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def attn_step_measure(ops, dev, w, lens, toks, steps, warmup, ws_n, keep_running_s=0.0):
    """Times `steps` steps (pack + forward + backward, bf16 gradients) of one
    workload with inputs resident in HBM: CUDA events on the launching stream
    around the whole region (barrier + synchronize on both sides) and, recorded
    by the library, around the forward and backward main kernels of every
    step. With keep_running_s, the same step keeps running (untimed) until the
    host window covers that many seconds, so a clock sampler sees it."""
    import torch
    from sample_packing_document_gb300 import workloads as W
    seg_lens = segment_lengths(lens, w)
    T = int(seg_lens.sum())
    d, Hq, Hkv = w.head_dim, w.Hq, w.Hkv
    toks_d = torch.tensor(toks, device=dev)
    lens_d = torch.tensor(lens, device=dev)
    q, k, v, do = W.qkv(T, Hq, Hkv, d, w.seed, device=dev, q_scale=w.q_scale)
    pk = ops.alloc_pack_outputs(len(lens), len(toks), w.micro_bsz, w.seq_len, w.use_packed_dataset, dev)
    ops.pack_tokens(toks_d, lens_d, w.micro_bsz, w.seq_len, w.use_packed_dataset, out=pk)
    ns = int(pk["num_segs"].item())    # same documents every step: read back once
    assert ns == len(seg_lens), (ns, len(seg_lens))
    cu = pk["cu_seqlens"]
    out = torch.empty_like(q)
    lse = torch.empty(Hq, T, dtype=torch.float32, device=dev)
    dq = torch.empty_like(q)
    dk = torch.empty_like(k)
    dv = torch.empty_like(v)
    ws_f = ops.workspace(ops.attn_workspace_size(T, ns, Hq, Hkv, d, False), dev)
    ws_b = ops.workspace(ops.attn_workspace_size(T, ns, Hq, Hkv, d, True), dev)

    def step():
        ops.pack_tokens(toks_d, lens_d, w.micro_bsz, w.seq_len, w.use_packed_dataset, out=pk)
        ops.varlen_attn_fwd(q, k, v, cu, ns, out=out, lse=lse, ws=ws_f)
        ops.varlen_attn_bwd(q, k, v, out, do, lse, cu, ns, dq=dq, dk=dk, dv=dv, ws=ws_b)

    # pack: one fused launch (few documents) or scan + stream; fwd: schedule + main;
    # bwd: schedule + pre + main + dq
    launches_per_step = (1 if (w.use_packed_dataset and len(lens) <= 1024) else 2) + 2 + 4
    for _ in range(max(warmup, 3)):
        step()
    torch.cuda.synchronize()
    for wsp in (pk["ws"], ws_f, ws_b):
        st = ops.read_status(wsp)
        if st != 0:
            raise RuntimeError("device status %d (%s)" % (st, ops.status_string(st)))

    stream = torch.cuda.current_stream()
    ev = {kname: [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                  for _ in range(steps)] for kname in ("fwd", "bwd")}
    for pair in ev["fwd"] + ev["bwd"]:
        for e in pair:
            e.record(stream)    # creates the CUDA event; the library re-records it around its kernel
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if keep_running_s:
        time.sleep(0.5)                      # nvidia-smi has started sampling
    dist_barrier(ws_n)
    torch.cuda.synchronize()
    host_t0 = time.time()
    t_start.record(stream)
    for i in range(steps):
        ops.pack_tokens(toks_d, lens_d, w.micro_bsz, w.seq_len, w.use_packed_dataset, out=pk)
        ops.set_profile_events(*ev["fwd"][i], ops.PROFILE_ATTN_FWD)
        ops.varlen_attn_fwd(q, k, v, cu, ns, out=out, lse=lse, ws=ws_f)
        ops.set_profile_events(*ev["bwd"][i], ops.PROFILE_ATTN_BWD)
        ops.varlen_attn_bwd(q, k, v, out, do, lse, cu, ns, dq=dq, dk=dk, dv=dv, ws=ws_b)
        ops.set_profile_events(None, None, ops.PROFILE_NONE)
    t_end.record(stream)
    torch.cuda.synchronize()
    host_t1 = time.time()
    dist_barrier(ws_n)
    extra = 0
    if host_t1 - host_t0 < keep_running_s:
        # A short timed region holds few 200 ms samples: keep running the
        # same step (untimed) so the clock record covers the window.
        while time.time() - host_t0 < keep_running_s:
            step()
            torch.cuda.synchronize()
            extra += 1
    host_t2 = time.time()
    for wsp in (pk["ws"], ws_f, ws_b):
        st = ops.read_status(wsp)
        if st != 0:
            raise RuntimeError("device status %d (%s)" % (st, ops.status_string(st)))
    return {"ms": t_start.elapsed_time(t_end) / steps,
            "fwd_ms": statistics.mean(a.elapsed_time(b) for a, b in ev["fwd"]),
            "bwd_ms": statistics.mean(a.elapsed_time(b) for a, b in ev["bwd"]),
            "host_t0": host_t0, "host_t2": host_t2, "extra": extra, "launches_per_step": launches_per_step}


def _time_kernel(ops, which, fn, flush, reps):
    """Median device time (ms) of the one library kernel `which` that fn()
    launches, L2 flushed before every repetition."""
    import torch
    times = []
    for it in range(reps + 3):
        flush.zero_()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        b.record()
        ops.set_profile_events(a, b, which)
        fn()
        ops.set_profile_events(None, None, ops.PROFILE_NONE)
        torch.cuda.synchronize()
        if it >= 3:
            times.append(a.elapsed_time(b))
    return statistics.median(times)


def data_measure(ops, dev, reps=20):
    """The data steps after packing, each alone on device-resident inputs:
    spd_unpack_data on the c3 documents packed with use_packed_dataset=False
    (micro_bsz 4, SEQ_LEN 8192), spd_split_sequence_parallel of the c5 packed
    row (input_ids, indexes, labels) at sp_size 8, spd_pad_for_sequence_parallel
    of a ragged labels row, RoPE and the masked token loss. Algorithmic bytes /
    time."""
    import torch
    torch.manual_seed(7)       # the random tensors below are seeded like every other input
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    pk, how = peaks()
    hbm = pk.get("hbm_gbs", 6800.0)
    out = {}
    # the unpack inputs are the library's own pack of the c3 documents (use_packed_dataset=False)
    w, lens, toks = workload_docs("c3_unpack")
    packed = ops.pack_tokens(torch.tensor(toks, dtype=torch.int32, device=dev),
                             torch.tensor(lens, dtype=torch.int32, device=dev), w.micro_bsz, w.seq_len, False)
    ids, labs, cu, rsp = packed["input_ids"], packed["labels"], packed["cu_seqlens"], packed["row_seg_ptr"]
    rows = packed["rows"]
    o_ids = torch.empty((rows, w.micro_bsz, w.seq_len), dtype=torch.int32, device=dev)
    o_lab = torch.empty_like(o_ids)
    ms = _time_kernel(ops, ops.PROFILE_UNPACK, lambda: ops.unpack_data(ids, labs, cu, rsp, rows, w.micro_bsz,
                                                                       w.seq_len, o_ids, o_lab), flush, reps)
    kept = int(sum(min(int(n), w.seq_len) for n in lens))
    nbytes = int(8 * kept + 8 * o_ids.numel() + 4 * (2 * rows * w.micro_bsz + rows + 1))
    out["unpack_data"] = {"workload": "c3 documents, use_packed_dataset=False: %d rows x %d x %d" % (
        rows, w.micro_bsz, w.seq_len), "ms": ms, "bytes": nbytes, "GB/s": nbytes / (ms * 1e-3) / 1e9,
        "frac_hbm": nbytes / (ms * 1e-3) / 1e9 / hbm}
    T, sp = 1 << 20, 8
    src = [torch.randint(0, 50000, (1, T), dtype=torch.int32, device=dev) for _ in range(3)]
    dst = [torch.empty((1, T // sp), dtype=torch.int32, device=dev) for _ in range(3)]
    ms = _time_kernel(ops, ops.PROFILE_SPLIT, lambda: ops.split_sequence_parallel(src, sp, 3, out=dst), flush, reps)
    nbytes = 3 * 2 * 4 * (T // sp)
    out["split_sequence_parallel"] = {"workload": "c5 packed row (input_ids, indexes, labels), %d tokens, sp_size %d,"
                                      " rank 3" % (T, sp), "ms": ms, "bytes": nbytes,
                                      "GB/s": nbytes / (ms * 1e-3) / 1e9, "frac_hbm": nbytes / (ms * 1e-3) / 1e9 / hbm}
    # sequence-parallel padding of a ragged row: the c5 row cut to 1048573 tokens, labels padded to sp_size 8
    T = (1 << 20) - 3
    lab = torch.randint(-100, 50000, (1, T), dtype=torch.int32, device=dev)
    ms = _time_kernel(ops, ops.PROFILE_PAD, lambda: ops.pad_for_sequence_parallel(sp, labels=lab), flush, reps)
    padded = -(-T // sp) * sp
    nbytes = 4 * T + 4 * padded
    out["pad_for_sequence_parallel"] = {"workload": "labels row of %d tokens padded to %d (sp_size %d)" % (
        T, padded, sp), "ms": ms, "bytes": nbytes, "GB/s": nbytes / (ms * 1e-3) / 1e9,
        "frac_hbm": nbytes / (ms * 1e-3) / 1e9 / hbm}
    # the same two steps on 16 rows of the c5 row's length (a size at which the launch no longer
    # dominates): sequence split of three [16, 1048576] tensors, padding of a [16, 1048573] labels tensor
    rows16 = 16
    T = 1 << 20
    src = [torch.randint(0, 50000, (rows16, T), dtype=torch.int32, device=dev) for _ in range(3)]
    dst = [torch.empty((rows16, T // sp), dtype=torch.int32, device=dev) for _ in range(3)]
    ms = _time_kernel(ops, ops.PROFILE_SPLIT, lambda: ops.split_sequence_parallel(src, sp, 3, out=dst), flush, reps)
    nbytes = 3 * 2 * 4 * rows16 * (T // sp)
    out["split_sequence_parallel_16_rows"] = {
        "workload": "16 rows of %d tokens (three tensors), sp_size %d, rank 3" % (T, sp), "ms": ms, "bytes": nbytes,
        "GB/s": nbytes / (ms * 1e-3) / 1e9, "frac_hbm": nbytes / (ms * 1e-3) / 1e9 / hbm}
    del src, dst
    T = (1 << 20) - 3
    lab = torch.randint(-100, 50000, (rows16, T), dtype=torch.int32, device=dev)
    ms = _time_kernel(ops, ops.PROFILE_PAD, lambda: ops.pad_for_sequence_parallel(sp, labels=lab), flush, reps)
    padded = -(-T // sp) * sp
    nbytes = rows16 * (4 * T + 4 * padded)
    out["pad_for_sequence_parallel_16_rows"] = {
        "workload": "16 labels rows of %d tokens padded to %d (sp_size %d)" % (T, padded, sp), "ms": ms,
        "bytes": nbytes, "GB/s": nbytes / (ms * 1e-3) / 1e9, "frac_hbm": nbytes / (ms * 1e-3) / 1e9 / hbm}
    del lab
    # RoPE in place on the c2 batch's q and k (32 + 32 heads x 32768 tokens x 128), positions restarting
    # at every document (the library's pack of the c2 documents gives them as indexes)
    w, lens, toks = workload_docs("c2")
    packed = ops.pack_tokens(torch.tensor(toks, dtype=torch.int32, device=dev),
                             torch.tensor(lens, dtype=torch.int32, device=dev), w.micro_bsz, w.seq_len, True)
    pos = packed["indexes"]
    T = pos.numel()
    q = torch.randn((T, w.Hq, w.head_dim), device=dev).to(torch.bfloat16)
    k = torch.randn((T, w.Hkv, w.head_dim), device=dev).to(torch.bfloat16)
    ms = _time_kernel(ops, ops.PROFILE_ROPE, lambda: ops.rope(q, k, pos), flush, reps)
    nbytes = 2 * 2 * (w.Hq + w.Hkv) * T * w.head_dim + 4 * T
    out["rope"] = {"workload": "c2 q / k in place: %d tokens, %d + %d heads, d %d, positions = indexes" % (
        T, w.Hq, w.Hkv, w.head_dim), "ms": ms, "bytes": int(nbytes), "GB/s": nbytes / (ms * 1e-3) / 1e9,
        "frac_hbm": nbytes / (ms * 1e-3) / 1e9 / hbm}
    # RoPE fused into the forward attention's prologue, against the same forward without RoPE and
    # against the unfused path (the RoPE pass over q and k, then the forward): c2's batch, 32 / 32 heads
    v = torch.randn((T, w.Hkv, w.head_dim), device=dev).to(torch.bfloat16)
    ns = int(packed["num_segs"].item())
    cu_t = packed["cu_seqlens"][:ns + 1].contiguous()
    ws_f = ops.workspace(ops.attn_workspace_size(T, ns, w.Hq, w.Hkv, w.head_dim, False), dev)
    o_buf = torch.empty_like(q)
    l_buf = torch.empty(w.Hq, T, dtype=torch.float32, device=dev)
    ms_plain = _time_kernel(ops, ops.PROFILE_ATTN_FWD, lambda: ops.varlen_attn_fwd(q, k, v, cu_t, ns, out=o_buf,
                                                                                   lse=l_buf, ws=ws_f), flush, reps)
    ms_fused = _time_kernel(ops, ops.PROFILE_ATTN_FWD, lambda: ops.varlen_attn_fwd_rope(
        q, k, v, cu_t, ns, rope_theta=10000.0, out=o_buf, lse=l_buf, ws=ws_f), flush, reps)
    out["rope_fused_forward"] = {
        "workload": "c2 batch (%d tokens, %d / %d heads, d %d), positions restarting at every segment" % (
            T, w.Hq, w.Hkv, w.head_dim),
        "forward_ms": ms_plain, "forward_with_rope_ms": ms_fused,
        "unfused_rope_pass_ms": out["rope"]["ms"],
        "saved_ms": ms_plain + out["rope"]["ms"] - ms_fused,
        "timing": "main forward kernel (CUDA events recorded by the library), L2 flushed, median of %d" % reps}
    del v, o_buf, l_buf
    # masked token loss and its gradient over the c2 batch's labels (the same pack), synthetic bf16 logits
    # over a 50000-token vocabulary (the token ids' range)
    V = 50000
    labels = packed["labels"]
    logits = (torch.randn((T, V), device=dev) * 2).to(torch.bfloat16)
    dlogits = torch.empty_like(logits)
    tok_loss = torch.empty(T, dtype=torch.float32, device=dev)
    ms = _time_kernel(ops, ops.PROFILE_LOSS, lambda: ops.masked_token_loss(logits, labels, dlogits=dlogits,
                                                                           grad_scale=1.0 / T, token_loss=tok_loss),
                      flush, reps)
    nbytes = 2 * 2 * T * V + 12 * T
    out["masked_token_loss"] = {"workload": "c2 labels (%d tokens) with bf16 logits over %d classes, loss + gradient"
                                % (T, V), "ms": ms, "bytes": int(nbytes), "GB/s": nbytes / (ms * 1e-3) / 1e9,
                                "frac_hbm": nbytes / (ms * 1e-3) / 1e9 / hbm}
    del logits, dlogits
    out["timing"] = "CUDA events recorded by the library around the kernel, L2 flushed, median of %d" % reps
    return out


def pack_measure(ops, dev, name="c5", reps=20):
    """spd_pack_tokens alone on a workload's documents (device-resident),
    L2 flushed between repetitions; algorithmic bytes / time."""
    import torch
    w, lens, toks = workload_docs(name)
    toks_d, lens_d = torch.tensor(toks, device=dev), torch.tensor(lens, device=dev)
    out = ops.alloc_pack_outputs(len(lens), len(toks), w.micro_bsz, w.seq_len, w.use_packed_dataset, dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    segs = len(segment_lengths(lens, w))
    npos = out["rows"] * w.micro_bsz * w.seq_len
    nbytes = 4 * len(toks) + 4 * len(lens) + 12 * npos + 4 * (segs + 1) + 4 * (2 * out["rows"] + 2)
    times = []
    fused = len(lens) <= 1024 and (not w.use_packed_dataset or out["rows"] <= 512)   # one-launch paths
    for it in range(reps + 3):
        flush.zero_()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        b.record()
        # events recorded by the library right around the kernel launch, so the
        # host's call overhead is not timed (one fused launch for this case)
        ops.set_profile_events(a, b, ops.PROFILE_PACK_STREAM)
        ops.pack_tokens(toks_d, lens_d, w.micro_bsz, w.seq_len, w.use_packed_dataset, out=out)
        ops.set_profile_events(None, None, ops.PROFILE_NONE)
        torch.cuda.synchronize()
        if it >= 3:
            times.append(a.elapsed_time(b))
    if ops.read_status(out["ws"]) != 0:
        raise RuntimeError("pack status")
    ms = statistics.median(times)
    pk, how = peaks()
    gbs = nbytes / (ms * 1e-3) / 1e9
    return {"workload": "%s documents: %d tokens, %d documents, one row of %d" % (name, len(toks), len(lens), npos),
            "ms": ms, "bytes": nbytes, "GB/s": gbs, "frac_hbm": gbs / pk.get("hbm_gbs", 6800.0),
            "frac_8TBs": gbs / 8000.0,
            "timing": ("%s, CUDA events around the launch, L2 flushed, median of %d" %
                       ("the whole call (one fused kernel)" if fused else "the token-stream kernel only", reps)),
            "graph": pack_graph_measure(ops, dev, w, toks_d, lens_d, nbytes, pk.get("hbm_gbs", 6800.0)),
            "graph_16_rows": pack_graph_16_rows(ops, dev, w, toks_d, lens_d, segs, pk.get("hbm_gbs", 6800.0)),
            "graph_many_docs": pack_graph_many_docs(ops, dev, w, pk.get("hbm_gbs", 6800.0)),
            "graph_unpack_16x": pack_graph_unpack(ops, dev, pk.get("hbm_gbs", 6800.0))}


def pack_graph_unpack(ops, dev, hbm, times=16):
    """build_unpack (use_packed_dataset=False) on the 32K workload's documents
    sixteen times over: rows of micro_bsz 4 documents, each cut to SEQ_LEN 8192,
    then padding. Algorithmic bytes: 4 B read per kept token and per document
    length, 12 B written per output position, the segment fields."""
    import torch
    w, lens, toks = workload_docs("c3_unpack")
    lens16 = list(lens) * times
    toks_d = torch.tensor(toks, dtype=torch.int32, device=dev).repeat(times)
    lens_d = torch.tensor(lens16, dtype=torch.int32, device=dev)
    rows, _ = ops.pack_rows(len(lens16), toks_d.numel(), w.micro_bsz, w.seq_len, False)
    npos = rows * w.micro_bsz * w.seq_len
    kept = sum(min(int(n), w.seq_len) for n in lens16)
    segs = ops.pack_num_segs(lens16, w.micro_bsz, w.seq_len, False)
    nbytes = 4 * kept + 4 * len(lens16) + 12 * npos + 4 * (segs + 1) + 4 * (2 * rows + 2)
    r = pack_graph_measure(ops, dev, w, toks_d, lens_d, nbytes, hbm)
    r["workload"] = "%d documents (the 32K workload's, %d times over), use_packed_dataset=False, %d rows of %d x %d" % (
        len(lens16), times, rows, w.micro_bsz, w.seq_len)
    r["bytes"] = nbytes
    return r


def pack_graph_many_docs(ops, dev, w, hbm):
    """The workload's row length filled with very short documents (lengths
    uniform in [1, 8], seeded): about 233,000 documents in one 1M-token row, so
    the document-start prefix runs over some 57 CTAs chained by a look-back."""
    import torch
    from sample_packing_document_gb300 import workloads as W
    rng = np.random.default_rng(5)
    npos = w.micro_bsz * w.seq_len
    lens, toks = W.random_docs(rng, npos // 3, 1, 8)
    c = np.cumsum(lens)
    n = int(np.searchsorted(c, npos, side="left"))   # documents until the row is full, the last one cut
    lens = lens[:n + 1].copy()
    lens[n] -= int(c[n] - npos)
    if lens[n] == 0:
        lens = lens[:n]
    toks = toks[:npos]
    segs = ops.pack_num_segs(lens, w.micro_bsz, w.seq_len, True)
    rows = 1
    nbytes = 4 * npos + 4 * len(lens) + 12 * npos + 4 * (segs + 1) + 4 * (2 * rows + 2)
    wm = W.Workload("many_docs", 5, w.micro_bsz, w.seq_len, True, npos, 1, 1, 128)
    r = pack_graph_measure(ops, dev, wm, torch.tensor(toks, device=dev), torch.tensor(lens, device=dev), nbytes, hbm)
    r["workload"] = "%d tokens, %d documents of 1-8 tokens, one row of %d" % (npos, len(lens), npos)
    r["bytes"] = nbytes
    return r


def pack_graph_16_rows(ops, dev, w, toks_d, lens_d, segs, hbm):
    """The same documents sixteen times over: sixteen rows of the workload's
    row length (268 MB moved for c5), a size at which launch and scan latency
    no longer dominate (more than 1024 documents: the scan and token-stream
    launches)."""
    toks16, lens16 = toks_d.repeat(16), lens_d.repeat(16)
    rows, _ = ops.pack_rows(lens16.numel(), toks16.numel(), w.micro_bsz, w.seq_len, w.use_packed_dataset)
    npos = rows * w.micro_bsz * w.seq_len
    nbytes = 4 * toks16.numel() + 4 * lens16.numel() + 12 * npos + 4 * (16 * segs + 1) + 4 * (2 * rows + 2)
    r = pack_graph_measure(ops, dev, w, toks16, lens16, nbytes, hbm)
    r["workload"] = "%d tokens, %d documents, %d rows of %d" % (toks16.numel(), lens16.numel(), rows, npos // rows)
    r["bytes"] = nbytes
    return r


def pack_graph_measure(ops, dev, w, toks_d, lens_d, nbytes, hbm, replays=10):
    """Back-to-back packs: one CUDA graph holding one spd_pack_tokens call per
    buffer set (inputs and outputs of its own), enough sets that together they
    exceed twice the L2, replayed; device time per pack from CUDA events around
    the replays. The throughput a stream of batches sees, without host launch
    gaps and without L2 reuse between calls."""
    import torch
    l2 = getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 126 << 20)
    nsets = max(4, int(2 * l2 // nbytes) + 2)
    sets = [(toks_d.clone(), lens_d.clone(),
             ops.alloc_pack_outputs(lens_d.numel(), toks_d.numel(), w.micro_bsz, w.seq_len, w.use_packed_dataset, dev))
            for _ in range(nsets)]
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())

    def run():
        for tk, ln, out in sets:
            ops.pack_tokens(tk, ln, w.micro_bsz, w.seq_len, w.use_packed_dataset, out=out, stream=s)

    with torch.cuda.stream(s):
        run()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    try:
        with torch.cuda.graph(g, stream=s):
            run()
    except RuntimeError as e:
        return {"error": "graph capture failed: %s" % str(e).splitlines()[0]}
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(replays):
        g.replay()
    b.record()
    torch.cuda.synchronize()
    if any(ops.read_status(out["ws"]) != 0 for _, _, out in sets):
        raise RuntimeError("pack status")
    ms = a.elapsed_time(b) / (replays * nsets)
    gbs = nbytes / (ms * 1e-3) / 1e9
    del sets
    copy = same_traffic_copy(dev, toks_d.numel(), nbytes, hbm, replays)
    return {"ms_per_pack": ms, "GB/s": gbs, "frac_hbm": gbs / hbm, "frac_8TBs": gbs / 8000.0,
            "timing": "one CUDA graph of %d packs over %d buffer sets (%.0f MB, > 2x L2), %d replays, CUDA events "
                      "around the replays" % (nsets, nsets, nsets * nbytes / 1e6, replays),
            "same_traffic_copy": copy, "frac_of_copy": copy["ms_per_call"] / ms}


def same_traffic_copy(dev, n, nbytes, hbm, replays=10):
    """What a plain copy of the pack's traffic shape reaches at the same size in
    the same harness: torch's copy kernel reading n int32 and writing them three
    times (4 B read + 12 B written per position, one launch per call), in a CUDA
    graph over rotating buffer sets larger than twice the L2. The HBM copy peak
    is measured on 1 GiB; at a few MB per launch, launch and ramp latency bound
    any kernel below it, and this is that bound."""
    import torch
    l2 = getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 126 << 20)
    per = 16 * n
    nsets = max(4, int(2 * l2 // per) + 2)
    sets = [(torch.randint(0, 50000, (n,), dtype=torch.int32, device=dev),
             torch.empty((3, n), dtype=torch.int32, device=dev)) for _ in range(nsets)]
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())

    def run():
        for src, dst in sets:
            dst.copy_(src.unsqueeze(0).expand(3, n))

    with torch.cuda.stream(s):
        run()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        run()
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(replays):
        g.replay()
    b.record()
    torch.cuda.synchronize()
    ms = a.elapsed_time(b) / (replays * nsets)
    return {"ms_per_call": ms, "GB/s": per / (ms * 1e-3) / 1e9, "frac_hbm": per / (ms * 1e-3) / 1e9 / hbm,
            "bytes": per, "what": "torch copy_ of int32 [n] into [3, n], n = %d, %d sets in one graph" % (n, nsets)}


def e2e_measure(args, ops, w, toks, lens, dev, step_ms=0.0):
    """Same metric through the public API with host buffers, pipelined the way
    a training loop feeds the GPU: every step copies its documents and q / k /
    v / dO from pinned host memory (copy stream in; dO last, the backward waits
    for it alone), packs and runs forward and backward (compute stream), and
    reads dQ / dK / dV back to pinned host memory (copy stream out); the next
    steps' inputs load and the previous steps' results drain while a step
    computes (three buffer sets). The segment count comes from
    the host document lengths (spd_pack_num_segs), so no step waits on the
    device. Timed from before the first copy in to after the last copy out."""
    import torch
    from sample_packing_document_gb300 import workloads as W
    NB = 3
    ns = ops.pack_num_segs(lens, w.micro_bsz, w.seq_len, w.use_packed_dataset)
    T = int(np.sum(lens))
    q, k, v, do = W.qkv(T, w.Hq, w.Hkv, w.head_dim, w.seed, device=dev, q_scale=w.q_scale)
    pin = lambda t: t.cpu().pin_memory()
    toks_h, lens_h = torch.tensor(toks).pin_memory(), torch.tensor(lens).pin_memory()
    in_h = (toks_h, lens_h, pin(q), pin(k), pin(v), pin(do))
    in_d = [tuple(torch.empty_like(x, device=dev) for x in in_h) for _ in range(NB)]
    out_h = [tuple(torch.empty(x.shape, dtype=x.dtype).pin_memory() for x in (q, k, v)) for _ in range(NB)]
    out_d = [tuple(torch.empty_like(x) for x in (q, k, v)) for _ in range(NB)]
    pk = ops.alloc_pack_outputs(len(lens), len(toks), w.micro_bsz, w.seq_len, w.use_packed_dataset, dev)
    T, Hq, Hkv, d = q.shape[0], w.Hq, w.Hkv, w.head_dim
    o = torch.empty_like(q)
    lse = torch.empty(Hq, T, dtype=torch.float32, device=dev)
    ws_f = ops.workspace(ops.attn_workspace_size(T, ns, Hq, Hkv, d, False), dev)
    ws_b = ops.workspace(ops.attn_workspace_size(T, ns, Hq, Hkv, d, True), dev)
    s_comp = torch.cuda.current_stream()
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    ev = lambda: torch.cuda.Event()
    in_ready, comp_done, out_read = [ev() for _ in range(NB)], [ev() for _ in range(NB)], [ev() for _ in range(NB)]
    do_ready = [ev() for _ in range(NB)]
    seg_lens = segment_lengths(lens, w)
    fl = flops(seg_lens, w.Hq, w.head_dim)

    def step(kk):
        b = kk % NB
        with torch.cuda.stream(s_in):
            if kk >= NB:
                s_in.wait_event(comp_done[b])     # step kk - NB has finished reading these inputs
            for dst, src in zip(in_d[b][:5], in_h[:5]):   # documents, q, k, v: what the pack and forward read
                dst.copy_(src, non_blocking=True)
            in_ready[b].record(s_in)
            in_d[b][5].copy_(in_h[5], non_blocking=True)    # dO, read by the backward only
            do_ready[b].record(s_in)
        s_comp.wait_event(in_ready[b])
        if kk >= NB:
            s_comp.wait_event(out_read[b])        # step kk - NB's results have been read back
        d_toks, d_lens, d_q, d_k, d_v, d_do = in_d[b]
        ns = ops.pack_num_segs(lens, w.micro_bsz, w.seq_len, w.use_packed_dataset)   # host: this step's documents
        ops.pack_tokens(d_toks, d_lens, w.micro_bsz, w.seq_len, w.use_packed_dataset, out=pk, stream=s_comp)
        ops.varlen_attn_fwd(d_q, d_k, d_v, pk["cu_seqlens"], ns, out=o, lse=lse, ws=ws_f, stream=s_comp)
        s_comp.wait_event(do_ready[b])
        ops.varlen_attn_bwd(d_q, d_k, d_v, o, d_do, lse, pk["cu_seqlens"], ns, dq=out_d[b][0], dk=out_d[b][1],
                            dv=out_d[b][2], ws=ws_b, stream=s_comp)
        comp_done[b].record(s_comp)
        with torch.cuda.stream(s_out):
            s_out.wait_event(comp_done[b])
            for dst, src in zip(out_h[b], out_d[b]):
                dst.copy_(src, non_blocking=True)
            out_read[b].record(s_out)

    del q, k, v, do
    for kk in range(2 * NB):
        step(kk)
    torch.cuda.synchronize()
    # A window long enough that one fill and one drain (the first step's copies
    # in, the last ones' copies out) weigh little per step. While the attention
    # kernels run, the copy engines move data far below their idle rate (a
    # 3.2 GB read-back took 58-228 ms instead of 17), so the drain after the
    # last step is long.
    n = max(24, args.steps)
    a, bev = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(torch.cuda.current_device()) as clk:
        time.sleep(0.5)                           # nvidia-smi has started sampling
        host_t0 = time.time()
        a.record(s_comp)
        s_in.wait_event(a)                        # no copy of the timed steps starts before `a`
        for kk in range(n):
            step(kk)
        for bb in range(NB):
            s_comp.wait_event(out_read[bb])       # every read-back has landed
        bev.record(s_comp)
        torch.cuda.synchronize()
        host_t1 = time.time()
    clocks = clk.summary(host_t0, host_t1)
    if ops.read_status(ws_b) != 0 or ops.read_status(pk["ws"]) != 0:
        raise RuntimeError("e2e status")
    ms = a.elapsed_time(bev) / n
    h2d = sum(x.numel() * x.element_size() for x in in_h)
    d2h = sum(x.numel() * x.element_size() for x in out_h[0])
    return {"value": fl["total"] / (ms * 1e-3) / 1e12, "unit": UNIT, "ms_per_step": ms,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "clocks": clocks,
            "pipeline": "%d buffer sets; copies in / compute / copies out on three streams (dO after the "
                        "forward's inputs); segment count from the host document lengths; %d steps timed from the "
                        "first copy in to the last copy out" % (NB, n)}


if __name__ == "__main__":
    sys.exit(main())
