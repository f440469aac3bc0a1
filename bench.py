"""Benchmark of paged decode attention on GB300 (one JSON line on rank 0).

Default workload: the Llama-3-8B-shaped decode (B64 Hq32 Hkv8 D128, page 64,
HND, seq_lens uniform in [1024, 8192], bf16).  A step is one decode call over
the whole batch (one launch of the decode kernel).  value = algorithmic KV
GB/s (every visible token's K and V row read once) over all ranks;
decode tokens/s = B * q_seq_len / step time.  The KV cache (1.2 GB) is larger
than L2, so no flush is needed between steps.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload 1..5]
  python bench.py --impl reference ...   (the float64 CPU oracle, bounded sample)
  python bench.py --op merge ...         (merge_attn_states on a chunked-prefill shape)
  python bench.py --op prep ...          (fused MLA decode prep on the MLA decode step)
  python bench.py --workload 3 --out-dtype e4m3   (fp8 output with the fp8 cache)

Multi-GPU: one process per GPU (torchrun); decode sequences are independent,
so every rank runs its own replica of the workload with no collective on the
data path (weak scaling); only the timing is reduced (max over ranks).
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
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from paged_kv_decode_20_gb300 import workloads as W  # noqa: E402

METRIC = "paged decode attention: KV GB/s & % of GB300 HBM peak; decode tokens/s"
FALLBACK_HBM_GBS = 6800.0
KERNEL_NAMES = {1: "gqa_decode_kernel", 2: "gqa_decode_kernel", 3: "gqa_decode_kernel",
                4: "gqa_decode_kernel", 5: "mla_decode_kernel", "large_group": "gqa_tc_kernel"}


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--workload", default="2", help="1..5 or large_group")
    ap.add_argument("--batch", type=int, default=None,
                    help="keep only the first B sequences (profiling a smaller case)")
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-read-probe", action="store_true",
                    help="skip the read-only HBM rate logged beside the copy peak")
    ap.add_argument("--op", default="decode", choices=["decode", "merge", "prep"])
    ap.add_argument("--out-dtype", default=None, choices=["e4m3"],
                    help="fp8 output (workloads with an fp8 cache)")
    ap.add_argument("--kv-dtype", default=None, choices=["e4m3"],
                    help="workload 5 with an e4m3 latent cache and query")
    ap.add_argument("--workloads", default="1,2,3,4,5,5e4m3,large_group",
                    help="named workloads also timed into the line's `workloads` object "
                         "(comma list, or 'none')")
    return ap.parse_args()


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def reduce_max(x, device=None):
    """Max of a float over all ranks (identity without torch.distributed)."""
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def tensor_peak():
    """Measured dense bf16 TFLOP/s (burst: the kernel is timed alone)."""
    try:
        d = json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))
        return float(d["bf16_tflops"]), "measured"
    except Exception:
        return 1900.0, "fallback"


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        d = json.load(open(path))
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def read_only_rate(dev, gib=4, reps=10):
    """The device's read-only HBM rate, measured now by the library's streaming
    read kernel over `gib` GiB (larger than L2), back to back between one event
    pair after 3 warm-up launches.  Context beside the copy peak: the decode
    kernels read the cache and write little, and a copy writes a byte for every
    byte it reads."""
    from paged_kv_decode_20_gb300 import xqa as X
    buf = torch.ones(gib << 28, dtype=torch.int32, device=dev)
    sink = torch.zeros(4096, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev)
    for _ in range(3):
        X.read_bandwidth_probe(buf, sink, stream)
    torch.cuda.synchronize(dev)
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for _ in range(reps):
        X.read_bandwidth_probe(buf, sink, stream)
    t1.record(stream)
    torch.cuda.synchronize(dev)
    ms = t0.elapsed_time(t1) / reps
    nbytes = buf.numel() * buf.element_size()
    del buf, sink
    torch.cuda.empty_cache()
    return {"value": round(nbytes / (ms * 1e-3) / 1e9, 1), "unit": "GB/s", "bytes": nbytes,
            "kernel": "read_stream_kernel (16-byte non-temporal loads, 4 CTAs per SM)"}


KERNEL_FILES = {
    "gqa_decode_kernel": ("gqa_kernel.cuh", "gqa_launch", "gqa_bf16.cu", "gqa_f16.cu", "gqa_e4m3.cu", "ptx.cuh",
                          "kernel_args.h", "finalize.cuh", "xqa_api.cu"),
    "gqa_tc_kernel": ("gqa_tc.cu", "umma.cuh", "ptx.cuh", "kernel_args.h", "finalize.cuh", "xqa_api.cu"),
    "mla_decode_kernel": ("mla_decode.cu", "umma.cuh", "ptx.cuh", "kernel_args.h", "finalize.cuh"),
}


def _code_only(text):
    """Source text without comments and with whitespace collapsed, so that an
    edit to comments alone keeps a kernel's hash."""
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return " ".join(text.split())


def kernel_source_hash(kernel):
    """Hash of the code (comments aside) of the source files that make up one kernel."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "paged_kv_decode_20_gb300", "csrc")
    for f in sorted(os.listdir(csrc)):
        if f.startswith(KERNEL_FILES[kernel]):
            h.update(f.encode())
            h.update(_code_only(open(os.path.join(csrc, f), encoding="utf-8").read()).encode())
    return h.hexdigest()[:16]


def recorded_traffic(workload):
    """DRAM bytes per launch from a committed ncu summary, if it was taken on
    the current kernel sources; else None.  workload: 1..5 or '5e4m3'."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        d = json.load(open(path))[str(workload)]
    except Exception:
        return None
    same = d.get("kernel_hash") == kernel_source_hash(KERNEL_NAMES[workload_key(workload)[0]])
    return d["dram_bytes_per_launch"] if same else None


class Clocks:
    """Samples SM clocks and throttle reasons with nvidia-smi while running."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except Exception:
                self.proc.kill()
                out = ""
            self.lines = [x for x in out.splitlines() if x.strip()]

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in getattr(self, "lines", []):
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


def workload_key(key):
    """'5' -> (5, None); '5e4m3' -> (5, torch.float8_e4m3fn); 'large_group' -> ('large_group', None)."""
    key = str(key)
    if key == "large_group":
        return key, None
    if key.endswith("e4m3"):
        return int(key[:-4]), torch.float8_e4m3fn
    return int(key), None


def workload_name(idx, kv_dtype=None):
    if idx == "large_group":
        return W.LARGE_GROUP
    return W.WORKLOAD_5_E4M3 if kv_dtype is not None else W.WORKLOADS[idx]


def build_case(idx, device, batch=None, kv_dtype=None):
    if idx == "large_group":
        return W.large_group_workload(device=device, poison=False, batch=batch)
    return W.workload(idx, device=device, poison=False, batch=batch, kv_dtype=kv_dtype)


L2_FLUSH_BYTES = 256 * 1024 * 1024  # twice the GB300's L2


def tensor_roofline(case, ms):
    """Tensor-pipe roofline of the MLA latent decode: Q K^T over 576 dims and
    P V over 512, 2 flops per multiply-add, per visible token and query row.
    Each contraction is priced at the peak of its own type: bf16 at the
    measured bf16 peak; an e4m3 Q K^T at twice it (the nominal fp8 : bf16
    ratio), its P V (f16 against the widened V) at the bf16 peak.  frac = the
    time both would take at those peaks / the measured time."""
    rows = case.visible_tokens() * case.q_seq_len * case.q.shape[2]
    qk, pv = rows * 2 * case.q.shape[3], rows * 2 * case.dv
    tpeak, tkind = tensor_peak()
    qk_peak = tpeak * (2.0 if case.k_cache.dtype == torch.float8_e4m3fn else 1.0)
    t_ideal = qk / (qk_peak * 1e12) + pv / (tpeak * 1e12)
    return {"bound": "tensor", "achieved": round((qk + pv) / (ms * 1e-3) / 1e12, 2),
            "peak": round((qk + pv) / t_ideal / 1e12, 1), "unit": "TFLOP/s",
            "frac": round(t_ideal / (ms * 1e-3), 4), "peak_source": tkind + " (bf16; fp8 at 2x)",
            "flops_per_launch": qk + pv}


WORKLOAD_REST_S = 1.0


def time_workload(key, dev, launches, flush):
    """Times one named workload's decode call on `dev` and returns its summary
    for the bench line's `workloads` object.

    Each workload's timed calls start after a 1 s rest.  Workloads whose KV
    exceeds L2 are timed back to back (one event pair
    around all calls; consecutive calls overlap their launch latency through
    programmatic dependent launch).  The small ones (KV inside L2) are timed
    twice: with L2 flushed before every call (a 256 MB write outside the
    event pair around each call), which is the number reported, and back to
    back."""
    from paged_kv_decode_20_gb300.runner import Decoder

    idx, kv_dtype = workload_key(key)
    case = build_case(idx, dev, kv_dtype=kv_dtype)
    dec = Decoder(case, error_word=False)
    stream = torch.cuda.current_stream(dev)
    kv, qb = case.kv_bytes(), case.q_bytes()
    small = kv <= 129e6
    for _ in range(5):
        dec.run(stream)
    torch.cuda.synchronize(dev)
    # a rest before the timed calls: the previous workload's (and the input
    # generation's) power draw must not carry over into this one's clocks
    time.sleep(WORKLOAD_REST_S)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(launches)]
    with Clocks(dev.index) as clk:
        b2b = None
        if small:
            for k in range(launches):
                flush.fill_(float(k))
                ev[k][0].record(stream)
                dec.run(stream)
                ev[k][1].record(stream)
            torch.cuda.synchronize(dev)
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0.record(stream)
        for _ in range(launches):
            dec.run(stream)
        t1.record(stream)
        torch.cuda.synchronize(dev)
        b2b = t0.elapsed_time(t1) / launches
    ms = sum(a.elapsed_time(b) for a, b in ev) / launches if small else b2b
    peak, kind = peaks()
    achieved = (kv + qb) / (ms * 1e-3) / 1e9
    out = {"workload": workload_name(idx, kv_dtype), "kernel": KERNEL_NAMES[idx],
           "ms_per_launch": round(ms, 5),
           "kernel_launches_per_call": dec.launches_per_call,
           "timing": "L2 flushed before every call" if small else "inputs larger than L2 (no flush), calls back to back",
           "kv_bytes": kv, "q_bytes": qb,
           "kv_gbs": round(kv / (ms * 1e-3) / 1e9, 2),
           "decode_tokens_per_s": round(case.batch * case.q_seq_len / (ms * 1e-3), 1),
           "roofline": {"bound": "hbm", "achieved": round(achieved, 2), "peak": peak, "unit": "GB/s",
                        "frac": round(achieved / peak, 4), "peak_source": kind}}
    if small:
        out["back_to_back_ms_per_launch"] = round(b2b, 5)
    traffic = recorded_traffic(key)
    if traffic is not None:
        out["traffic_over_algorithmic"] = round(traffic / (kv + qb), 4)
    if case.mla:
        out["roofline_tensor"] = tensor_roofline(case, ms)
    out["clocks"] = clk.summary()
    del dec, case
    torch.cuda.empty_cache()
    return out


def run_gb300(args):
    from paged_kv_decode_20_gb300 import build as B
    from paged_kv_decode_20_gb300 import xqa as X
    from paged_kv_decode_20_gb300.runner import Decoder

    world, rank, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    if rank == 0 or world == 1:
        B.build()
    if world > 1:
        dist.barrier()
    X.load()

    kv_dtype = torch.float8_e4m3fn if args.kv_dtype == "e4m3" else None
    case = build_case(args.workload, dev, args.batch, kv_dtype)
    dec = Decoder(case, error_word=False,
                  out_dtype=torch.float8_e4m3fn if args.out_dtype == "e4m3" else None)
    stream = torch.cuda.current_stream(dev)
    launches_per_call = dec.launches_per_call
    kv_bytes = case.kv_bytes()
    q_bytes = case.q_bytes()
    tokens = case.batch * case.q_seq_len
    batch = case.batch
    mla = case.mla
    dtype_name = {torch.bfloat16: "bf16", torch.float16: "f16",
                  torch.float8_e4m3fn: "e4m3 kv, bf16 q"}[case.k_cache.dtype]
    if case.q.dtype == torch.float8_e4m3fn:
        dtype_name = "e4m3 kv and q, bf16 out"

    # ---- device-resident timing: K steps back to back between one event pair
    # (an event between two calls would end the programmatic dependent launch
    # that lets a call's CTAs start while the previous call drains); a call's
    # duration is the step time.  The latent workload's call is two launches,
    # the decode and its split merge, both inside the step.
    for _ in range(args.warmup):
        dec.run(stream)
    torch.cuda.synchronize(dev)
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    with Clocks(local) as clk:
        torch.cuda.nvtx.range_push("timed")
        t0.record(stream)
        for s in range(args.steps):
            dec.run(stream)
        t1.record(stream)
        torch.cuda.synchronize(dev)
        torch.cuda.nvtx.range_pop()
    if world > 1:
        dist.barrier()
    total_ms = reduce_max(t0.elapsed_time(t1), dev)
    ms_per_step = total_ms / args.steps
    avg_launch_ms = ms_per_step
    tensor_rl = tensor_roofline(case, avg_launch_ms) if mla else None

    # ---- end to end through the C ABI with host buffers
    e2e = None
    if not args.no_e2e:
        host = {n: getattr(case, n).cpu().pin_memory() for n in
                ("q", "k_cache", "v_cache", "page_table", "seq_lens")}
        if case.mla:
            host["v_cache"] = host["k_cache"]
        out_host = torch.empty(dec.output.shape, dtype=dec.output.dtype).pin_memory()
        names = ["q", "k_cache", "page_table", "seq_lens"] + ([] if case.mla else ["v_cache"])
        h2d = sum(host[n].numel() * host[n].element_size() for n in names)
        d2h = out_host.numel() * out_host.element_size()

        def e2e_step():
            for n in names:
                getattr(case, n).copy_(host[n], non_blocking=True)
            dec.run(stream)
            out_host.copy_(dec.output, non_blocking=True)

        for _ in range(max(1, args.warmup // 2)):
            e2e_step()
        torch.cuda.synchronize(dev)
        if world > 1:
            dist.barrier()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e_steps = max(3, args.steps // 4)
        e0.record(stream)
        for _ in range(e_steps):
            e2e_step()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        e_ms = reduce_max(e0.elapsed_time(e1) / e_steps, dev)
        e2e = {"value": round(kv_bytes * world / (e_ms * 1e-3) / 1e9, 2), "unit": "GB/s",
               "ms_per_step": round(e_ms, 4), "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h}

    # ---- CPU baseline: the oracle on this workload, on all host threads and
    # on one (rank 0)
    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        cpu_case = case.to("cpu")
        cpu = cpu_baseline(cpu_case, args.workload, min_seconds=6.0)
        one = cpu_baseline(cpu_case, args.workload, max_rows=64, min_seconds=3.0, threads=1)
        cpu["single_thread"] = {k: one[k] for k in ("value", "unit", "cores", "sample", "seconds")}

    # ---- every named workload, one after another (rank 0 reports them)
    per_workload = None
    if rank == 0 and args.workloads != "none" and args.batch is None:
        del dec, case
        torch.cuda.empty_cache()
        flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
        per_workload = {}
        for key in args.workloads.split(","):
            per_workload[key] = time_workload(key, dev, max(args.steps, 20), flush)
        del flush

    if world > 1:
        dist.barrier()
    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return
    read_only = None
    if not args.no_read_probe:
        if per_workload is None:
            del dec, case
            torch.cuda.empty_cache()
        read_only = read_only_rate(dev)
    peak, peak_kind = peaks()
    achieved = (kv_bytes + q_bytes) / (avg_launch_ms * 1e-3) / 1e9
    value = kv_bytes * world / (ms_per_step * 1e-3) / 1e9
    line = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_per_step, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": dtype_name,
        "data": "synthetic (seeded N(0,1) q/K/V, shuffled page pool)",
        "config": {"workload": workload_name(args.workload, kv_dtype) + (", fp8 output" if args.out_dtype else ""),
                   "global_batch": batch * world,
                   "kv_bytes_per_step": kv_bytes * world, "q_bytes_per_step": q_bytes * world,
                   "l2": "inputs larger than L2 (no flush)" if kv_bytes > 129e6
                   else "KV fits in L2: numbers are L2-assisted",
                   "parallelism": f"replicas x{world} (no collective)"},
        "decode_tokens_per_s": round(tokens * world / (ms_per_step * 1e-3), 1),
        "pct_hbm_peak": round(100 * achieved / peak, 2),
        "roofline": {"bound": "hbm", "achieved": round(achieved, 2), "peak": peak,
                     "unit": "GB/s", "frac": round(achieved / peak, 4),
                     "peak_source": peak_kind,
                     "traffic": recorded_traffic(f"{args.workload}e4m3" if kv_dtype is not None
                                                 else args.workload),
                     "kernel": KERNEL_NAMES[args.workload],
                     "algorithmic_bytes_per_launch": kv_bytes + q_bytes,
                     "avg_launch_ms": round(avg_launch_ms, 5)},
        "read_only_gbs": read_only,
        "gpu_launches": args.steps * launches_per_call,
        "e2e": e2e,
        "cpu_baseline": cpu,
        "clocks": clk.summary(),
    }
    if per_workload is not None:
        line["workloads"] = per_workload
    if mla:
        # the latent workload sits near the ridge: report the tensor pipe too
        line["roofline_tensor"] = tensor_rl
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def cpu_baseline(case, idx, max_rows=None, min_seconds=10.0, threads=None):
    """Time the float64 oracle on all rows of the workload (or a bounded
    sample of whole (b, kv head) units) with every host thread (or `threads`)."""
    import oracle
    B, qs, Hq, _ = case.q.shape
    G = Hq // case.num_kv_heads
    threads = threads or os.cpu_count() or 1
    units = None
    frac = 1.0
    rows = B * qs * Hq
    budget_rows = max_rows if max_rows is not None else {1: rows, 2: rows, 3: 256, 4: rows, 5: 128,
                                                         "large_group": 512}[idx]
    if budget_rows < rows:
        # whole (b, kvh) units, spread over the batch
        per_unit = qs * G
        n_units = max(1, budget_rows // per_unit)
        sel = torch.linspace(0, B * case.num_kv_heads - 1, n_units).round().long().unique()
        ids = []
        for u in sel.tolist():
            b, kvh = divmod(u, case.num_kv_heads)
            for i in range(qs):
                for g in range(G):
                    ids.append((b * qs + i) * Hq + kvh * G + g)
        units = torch.tensor(ids, dtype=torch.int64)
        lens = case.seq_lens.to(torch.int64)
        if case.sliding_win_size > 0:
            lens = lens.clamp(max=case.sliding_win_size + qs - 1)
        per_b = lens.to(torch.float64)
        frac = float(sum(per_b[u // case.num_kv_heads] for u in sel.tolist()) /
                     (per_b.sum() * case.num_kv_heads))
        sample = f"{len(sel)} of {B * case.num_kv_heads} (sequence, kv head) units, all their rows"
    else:
        sample = f"all {rows} output rows of the workload"
    kw = case.kwargs()
    reps = 0
    t = time.perf_counter()
    while True:
        oracle.xqa_attention(case.q, case.k_cache, case.v_cache, case.page_table, case.seq_lens,
                             units=units, threads=threads, **kw)
        reps += 1
        if time.perf_counter() - t >= min_seconds or reps >= 500:
            break
    dt = (time.perf_counter() - t) / reps
    sample += f" (mean of {reps} repetitions)"
    kv = case.kv_bytes() * frac
    return {"value": round(kv / dt / 1e9, 4), "unit": "GB/s", "cores": threads, "kind": "oracle",
            "sample": sample, "seconds": round(dt, 3)}


def run_reference(args):
    """The reference arm: the float64 CPU oracle as it stands, each step a
    bounded sample of the workload, on the host cores of rank 0."""
    world, rank, _ = dist_env()
    if rank != 0:
        return
    case = build_case(args.workload, "cpu", args.batch)
    B = case.batch
    # each step: a few whole (sequence, kv head) units
    rows_per_step = {1: 16, 2: 32, 3: 8, 4: 64, 5: 128, "large_group": 64}[args.workload]
    for _ in range(args.warmup):
        cpu_baseline(case, args.workload, max_rows=rows_per_step, min_seconds=0.0)
    times, vals = [], []
    t0 = time.perf_counter()
    for _ in range(args.steps):
        r = cpu_baseline(case, args.workload, max_rows=rows_per_step, min_seconds=0.0)
        times.append(r["seconds"])
        vals.append(r["value"])
    total = time.perf_counter() - t0
    value = statistics.median(vals)
    line = {
        "impl": "reference",
        "metric": METRIC,
        "value": value,
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(1e3 * total / args.steps, 3),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64",
        "data": "synthetic (seeded N(0,1) q/K/V, shuffled page pool)",
        "config": {"workload": workload_name(args.workload), "global_batch": B,
                   "parallelism": "CPU oracle, rank 0 only"},
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": os.cpu_count(),
                         "kind": "oracle", "sample": r["sample"] + " per step"},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)


# merge_attn_states on the shape of Kimi-K3's prefill with chunked context (vLLM
# MultiHeadLatentAttention page): 8192 new tokens, 128 heads, v_head_dim 128.
MERGE_SHAPE = (8192, 128, 128)
MERGE_METRIC = "merge_attn_states: GB/s moved (two results + lse in, one out) & % of HBM peak"


def merge_inputs(device, T, H, D):
    g = torch.Generator(device="cpu").manual_seed(12)
    po = torch.randn((T, H, D), generator=g).to(torch.bfloat16)
    so = torch.randn((T, H, D), generator=g).to(torch.bfloat16)
    pl = torch.randn((T, H), generator=g) * 3
    sl = torch.randn((T, H), generator=g) * 3
    return [x.to(device) for x in (po, pl, so, sl)]


def run_merge(args):
    """One step = one merge_attn_states call over MERGE_SHAPE (bf16)."""
    T, H, D = MERGE_SHAPE
    moved = 3 * T * H * D * 2 + 3 * T * H * 4
    cfg = {"workload": f"merge_attn_states T{T} H{H} D{D} bf16 (chunked-context prefill)",
           "global_batch": T, "bytes_per_step": moved,
           "l2": "inputs larger than L2 (no flush)", "parallelism": "replicas x1 (no collective)"}
    world, rank, local = dist_env()
    if rank != 0:
        return
    if args.impl == "reference":
        import oracle
        n = 64  # tokens per sample
        po, pl, so, sl = [x[:n].to(torch.float64) for x in merge_inputs("cpu", T, H, D)]
        for _ in range(args.warmup):
            oracle.merge_attn_states(po, pl, so, sl)
        t = time.perf_counter()
        for _ in range(args.steps):
            oracle.merge_attn_states(po, pl, so, sl)
        dt = (time.perf_counter() - t) / args.steps * (T / n)  # scaled to a full step
        v = moved / dt / 1e9
        print(json.dumps({"metric": MERGE_METRIC, "value": round(v, 3), "unit": "GB/s", "n_gpus": world,
                          "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt * 1e3, 3),
                          "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
                          "dtype": "f64", "data": "synthetic (seeded N(0,1))", "config": cfg,
                          "impl": "reference",
                          "cpu_baseline": {"value": round(v, 3), "unit": "GB/s", "cores": 1,
                                           "kind": "oracle", "sample": f"{n} of {T} tokens per step"},
                          "e2e": {"value": round(v, 3), "unit": "GB/s", "h2d_bytes_per_step": 0,
                                  "d2h_bytes_per_step": 0}}), flush=True)
        return
    from paged_kv_decode_20_gb300 import build as B
    from paged_kv_decode_20_gb300 import xqa as X
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    B.build()
    po, pl, so, sl = merge_inputs(dev, T, H, D)
    out = torch.empty_like(so)
    out_lse = torch.empty_like(sl)
    stream = torch.cuda.current_stream(dev)

    def step():
        X.merge_attn_states(out, po, pl, so, sl, output_lse=out_lse, stream=stream)

    for _ in range(args.warmup):
        step()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize(dev)
    with Clocks(local) as clk:
        t0.record(stream)
        for s_ in range(args.steps):
            ev[s_][0].record(stream)
            step()
            ev[s_][1].record(stream)
        t1.record(stream)
        torch.cuda.synchronize(dev)
    ms = t0.elapsed_time(t1) / args.steps
    launch = sum(a.elapsed_time(b) for a, b in ev) / args.steps
    # end to end: inputs from pinned host memory, result and lse back
    hosts = [x.cpu().pin_memory() for x in (po, pl, so, sl)]
    oh, lh = torch.empty(out.shape, dtype=out.dtype).pin_memory(), torch.empty(sl.shape).pin_memory()

    def e2e_step():
        for d_, h_ in zip((po, pl, so, sl), hosts):
            d_.copy_(h_, non_blocking=True)
        step()
        oh.copy_(out, non_blocking=True)
        lh.copy_(out_lse, non_blocking=True)

    e2e_step()
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ne = max(3, args.steps // 10)
    e0.record(stream)
    for _ in range(ne):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    e_ms = e0.elapsed_time(e1) / ne
    peak, kind = peaks()
    achieved = moved / (launch * 1e-3) / 1e9
    print(json.dumps({
        "metric": MERGE_METRIC, "value": round(moved / (ms * 1e-3) / 1e9, 2), "unit": "GB/s",
        "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,1))", "config": cfg,
        "roofline": {"bound": "hbm", "achieved": round(achieved, 2), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "peak_source": kind, "traffic": None,
                     "kernel": "merge_kernel", "algorithmic_bytes_per_launch": moved,
                     "avg_launch_ms": round(launch, 5)},
        "gpu_launches": args.steps,
        "e2e": {"value": round(moved / (e_ms * 1e-3) / 1e9, 2), "unit": "GB/s", "ms_per_step": round(e_ms, 4),
                "h2d_bytes_per_step": sum(h.numel() * h.element_size() for h in hosts),
                "d2h_bytes_per_step": oh.numel() * 2 + lh.numel() * 4},
        "cpu_baseline": None, "clocks": clk.summary()}), flush=True)


# the fused MLA decode prep on the MLA latent workload's decode step: 64 tokens,
# 128 heads, kv_lora_rank 512, rope 64 (Kimi-K3 MultiHeadLatentAttention page)
PREP_SHAPE = (64, 128, 512, 64)
PREP_METRIC = "MLA decode prep (q concat + RoPE + latent cache insert): GB/s moved & % of HBM peak"


def run_prep(args):
    """One step = one xqa_mla_decode_prep call; L2 is flushed (a 256 MB write)
    before every timed launch because the step's bytes fit in L2."""
    T, H, Lr, R = PREP_SHAPE
    moved = 2 * T * H * (Lr + R) * 2 + 2 * T * (Lr + R) * 2 + T * 16 + T * R * 4
    cfg = {"workload": f"MLA decode prep T{T} H{H} latent {Lr} rope {R} bf16",
           "global_batch": T, "bytes_per_step": moved, "l2": "flushed before every launch (256 MB write)",
           "parallelism": "replicas x1 (no collective)"}
    world, rank, local = dist_env()
    if rank != 0:
        return
    g = torch.Generator().manual_seed(13)
    P = 32768
    inv = 10000.0 ** (-torch.arange(0, R, 2, dtype=torch.float64) / R)
    ang = torch.arange(P, dtype=torch.float64)[:, None] * inv[None, :]
    cs = torch.cat([ang.cos(), ang.sin()], dim=1).to(torch.float32)
    ql = torch.randn(T, H, Lr, generator=g).to(torch.bfloat16)
    qp = torch.randn(T, H, R, generator=g).to(torch.bfloat16)
    kc = torch.randn(T, Lr, generator=g).to(torch.bfloat16)
    kp = torch.randn(T, R, generator=g).to(torch.bfloat16)
    pos = torch.randint(0, P, (T,), generator=g)
    slots = torch.randperm(64 * 512, generator=g)[:T]
    if args.impl == "reference":
        import oracle
        cache = torch.zeros(64 * 512, Lr + R, dtype=torch.bfloat16)
        t0 = time.perf_counter()
        n = max(1, args.steps)
        for _ in range(n):
            oracle.mla_decode_prep(ql, qp, kc, kp, pos, cs, slots, cache)
        dt = (time.perf_counter() - t0) / n
        v = moved / dt / 1e9
        print(json.dumps({"metric": PREP_METRIC, "value": round(v, 4), "unit": "GB/s", "n_gpus": world,
                          "steps": n, "warmup": args.warmup, "ms_per_step": round(dt * 1e3, 3),
                          "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
                          "data": "synthetic (seeded N(0,1))", "config": cfg, "impl": "reference",
                          "cpu_baseline": {"value": round(v, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
                                           "sample": "the whole step"},
                          "e2e": {"value": round(v, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                                  "d2h_bytes_per_step": 0}}), flush=True)
        return
    from paged_kv_decode_20_gb300 import build as B
    from paged_kv_decode_20_gb300 import xqa as X
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    B.build()
    d = [x.to(dev) for x in (ql, qp, kc, kp, pos, cs, slots)]
    cache = torch.zeros(64, 512, 1, Lr + R, dtype=torch.bfloat16, device=dev)
    q_out = torch.empty(T, H, Lr + R, dtype=torch.bfloat16, device=dev)
    flush = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        X.mla_decode_prep(d[0], d[1], d[2], d[3], d[4], d[5], d[6], cache, q_out=q_out, stream=stream)

    for _ in range(args.warmup):
        step()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    torch.cuda.synchronize(dev)
    with Clocks(local) as clk:
        for s_ in range(args.steps):
            flush.fill_(float(s_))
            ev[s_][0].record(stream)
            step()
            ev[s_][1].record(stream)
        torch.cuda.synchronize(dev)
    launch = sum(a.elapsed_time(b) for a, b in ev) / args.steps
    hosts = [x.cpu().pin_memory() for x in d]
    qh = torch.empty(q_out.shape, dtype=q_out.dtype).pin_memory()

    def e2e_step():
        for dd, hh in zip(d, hosts):
            dd.copy_(hh, non_blocking=True)
        step()
        qh.copy_(q_out, non_blocking=True)

    e2e_step()
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ne = max(3, args.steps // 10)
    e0.record(stream)
    for _ in range(ne):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    e_ms = e0.elapsed_time(e1) / ne
    peak, kind = peaks()
    achieved = moved / (launch * 1e-3) / 1e9
    print(json.dumps({
        "metric": PREP_METRIC, "value": round(achieved, 2), "unit": "GB/s", "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(launch, 5), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded N(0,1))", "config": cfg,
        "roofline": {"bound": "hbm", "achieved": round(achieved, 2), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "peak_source": kind, "traffic": None,
                     "kernel": "prep_kernel", "algorithmic_bytes_per_launch": moved,
                     "avg_launch_ms": round(launch, 5)},
        "gpu_launches": args.steps,
        "e2e": {"value": round(moved / (e_ms * 1e-3) / 1e9, 2), "unit": "GB/s", "ms_per_step": round(e_ms, 4),
                "h2d_bytes_per_step": sum(h.numel() * h.element_size() for h in hosts),
                "d2h_bytes_per_step": qh.numel() * 2},
        "cpu_baseline": None, "clocks": clk.summary()}), flush=True)


def main():
    args = parse()
    args.workload = int(args.workload) if str(args.workload).isdigit() else args.workload
    if args.op == "merge":
        run_merge(args)
    elif args.op == "prep":
        run_prep(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_gb300(args)


if __name__ == "__main__":
    main()
