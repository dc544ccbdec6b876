"""Benchmark of the NVFP4 sparse-MLA decode path on one GB300.

Workload (default): the pages' decode point -- 15 query tokens of one
sequence, 64 heads, 200K-token context in 64-token pages behind a shuffled
block table, top-2048 distinct uniform positions per token, NVFP4 cache
(352-byte rows). One step is one pass of the whole path: nvfp4_mla_pack of
the step's 15 new tokens into fresh slots, then sparse_mla_decode of the 15
query tokens. L2 (126 MB) is flushed before every step by writing a 256 MiB
buffer. The metric is the decode call's device time (CUDA events on the
launching stream), in microseconds per call.

Printed: one JSON line (rank 0). `--impl reference` times the CPU oracle on
the same workload instead (the reference arm of this build).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "sparse-MLA NVFP4 decode µs/call & % roofline (15 q-tok × top-2048, 1 GB300)"
UNIT = "us/call"
FLUSH_BYTES = 256 << 20
GROUP = 16                       # steps enqueued behind one GPU sleep
LEAD_CYCLES_PER_STEP = 400_000   # ~0.2 ms of sleep per queued step
PEAKS_FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
WORKLOAD_DESC = ("decode_point: 15 query tokens (1 sequence) x top-2048 distinct uniform positions, 64 heads, "
                 "200K-token context, 64-token pages, NVFP4 latent 512 + FP8 RoPE 64 (352 B/row)")


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--kernel", default="auto", choices=["auto", "mma", "tcgen05"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--no-staged", action="store_true")
    ap.add_argument("--no-layered", action="store_true")
    ap.add_argument("--no-topk", action="store_true")
    ap.add_argument("--no-fp8", action="store_true")
    ap.add_argument("--no-configs", action="store_true")
    return ap.parse_args()


def max_over_ranks(values, world, device):
    """The element-wise maximum of `values` (floats) over the job's ranks (a
    no-op for one rank). Replicas exchange nothing but this and barriers."""
    if world <= 1:
        return [float(v) for v in values]
    import torch
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return [float(v) for v in t.tolist()]


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(PEAKS_FALLBACK), "fallback"


def algorithmic(w):
    """Algorithmic bytes and flops of one decode call: per valid slot one
    352-byte row and 64 heads x (2*576 + 2*512) flops; plus the queries,
    index lists, block table entries read, outputs and lse."""
    valid = int((w.topk_idx >= 0).sum())
    T, H, K = w.T, w.H, w.topk
    rows = valid * 352
    q = T * H * 576 * 2
    idx = T * K * 4
    bt = int(w.block_table.numel()) * 4
    out = T * H * 512 * 2 + T * H * 4
    flops = valid * H * (2 * 576 + 2 * 512)
    return {"bytes": rows + q + idx + bt + out, "row_bytes": rows, "flops": flops, "valid_slots": valid}


def graph_us(fn, reps=5):
    """Median device time of one replay of a CUDA graph that runs `fn` (which
    enqueues on the current stream), in microseconds."""
    import torch
    g = torch.cuda.CUDAGraph()
    cap = torch.cuda.Stream()
    cap.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(cap):
        fn()  # warm-up outside the capture (library set-up, allocator)
    torch.cuda.current_stream().wait_stream(cap)
    torch.cuda.synchronize()
    with torch.cuda.graph(g):
        fn()
    g.replay()
    torch.cuda.synchronize()
    ts = []
    for _ in range(reps):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        g.replay()
        b.record()
        b.synchronize()
        ts.append(a.elapsed_time(b) * 1e3)
    del g
    return statistics.median(ts)


def kernel_only_us(call, flush, n=20):
    """Device time of `call` alone: a CUDA graph of n x (L2 flush, call) less
    a graph of the n flushes, per call (cold L2); and a graph of n calls back
    to back, per call (warm L2). Graph replay keeps the host's launch latency
    out of both."""
    def flushed():
        for k in range(n):
            flush.fill_(float(k))
            call()

    def flushes():
        for k in range(n):
            flush.fill_(float(k))

    def warm():
        for _ in range(n):
            call()

    cold = (graph_us(flushed) - graph_us(flushes)) / n
    return {"cold_l2_us": cold, "warm_l2_us": graph_us(warm) / n, "calls_per_graph": n,
            "how": "CUDA graph of n x (256 MiB L2 flush, call) minus a graph of the n flushes, per call; "
                   "warm: a graph of n calls back to back, per call"}


def event_us(call, flush, steps, before=None):
    """Mean event time of `call` per step, L2 flushed before every step, steps
    queued behind a GPU sleep so that the events bracket device work only."""
    import torch
    evs = []
    for k in range(steps):
        if k % GROUP == 0:
            torch.cuda._sleep(LEAD_CYCLES_PER_STEP * min(GROUP, steps - k))
        flush.fill_(float(k))
        if before is not None:
            before()
        e = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
        e[0].record()
        call()
        e[1].record()
        evs.append(e)
    torch.cuda.synchronize()
    return statistics.mean([e[0].elapsed_time(e[1]) for e in evs]) * 1e3


def roofline_of(alg, us, pk):
    """Achieved rate of one call against the bound that limits it."""
    bw, tf = pk["hbm_gbs"], pk["bf16_tflops"]
    t_bytes = alg["bytes"] / (bw * 1e9) * 1e6
    t_flops = alg["flops"] / (tf * 1e12) * 1e6
    if t_flops >= t_bytes:
        ach = alg["flops"] / (us * 1e-6) / 1e12
        return {"bound": "tensor", "achieved": ach, "peak": tf, "unit": "TFLOP/s", "frac": ach / tf,
                "roofline_us": t_flops}
    ach = alg["bytes"] / (us * 1e-6) / 1e9
    return {"bound": "hbm", "achieved": ach, "peak": bw, "unit": "GB/s", "frac": ach / bw, "roofline_us": t_bytes}


class ClockSampler:
    """nvidia-smi clock and throttle-reason samples (every 20 ms) taken in the
    background; stop() keeps the samples that fall inside a wall-clock window
    around the timed region."""

    NAMES = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]

    def __init__(self, gpu_index: int):
        self.proc = None
        self.path = os.path.join(tempfile.gettempdir(), f"nvmla_clocks_{os.getpid()}.csv")
        q = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(gpu_index), f"--query-gpu={q}",
                                          "--format=csv,noheader,nounits", "-lms", "20"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    @staticmethod
    def _ts(text):
        import datetime
        for fmt in ("%Y/%m/%d %H:%M:%S.%f", "%Y/%m/%d %H:%M:%S"):
            try:
                return datetime.datetime.strptime(text.strip(), fmt).timestamp()
            except ValueError:
                pass
        return None

    def stop(self, t0: float, t1: float, pad: float = 0.05):
        if self.proc is None:
            return None
        time.sleep(0.1)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        rows = []
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 10:
                continue
            try:
                rows.append((self._ts(parts[0]), float(parts[2]), float(parts[3]), float(parts[4]), parts[6:10]))
            except ValueError:
                continue
        if not rows:
            return None
        inside = [r for r in rows if r[0] is not None and t0 - pad <= r[0] <= t1 + pad]
        window = "timed region +-50 ms"
        if not inside:
            inside = sorted(rows, key=lambda r: abs((r[0] or t0) - (t0 + t1) / 2))[:3]
            window = "3 samples nearest the timed region"
        reasons = sorted({n for r in inside for n, v in zip(self.NAMES, r[4]) if v.lower().startswith("active")})
        return {"sm_mhz": statistics.median(r[1] for r in inside), "sm_max_mhz": max(r[2] for r in inside),
                "power_w_max": max(r[3] for r in inside), "samples": len(inside), "window": window,
                "reasons": reasons}


def strip_comments(src):
    """C/C++/CUDA source without its comments and blank lines, trailing spaces
    removed: what a comment-only edit leaves unchanged."""
    out, i, n = [], 0, len(src)
    while i < n:
        c = src[i]
        if c == '"' or c == "'":  # a literal: copied through, escapes included
            j = i + 1
            while j < n and src[j] != c:
                j += 2 if src[j] == "\\" else 1
            out.append(src[i:j + 1])
            i = j + 1
        elif src.startswith("//", i):
            j = src.find("\n", i)
            i = n if j < 0 else j
        elif src.startswith("/*", i):
            j = src.find("*/", i + 2)
            i = n if j < 0 else j + 2
            out.append(" ")
        else:
            out.append(c)
            i += 1
    lines = ("".join(out)).split("\n")
    return "\n".join(l.rstrip() for l in lines if l.strip())


def source_hash(names):
    """Hash of a kernel's source files, comments left out: the traffic record
    stays valid across comment-only edits and lapses on any code change."""
    h = hashlib.sha256()
    for n in names:
        with open(os.path.join(ROOT, "nvfp4_sparse_mla_gb300", "csrc", n), encoding="utf-8") as f:
            h.update(strip_comments(f.read()).encode("utf-8"))
    return h.hexdigest()[:16]


KERNEL_FILES = {"decode_tc_kernel": ["decode_tc.cu", "decode_tc_layout.h", "format.h", "common.cuh"],
                "decode_mma_kernel": ["decode_mma.cu", "format.h", "common.cuh"]}


def traffic_record(kernel):
    """DRAM bytes per launch of `kernel` on this workload from the committed
    ncu summary (profiles/traffic.json), or None when the kernel's source
    changed since the counters were taken."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    rec = d.get(kernel)
    if not rec or rec.get("source_hash") != source_hash(KERNEL_FILES[kernel]):
        return None
    return rec.get("dram_bytes_per_launch")


def cpu_baseline(w, seconds: float):
    """The oracle, as it stands, on the host cores: whole decode calls of the
    same workload, repeated until `seconds` have elapsed (at least one)."""
    import numpy as np
    from oracle import attention as oatt
    from oracle import pack as opack

    lat, rope, slots = w.all_written()
    cache = np.zeros((w.num_pages + 1, 64, 352), dtype=np.uint8)
    opack.pack_into_cache(lat.double().numpy(), rope.double().numpy(), slots.numpy(), cache)
    n, t0 = 0, time.perf_counter()
    while True:
        oatt.sparse_mla_decode(w.q_latent, w.q_rope, cache, w.block_table, w.topk_idx, w.sm_scale,
                               w.q_seq_idx, w.seq_lens)
        n += 1
        el = time.perf_counter() - t0
        if el >= seconds:
            break
    threads = blas_threads()
    res = {"value": el / n * 1e6, "unit": UNIT, "cores": threads, "kind": "oracle",
           "sample": f"{n} whole decode calls of the workload (15 tokens x 2048 slots each), "
                     f"numpy float64 with a {threads}-thread BLAS on {os.cpu_count()} host cores"}
    # the same oracle on one host thread: a child process whose BLAS is held
    # to one thread from the start
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1")
    code = ("import sys, time; sys.path.insert(0, %r); import numpy as np; "
            "from nvfp4_sparse_mla_gb300 import workloads; from oracle import attention as oatt; "
            "from oracle import pack as opack; w = workloads.decode_point(); lat, rope, slots = w.all_written(); "
            "cache = np.zeros((w.num_pages + 1, 64, 352), dtype=np.uint8); "
            "opack.pack_into_cache(lat.double().numpy(), rope.double().numpy(), slots.numpy(), cache); "
            "n, t0 = 0, time.perf_counter()\n"
            "while True:\n"
            "    oatt.sparse_mla_decode(w.q_latent, w.q_rope, cache, w.block_table, w.topk_idx, w.sm_scale, "
            "w.q_seq_idx, w.seq_lens); n += 1; el = time.perf_counter() - t0\n"
            "    if el >= %f: break\n"
            "print(n, el / n * 1e6)") % (ROOT, seconds / 2)
    try:
        r = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True, timeout=300)
        n1, us1 = r.stdout.split()
        res["one_thread"] = {"value": float(us1), "unit": UNIT, "cores": 1,
                             "sample": f"{n1} whole decode calls in a child process with a one-thread BLAS"}
    except Exception as e:  # the all-cores figure stands on its own
        res["one_thread"] = {"error": str(e)[:200]}
    return res


def blas_threads():
    for var in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
        if os.environ.get(var):
            try:
                return int(os.environ[var])
            except ValueError:
                pass
    try:
        import threadpoolctl
        info = threadpoolctl.threadpool_info()
        if info:
            return max(int(i.get("num_threads", 1)) for i in info)
    except Exception:
        pass
    return os.cpu_count() or 1


def run_reference(args, rank, world):
    """Reference arm: the CPU oracle timed on this machine's host cores."""
    if rank != 0:
        return
    from nvfp4_sparse_mla_gb300 import workloads
    import numpy as np
    from oracle import attention as oatt
    from oracle import pack as opack
    w = workloads.decode_point()
    lat, rope, slots = w.all_written()
    cache = np.zeros((w.num_pages + 1, 64, 352), dtype=np.uint8)
    opack.pack_into_cache(lat.double().numpy(), rope.double().numpy(), slots.numpy(), cache)
    call = lambda: oatt.sparse_mla_decode(w.q_latent, w.q_rope, cache, w.block_table, w.topk_idx, w.sm_scale,
                                          w.q_seq_idx, w.seq_lens)
    for _ in range(args.warmup):
        call()
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        call()
        times.append(time.perf_counter() - t0)
    v = statistics.mean(times) * 1e6
    threads = blas_threads()
    line = {
        "impl": "reference", "metric": METRIC, "value": v, "unit": UNIT, "n_gpus": args.gpus, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": v / 1e3, "higher_is_better": False, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOAD_DESC, "T": w.T, "H": w.H, "topk": w.topk, "ctx": int(w.seq_lens[0]),
                   "l2": "n/a (CPU)"},
        "cpu_baseline": {"value": v, "unit": UNIT, "cores": threads, "kind": "oracle",
                         "sample": f"each step one whole decode call (15 tokens x 2048 slots), numpy float64, "
                                   f"{threads}-thread BLAS on {os.cpu_count()} host cores"},
        "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)


def config_line(name, args, flush, dev, pk, impl):
    """One of the baseline's other workloads on the GPU: the decode call's
    event time (L2 flushed before every call), its kernel-only times and its
    roofline from the workload's actual valid slots; for write+read also the
    pack of the 6,144-token chunk, the whole step (pack, then decode) and the
    staged dequant-to-FP8 path timed the same way."""
    import torch
    import nvfp4_sparse_mla_gb300 as nvmla
    from nvfp4_sparse_mla_gb300 import workloads
    w = workloads.make(name)
    alg = algorithmic(w)
    cache = torch.zeros((w.num_pages, 64, 352), dtype=torch.uint8, device=dev)
    nvmla.nvfp4_mla_pack(w.hist_latent.to(dev), w.hist_rope.to(dev), w.hist_slots.to(dev), cache)
    nl, nr, ns = w.new_latent.to(dev), w.new_rope.to(dev), w.new_slots.to(dev)
    if ns.numel():
        nvmla.nvfp4_mla_pack(nl, nr, ns, cache)
    ql, qr = w.q_latent.to(dev), w.q_rope.to(dev)
    bt, tk = w.block_table.to(dev), w.topk_idx.to(dev)
    qs, sl = w.q_seq_idx.to(dev), w.seq_lens.to(dev)
    out = torch.empty((w.T, w.H, 512), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((w.T, w.H), dtype=torch.float32, device=dev)
    ws_n = nvmla.sparse_mla_decode_workspace_size(w.T, w.H, w.topk, impl=impl)
    ws = torch.empty(max(ws_n, 16), dtype=torch.uint8, device=dev)

    def decode():
        nvmla.sparse_mla_decode(ql, qr, cache, bt, tk, w.sm_scale, out=out, lse=lse, q_seq_idx=qs, seq_lens=sl,
                                workspace=ws, impl=impl)

    for _ in range(3):
        flush.fill_(1.0)
        decode()
    torch.cuda.synchronize()
    steps = max(20, args.steps // 4)
    us = event_us(decode, flush, steps)
    ko = kernel_only_us(decode, flush)
    line = {"workload": workloads.describe(w), "decode_us": us, "decode_kernel_only": ko,
            "splits": nvmla.sparse_mla_decode_splits(w.T, w.H, w.topk, impl=impl),
            "algorithmic_bytes": alg["bytes"], "algorithmic_flops": alg["flops"],
            "roofline": roofline_of(alg, us, pk), "roofline_kernel": roofline_of(alg, ko["cold_l2_us"], pk)}
    if name == "write_read":
        def pack():
            nvmla.nvfp4_mla_pack(nl, nr, ns, cache)

        def step():
            pack()
            decode()

        line["pack_us"] = event_us(pack, flush, steps)
        line["step_us"] = event_us(step, flush, steps)
        line["pack_tokens"] = int(ns.numel())
        # the staged baseline over the same rows: dequantise to 576-byte FP8
        # rows in GPU memory, then attend over them on the tcgen05 kernel (the
        # buffer read as a paged FP8 cache, one block-table row per token)
        buf = torch.empty((w.T, w.topk, 576), dtype=torch.uint8, device=dev)
        ridx = torch.empty((w.T, w.topk), dtype=torch.int32, device=dev)
        ppt = w.topk // 64
        sbt = torch.arange(w.T * ppt, dtype=torch.int32, device=dev).view(w.T, ppt)
        sqs = torch.arange(w.T, dtype=torch.int32, device=dev)
        sview = buf.view(w.T * ppt, 64, 576)
        fo, fl = torch.empty_like(out), torch.empty_like(lse)
        ws2 = torch.empty(max(nvmla.sparse_mla_decode_workspace_size(w.T, w.H, w.topk), 16), dtype=torch.uint8,
                          device=dev)

        def dequant():
            nvmla.nvfp4_stage_dequant_fp8(cache, bt, tk, qs, sl, fp8_rows=buf, row_idx=ridx)

        def attend():
            nvmla.sparse_mla_decode_fp8cache(ql, qr, sview, sbt, ridx, w.sm_scale, out=fo, lse=fl, q_seq_idx=sqs,
                                             workspace=ws2)

        def staged_step():
            pack()
            dequant()
            attend()

        dequant()
        attend()
        torch.cuda.synchronize()
        st = {"dequant_us": event_us(dequant, flush, steps), "attend_us": event_us(attend, flush, steps, before=dequant),
              "step_us": event_us(staged_step, flush, steps), "fp8_buffer_bytes": int(buf.numel())}
        st["us_per_call"] = st["dequant_us"] + st["attend_us"]
        line["staged"] = st
        del buf, ridx
    del cache
    return line


def main():
    args = parse()
    rank, world, local = dist_env()
    if args.impl == "reference":
        return run_reference(args, rank, world)

    import numpy as np
    import torch
    import nvfp4_sparse_mla_gb300 as nvmla
    from nvfp4_sparse_mla_gb300 import workloads

    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    nvmla.load()
    impl = {"auto": None, "mma": nvmla.IMPL_MMA, "tcgen05": nvmla.IMPL_TCGEN05}[args.kernel]

    # ---------------- workload resident in HBM (replica per rank)
    w = workloads.decode_point()
    alg = algorithmic(w)
    new_pages = 1
    cache = torch.zeros((w.num_pages + new_pages, 64, 352), dtype=torch.uint8, device=dev)
    lat, rope, slots = w.all_written()
    nvmla.nvfp4_mla_pack(lat.to(dev), rope.to(dev), slots.to(dev), cache)
    g = torch.Generator().manual_seed(77)
    new_lat = torch.randn((w.T, 512), generator=g).to(torch.bfloat16)
    new_rope = torch.randn((w.T, 64), generator=g).to(torch.bfloat16)
    new_slots = torch.arange(w.num_pages * 64, w.num_pages * 64 + w.T, dtype=torch.int32)
    d_new_lat, d_new_rope, d_new_slots = new_lat.to(dev), new_rope.to(dev), new_slots.to(dev)
    ql, qr = w.q_latent.to(dev), w.q_rope.to(dev)
    bt, tk = w.block_table.to(dev), w.topk_idx.to(dev)
    qs, sl = w.q_seq_idx.to(dev), w.seq_lens.to(dev)
    out = torch.empty((w.T, w.H, 512), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((w.T, w.H), dtype=torch.float32, device=dev)
    ws_bytes = nvmla.sparse_mla_decode_workspace_size(w.T, w.H, w.topk, impl=impl)
    ws = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device=dev)
    flush = torch.empty(FLUSH_BYTES // 4, dtype=torch.float32, device=dev)

    def decode():
        nvmla.sparse_mla_decode(ql, qr, cache, bt, tk, w.sm_scale, out=out, lse=lse, q_seq_idx=qs, seq_lens=sl,
                                workspace=ws, impl=impl)

    def pack_new():
        nvmla.nvfp4_mla_pack(d_new_lat, d_new_rope, d_new_slots, cache)

    for _ in range(max(3, args.warmup)):
        flush.fill_(1.0)
        pack_new()
        decode()
    torch.cuda.synchronize()

    # ---------------- timed region
    # Steps are enqueued in groups behind a GPU sleep, so that the host has
    # queued a whole group before the GPU reaches it: the events of a step
    # then bracket device work only, never host enqueue time. The sleeps,
    # like the L2 flushes, sit between steps.
    K = args.steps
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(K)]
    sampler = ClockSampler(local) if rank == 0 else None
    time.sleep(0.3 if sampler else 0.0)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    launches0 = nvmla.launch_count()
    t_wall0 = time.perf_counter()
    t_epoch0 = time.time()
    for k in range(K):
        if k % GROUP == 0:
            torch.cuda._sleep(LEAD_CYCLES_PER_STEP * min(GROUP, K - k))
        flush.fill_(float(k))
        ev[k][0].record()
        pack_new()
        ev[k][1].record()
        decode()
        ev[k][2].record()
    torch.cuda.synchronize()
    t_wall = time.perf_counter() - t_wall0
    t_epoch1 = time.time()
    launches = nvmla.launch_count() - launches0
    if world > 1:
        torch.distributed.barrier()
    clocks = sampler.stop(t_epoch0, t_epoch1) if sampler else None
    step_ms = [ev[k][0].elapsed_time(ev[k][2]) for k in range(K)]
    dec_ms = [ev[k][1].elapsed_time(ev[k][2]) for k in range(K)]
    pack_ms = [ev[k][0].elapsed_time(ev[k][1]) for k in range(K)]
    dec_us = statistics.mean(dec_ms) * 1e3
    step_mean = statistics.mean(step_ms)
    dec_us, step_mean = max_over_ranks([dec_us, step_mean], world, dev)
    # the decode call's device time without the event and launch overhead
    dec_kernel = kernel_only_us(decode, flush)

    # ---------------- end to end through the public API with host buffers
    # Every per-step input (queries, index lists, the new tokens) lives in
    # one pinned host buffer and goes up with one copy; out and lse come back
    # with one copy. The library calls take views of the device mirrors.
    def packed(parts, align=256):
        offs, total = [], 0
        for t in parts:
            offs.append(total)
            total += (t.numel() * t.element_size() + align - 1) // align * align
        return offs, total

    in_parts = [w.q_latent, w.q_rope, w.topk_idx, new_lat, new_rope, new_slots]
    in_offs, in_total = packed(in_parts)
    h_in = torch.zeros(in_total, dtype=torch.uint8).pin_memory()
    for t, o in zip(in_parts, in_offs):
        n = t.numel() * t.element_size()
        h_in[o:o + n].copy_(t.contiguous().view(-1).view(torch.uint8))
    d_in = torch.empty(in_total, dtype=torch.uint8, device=dev)

    def view(buf, off, like):
        n = like.numel() * like.element_size()
        return buf[off:off + n].view(like.dtype).view(like.shape)

    d_ql, d_qr, d_tk, d_nl, d_nr, d_ns = (view(d_in, o, t) for t, o in zip(in_parts, in_offs))
    out_like = torch.empty((w.T, w.H, 512), dtype=torch.bfloat16)
    lse_like = torch.empty((w.T, w.H), dtype=torch.float32)
    res_offs, res_total = packed([out_like, lse_like])
    d_res = torch.empty(res_total, dtype=torch.uint8, device=dev)
    h_res = torch.empty(res_total, dtype=torch.uint8).pin_memory()
    d_out, d_lse = view(d_res, res_offs[0], out_like), view(d_res, res_offs[1], lse_like)
    h2d = in_total
    d2h = res_total

    def e2e_step():
        d_in.copy_(h_in, non_blocking=True)
        nvmla.nvfp4_mla_pack(d_nl, d_nr, d_ns, cache)
        nvmla.sparse_mla_decode(d_ql, d_qr, cache, bt, d_tk, w.sm_scale, out=d_out, lse=d_lse, q_seq_idx=qs,
                                seq_lens=sl, workspace=ws, impl=impl)
        h_res.copy_(d_res, non_blocking=True)

    for _ in range(3):
        e2e_step()
    torch.cuda.synchronize()
    # the host copy of the result matches the device-resident path's
    if not (torch.equal(view(h_res, res_offs[0], out_like), out.cpu()) and
            torch.equal(view(h_res, res_offs[1], lse_like), lse.cpu())):
        raise RuntimeError("end-to-end result differs from the device-resident decode")
    def time_steps(step):
        ms = []
        for k in range(K):
            flush.fill_(float(k))
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            step()
            b.record()
            b.synchronize()
            ms.append(a.elapsed_time(b))
        return statistics.mean(ms) * 1e3

    # eager: the host enqueues the four operations of the step itself
    e2e_eager_us = time_steps(e2e_step)
    # serving-style: the same four operations recorded once as a CUDA graph
    # (the library's calls are capture-safe once a call has set the device
    # up) and replayed per step
    graph = torch.cuda.CUDAGraph()
    cap = torch.cuda.Stream()
    cap.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(cap):
        e2e_step()
    torch.cuda.current_stream().wait_stream(cap)
    with torch.cuda.graph(graph):
        e2e_step()
    for _ in range(3):
        graph.replay()
    torch.cuda.synchronize()
    if not torch.equal(view(h_res, res_offs[0], out_like), out.cpu()):
        raise RuntimeError("graph end-to-end result differs from the device-resident decode")
    e2e_us = time_steps(graph.replay)

    # ---------------- staged baseline (same workload, same protocol)
    staged = None
    if not args.no_staged:
        buf = torch.empty((w.T, w.topk, 576), dtype=torch.uint8, device=dev)
        ridx = torch.empty((w.T, w.topk), dtype=torch.int32, device=dev)
        ws2 = nvmla.sparse_mla_decode_fp8rows_workspace_size(w.T, w.H, w.topk, impl=impl)
        ws2 = torch.empty(max(ws2, 16), dtype=torch.uint8, device=dev)

        # stage 2 on the tcgen05 kernel: the staging buffer read as a paged
        # FP8 cache, token t's rows being pages t * topk / 64 onwards (one
        # block-table row per token; the list entries are the row indices)
        tc_stage2 = args.kernel != "mma" and w.H % 64 == 0 and w.topk % 64 == 0
        if tc_stage2:
            ppt = w.topk // 64
            sbt = torch.arange(w.T * ppt, dtype=torch.int32, device=dev).view(w.T, ppt)
            sqs = torch.arange(w.T, dtype=torch.int32, device=dev)
            sview = buf.view(w.T * ppt, 64, 576)

        def attend_tc():
            nvmla.sparse_mla_decode_fp8cache(ql, qr, sview, sbt, ridx, w.sm_scale, out=out, lse=lse, q_seq_idx=sqs,
                                             workspace=ws)

        def attend_mma():
            nvmla.sparse_mla_decode_fp8rows(ql, qr, buf, ridx, w.sm_scale, out=out, lse=lse, workspace=ws2,
                                            impl=impl)

        def staged_call():
            nvmla.nvfp4_stage_dequant_fp8(cache, bt, tk, qs, sl, fp8_rows=buf, row_idx=ridx)
            attend_mma()
            if tc_stage2:
                attend_tc()

        for _ in range(3):
            flush.fill_(1.0)
            staged_call()
        torch.cuda.synchronize()
        sev = []
        for k in range(K):
            if k % GROUP == 0:
                torch.cuda._sleep(LEAD_CYCLES_PER_STEP * min(GROUP, K - k))
            flush.fill_(float(k))
            e = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
            e[0].record()
            nvmla.nvfp4_stage_dequant_fp8(cache, bt, tk, qs, sl, fp8_rows=buf, row_idx=ridx)
            e[1].record()
            attend_mma()
            e[2].record()
            sev.append(e)
        torch.cuda.synchronize()
        s1 = [e[0].elapsed_time(e[1]) for e in sev]
        s2 = [e[1].elapsed_time(e[2]) for e in sev]
        attend_us = statistics.mean(s2) * 1e3
        how = "stage 2 on the mma.sync kernel (FP8 rows by index)"
        staged = {"dequant_us": statistics.mean(s1) * 1e3, "attend_mma_us": attend_us,
                  "fp8_buffer_bytes": w.T * w.topk * 576}
        if tc_stage2:
            # the tcgen05 stage 2 timed right after an untimed stage 1, as the
            # mma one is (the buffer partly in L2)
            tcev = []
            for k in range(K):
                if k % GROUP == 0:
                    torch.cuda._sleep(LEAD_CYCLES_PER_STEP * min(GROUP, K - k))
                flush.fill_(float(k))
                nvmla.nvfp4_stage_dequant_fp8(cache, bt, tk, qs, sl, fp8_rows=buf, row_idx=ridx)
                e = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
                e[0].record()
                attend_tc()
                e[1].record()
                tcev.append(e)
            torch.cuda.synchronize()
            staged["attend_tcgen05_us"] = statistics.mean([e[0].elapsed_time(e[1]) for e in tcev]) * 1e3
            attend_us = min(attend_us, staged["attend_tcgen05_us"])
            how = "stage 2 on the faster of the mma.sync kernel (FP8 rows by index) and the tcgen05 kernel (the " \
                  "buffer read as a paged FP8 cache)"
        staged["attend_us"] = attend_us
        staged["us_per_call"] = staged["dequant_us"] + attend_us
        staged["how"] = how

    # ---------------- the same decode over one layer of a block-major cache
    # of 4 layers (the rows of this workload in layer 2); same protocol
    layered = None
    if not args.no_layered:
        n_layers, layer = 4, 2
        lcache = torch.zeros((cache.shape[0], n_layers, 64, 352), dtype=torch.uint8, device=dev)
        lcache[:, layer] = cache
        lo, ll = torch.empty_like(out), torch.empty_like(lse)

        def layered_call():
            nvmla.sparse_mla_decode_layered(ql, qr, lcache, layer, bt, tk, w.sm_scale, out=lo, lse=ll, q_seq_idx=qs,
                                            seq_lens=sl, workspace=ws, impl=impl)

        decode()
        for _ in range(3):
            flush.fill_(1.0)
            layered_call()
        torch.cuda.synchronize()
        same = bool(torch.equal(lo, out) and torch.equal(ll, lse))
        if not same:
            raise RuntimeError("the layered decode differs from the one-layer decode of the same rows")
        lev = []
        for k in range(K):
            if k % GROUP == 0:
                torch.cuda._sleep(LEAD_CYCLES_PER_STEP * min(GROUP, K - k))
            flush.fill_(float(k))
            e = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
            e[0].record()
            layered_call()
            e[1].record()
            lev.append(e)
        torch.cuda.synchronize()
        layered = {"us_per_call": statistics.mean([e[0].elapsed_time(e[1]) for e in lev]) * 1e3,
                   "num_layers": n_layers, "layer": layer, "cache_bytes": lcache.numel(),
                   "bitwise_equal_to_one_layer_decode": same}
        del lcache

    # ---------------- the same decode over the FP8 cache (576-byte rows of the
    # same tokens) on the same kernel design, same protocol
    fp8 = None
    if not args.no_fp8 and args.kernel != "mma" and w.H % 64 == 0:
        lat_all, rope_all, slots_all = w.all_written()
        fcache = torch.zeros((cache.shape[0], 64, 576), dtype=torch.uint8, device=dev)
        nvmla.fp8_mla_pack(lat_all.to(dev), rope_all.to(dev), slots_all.to(dev), fcache)
        nvmla.fp8_mla_pack(d_new_lat, d_new_rope, d_new_slots, fcache)
        fo, fl = torch.empty_like(out), torch.empty_like(lse)

        def fp8_call():
            nvmla.sparse_mla_decode_fp8cache(ql, qr, fcache, bt, tk, w.sm_scale, out=fo, lse=fl, q_seq_idx=qs,
                                             seq_lens=sl, workspace=ws)

        for _ in range(3):
            flush.fill_(1.0)
            fp8_call()
        torch.cuda.synchronize()
        fev = []
        for k in range(K):
            if k % GROUP == 0:
                torch.cuda._sleep(LEAD_CYCLES_PER_STEP * min(GROUP, K - k))
            flush.fill_(float(k))
            e = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
            e[0].record()
            fp8_call()
            e[1].record()
            fev.append(e)
        torch.cuda.synchronize()
        f_us = statistics.mean([e[0].elapsed_time(e[1]) for e in fev]) * 1e3
        f_bytes = alg["bytes"] - alg["valid_slots"] * (352 - 576)
        fp8 = {"us_per_call": f_us, "row_bytes": 576, "cache_bytes": fcache.numel(),
               "algorithmic_bytes": f_bytes, "effective_hbm_gbs": f_bytes / (f_us * 1e-6) / 1e9,
               "nvfp4_cache_bytes": cache.numel()}
        del fcache

    # ---------------- the step upstream: top-2048 lists from scores of the
    # whole context (synthetic N(0,1) scores, seeded), same protocol
    topk_sel = None
    if not args.no_topk:
        gen = torch.Generator(device="cpu").manual_seed(7)
        ctx = int(w.seq_lens[0])
        sc = torch.randn((w.T, ctx), generator=gen, dtype=torch.float32).to(dev)
        tko = torch.empty((w.T, w.topk), dtype=torch.int32, device=dev)
        for _ in range(3):
            flush.fill_(1.0)
            nvmla.nvmla_topk_select(sc, w.topk, out=tko)
        torch.cuda.synchronize()
        tev = []
        for k in range(K):
            if k % GROUP == 0:
                torch.cuda._sleep(LEAD_CYCLES_PER_STEP * min(GROUP, K - k))
            flush.fill_(float(k))
            e = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
            e[0].record()
            nvmla.nvmla_topk_select(sc, w.topk, out=tko)
            e[1].record()
            tev.append(e)
        torch.cuda.synchronize()
        t_us = statistics.mean([e[0].elapsed_time(e[1]) for e in tev]) * 1e3
        t_kernel = kernel_only_us(lambda: nvmla.nvmla_topk_select(sc, w.topk, out=tko), flush)
        topk_sel = {"us_per_call": t_us, "T": w.T, "candidates": ctx, "topk": w.topk,
                    "score_bytes": w.T * ctx * 4, "gbs": w.T * ctx * 4 / (t_us * 1e-6) / 1e9,
                    "kernel_only": t_kernel}
        del sc

    # ---------------- pack of the write+read workload's 6144-token chunk
    plat, prope, pslots = workloads.pack_chunk(seed=4, n=6144, num_pages=2188)
    pcache = torch.zeros((2188, 64, 352), dtype=torch.uint8, device=dev)
    plat, prope, pslots = plat.to(dev), prope.to(dev), pslots.to(dev)
    for _ in range(3):
        nvmla.nvfp4_mla_pack(plat, prope, pslots, pcache)
    pk = []
    for k in range(K):
        if k % GROUP == 0:
            torch.cuda._sleep(LEAD_CYCLES_PER_STEP * min(GROUP, K - k))
        flush.fill_(float(k))
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        nvmla.nvfp4_mla_pack(plat, prope, pslots, pcache)
        b.record()
        pk.append(a)
        pk.append(b)
    torch.cuda.synchronize()
    pack_us = statistics.mean([pk[2 * i].elapsed_time(pk[2 * i + 1]) for i in range(K)]) * 1e3
    pack_bytes = 6144 * (1152 + 352 + 4)
    pack_kernel = kernel_only_us(lambda: nvmla.nvfp4_mla_pack(plat, prope, pslots, pcache), flush)
    # the same measure of a launch that does no work (torch's GPU sleep for
    # one cycle): the floor under every kernel-only figure of this line
    floor = kernel_only_us(lambda: torch.cuda._sleep(1), flush)

    # ---------------- the other workloads the baseline names, same protocol
    configs = None
    if not args.no_configs:
        configs = {}
        pk_c, _ = peaks()
        for cname in ("padded", "batched", "write_read"):
            configs[cname] = config_line(cname, args, flush, dev, pk_c, impl)
            torch.cuda.empty_cache()

    if rank != 0:
        return
    pk_peaks, peak_src = peaks()
    bw = pk_peaks["hbm_gbs"]
    tf = pk_peaks["bf16_tflops"]
    t_bytes = alg["bytes"] / (bw * 1e9) * 1e6
    t_flops = alg["flops"] / (tf * 1e12) * 1e6
    bound = "tensor" if t_flops >= t_bytes else "hbm"
    if bound == "tensor":
        achieved = alg["flops"] / (dec_us * 1e-6) / 1e12
        peak, unit = tf, "TFLOP/s"
    else:
        achieved = alg["bytes"] / (dec_us * 1e-6) / 1e9
        peak, unit = bw, "GB/s"
    kernel = "decode_tc_kernel" if args.kernel in ("auto", "tcgen05") and w.H % 64 == 0 else "decode_mma_kernel"
    traffic = traffic_record(kernel)
    cpu = None
    if not args.no_cpu_baseline:
        cpu = cpu_baseline(w, args.cpu_seconds)
    line = {
        "metric": METRIC, "value": dec_us, "unit": UNIT, "n_gpus": world, "steps": K, "warmup": args.warmup,
        "ms_per_step": step_mean, "higher_is_better": False, "scaling": "weak", "vs_baseline": None,
        "dtype": "f16", "data": "synthetic",
        "config": {"workload": WORKLOAD_DESC, "T": w.T, "H": w.H, "topk": w.topk, "ctx": int(w.seq_lens[0]),
                   "valid_slots": alg["valid_slots"], "kernel": args.kernel,
                   "l2": f"flushed before every step ({FLUSH_BYTES >> 20} MiB write)",
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        "roofline": {"bound": bound, "achieved": achieved, "peak": peak, "unit": unit, "frac": achieved / peak,
                     "peak_source": f"{peak_src} ({'bf16 burst; fp16 nominal rate equals bf16' if bound == 'tensor' else 'HBM copy'})",
                     "roofline_us": max(t_bytes, t_flops), "bytes_us": t_bytes, "flops_us": t_flops,
                     "algorithmic_bytes": alg["bytes"], "algorithmic_flops": alg["flops"],
                     "effective_hbm_gbs": alg["bytes"] / (dec_us * 1e-6) / 1e9,
                     "kernel": kernel, "timed": "whole decode call (CUDA events on the launching stream)",
                     "traffic": traffic,
                     "kernel_us": dec_kernel["cold_l2_us"],
                     "frac_kernel": (alg["flops"] / (dec_kernel["cold_l2_us"] * 1e-6) / 1e12) / peak
                     if bound == "tensor" else (alg["bytes"] / (dec_kernel["cold_l2_us"] * 1e-6) / 1e9) / peak},
        "decode_kernel_only": dec_kernel,
        "kernel_only_floor": dict(floor, what="an empty launch (one-cycle GPU sleep) under the same "
                                              "kernel-only measure: context, not subtracted"),
        "decode_us": {"mean": dec_us, "median": statistics.median(dec_ms) * 1e3, "min": min(dec_ms) * 1e3},
        "pack_step_us": statistics.mean(pack_ms) * 1e3,
        "pack_chunk": {"tokens": 6144, "bytes": pack_bytes, "us_per_call": pack_us,
                       "gbs": pack_bytes / (pack_us * 1e-6) / 1e9,
                       "frac_hbm": pack_bytes / (pack_us * 1e-6) / 1e9 / bw,
                       "kernel_only": pack_kernel,
                       "frac_hbm_kernel": pack_bytes / (pack_kernel["cold_l2_us"] * 1e-6) / 1e9 / bw},
        "staged": staged,
        "layered": layered,
        "topk_select": (dict(topk_sel, frac_hbm=topk_sel["gbs"] / bw,
                             frac_hbm_kernel=topk_sel["score_bytes"] / (topk_sel["kernel_only"]["cold_l2_us"] * 1e-6)
                             / 1e9 / bw,
                             kernel="topk_resident_kernel (rows of up to 262,144 scores)")
                        if topk_sel else None),
        "fp8_cache": fp8,
        "configs": configs,
        "e2e": {"value": e2e_us, "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "how": "per step: one host-to-device copy of every input from pinned memory, nvfp4_mla_pack, "
                       "sparse_mla_decode, one device-to-host copy of out and lse, replayed as a CUDA graph; "
                       "host synchronised after every step",
                "eager_value": e2e_eager_us},
        "gpu_launches": int(launches),
        "clocks": clocks,
        "cpu_baseline": cpu,
        "wall_s_timed_region": t_wall,
    }
    print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
