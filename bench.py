"""Benchmark of the paged-attention forward hot path on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Main line (`value`): paged decode of the bf16 GQA workload (64 sequences,
32 q / 8 kv heads, head_dim 128, block size 16, cached lengths U[512, 4096]),
one pa_decode call (in-place append + attention through the block table)
per step, reported as KV-read GB/s over the DISTINCT pool bytes the step
reads, with the roofline of the decode kernel against the measured HBM
copy bandwidth.  Extra keys report the other decode workloads (long-context
split-K, shared-prefix mixed) and the varlen prefill leg (pa_cache_update +
causal pa_varlen) in TFLOP/s against the measured bf16 tensor peak.

`--impl reference` times the fp64 CPU oracle (test infrastructure, the only
other place this script runs it) on a bounded sample of the same workload.

Inputs are seeded and synthetic (CPU generator, then copied to the GPU).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "paged decode KV-read GB/s (% of GB300 HBM peak), seq/s; varlen prefill TFLOP/s"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def code_text(src: str) -> str:
    """C++/CUDA source with comments and all whitespace removed (string
    literals kept): two files with equal code text compile to the same
    kernel, whatever their comments say."""
    out, i, n = [], 0, len(src)
    while i < n:
        c = src[i]
        if src.startswith("//", i):
            j = src.find("\n", i)
            i = n if j < 0 else j
        elif src.startswith("/*", i):
            j = src.find("*/", i + 2)
            i = n if j < 0 else j + 2
        elif c in "\"'":
            j = i + 1
            while j < n and src[j] != c:
                j += 2 if src[j] == "\\" else 1
            out.append(src[i:j + 1])
            i = j + 1
        else:
            if not c.isspace():
                out.append(c)
            i += 1
    return "".join(out)


def source_hash(name: str) -> str:
    """Hash of a kernel file's code text (comments and layout excluded)."""
    with open(os.path.join(ROOT, "paged_kv_cache_300_gb300", "csrc", name), encoding="utf-8") as f:
        return hashlib.sha256(code_text(f.read()).encode()).hexdigest()[:16]


# DRAM traffic per launch taken from ncu captures (profiles/), valid only for
# the kernel code they were measured on (source_hash: code text without
# comments, so a comment edit keeps a capture valid and a code edit does not).
NCU_TRAFFIC = {
    ("pa_decode.cu", "workload2"): {"src": "dd4f6d587e86c182", "bytes": 561_159_680},
    ("pa_varlen_tc.cu", "workload4"): {"src": "bda691fcb9927be7", "bytes": 661_326_848},
}


def traffic_for(kernel_file: str, workload: str):
    rec = NCU_TRAFFIC.get((kernel_file, workload))
    if rec and rec["src"] == source_hash(kernel_file):
        return rec["bytes"]
    return None


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled every 100 ms."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                smax = float(parts[1])
            except ValueError:
                continue
            for n, v in zip(names, parts[3:7]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        sm.sort()
        return {"sm_mhz": sm[len(sm) // 2] if sm else None, "sm_max_mhz": smax,
                "reasons": sorted(reasons), "samples": len(sm)}


class L2Flush:
    """Evicts the previous step's data from L2 between timed steps: writes a
    buffer of 2x L2, then reads another 2x L2 buffer, so that the timed step
    starts with an L2 holding none of its inputs and no dirty lines whose
    write-back it would otherwise pay for."""

    def __init__(self, torch, nbytes):
        self.w = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
        self.r = torch.ones(nbytes // 4, dtype=torch.float32, device="cuda")
        self.acc = torch.empty((), dtype=torch.float32, device="cuda")
        self.torch = torch

    def zero_(self):
        self.w.zero_()
        self.torch.sum(self.r, dim=(0,), out=self.acc)


# --------------------------------------------------------------------------
# distributed plumbing (one process per GPU; the workload shards by sequence,
# no data-path collective)
# --------------------------------------------------------------------------

class Dist:
    def __init__(self):
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local = int(os.environ.get("LOCAL_RANK", "0"))
        self.pg = None

    def init(self, torch, backend: str = "nccl"):
        """nccl on GPUs; gloo (CPU tensors) for the host-side tests."""
        self.device = "cuda" if backend == "nccl" else "cpu"
        if self.world > 1:
            import torch.distributed as dist
            os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
            if backend == "nccl":
                torch.cuda.set_device(self.local)
            dist.init_process_group(backend, rank=self.rank, world_size=self.world)
            self.pg = dist

    def barrier(self, torch):
        if self.pg is not None:
            self.pg.barrier()

    def _reduce(self, torch, x: float, op) -> float:
        if self.pg is None:
            return x
        t = torch.tensor([x], dtype=torch.float64, device=self.device)
        self.pg.all_reduce(t, op=op)
        return float(t.item())

    def max(self, torch, x: float) -> float:
        return self._reduce(torch, x, None if self.pg is None else self.pg.ReduceOp.MAX)

    def sum(self, torch, x: float) -> float:
        return self._reduce(torch, x, None if self.pg is None else self.pg.ReduceOp.SUM)

    def close(self):
        if self.pg is not None:
            self.pg.destroy_process_group()


# --------------------------------------------------------------------------
# decode legs
# --------------------------------------------------------------------------

def decode_alg_bytes(case) -> int:
    """Algorithmic bytes of one decode step: distinct KV rows read, q and
    out, k_new/v_new read, the appended rows written, table entries read."""
    import numpy as np
    bs = case.block_size
    L = case.cache_seqlens.numpy().astype(np.int64)
    table = int(((L + bs) // bs).sum()) * 4 + 4 * case.batch
    return case.unique_kv_bytes() + case.io_bytes() + table


def run_decode_leg(torch, pa, case, steps, warmup, dist=None, sync_ranks=False,
                   contiguous=False):
    """Device time of `steps` pa_decode calls run back to back, as a serving
    loop runs them: the steps are captured as one CUDA graph of `steps`
    launches and the graph is timed with one pair of events.  No L2 flush:
    the KV a step reads (0.55-6.5 GB on the decode workloads) is several
    times the 129 MB L2, and consecutive launches read as many bytes from
    DRAM as a launch after a flush.  Each launch allows programmatic
    dependence, so a step's start-up overlaps the previous step's end.
    Returns dict with the per-step ms (total / steps) and wall seconds.
    `contiguous`: the same logical cache laid out as [B, max_seqlen, Hkv, D]
    and decoded by the contiguous-cache twin (pa_decode_contiguous)."""
    dev = "cuda"
    t = lambda x: x.to(dev)
    q, bt, sl, kn, vn = map(t, (case.q, case.block_table, case.cache_seqlens, case.k_new,
                                case.v_new))
    if contiguous:
        kc, vc = case.contiguous_cache(device=dev)
        need = pa.pa_decode_contiguous_workspace_size(case.batch, case.num_heads,
                                                      case.num_kv_heads, case.head_dim)
    else:
        kc, vc = t(case.k_cache), t(case.v_cache)
        need = pa.pa_decode_workspace_size(case.batch, case.num_heads, case.num_kv_heads,
                                           case.head_dim, case.block_size, case.q.dtype)
    out = torch.empty_like(q)
    ws = torch.zeros(max(need, 16), dtype=torch.uint8, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    args = (q, kc, vc, bt, sl, kn, vn, out)
    if contiguous:
        step = lambda: pa.pa_decode_contiguous(q, kc, vc, sl, kn, vn, out, workspace=ws,
                                               dev_err=err)
    else:
        step = lambda: pa.pa_decode(*args, workspace=ws, dev_err=err)
    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    # the timed steps captured as one CUDA graph, so the per-step host work
    # (argument checks, descriptor lookup) is paid once, as a serving loop
    # would; the graph is replayed once untimed before the timed replay
    graph = None
    try:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for _ in range(steps):
                step()
        graph = g
        graph.replay()
        torch.cuda.synchronize()
    except Exception as e:  # capture refused: time the direct calls
        graph = None
        print(f"note: CUDA graph capture unavailable ({e}); timing direct calls",
              file=sys.stderr)
        torch.cuda.synchronize()

    def run():
        if graph is not None:
            graph.replay()
        else:
            for _ in range(steps):
                step()

    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if sync_ranks and dist is not None:
        dist.barrier(torch)
    torch.cuda.synchronize()
    w0 = time.perf_counter()
    e0.record()
    run()
    e1.record()
    torch.cuda.synchronize()
    if sync_ranks and dist is not None:
        dist.barrier(torch)
    wall = time.perf_counter() - w0
    per = e0.elapsed_time(e1) / steps
    if int(err.item()) != 0:
        raise RuntimeError(f"device error bits {int(err.item())} during the benchmark")
    res = {"ms": [per] * steps, "wall_s": wall,
           "tensors": (q, kn, vn, bt, sl, out, kc, vc, ws, err),
           "launch": (f"one CUDA graph of {steps} back-to-back steps" if graph is not None
                      else "direct calls, back to back")}
    return res


def run_decode_e2e(torch, pa, case, res, steps):
    """The same step through the public API with the step's tensors in HOST
    memory: q, k_new, v_new, block_table and cache_seqlens in page-locked
    host buffers, the output into a page-locked host buffer.  pa_decode is
    called on the host tensors every step, back to back (host-side checks
    and launch included; one pair of events around all steps); on GB300 the kernel reads the inputs and writes the output in
    place over NVLink-C2C, so the host<->device transfer of every input and
    output byte happens inside the timed region.  The KV pool stays resident
    in HBM, as a KV cache does.  Returns (ms, h2d_bytes, d2h_bytes)."""
    q, kn, vn, bt, sl, out, kc, vc, ws, err = res["tensors"]
    pin = lambda x: x.clone().pin_memory()
    hq, hkn, hvn, hbt, hsl = (pin(x) for x in (case.q, case.k_new, case.v_new, case.block_table,
                                               case.cache_seqlens))
    hout = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    h2d = sum(x.numel() * x.element_size() for x in (hq, hkn, hvn, hbt, hsl))
    d2h = hout.numel() * hout.element_size()
    step = lambda: pa.pa_decode(hq, kc, vc, hbt, hsl, hkn, hvn, hout, workspace=ws, dev_err=err)
    for _ in range(3):
        step()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record()
    for _ in range(steps):
        step()
    e1.record()
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / steps
    if int(err.item()) != 0:
        raise RuntimeError(f"device error bits {int(err.item())} in the e2e leg")
    if not torch.equal(hout.view(torch.int16), out.cpu().view(torch.int16)):
        raise RuntimeError("host-buffer decode differs from the device-buffer decode")
    return ms, h2d, d2h


def run_decode_e2e_copies(torch, pa, case, res, steps):
    """The step with explicit copies instead: the five inputs go host->device
    in one copy from a pinned staging buffer, pa_decode runs on device
    views, the output comes back device->host (copy engines)."""
    q, kn, vn, bt, sl, out, kc, vc, ws, err = res["tensors"]
    srcs = (case.q, case.k_new, case.v_new, case.block_table, case.cache_seqlens)
    offs, total = [], 0
    for x in srcs:  # 256-byte aligned slices of one buffer
        offs.append(total)
        total += (x.numel() * x.element_size() + 255) // 256 * 256
    hbuf = torch.empty(total, dtype=torch.uint8).pin_memory()
    dbuf = torch.empty(total, dtype=torch.uint8, device="cuda")

    def views(buf):
        return [buf[o:o + x.numel() * x.element_size()].view(x.dtype).view(x.shape)
                for o, x in zip(offs, srcs)]

    for h, x in zip(views(hbuf), srcs):
        h.copy_(x)
    dq, dkn, dvn, dbt, dsl = views(dbuf)
    hout = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(steps)]
    torch.cuda.synchronize()
    for e in evs:
        e[0].record()
        dbuf.copy_(hbuf, non_blocking=True)
        e[1].record()
        pa.pa_decode(dq, kc, vc, dbt, dsl, dkn, dvn, out, workspace=ws, dev_err=err)
        e[2].record()
        hout.copy_(out, non_blocking=True)
        e[3].record()
    torch.cuda.synchronize()
    n = len(evs)
    return {"ms_per_step": round(sum(e[0].elapsed_time(e[3]) for e in evs) / n, 5),
            "h2d_ms": round(sum(e[0].elapsed_time(e[1]) for e in evs) / n, 5),
            "call_ms": round(sum(e[1].elapsed_time(e[2]) for e in evs) / n, 5),
            "d2h_ms": round(sum(e[2].elapsed_time(e[3]) for e in evs) / n, 5)}


# --------------------------------------------------------------------------
# varlen leg: pa_cache_update (scatter + gather) then causal pa_varlen
# --------------------------------------------------------------------------

def run_varlen_leg(torch, pa, case, steps, warmup, flush):
    dev = "cuda"
    t = lambda x: x.to(dev)
    q, kch, vch = t(case.q), t(case.k_chunk), t(case.v_chunk)
    kc, vc, bt = t(case.k_cache), t(case.v_cache), t(case.block_table)
    pl, cq, ck = t(case.prefix_lens), t(case.cu_seq_lens_q), t(case.cu_seq_lens_k)
    tk = int(case.cu_seq_lens_k[-1])
    kf = torch.empty(tk, *case.k_chunk.shape[1:], dtype=case.k_chunk.dtype, device=dev)
    vf = torch.empty_like(kf)
    out = torch.empty_like(q)
    err = torch.zeros(1, dtype=torch.int32, device=dev)

    def upd():
        pa.pa_cache_update(kch, vch, cq, pl, bt, kc, vc, kf, vf, ck, dev_err=err)

    def att():
        pa.pa_varlen(q, kf, vf, cq, ck, case.max_length_q, case.max_length_k, case.causal,
                     out=out, dev_err=err)

    for _ in range(warmup):
        upd()
        att()
    torch.cuda.synchronize()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(steps)]
    for e in ev:
        flush.zero_()
        e[0].record()
        upd()
        e[1].record()
        att()
        e[2].record()
    torch.cuda.synchronize()
    if int(err.item()) != 0:
        raise RuntimeError(f"device error bits {int(err.item())} in the varlen leg")
    upd_ms = [a.elapsed_time(b) for a, b, _ in ev]
    att_ms = [b.elapsed_time(c) for _, b, c in ev]

    # fused path: scatter only, then attention reading keys through the table
    seqlens_k = (ck[1:] - ck[:-1]).to(torch.int32)

    def scat():
        pa.pa_cache_update(kch, vch, cq, pl, bt, kc, vc, dev_err=err)

    def patt():
        pa.pa_varlen_paged(q, kc, vc, bt, cq, seqlens_k, case.max_length_q, case.max_length_k,
                           case.causal, out=out, dev_err=err)

    for _ in range(warmup):
        scat()
        patt()
    torch.cuda.synchronize()
    for e in ev:
        flush.zero_()
        e[0].record()
        scat()
        e[1].record()
        patt()
        e[2].record()
    torch.cuda.synchronize()
    if int(err.item()) != 0:
        raise RuntimeError(f"device error bits {int(err.item())} in the fused varlen leg")
    scat_ms = sum(a.elapsed_time(b) for a, b, _ in ev) / steps
    patt_ms = sum(b.elapsed_time(c) for _, b, c in ev) / steps
    return sum(upd_ms) / steps, sum(att_ms) / steps, scat_ms, patt_ms


# --------------------------------------------------------------------------
# CPU oracle timing (the reported baseline; never tuned)
# --------------------------------------------------------------------------

def oracle_decode_sample(case, rows, cores):
    import numpy as np
    import oracle
    from workloads import to_numpy
    q, kn, vn = (np.ascontiguousarray(to_numpy(x)[rows]) for x in (case.q, case.k_new, case.v_new))
    tab = np.ascontiguousarray(case.block_table.numpy()[rows])
    sl = np.ascontiguousarray(case.cache_seqlens.numpy()[rows])
    kc, vc = to_numpy(case.k_cache).copy(), to_numpy(case.v_cache).copy()
    t0 = time.perf_counter()
    oracle.decode(q, kc, vc, tab, sl, kn, vn, nthreads=cores)
    dt = time.perf_counter() - t0
    bs = case.block_size
    ub = 0
    for b in rows:
        ub += (int(case.cache_seqlens[b]) + 1)
    kv_bytes = ub * case.num_kv_heads * case.head_dim * case.elt() * 2
    return dt, kv_bytes


def cpu_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


# --------------------------------------------------------------------------
# main
# --------------------------------------------------------------------------

def leg_summary(case, ms_list, peaks, wall=None):
    ms = sum(ms_list) / len(ms_list)
    ub, lb, ab = case.unique_kv_bytes(), case.logical_kv_bytes(), decode_alg_bytes(case)
    return {
        "workload": case.name,
        "ms": round(ms, 5),
        "kv_unique_GBps": round(ub / ms / 1e6, 1),
        "kv_logical_GBps": round(lb / ms / 1e6, 1),
        "seq_per_s": round(case.batch / ms * 1e3, 1),
        "roofline": {"bound": "hbm", "achieved": round(ab / ms / 1e6, 1),
                     "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": round(ab / ms / 1e6 / peaks["hbm_gbs"], 4)},
    }


def reference_main(args, dist):
    """The reference arm: the fp64 CPU oracle on a bounded sample."""
    if dist.rank != 0:
        return 0
    from workloads import decode_config
    case = decode_config(2)
    cores = cpu_cores()
    rows = list(range(0, case.batch, 4))  # 16 of the 64 sequences
    for _ in range(args.warmup):
        oracle_decode_sample(case, rows[:2], cores)
    tot_t, tot_b = 0.0, 0
    for _ in range(args.steps):
        dt, kvb = oracle_decode_sample(case, rows, cores)
        tot_t += dt
        tot_b += kvb
    gbps = tot_b / tot_t / 1e9
    sample = f"{len(rows)} of the 64 sequences of the workload per step (every 4th)"
    line = {
        "impl": "reference", "metric": METRIC, "value": round(gbps, 4), "unit": "GB/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(tot_t / args.steps * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": case.name, "sample": sample},
        "cpu_baseline": {"value": round(gbps, 4), "unit": "GB/s", "cores": cores,
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(gbps, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--main-only", action="store_true",
                    help="skip the extra workloads and the CPU baseline")
    ap.add_argument("--leg", choices=["all", "varlen"], default="all",
                    help="varlen: time only the varlen prefill leg (for profiling)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    dist = Dist()
    if args.impl == "reference":
        return reference_main(args, dist)

    import torch
    import paged_kv_cache_300_gb300 as pa
    from workloads import decode_config, varlen_config

    dist.init(torch)
    torch.cuda.set_device(dist.local)
    pa.load()
    peaks, peak_kind = load_peaks()
    l2 = torch.cuda.get_device_properties(dist.local).L2_cache_size
    flush = L2Flush(torch, max(2 * l2, 256 << 20))
    clocks = ClockSampler(dist.local)
    clocks.start()

    if args.leg == "varlen":
        vc = varlen_config(4)
        upd_ms, att_ms, scat_ms, patt_ms = run_varlen_leg(torch, pa, vc, args.steps, args.warmup,
                                                          flush)
        flops = 4.0 * vc.q.shape[2] * vc.q.shape[1] * vc.causal_pairs()
        clk = clocks.stop()
        if dist.rank == 0:
            print(json.dumps({"leg": "varlen", "workload": vc.name, "varlen_ms": round(att_ms, 5),
                              "cache_update_ms": round(upd_ms, 5),
                              "tflops": round(flops / att_ms / 1e9, 2),
                              "fused_scatter_ms": round(scat_ms, 5),
                              "fused_varlen_paged_ms": round(patt_ms, 5),
                              "fused_tflops": round(flops / patt_ms / 1e9, 2), "clocks": clk}))
        return 0

    # ---- main line: decode workload 2 (each rank decodes its own batch)
    case = decode_config(2, seed_offset=dist.rank)
    res = run_decode_leg(torch, pa, case, args.steps, args.warmup, dist, sync_ranks=True)
    dev_ms_total = dist.max(torch, sum(res["ms"]))
    ms = dev_ms_total / args.steps
    ub_all = dist.sum(torch, float(case.unique_kv_bytes()))
    seqs_all = dist.sum(torch, float(case.batch))
    value = ub_all / ms / 1e6
    main = leg_summary(case, res["ms"], peaks)
    main_launch = res["launch"]
    e2e_steps = max(10, args.steps // 2)
    e2e_ms, h2d, d2h = run_decode_e2e(torch, pa, case, res, e2e_steps)
    e2e_ms = dist.max(torch, e2e_ms)
    e2e_copies = run_decode_e2e_copies(torch, pa, case, res, e2e_steps)
    del res
    torch.cuda.empty_cache()

    extra = {}
    if not args.main_only:
        for idx, key in ((3, "decode_long_context"), (5, "decode_shared_prefix")):
            c = decode_config(idx)
            r = run_decode_leg(torch, pa, c, min(args.steps, 20), args.warmup)
            extra[key] = leg_summary(c, r["ms"], peaks)
            del r, c
            torch.cuda.empty_cache()
        # paging overhead, two ways.  (1) Placement: the main workload again
        # with every sequence's blocks adjacent in the pool, same kernel.
        # (2) The contiguous-cache twin: the same logical cache laid out as
        # [B, max_seqlen, Hkv, D] and decoded by pa_decode_contiguous (no
        # block table), against pa_decode on the paged pool.
        c = decode_config(2, seed_offset=dist.rank, contiguous=True)
        r = run_decode_leg(torch, pa, c, min(args.steps, 20), args.warmup)
        cms = sum(r["ms"]) / len(r["ms"])
        overhead = {"placement": {
            "workload": c.name,
            "adjacent_blocks_ms": round(cms, 5), "scattered_blocks_ms": round(ms, 5),
            "scattered_over_adjacent": round(ms / cms, 4),
            "note": "same paged kernel and data; only the physical placement of the blocks "
                    "differs"}}
        del r, c
        torch.cuda.empty_cache()
        for idx, paged_ms in ((2, ms), (3, extra["decode_long_context"]["ms"])):
            c = decode_config(idx, seed_offset=dist.rank if idx == 2 else 0)
            r = run_decode_leg(torch, pa, c, min(args.steps, 20), args.warmup,
                               contiguous=True)
            cms = sum(r["ms"]) / len(r["ms"])
            overhead[f"paged_over_contiguous_workload{idx}"] = {
                "workload": c.name, "paged_ms": round(paged_ms, 5),
                "contiguous_ms": round(cms, 5), "paged_over_contiguous": round(paged_ms / cms, 4),
                "contiguous_kv_GBps": round(c.unique_kv_bytes() / cms / 1e6, 1),
                "note": "pa_decode (block table, scattered blocks) vs pa_decode_contiguous "
                        "(the same kernel code over a [B, max_seqlen, Hkv, D] cache, no table)"}
            del r, c
            torch.cuda.empty_cache()
        extra["paging_overhead"] = overhead
        vc = varlen_config(4)
        try:
            upd_ms, att_ms, scat_ms, patt_ms = run_varlen_leg(torch, pa, vc, min(args.steps, 20),
                                                              args.warmup, flush)
            flops = 4.0 * vc.q.shape[2] * vc.q.shape[1] * vc.causal_pairs()
            tk = int(vc.cu_seq_lens_k[-1])
            row = vc.k_chunk.shape[1] * vc.k_chunk.shape[2] * vc.k_chunk.element_size()
            tq = vc.q.shape[0]
            upd_bytes = 2 * (2 * tq * row) + 2 * (2 * (tk - tq) * row) + 2 * (tq * row)
            extra["varlen_prefill"] = {
                "workload": vc.name, "causal_pairs": vc.causal_pairs(),
                "varlen_ms": round(att_ms, 5), "cache_update_ms": round(upd_ms, 5),
                "tflops": round(flops / att_ms / 1e9, 2),
                "roofline": {"bound": "tensor", "achieved": round(flops / att_ms / 1e9, 2),
                             "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                             "frac": round(flops / att_ms / 1e9 / peaks["bf16_tflops"], 4),
                             "traffic": traffic_for("pa_varlen_tc.cu", "workload4"),
                             "peak_source": f"{peak_kind} bf16_tflops (burst)"},
                "cache_update_GBps": round(upd_bytes / upd_ms / 1e6, 1),
                "step_tflops": round(flops / (att_ms + upd_ms) / 1e9, 2),
                "fused_paged": {
                    "note": "scatter-only pa_cache_update, then pa_varlen_paged reading the "
                            "keys through block_table (no gather copy)",
                    "scatter_ms": round(scat_ms, 5), "varlen_paged_ms": round(patt_ms, 5),
                    "tflops": round(flops / patt_ms / 1e9, 2),
                    "step_tflops": round(flops / (patt_ms + scat_ms) / 1e9, 2)},
            }
        except pa.PAError as e:
            extra["varlen_prefill"] = {"unavailable": str(e)}
        del vc
        torch.cuda.empty_cache()
    clk = clocks.stop()

    if dist.rank != 0:
        return 0
    line = {
        "metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": dist.world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": case.name, "batch": case.batch, "num_heads": case.num_heads,
                   "num_kv_heads": case.num_kv_heads, "head_dim": case.head_dim,
                   "block_size": case.block_size, "kv_unique_bytes": case.unique_kv_bytes(),
                   "l2": "decode legs: no flush; inputs larger than L2 (552 MB of distinct KV per step against a 129 MB L2), steps back to back, and consecutive launches each read as many bytes from DRAM as a launch after a flush (ncu); varlen leg: L2 flushed before every step outside the timed events (2x L2 written, then 2x L2 read)",
                   "parallelism": f"replicas x{dist.world} (sequences shard, no collective)",
                   "launch": main_launch},
        "pct_of_hbm_peak": round(100 * value / dist.world / peaks["hbm_gbs"], 2),
        "seq_per_s": round(seqs_all / ms * 1e3, 1),
        "roofline": dict(main["roofline"], traffic=traffic_for("pa_decode.cu", "workload2"),
                         peak_source=f"{peak_kind} hbm_gbs (copy)"),
        "e2e": {"value": round(ub_all / e2e_ms / 1e6, 1), "unit": "GB/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": round(e2e_ms, 5),
                "how": "pa_decode called every step on page-locked host tensors (q, k_new, "
                       "v_new, block_table, cache_seqlens in, out back): the kernel reads and "
                       "writes them in place over NVLink-C2C; KV pool resident in HBM",
                "explicit_copies": dict(e2e_copies, value=round(
                    ub_all / e2e_copies["ms_per_step"] / 1e6, 1), unit="GB/s",
                    how="one pinned host->device copy of the inputs, pa_decode on device "
                        "buffers, one device->host copy of out (copy engines)")},
        "gpu_launches": args.steps,
        "clocks": clk,
    }
    line.update(extra)
    if dist.world == 1 and not args.main_only:
        cores = cpu_cores()
        rows = list(range(case.batch))
        tot_t, tot_b, passes = 0.0, 0, 0
        while tot_t < 10.0 and passes < 200:
            dt, kvb = oracle_decode_sample(case, rows, cores)
            tot_t, tot_b, passes = tot_t + dt, tot_b + kvb, passes + 1
        line["cpu_baseline"] = {"value": round(tot_b / tot_t / 1e9, 4), "unit": "GB/s",
                                "cores": cores, "kind": "oracle", "seconds": round(tot_t, 2),
                                "sample": f"{passes} full passes of the main workload "
                                          "(64 sequences each), about 10 s of CPU work"}
    print(json.dumps(line), flush=True)
    return 0


if __name__ == "__main__":
    sys.exit(main())
