"""Benchmark of split-KV decode attention (FlashDecoding) on GB300.

One step = one fused decode (split kernel + in-kernel merge, automatic
decomposition) over the whole workload, inputs resident in HBM.  Prints ONE
JSON line (rank 0):

  value      KV-GB/s over all ranks: valid K+V bytes of every rank's step
             divided by the max over ranks of the device time per step
  roofline   the split kernel's achieved bytes/s (algorithmic bytes per
             launch / mean launch time from CUDA events on its stream)
             against the measured HBM copy bandwidth
  e2e        the same metric through the public API from pinned host
             buffers: every step copies q, K, V, lengths to the device,
             decodes, and reads out and lse back
  cpu_baseline  the float64 oracle timed on the host's cores on a bounded
             sample of the same workload (rank 0, one GPU only)

`--impl reference` times the oracle itself as the reference arm (host cores,
bounded sample per step) and prints the same line with "impl": "reference".
Multi-GPU (torchrun): every rank runs its own replica of the workload (the
(b, h) problems are independent; no data-path collective), weak scaling.
"""
from __future__ import annotations

import argparse
import hashlib
import re
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

from split_kv_fd_gb300.workloads import BENCH_DEFAULT, ELEMENT_BYTES, WORKLOADS  # noqa: E402

METRIC = "split-KV decode attention KV-GB/s and % of GB300 HBM peak (~8 TB/s), 1 GPU"
NOMINAL_HBM_GBS = 8000.0
L2_BYTES = 129 * 1024 * 1024
# the sources each profiled kernel is compiled from (the hash of a kernel's
# sources keys its committed ncu traffic record)
KERNEL_SOURCES = {
    "split_kernel": ["fd_split.cuh", "fd_device.cuh", "fd_internal.h", "fd_split_bf16.cu",
                     "fd_split_f16.cu", "fd_split_f32.cu", "fd_split_fp8.cu"],
    "gqa_kernel": ["fd_gqa.cuh", "fd_gqa_kernel.cuh", "fd_gqa_bf16.cu", "fd_gqa_f16.cu", "fd_split.cuh",
                   "fd_device.cuh", "fd_internal.h"],
    "gqa_tc_kernel": ["fd_gqa_tc.cuh", "fd_tc.cuh", "fd_gqa_tc.cu", "fd_gqa.cuh", "fd_split.cuh",
                      "fd_device.cuh", "fd_internal.h"],
    "gqa_tc8_kernel": ["fd_gqa_tc8.cuh", "fd_gqa_tc8.cu", "fd_gqa_tc.cuh", "fd_tc.cuh", "fd_gqa.cuh",
                       "fd_split.cuh", "fd_device.cuh", "fd_internal.h"],
}


# ----------------------------------------------------------------- helpers

def kv_bytes(w, lens) -> int:
    """Valid K and V bytes of one step: 2 * Hkv * d * elt * sum_b len_b."""
    return 2 * w.kv_heads * w.d * ELEMENT_BYTES[w.dtype] * int(sum(int(x) for x in lens))


def algorithmic_bytes(w, lens) -> int:
    """Compulsory DRAM traffic of one launch: K/V valid rows, q, out, lse, lengths."""
    e = ELEMENT_BYTES[w.dtype]
    out_e = ELEMENT_BYTES[w.out_dtype]
    return kv_bytes(w, lens) + w.B * w.H * w.d * (e + out_e) + w.B * w.H * 4 + w.B * 4


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            return json.load(f), "measured"
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0}, "fallback"


def kernel_source_hash(kernel: str = "split_kernel") -> str:
    """Hash of a kernel's code: its sources without comments and with
    whitespace collapsed, so that editing a comment keeps the ncu records
    taken from the same code valid."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "split_kv_fd_gb300", "csrc")
    for f in KERNEL_SOURCES[kernel]:
        with open(os.path.join(csrc, f), encoding="utf-8") as fh:
            src = fh.read()
        src = re.sub(r"/\*.*?\*/", " ", src, flags=re.S)
        src = re.sub(r"//[^\n]*", " ", src)
        h.update(" ".join(src.split()).encode())
    return h.hexdigest()[:16]


# groups of at least this many query heads per K/V head run the tcgen05
# kernel (contiguous 16-bit K/V, head dim 64 or 128)
GQA_TC_MIN_G = 17


def kernel_key(w, fp8: bool, paged: bool, page_size: int = 0) -> str:
    """Which kernel does the timed work: split_kernel, gqa_kernel,
    gqa_tc_kernel or gqa_tc8_kernel."""
    if w.kv_heads == w.H:
        return "split_kernel"
    if not fp8 and not paged and w.d <= 128 and w.H // w.kv_heads >= GQA_TC_MIN_G:
        return "gqa_tc_kernel"
    if fp8 and w.d == 128 and (not paged or page_size % 128 == 0):
        return "gqa_tc8_kernel"
    return "gqa_kernel"


def kernel_name(w, fp8: bool, paged: bool, page_size: int = 0) -> str:
    """The kernel that does the timed work, as ncu names it."""
    key = kernel_key(w, fp8, paged, page_size)
    elt = "e4m3" if fp8 else w.dtype
    return f"fd::{key}<{elt}, {w.d}>" + (" (paged)" if paged else "")


def profiled_traffic(workload: str, kernel: str = "split_kernel"):
    """DRAM bytes per launch from the committed ncu summary of `kernel`, if
    it was taken from the kernel's current sources on this workload; else
    None."""
    p = os.path.join(ROOT, "profiles", f"{kernel}_traffic.json")
    if not os.path.exists(p):
        return None
    try:
        with open(p) as f:
            rec = json.load(f)
        ent = rec.get(workload)
        if ent and ent.get("kernel_source_hash") == kernel_source_hash(kernel):
            return ent.get("dram_bytes_per_launch")
    except Exception:
        return None
    return None


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms."""
    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.t0 = self.t1 = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, FileNotFoundError):
            self.proc = None

    def mark(self, which):
        setattr(self, which, time.time())

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        rows = []
        for line in out.strip().splitlines():
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 10:
                continue
            try:
                ts = time.mktime(time.strptime(parts[0].split(".")[0], "%Y/%m/%d %H:%M:%S"))
                rows.append(dict(ts=ts, sm=float(parts[2]), smax=float(parts[3]),
                                 hw=parts[6], hwt=parts[7], swt=parts[8], pcap=parts[9]))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        win = [r for r in rows if self.t0 is not None and self.t0 - 1 <= r["ts"] <= self.t1 + 1]
        window = "timed"
        if not win:
            win, window = rows, "warmup+timed"
        reasons = set()
        for r in win:
            for key, name in (("hw", "hw_slowdown"), ("hwt", "hw_thermal_slowdown"),
                              ("swt", "sw_thermal_slowdown"), ("pcap", "sw_power_cap")):
                if r[key].lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(r["sm"] for r in win),
                "sm_max_mhz": max(r["smax"] for r in win), "reasons": sorted(reasons),
                "samples": len(win), "window": window}


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def reduce_max(x: float, ws: int, device) -> float:
    if ws == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(ws: int):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


# ------------------------------------------------------------ oracle timing

def host_sample(w, rows: int, q=None, k=None, v=None, lens=None, seed=1):
    """``rows`` (b, K/V head) rows of the workload as host tensors.

    Each row is one sequence with one K/V head and its G query heads:
    q [rows, G, d], K/V [rows, 1, n, d] (G = 1 unless grouped-query).  Taken
    from the device tensors when given (the exact workload bytes), else drawn
    on the CPU with the workload's distributions."""
    G = w.H // w.kv_heads
    if k is not None:
        lens_h = lens.cpu().tolist()
        pairs = [(i // w.kv_heads % w.B, i % w.kv_heads) for i in range(rows)]
        n = max(lens_h[b] for b, _ in pairs)
        qs = torch.stack([q[b, h * G:(h + 1) * G] for b, h in pairs]).cpu()
        ks = torch.stack([k[b, h, :n] for b, h in pairs]).unsqueeze(1).cpu()
        vs = torch.stack([v[b, h, :n] for b, h in pairs]).unsqueeze(1).cpu()
        ls = torch.tensor([lens_h[b] for b, _ in pairs], dtype=torch.int32)
        return qs, ks, vs, ls
    from split_kv_fd_gb300.inputs import TORCH_DTYPES, random_case
    if w.ragged:
        g = torch.Generator().manual_seed(w.seed)
        lens_l = torch.randint(1, w.N + 1, (rows,), generator=g).tolist()
    else:
        lens_l = [w.N] * rows
    qs, ks, vs, ls = random_case(rows, 1, max(lens_l), w.d, w.dtype, lens=lens_l, seed=seed,
                                 k_scale=w.k_scale)
    if G > 1:
        g = torch.Generator().manual_seed(seed + 1)
        qs = torch.randn(rows, G, w.d, generator=g).to(TORCH_DTYPES[w.dtype])
    return qs, ks, vs, ls


def time_oracle(w, sample, nthreads):
    import oracle
    qs, ks, vs, ls = sample
    t0 = time.perf_counter()
    if qs.shape[1] != ks.shape[1]:
        oracle.attention_gqa(qs, ks, vs, lens=ls, scale=w.scale, nthreads=nthreads)
    else:
        oracle.attention(qs, ks, vs, lens=ls, scale=w.scale, nthreads=nthreads)
    return time.perf_counter() - t0


def sample_bytes(w, ls) -> int:
    return 2 * w.d * ELEMENT_BYTES[w.dtype] * int(ls.sum())


def cpu_baseline(w, q, k, v, lens, budget_s=8.0):
    """Oracle on a bounded sample: grow the sample until ~budget_s of wall time."""
    import oracle
    oracle.build()
    cores = oracle.default_threads()
    rows = cores
    total = w.B * w.kv_heads
    while True:
        sample = host_sample(w, min(rows, total), q, k, v, lens)
        dt = time_oracle(w, sample, cores)
        if dt * 2 > budget_s or rows >= total:
            break
        rows = min(total, max(rows * 2, int(rows * budget_s / max(dt, 1e-3) * 0.8)))
    nb = sample_bytes(w, sample[3])
    return {"value": nb / dt / 1e9, "unit": "GB/s", "cores": cores, "kind": "oracle",
            "sample": f"{sample[0].shape[0]} of {total} (b, kv head) rows of {w.name}, full length "
                      f"({int(sample[3].sum())} tokens), float64 C oracle, {cores} threads, "
                      f"{dt:.2f} s wall"}


# --------------------------------------------------------------- the arms

def run_reference(args, w):
    ws, rank, _ = dist_env()
    if rank != 0:
        return 0
    import oracle
    oracle.build()
    cores = oracle.default_threads()
    rows = max(1, min(cores, w.B * w.kv_heads))
    sample = host_sample(w, rows)
    for _ in range(args.warmup):
        time_oracle(w, sample, cores)
    times = [time_oracle(w, sample, cores) for _ in range(args.steps)]
    nb = sample_bytes(w, sample[3])
    total = sum(times)
    value = nb * args.steps / total / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": total / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": config_of(w, w.num_splits or "auto", args.page_size, args.kv_dtype),
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": cores, "kind": "oracle",
                         "sample": f"each step: {rows} of {w.B * w.kv_heads} (b, kv head) rows of {w.name}, "
                                   f"full length, drawn on the host with the workload's "
                                   f"distributions; float64 C oracle, {cores} threads"},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def config_of(w, num_splits, page_size=0, kv_dtype="native", path="fused"):
    return {"workload": w.name, "path": path, "batch": w.B, "heads": w.H, "kv_heads": w.kv_heads,
            "kv_len": w.N, "head_dim": w.d,
            "kv_dtype": (w.dtype if kv_dtype == "native"
                         else f"e4m3 with per-(b,h) scales (q {w.dtype})"),
            "out_dtype": w.out_dtype, "num_splits": num_splits,
            "kv_layout": (f"paged, {page_size}-token pages in shuffled order" if page_size
                          else "contiguous [B,H,N,d]"),
            "lengths": "uniform[1,N] seeded" if w.ragged else "all N",
            "k_scale": w.k_scale,
            "l2": ("inputs larger than L2, no flush"
                   if 2 * w.B * w.kv_heads * w.N * w.d * ELEMENT_BYTES[w.dtype] > 4 * L2_BYTES
                   else "L2 flushed before every step (256 MiB write, then 256 MiB read), "
                        "outside the steps' CUDA events")}


# the workloads the >= 80 %-of-HBM gate covers (uniform 32K, one 128K
# sequence with peaked scores, ragged 16 x 32); the first is the headline
GATED = ["decode_b8_h32_n32k_d128_bf16", "decode_b1_h32_n128k_d128_bf16_k8",
         "decode_ragged_b16_h32_n64k_d128_bf16"]


def check_device_status(fd):
    """A timed run counts only if no kernel gave up a bounded wait in it."""
    st = fd.device_status()
    if st != 0:
        raise SystemExit(f"bench: a kernel reported device status {st} during the timed steps")


def time_gated(fd, name, steps, warmup, dev, ws, peaks):
    """One gated workload through the fused call (automatic decomposition),
    timed like the headline: `steps` launches, each inside its own CUDA
    events on the launching stream, after `warmup` untimed ones.  The ragged
    workload also times the two-call form with both merges (split kernel +
    combine per step).  Inputs are larger than L2, so no flush is needed."""
    from split_kv_fd_gb300.inputs import make_inputs
    w = WORKLOADS[name]
    q, k, v, lens = make_inputs(w, device=dev)
    lens_h = lens.cpu().tolist()
    out = torch.empty((w.B, w.H, w.d), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((w.B, w.H), dtype=torch.float32, device=dev)
    wsbuf = fd.new_workspace(w.B, w.H, w.N, w.d, 0, device=dev)
    stream = torch.cuda.current_stream(dev)
    kvb = kv_bytes(w, lens_h)
    alg = algorithmic_bytes(w, lens_h)

    def timed(fn):
        for _ in range(max(3, warmup)):
            fn()
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(steps)]
        barrier(ws)
        torch.cuda.synchronize(dev)
        for a, b in evs:
            a.record(stream)
            fn()
            b.record(stream)
        torch.cuda.synchronize(dev)
        barrier(ws)
        ms = [a.elapsed_time(b) for a, b in evs]
        return reduce_max(sum(ms), ws, dev) / steps, statistics.mean(ms)

    step_ms, launch_ms = timed(lambda: fd.decode(q, k, v, lens, scale=w.scale, out=out, lse=lse,
                                                 workspace=wsbuf, stream=stream))
    check_device_status(fd)
    ent = {"value": ws * kvb / (step_ms * 1e-3) / 1e9, "unit": "GB/s", "ms_per_step": step_ms,
           "pct_of_nominal_8tbs": 100.0 * kvb / (step_ms * 1e-3) / 1e9 / NOMINAL_HBM_GBS,
           "roofline": {"frac": alg / (launch_ms * 1e-3) / 1e9 / peaks["hbm_gbs"],
                        "achieved": alg / (launch_ms * 1e-3) / 1e9,
                        "traffic": profiled_traffic(w.name, "split_kernel")},
           "mean_launch_ms": launch_ms, "gpu_launches": steps}
    if w.ragged:
        P = fd.auto_num_splits(w.B, w.H, w.N, w.d)
        parts = fd.decode_split(q, k, v, P, seqlens=lens, scale=w.scale, stream=stream)
        o_p, m_p, l_p, s_p = parts
        for path, comb in (("split-mlo", lambda: fd.combine_mlo(o_p, m_p, l_p, out=out, lse=lse,
                                                                stream=stream)),
                           ("split-lse", lambda: fd.combine_lse(o_p, s_p, out=out, lse=lse,
                                                                stream=stream))):
            def two_call(comb=comb):
                fd.decode_split(q, k, v, P, seqlens=lens, scale=w.scale, stream=stream,
                                o_part=o_p, m_part=m_p, l_part=l_p, lse_part=s_p)
                comb()
            sm, _ = timed(two_call)
            ent[path] = {"value": ws * kvb / (sm * 1e-3) / 1e9, "ms_per_step": sm,
                         "num_splits": P, "gpu_launches": 2 * steps}
        del parts, o_p, m_p, l_p, s_p
    del q, k, v, lens, wsbuf
    torch.cuda.synchronize(dev)
    torch.cuda.empty_cache()
    return ent


def run_ours(args, w):
    ws, rank, local = dist_env()
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    import split_kv_fd_gb300 as fd
    from split_kv_fd_gb300.inputs import make_inputs
    from split_kv_fd_gb300.workloads import ELEMENT_BYTES as EB
    fd.load(build_if_missing=True)

    q, k, v, lens = make_inputs(w, device=dev)
    lens_h = lens.cpu().tolist()
    table = None
    k_scale = v_scale = None
    if args.kv_dtype == "e4m3":
        from split_kv_fd_gb300.inputs import quantize_e4m3
        k, k_scale = quantize_e4m3(k)
        v, v_scale = quantize_e4m3(v)
        torch.cuda.empty_cache()
    if args.page_size and k_scale is not None:
        from split_kv_fd_gb300.inputs import to_paged_bytes
        k, table = to_paged_bytes(k, args.page_size, seed=w.seed)
        v, _ = to_paged_bytes(v, args.page_size, seed=w.seed)
        torch.cuda.empty_cache()
    elif args.page_size:
        from split_kv_fd_gb300.inputs import to_paged
        k, v, table = to_paged(k, v, args.page_size, seed=w.seed)
        torch.cuda.empty_cache()

    # the two-call form: fd_decode_split then a combine, with its own split count
    P_split = 0
    if args.path != "fused":
        P_split = args.num_splits or w.num_splits or fd.auto_num_splits(w.B, w.H, w.N, w.d)
    # fused: the workload's split count, else the automatic decomposition (0)
    P_fused = args.num_splits or w.num_splits

    def decode(out, lse, stream, mid=None):
        if args.path != "fused":
            o_p, m_p, l_p, s_p = fd.decode_split(q, k, v, P_split, seqlens=lens, scale=w.scale,
                                                 stream=stream)
            if mid is not None:
                mid.record(stream)
            if args.path == "split-mlo":
                fd.combine_mlo(o_p, m_p, l_p, out=out, lse=lse, stream=stream)
            else:
                fd.combine_lse(o_p, s_p, out=out, lse=lse, stream=stream)
            return
        if w.kv_heads != w.H and k_scale is not None and table is not None:
            fd.decode_gqa_paged_fp8(q, k, v, k_scale, v_scale, table, lens, num_splits=P_fused, scale=w.scale,
                                    out=out, lse=lse, workspace=wsbuf, stream=stream)
        elif w.kv_heads != w.H and k_scale is not None:
            fd.decode_gqa_fp8(q, k, v, k_scale, v_scale, seqlens=lens, num_splits=P_fused, scale=w.scale,
                              out=out, lse=lse, workspace=wsbuf, stream=stream)
        elif w.kv_heads != w.H and table is None:
            fd.decode_gqa(q, k, v, lens, num_splits=P_fused, scale=w.scale, out=out, lse=lse,
                          workspace=wsbuf, stream=stream)
        elif w.kv_heads != w.H:
            fd.decode_gqa_paged(q, k, v, table, lens, num_splits=P_fused, scale=w.scale, out=out,
                                lse=lse, workspace=wsbuf, stream=stream)
        elif k_scale is not None:
            fd.decode_fp8(q, k, v, k_scale, v_scale, seqlens=lens, num_splits=P_fused, scale=w.scale,
                          out=out, lse=lse, workspace=wsbuf, stream=stream)
        elif table is None:
            fd.decode(q, k, v, lens, num_splits=P_fused, scale=w.scale, out=out, lse=lse,
                      workspace=wsbuf, stream=stream)
        else:
            fd.decode_paged(q, k, v, table, lens, num_splits=P_fused, scale=w.scale, out=out, lse=lse,
                            workspace=wsbuf, stream=stream)
    out = torch.empty((w.B, w.H, w.d), dtype=getattr(torch, {"bf16": "bfloat16", "f16": "float16",
                                                            "f32": "float32"}[w.out_dtype]),
                      device=dev)
    lse = torch.empty((w.B, w.H), dtype=torch.float32, device=dev)
    if w.kv_heads != w.H:
        wsbuf = torch.empty(max(256, fd.workspace_size_gqa(w.B, w.H, w.kv_heads, w.N, w.d, P_fused)),
                            dtype=torch.uint8, device=dev)
    else:
        wsbuf = fd.new_workspace(w.B, w.H, w.N, w.d, P_fused, device=dev)
    stream = torch.cuda.current_stream(dev)
    flush = None
    if 2 * w.B * w.kv_heads * w.N * w.d * EB[w.dtype] <= 4 * L2_BYTES:
        # write one buffer larger than L2, then read another, so that L2
        # holds none of the inputs and no dirty lines left to write back
        flush = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device=dev)
        flush_rd = torch.ones(64 * 1024 * 1024, dtype=torch.int32, device=dev)
        flush_sink = torch.empty((), dtype=torch.int64, device=dev)

    def do_flush():
        flush.fill_(1)
        torch.sum(flush_rd, dim=0, out=flush_sink)

    def step():
        if flush is not None:
            do_flush()
        decode(out, lse, stream)

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize(dev)

    sampler = ClockSampler(dev.index if dev.index is not None else 0)
    sampler.start()
    time.sleep(0.25)  # the sampler's first row
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.steps)]
    mids = [torch.cuda.Event(enable_timing=True) if args.path != "fused" else None
            for _ in range(args.steps)]
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    barrier(ws)
    torch.cuda.synchronize(dev)
    sampler.mark("t0")
    t_start.record(stream)
    for i in range(args.steps):
        if flush is not None:
            do_flush()
        evs[i][0].record(stream)
        decode(out, lse, stream, mids[i])
        evs[i][1].record(stream)
    t_end.record(stream)
    torch.cuda.synchronize(dev)
    # the other gated workloads, measured the same way in the same process
    # (inside the clock sampler's window)
    gated = None
    if (w.name == GATED[0] and args.path == "fused" and not args.page_size
            and args.kv_dtype == "native" and not args.num_splits and not args.no_gated):
        gated = {}
        for name in GATED[1:]:
            gated[name] = time_gated(fd, name, args.steps, args.warmup, dev, ws, measured_peaks()[0])
    sampler.mark("t1")
    barrier(ws)
    clocks = sampler.stop()
    check_device_status(fd)
    total_ms = t_start.elapsed_time(t_end)
    launch_ms = [a.elapsed_time(b) for a, b in evs]
    combine_ms = None
    if args.path != "fused":
        # the dominant kernel is the split kernel; the combine is timed apart
        combine_ms = statistics.mean(m.elapsed_time(b) for m, (_, b) in zip(mids, evs))
        split_ms = [a.elapsed_time(m) for m, (a, _) in zip(mids, evs)]
    if flush is not None:
        # the flush runs between the steps, outside their events: a step's
        # time is its own events' interval
        total_ms = sum(launch_ms)
    total_ms = reduce_max(total_ms, ws, dev)
    kern_ms = statistics.mean(launch_ms if args.path == "fused" else split_ms)

    kvb = kv_bytes(w, lens_h)
    if k_scale is not None:  # one byte per element, plus the scales
        kvb = kvb // ELEMENT_BYTES[w.dtype]
    ms_per_step = total_ms / args.steps
    value = ws * kvb / (ms_per_step * 1e-3) / 1e9
    peaks, peak_src = measured_peaks()
    alg = algorithmic_bytes(w, lens_h)
    if k_scale is not None:  # one byte per element, plus the K and V scales of each (b, K/V head)
        alg = alg - kv_bytes(w, lens_h) + kvb + 8 * w.B * w.kv_heads
    if table is not None:  # the block-table entries of the valid pages, read once
        alg += 4 * sum(-(-int(n) // args.page_size) for n in lens_h)
    if args.path != "fused":
        # the split kernel also writes the partials: P (d + 3) floats per (b, h)
        alg += 4 * w.B * w.H * P_split * (w.d + 3) - w.B * w.H * (w.d * ELEMENT_BYTES[w.out_dtype] + 4)
    achieved = alg / (kern_ms * 1e-3) / 1e9
    tokens = sum(lens_h) * w.H

    # end to end from pinned host buffers through the public API
    e2e = None
    if not args.no_e2e:
        hq = q.cpu().pin_memory()
        hk = k.cpu().pin_memory()
        hv = v.cpu().pin_memory()
        hl = lens.cpu().pin_memory()
        ht = table.cpu().pin_memory() if table is not None else None
        hks = k_scale.cpu().pin_memory() if k_scale is not None else None
        hvs = v_scale.cpu().pin_memory() if v_scale is not None else None
        hout = torch.empty(out.shape, dtype=out.dtype).pin_memory()
        hlse = torch.empty(lse.shape, dtype=lse.dtype).pin_memory()
        e2e_steps = max(1, min(args.steps, args.e2e_steps))

        def e2e_step():
            q.copy_(hq, non_blocking=True)
            k.copy_(hk, non_blocking=True)
            v.copy_(hv, non_blocking=True)
            lens.copy_(hl, non_blocking=True)
            if table is not None:
                table.copy_(ht, non_blocking=True)
            if k_scale is not None:
                k_scale.copy_(hks, non_blocking=True)
                v_scale.copy_(hvs, non_blocking=True)
            decode(out, lse, stream)
            hout.copy_(out, non_blocking=True)
            hlse.copy_(lse, non_blocking=True)

        e2e_step()
        torch.cuda.synchronize(dev)
        barrier(ws)
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(e2e_steps):
            e2e_step()
        b.record(stream)
        torch.cuda.synchronize(dev)
        e_ms = reduce_max(a.elapsed_time(b), ws, dev) / e2e_steps
        h2d = sum(t.numel() * t.element_size() for t in (hq, hk, hv, hl, ht, hks, hvs)
                  if t is not None)
        d2h = hout.numel() * hout.element_size() + hlse.numel() * hlse.element_size()
        e2e = {"value": ws * kvb / (e_ms * 1e-3) / 1e9, "unit": "GB/s", "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "steps": e2e_steps, "ms_per_step": e_ms}
        del hq, hk, hv

    cpu = None
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        if table is None and k_scale is None:
            cpu = cpu_baseline(w, q, k, v, lens)
        else:  # the oracle on host-drawn rows of the same workload in its native dtype
            cpu = cpu_baseline(w, None, None, None, None)
            cpu["sample"] += " (native-dtype contiguous rows drawn on the host)"

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None,
            "dtype": "e4m3" if k_scale is not None else w.dtype, "accumulate": "f32",
            "data": "synthetic",
            "config": config_of(w, (P_fused or "auto") if args.path == "fused" else P_split,
                                args.page_size, args.kv_dtype, args.path),
            "tokens_per_s": ws * tokens / (ms_per_step * 1e-3),
            "pct_of_nominal_8tbs": 100.0 * value / ws / NOMINAL_HBM_GBS,
            "pct_of_measured_hbm": 100.0 * value / ws / peaks["hbm_gbs"],
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"],
                         "unit": "GB/s", "frac": achieved / peaks["hbm_gbs"],
                         "traffic": (None if table is not None
                                     else profiled_traffic(w.name + ("+e4m3" if k_scale is not None
                                                                     else ""),
                                                           kernel_key(w, k_scale is not None,
                                                                      table is not None, args.page_size))),
                         "kernel": kernel_name(w, k_scale is not None, table is not None, args.page_size),
                         "peak_source": f"{peak_src} (hbm_gbs, STREAM-style copy)",
                         "algorithmic_bytes_per_launch": alg, "mean_launch_ms": kern_ms},
            "e2e": e2e,
            "gpu_launches": args.steps * (1 if args.path == "fused" else 2),
            "clocks": clocks,
            "cpu_baseline": cpu,
        }
        if combine_ms is not None:
            line["combine_ms"] = combine_ms
        if gated is not None:
            line["configs"] = {w.name: {
                "value": value, "unit": "GB/s", "ms_per_step": ms_per_step,
                "pct_of_nominal_8tbs": 100.0 * value / ws / NOMINAL_HBM_GBS,
                "roofline": {k_: line["roofline"][k_] for k_ in ("frac", "achieved", "traffic")},
                "mean_launch_ms": kern_ms, "gpu_launches": args.steps}}
            line["configs"].update(gated)
            line["gpu_launches"] += sum(e["gpu_launches"] + sum(e[p]["gpu_launches"]
                                                                for p in ("split-mlo", "split-lse")
                                                                if p in e)
                                        for e in gated.values())
        print(json.dumps(line), flush=True)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=BENCH_DEFAULT, choices=sorted(WORKLOADS))
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--kv-dtype", choices=["native", "e4m3"], default="native",
                    help="e4m3: store K/V in FP8 with per-(b,h) scales and time fd_decode_fp8")
    ap.add_argument("--num-splits", type=int, default=0,
                    help="split count (0: the workload's own, else the automatic decomposition)")
    ap.add_argument("--path", choices=["fused", "split-mlo", "split-lse"], default="fused",
                    help="fused fd_decode, or fd_decode_split then fd_combine_mlo / fd_combine_lse")
    ap.add_argument("--page-size", type=int, default=0,
                    help="time fd_decode_paged (fd_decode_gqa_paged for a GQA workload) on the "
                         "workload laid out in pages of this many tokens")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-gated", action="store_true",
                    help="time only the chosen workload, not the other two workloads of the "
                         "bandwidth gate")
    args = ap.parse_args(argv)
    w = WORKLOADS[args.workload]
    if args.path != "fused" and (args.page_size or args.kv_dtype != "native" or w.kv_heads != w.H):
        ap.error("--path split-* times the contiguous, native-dtype, one-query-per-K/V-head path")
    if args.kv_dtype != "native" and args.page_size and w.kv_heads == w.H:
        ap.error("--kv-dtype e4m3 with --page-size times the paged E4M3 grouped-query path")
    ws, _, _ = dist_env()
    if args.gpus > 1 and ws == 1 and "LOCAL_RANK" not in os.environ:
        # launch the per-GPU ranks ourselves
        cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1",
               f"--nproc-per-node={args.gpus}", "--master-addr", "127.0.0.1",
               "--master-port", os.environ.get("MASTER_PORT", "29511"),
               os.path.abspath(__file__), *(argv if argv is not None else sys.argv[1:])]
        return subprocess.call(cmd)
    if args.impl == "reference":
        return run_reference(args, w)
    return run_ours(args, w)


if __name__ == "__main__":
    sys.exit(main())
