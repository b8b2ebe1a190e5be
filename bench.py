"""Benchmark of the sparse MXFP4 decode step on GB300.

python bench.py [--gpus N] [--steps K] [--warmup W] [--impl smx|reference] [--config 5]

One step = the whole hot path (insert, q pack, index score of every page, top-k, split-K
attention, merge). The headline workload (--config, default 5) is the largest case of the sweep:
B = 4 rows x Q = 8 query tokens, 16 query heads on 1 KV head, ragged contexts up to 262144 tokens
(1158 to 1695 pages), top-k 128 pages. The metric is achieved HBM GB/s of the algorithmic bytes
(every index page of each row + the K and V pages of the selected set) per step; microseconds per
step are reported too. The same line carries `per_config`: the fixed 7-draft verify (2), FP8-KV
(3) and long-context (4) workloads and the verify workload with NVFP4 K/V and index pages (nv2,
six launches a step), each timed the same way. `--stage index` times the index scorer alone,
`--reuse` the step of a layer that reuses a selection.

The timed K steps are replayed from one CUDA graph; every step reads a different copy of the
three page pools, with enough copies that their bytes exceed 3x the L2 cache, so each step reads
from HBM. N > 1 (torchrun) runs N independent replicas (the path has no exchange step); value is
the bytes of all ranks over the slowest rank's time.

The reference arm (--impl reference) is the CPU oracle timed on this host's cores on a bounded
sample of the same workload (one batch row per step).
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

import numpy as np  # noqa: E402
import torch  # noqa: E402

from sparse_attention_decode_mxfp4_gb300 import workloads as wl  # noqa: E402

METRIC = "sparse MXFP4 decode step: µs/step and achieved HBM GB/s vs GB300 peak"
METRIC_REUSE = ("sparse MXFP4 decode step of a layer reusing an earlier layer's selection: µs/step and "
                "achieved HBM GB/s vs GB300 peak")


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="smx", choices=["smx", "reference"])
    ap.add_argument("--config", type=int, default=5)
    ap.add_argument("--per-config", default="2,3,4,nv2",
                    help="other workloads timed in the same run, reported under per_config ('' for none; "
                         "nvN: config N with NVFP4 K/V and index pages)")
    ap.add_argument("--splits", type=int, default=0,
                    help="partitions of the split stage (0 = about two CTAs per SM, at most one page each)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=100)
    ap.add_argument("--reuse", action="store_true",
                    help="time the step of a layer that reuses one full step's selection (K/V insert, "
                         "split and merge; no index scoring or selection); bytes = the selected K/V pages")
    ap.add_argument("--stage", default="step", choices=["step", "index"],
                    help="index: time the index scorer alone (smx_index_score over the workload's index "
                         "pages, rotating copies of the index pool); bytes = the index pages read")
    return ap.parse_args()


def algorithmic_bytes(w, ctx_len):
    n_pages = [(int(c) + 127) // 128 for c in ctx_len]
    idx = sum(n * w.idx_page_bytes for n in n_pages)
    kv = sum(min(w.topk, n) * 2 * w.Hkv * w.kv_page_bytes for n in n_pages)
    return idx, kv


def default_splits(w):
    """Partitions of the split stage, as the library suggests for this device: one wave of split
    CTAs, the same number of selected pages in every partition."""
    from sparse_attention_decode_mxfp4_gb300 import ops
    return ops.suggest_num_splits(ops.Shape.of(w, 1))


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def kernel_sources_sha():
    h = hashlib.sha256()
    for f in ("smx_step.cu", "smx_attend.cuh", "smx_attend_tc.cuh", "smx_tc.cuh", "smx_scan.cuh",
              "smx_select.cuh", "smx_device.cuh"):
        h.update(open(os.path.join(ROOT, "sparse_attention_decode_mxfp4_gb300", "csrc", f), "rb").read())
    return h.hexdigest()[:16]


def recorded_traffic(workload_name, reuse=False):
    """DRAM bytes per launch of the decode-step kernel (reuse: its reusing-layer variant) on this
    workload from a committed ncu summary (one record per workload), if it was taken on the current
    kernel source; else None."""
    p = os.path.join(ROOT, "profiles", "decode_step_reuse_traffic.json" if reuse else "decode_step_traffic.json")
    if not os.path.exists(p):
        return None
    try:
        d = json.load(open(p))
    except Exception:
        return None
    if d.get("kernel_sources_sha") != kernel_sources_sha():
        return None
    for r in d.get("records", [d]):
        if r.get("workload") == workload_name:
            return r.get("dram_bytes_per_launch")
    return None


def slowest_rank(x, device):
    """The largest x over the ranks of the process group (the slowest rank's time), x itself with
    no group or one rank. Any backend (NCCL on the GPUs, gloo in the host tests)."""
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_gbs(step_bytes, world, steps, seconds):
    """Every rank's step bytes over the slowest rank's time, GB/s (the replicas' aggregate)."""
    return step_bytes * world * steps / seconds / 1e9


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms during the timed region."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index):
        self.proc = None
        self.path = None
        vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
        self.gpu = vis.split(",")[device_index] if vis else str(device_index)

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                          "-lms", "200", "-i", self.gpu], stdout=open(self.path, "w"),
                                         stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        rows = []
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) >= 9:
                rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


# ------------------------------------------------------------------------------------------------
def run_reference(args):
    """The CPU oracle as it stands, one batch row of the workload per step, all host cores (with
    --reuse, the reusing layer's step over the oracle's own selection of that row)."""
    import oracle
    w = wl.config(args.config)
    data = wl.generate(w)
    rows = [wl.shrink(w, B=1, ctx_lens=(int(data["ctx_len"][b]),), name=w.name + f"_row{b}") for b in range(w.B)]
    samples = []
    for b, wb in enumerate(rows):
        db = {k: (v[b:b + 1] if isinstance(v, np.ndarray) and v.ndim >= 1 and v.shape[0] == w.B else v)
              for k, v in data.items()}
        db["page_table"] = np.arange(wb.max_pages, dtype=np.int32)[None]
        pools = wl.empty_pools(wb)
        sh = oracle.shape_of(wb)
        oracle.kv_fill(sh, db["k"], db["v"], db["kidx"], db["page_table"], db["n_hist"], *pools)
        samples.append([wb, sh, db, pools, None])
    idx_b, kv_b = algorithmic_bytes(w, data["ctx_len"])
    if args.reuse:
        idx_b = 0   # a reusing layer reads no index page
    per_row = (idx_b + kv_b) / w.B

    def full(sh, db, pools):
        return oracle.decode_step(sh, q_f32=db["q"], q_bf16=db["q_bf16"], qidx_bf16=db["qidx_bf16"],
                                  k_new=db["k_new"], v_new=db["v_new"], kidx_new=db["kidx_new"],
                                  page_table=db["page_table"], ctx_len=db["ctx_len"], k_pool=pools[0],
                                  v_pool=pools[1], idx_pool=pools[2])

    if args.reuse:
        for smp in samples:
            smp[4] = full(*smp[1:4])

    def one(i):
        wb, sh, db, pools, sel = samples[i % len(samples)]
        if sel is None:
            full(sh, db, pools)
        else:
            oracle.decode_step_reuse(sh, q_f32=db["q"], q_bf16=db["q_bf16"], k_new=db["k_new"], v_new=db["v_new"],
                                     page_table=db["page_table"], ctx_len=db["ctx_len"], k_pool=pools[0],
                                     v_pool=pools[1], topk_pages=sel["topk_pages"], topk_count=sel["topk_count"])

    for i in range(args.warmup):
        one(i)
    t0 = time.perf_counter()
    for i in range(args.steps):
        one(i)
    dt = time.perf_counter() - t0
    value = per_row * args.steps / dt / 1e9
    cores = oracle.max_threads()
    line = {
        "impl": "reference", "metric": METRIC_REUSE if args.reuse else METRIC, "value": value, "unit": "GB/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": dict(w.describe(), step="reusing layer" if args.reuse else "full",
                       sample="one batch row per step (rows cycled)",
                       parallelism="replicas" if args.gpus > 1 else "single"),
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": cores, "kind": "oracle",
                         "sample": "one batch row of the workload per step, rows cycled"},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def cpu_baseline(w, data, step_bytes, reuse=False):
    """Oracle on this host's cores: whole steps of the same workload, repeated for ~10 s (reuse:
    the reusing layer's step over the oracle's own selection)."""
    import oracle
    from oracle import shape_of
    pools = wl.empty_pools(w)
    sh = shape_of(w)
    oracle.kv_fill(sh, data["k"], data["v"], data["kidx"], data["page_table"], data["n_hist"], *pools)

    def full():
        return oracle.decode_step(sh, q_f32=data["q"], q_bf16=data["q_bf16"], qidx_bf16=data["qidx_bf16"],
                                  k_new=data["k_new"], v_new=data["v_new"], kidx_new=data["kidx_new"],
                                  page_table=data["page_table"], ctx_len=data["ctx_len"], k_pool=pools[0],
                                  v_pool=pools[1], idx_pool=pools[2])

    sel = full() if reuse else None

    def one():
        if reuse:
            oracle.decode_step_reuse(sh, q_f32=data["q"], q_bf16=data["q_bf16"], k_new=data["k_new"],
                                     v_new=data["v_new"], page_table=data["page_table"], ctx_len=data["ctx_len"],
                                     k_pool=pools[0], v_pool=pools[1], topk_pages=sel["topk_pages"],
                                     topk_count=sel["topk_count"])
        else:
            full()

    def timed(seconds, min_reps):
        reps, t0 = 0, time.perf_counter()
        while True:
            one()
            reps += 1
            dt = time.perf_counter() - t0
            if dt > seconds and reps >= min_reps:
                return reps, dt

    cores = oracle.max_threads()
    reps, dt = timed(10.0, 1)
    oracle.set_threads(1)        # the same steps on one core, a shorter sample
    try:
        reps1, dt1 = timed(4.0, 2)
    finally:
        oracle.set_threads(cores)
    return {"value": step_bytes * reps / dt / 1e9, "unit": "GB/s", "cores": cores,
            "kind": "oracle", "sample": f"{reps} whole {'reusing-layer ' if reuse else ''}steps of the workload "
                                       f"({dt:.1f} s) on {cores} threads; {reps1} more on one thread ({dt1:.1f} s)",
            "us_per_step": dt / reps * 1e6, "single_thread_us_per_step": dt1 / reps1 * 1e6}


class Prepared:
    """One workload on the device: pools prefilled by the library, R rotating copies (more than 3x
    L2 of bytes read per rotation), the step's inputs and outputs, and step(i) (one decode step over
    copy i mod R, through the binding of the C ABI)."""

    def __init__(self, w, args, dev, reuse=False):
        from sparse_attention_decode_mxfp4_gb300 import ops
        self.w = w
        self.shape = ops.Shape.of(w, args.splits or default_splits(w))
        self.data = data = wl.generate(w)
        idx_b, kv_b = algorithmic_bytes(w, data["ctx_len"])
        if reuse:
            idx_b = 0   # a reusing layer reads no index page
        self.idx_b, self.kv_b, self.step_bytes = idx_b, kv_b, idx_b + kv_b

        def T(a):
            return torch.from_numpy(np.ascontiguousarray(a)).to(dev)

        self.page_table, self.ctx_len = T(data["page_table"]), T(data["ctx_len"])
        base = tuple(torch.zeros(p.shape, dtype=torch.uint8, device=dev) for p in wl.empty_pools(w))
        ops.kv_prefill(self.shape, T(data["k"]), T(data["v"]), T(data["kidx"]), self.page_table, T(data["n_hist"]),
                       *base)
        torch.cuda.synchronize()
        self.l2 = torch.cuda.get_device_properties(dev).L2_cache_size
        self.pool_bytes = sum(p.numel() for p in base)
        self.R = R = max(2, math.ceil(3 * self.l2 / self.step_bytes))
        self.copies = [tuple(p.clone() for p in base) for _ in range(R)]
        del base
        self.inp = dict(q_f32=T(data["q"]) if w.kv_format != wl.KV_E4M3_ROWSCALE else None,
                        q_bf16=T(data["q_bf16"].view(np.int16)) if w.kv_format == wl.KV_E4M3_ROWSCALE else None,
                        qidx_bf16=T(data["qidx_bf16"].view(np.int16)), k_new=T(data["k_new"]),
                        v_new=T(data["v_new"]), kidx_new=T(data["kidx_new"]))
        self.out = torch.empty((w.B, w.Q, w.Hq, 128), dtype=torch.float32, device=dev)
        self.topk_pages = torch.empty((w.B, w.topk), dtype=torch.int32, device=dev)
        self.topk_count = torch.empty((w.B,), dtype=torch.int32, device=dev)
        self.workspace = ops.alloc_workspace(self.shape, dev)
        self.status = torch.zeros(1, dtype=torch.int32, device=dev)
        self.reuse = False
        if reuse:
            # an earlier layer's selection: one full step's output, then the reusing layer's step
            self.step(0)
            self.sel_pages, self.sel_count = self.topk_pages.clone(), self.topk_count.clone()
            del self.inp["qidx_bf16"], self.inp["kidx_new"]
            self.reuse = True

    def step(self, i, pt=None, cl=None, io=None, o=None):
        from sparse_attention_decode_mxfp4_gb300 import ops
        pt = self.page_table if pt is None else pt
        cl = self.ctx_len if cl is None else cl
        io = self.inp if io is None else io
        o = self.out if o is None else o
        kp, vp, ip = self.copies[i % self.R]
        if self.reuse:
            ops.decode_step_reuse(self.shape, **io, page_table=pt, ctx_len=cl, k_pool=kp, v_pool=vp,
                                  topk_pages=self.sel_pages, topk_count=self.sel_count, out=o,
                                  workspace=self.workspace, dev_status=self.status)
        else:
            ops.decode_step(self.shape, **io, page_table=pt, ctx_len=cl, k_pool=kp, v_pool=vp, idx_pool=ip,
                            topk_pages=self.topk_pages, topk_count=self.topk_count, out=o,
                            workspace=self.workspace, dev_status=self.status)

    def l2_note(self):
        return (f"rotating {self.R} pool copies ({self.R * self.pool_bytes / 1e6:.0f} MB, reads "
                f"{self.R * self.step_bytes / 1e6:.0f} MB per rotation > 3x L2 {self.l2 / 1e6:.0f} MB)")


def time_steps(prep, steps, warmup, world, dev, clocks=None):
    """Milliseconds of `steps` decode steps replayed from one CUDA graph (after a replayed graph of
    `warmup` steps), CUDA events on the replay stream, the slowest rank's; clocks sampled inside."""
    import torch.distributed as dist
    prep.step(0)
    torch.cuda.synchronize()
    s = torch.cuda.Stream(device=dev)
    s.wait_stream(torch.cuda.current_stream())
    g_warm, g_timed = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g_warm, stream=s):
            for i in range(max(3, warmup)):
                prep.step(i)
        with torch.cuda.graph(g_timed, stream=s):
            for i in range(steps):
                prep.step(i)
    torch.cuda.synchronize()
    g_warm.replay()
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    if clocks is not None:
        clocks.start()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    cur = torch.cuda.current_stream()
    e0.record(cur)
    g_timed.replay()
    e1.record(cur)
    e1.synchronize()
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1)
    clk = clocks.stop() if clocks is not None else None
    ms = slowest_rank(ms, dev)
    if world > 1:
        dist.barrier()
    assert prep.status.item() == 0, f"device status {prep.status.item()}"
    return ms, clk


def run_index_stage(args, world, dev, peak, peak_kind):
    """The index scorer (a3) alone on one workload: every index page of every row scored once per
    call, over rotating copies of the index pool (more than 3x L2 read per rotation), replayed from
    a CUDA graph and timed with CUDA events."""
    from sparse_attention_decode_mxfp4_gb300 import ops
    w = wl.config(args.config)
    shape = ops.Shape.of(w, 1)
    data = wl.generate(w)
    idx_b, _ = algorithmic_bytes(w, data["ctx_len"])

    def T(a):
        return torch.from_numpy(np.ascontiguousarray(a)).to(dev)

    base = tuple(torch.zeros(p.shape, dtype=torch.uint8, device=dev) for p in wl.empty_pools(w))
    pt, cl = T(data["page_table"]), T(data["ctx_len"])
    ops.kv_prefill(shape, T(data["k"]), T(data["v"]), T(data["kidx"]), pt, T(data["n_hist"]), *base)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    R = max(2, math.ceil(3 * l2 / idx_b))
    pools = [base[2].clone() for _ in range(R)]
    del base
    qidx = T(data["qidx_bf16"].view(np.int16))
    scores = torch.empty((w.B, w.max_pages), dtype=torch.float32, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    steps, warm = args.steps, max(3, args.warmup)
    s = torch.cuda.Stream(device=dev)
    s.wait_stream(torch.cuda.current_stream())
    g_warm, g = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g_warm, stream=s):
            for i in range(warm):
                ops.index_score(shape, qidx, pools[i % R], pt, cl, page_scores=scores, dev_status=status)
        with torch.cuda.graph(g, stream=s):
            for i in range(steps):
                ops.index_score(shape, qidx, pools[i % R], pt, cl, page_scores=scores, dev_status=status)
    torch.cuda.synchronize()
    g_warm.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    g.replay()
    e1.record()
    e1.synchronize()
    ms = e0.elapsed_time(e1)
    assert status.item() == 0, f"device status {status.item()}"
    us = ms * 1e3 / steps
    gbs = idx_b / (us * 1e-6) / 1e9
    print(json.dumps({
        "metric": "index scorer (a3) alone: us per call and achieved HBM GB/s vs GB300 peak", "value": gbs,
        "unit": "GB/s", "n_gpus": 1, "steps": steps, "warmup": warm, "us_per_call": us, "higher_is_better": True,
        "dtype": "f32", "data": "synthetic (seeded N(0,1) index-K rows quantised on the GPU)",
        "config": {"workload": w.name, "B": w.B, "Q": w.Q, "max_ctx": w.max_ctx, "index_bytes": idx_b,
                   "pages": int(idx_b // wl.MXFP4_PAGE_BYTES),
                   "l2": f"rotating {R} index pool copies ({R * idx_b / 1e6:.0f} MB read per rotation)"},
        "roofline": {"bound": "hbm", "kernel": "index_scan_kernel / index_score_mma_kernel", "achieved": gbs,
                     "peak": peak, "peak_kind": peak_kind, "unit": "GB/s", "frac": gbs / peak}}))


def main():
    args = parse()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        if rank == 0:
            run_reference(args)
        return
    import torch.distributed as dist
    from sparse_attention_decode_mxfp4_gb300 import build as smx_build
    from sparse_attention_decode_mxfp4_gb300 import ops

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)
    smx_build.build()
    peak, peak_kind = peaks()
    if args.stage == "index":
        if rank == 0:
            run_index_stage(args, world, dev, peak, peak_kind)
        return

    # ---- the other workloads first (their memory is freed before the headline one) ----
    per_config = {}
    for tok in [x.strip() for x in args.per_config.split(",") if x.strip()]:
        nv = tok.startswith("nv")
        n = int(tok[2:] if nv else tok)
        if n == args.config and not nv:
            continue
        w_n = wl.nvfp4_variant(wl.config(n)) if nv else wl.config(n)
        p = Prepared(w_n, args, dev, reuse=args.reuse)
        k = min(args.steps, 100)
        ms_n, _ = time_steps(p, k, max(3, args.warmup), world, dev)
        us_n = ms_n * 1e3 / k
        gbs = whole_job_gbs(p.step_bytes, world, k, ms_n * 1e-3)
        per_config[tok] = {"workload": p.w.name, "us_per_step": us_n, "value": gbs, "unit": "GB/s",
                              "roofline_frac": gbs / world / peak, "bytes_per_step": p.step_bytes,
                              "index_bytes": p.idx_b, "kv_bytes": p.kv_b, "num_splits": p.shape.num_splits,
                              "steps": k, "l2": p.l2_note(), "traffic": recorded_traffic(p.w.name, args.reuse),
                              "launches_per_step": ops.decode_step_launches(p.shape)}
        del p
        torch.cuda.empty_cache()

    prep = Prepared(wl.config(args.config), args, dev, reuse=args.reuse)
    w, shape, step_bytes = prep.w, prep.shape, prep.step_bytes
    clocks = ClockSampler(local)
    ms, clk = time_steps(prep, args.steps, args.warmup, world, dev, clocks)
    us_step = ms * 1e3 / args.steps
    value = whole_job_gbs(step_bytes, world, args.steps, ms * 1e-3)

    # ---- the dominant kernel: the step is one kernel (decode_step_kernel), timed above with CUDA
    # events on the replay stream; its algorithmic bytes per launch are the step's bytes
    launches_per_step = ops.decode_step_launches(shape)
    kernel_us = us_step / launches_per_step
    achieved = step_bytes / launches_per_step / (kernel_us * 1e-6) / 1e9

    # ---- end to end through the public API: pinned host inputs in, output back, every step ----
    # every input of a step in one pinned host buffer (256-byte aligned slices) with a device twin
    # of the same layout: one host->device copy per step, then one device->host copy of the output
    inp, out = prep.inp, prep.out
    srcs = {k: v for k, v in inp.items() if v is not None}
    srcs["page_table"], srcs["ctx_len"] = prep.page_table, prep.ctx_len
    offs, total = {}, 0
    for k, v in srcs.items():
        offs[k] = total
        total = (total + v.numel() * v.element_size() + 255) // 256 * 256
    host_buf = torch.empty(total, dtype=torch.uint8).pin_memory()

    def view(buf, k):
        v = srcs[k]
        return buf[offs[k]:offs[k] + v.numel() * v.element_size()].view(v.dtype).view(v.shape)

    for k, v in srcs.items():
        view(host_buf, k).copy_(v.cpu())
    # two device input buffers and two outputs, so a step's copies overlap its neighbours' work:
    # the serving loop's pipeline (inputs of step i + 1 in, and the output of step i - 1 out,
    # while step i runs); every step still copies its own inputs in and reads its result back
    dev_bufs = [torch.empty(total, dtype=torch.uint8, device=dev) for _ in range(2)]
    dev_ins = [{k: view(db, k) for k in srcs} for db in dev_bufs]
    io_e2es = [{k: (di[k] if v is not None else None) for k, v in inp.items()} for di in dev_ins]
    outs = [torch.empty_like(out) for _ in range(2)]
    host_outs = [torch.empty(out.shape, dtype=out.dtype).pin_memory() for _ in range(2)]
    h2d = sum(v.numel() * v.element_size() for v in srcs.values())
    d2h = host_outs[0].numel() * host_outs[0].element_size()
    s_in, s_out = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    s = torch.cuda.Stream(device=dev)

    def e2e_cycle(n):
        main = torch.cuda.current_stream()
        ev_in = [torch.cuda.Event() for _ in range(n)]
        ev_done = [torch.cuda.Event() for _ in range(n)]
        ev_out = [torch.cuda.Event() for _ in range(n)]
        s_in.wait_stream(main)
        s_out.wait_stream(main)
        for i in range(n):
            b = i % 2
            with torch.cuda.stream(s_in):
                if i >= 2:
                    s_in.wait_event(ev_done[i - 2])   # step i - 2 has read this input buffer
                dev_bufs[b].copy_(host_buf, non_blocking=True)
                ev_in[i].record(s_in)
            main.wait_event(ev_in[i])
            if i >= 2:
                main.wait_event(ev_out[i - 2])        # step i - 2's output has been read back
            prep.step(i, pt=dev_ins[b]["page_table"], cl=dev_ins[b]["ctx_len"], io=io_e2es[b], o=outs[b])
            ev_done[i].record(main)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev_done[i])
                host_outs[b].copy_(outs[b], non_blocking=True)
                ev_out[i].record(s_out)
        main.wait_stream(s_in)
        main.wait_stream(s_out)

    # captured once and replayed, as a serving loop would; pool copies rotate as in the timed
    # region; wall clock over whole replays
    n_e2e = max(prep.R, 2)
    with torch.cuda.stream(s):
        e2e_cycle(4)
    torch.cuda.synchronize()
    g_e2e = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g_e2e, stream=s):
            e2e_cycle(n_e2e)
    g_e2e.replay()
    torch.cuda.synchronize()
    reps = max(1, -(-args.e2e_steps // n_e2e))
    t0 = time.perf_counter()
    for _ in range(reps):
        g_e2e.replay()
    torch.cuda.synchronize()
    e2e_s = (time.perf_counter() - t0) / (reps * n_e2e)
    e2e_s = slowest_rank(e2e_s, dev)
    e2e_val = whole_job_gbs(step_bytes, world, 1, e2e_s)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(w, prep.data, step_bytes, reuse=args.reuse)

    if rank == 0:
        line = {
            "metric": METRIC_REUSE if args.reuse else METRIC, "value": value, "unit": "GB/s", "n_gpus": world,
            "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": us_step / 1e3, "us_per_step": us_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic (seeded N(0,1) rows quantised on the GPU; the benchmark workload's shapes)",
            "config": dict(w.describe(), step="reusing layer" if args.reuse else "full",
                           num_splits=shape.num_splits, bytes_per_step=step_bytes,
                           index_bytes=prep.idx_b, kv_bytes=prep.kv_b,
                           ctx_len=[int(x) for x in prep.data["ctx_len"]],
                           parallelism="replicas" if world > 1 else "single", l2=prep.l2_note()),
            "roofline": {"bound": "hbm", "kernel": "decode_step_kernel", "achieved": achieved, "peak": peak,
                         "peak_kind": peak_kind, "unit": "GB/s", "frac": achieved / peak,
                         "traffic": recorded_traffic(w.name, args.reuse), "us_per_launch": kernel_us,
                         "algorithmic_bytes_per_launch": step_bytes // launches_per_step},
            "per_config": per_config,
            "cpu_baseline": cpu,
            "e2e": {"value": e2e_val, "unit": "GB/s", "us_per_step": e2e_s * 1e6, "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h},
            "gpu_launches": ops.decode_step_launches(shape) * args.steps,
            "clocks": clk,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
