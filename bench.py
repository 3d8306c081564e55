"""Attention-forward throughput on GB300.

One step = one attention forward (the whole hot path: one kernel launch) over
the GQA long-context workload B=1, Hq=32, Hkv=4, Sq=Skv=8192, D=128, bf16,
causal, Q/K/V ~ N(0,1), scale = 1/sqrt(128).  Throughput is reported in
TFLOPS with 4*B*Hq*Sq*Skv*D FLOPs per step, halved for causal.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Under torchrun (N > 1) every rank runs an independent replica of the same
workload (the path has no exchange step); the value is the FLOPs of all
ranks over the slowest rank's time.  ``--impl reference`` times the fp64 CPU
oracle on the host cores instead (rank 0 only), a bounded sample per step.
"""
import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = ("attention fwd TFLOPS on 1 GB300 (causal-halved FLOPs) and % of "
          "dense bf16 peak")
UNIT = "TFLOPS"
FLUSH_BYTES = 256 << 20  # > 129 MB L2
# ex2.approx.ftz.f32 results per clock per SM, measured on GB300 with a
# probe kernel (one CTA per SM, dependent-free ex2 streams).
EX2_PER_CLK_PER_SM = 32
KERNEL_SOURCES = ["attention_attn_fwd_gb300/csrc/attn_fwd_kernel.cuh",
                  "attention_attn_fwd_gb300/csrc/sm103_ptx.cuh",
                  "attention_attn_fwd_gb300/csrc/attn_sync.cuh",
                  "attention_attn_fwd_gb300/csrc/fast_div.h"]
# DRAM bytes of one headline launch from an ncu capture (data file written
# from the capture's summary; see the .md of the same name for the command).
TRAFFIC_PROFILE = os.path.join(ROOT, "profiles",
                               "attn_fwd_sm103_gqa8k_traffic.json")


def kernel_source_hash():
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def measured_traffic():
    """(DRAM bytes per launch, source label) from the committed ncu capture
    data, or (None, reason) when it is missing or the kernel source changed
    since the capture (the counters then describe another kernel)."""
    try:
        with open(TRAFFIC_PROFILE) as f:
            d = json.load(f)
        h, nbytes = str(d["kernel_source_hash"]), int(d["dram_bytes_per_launch"])
    except (OSError, KeyError, ValueError, TypeError):
        return None, "no capture data"
    if h != kernel_source_hash():
        return None, "capture of kernel source %s, not the current %s" % (
            h, kernel_source_hash())
    return nbytes, "ncu capture (dram__bytes_read.sum + dram__bytes_write.sum)" \
        " of kernel source %s" % h


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["bf16_tflops"]), float(p["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return 1900.0, 6800.0, "fallback"


class ClockSampler:
    """nvidia-smi samples every 100 ms while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,"
              "clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index):
        self.dev = device_index
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.dev),
                 "--query-gpu=" + self.FIELDS, "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=open(self.path, "w"),
                stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if self.proc is None or not self.path:
            return {"sm_mhz": None, "sm_max_mhz": None,
                    "reasons": ["nvidia-smi unavailable"]}
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown",
                 "sw_power_cap"]
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax = float(parts[2])
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        os.unlink(self.path)
        # Median over the busier half of the samples (the kernel runs).
        busy = sorted(sm)[len(sm) // 2:] if sm else []
        return {"sm_mhz": statistics.median(busy) if busy else None,
                "sm_max_mhz": smax, "reasons": sorted(reasons),
                "samples": len(sm)}


def exp2_roofline(w, ms, clocks, sms):
    """One exp2 per visible score: achieved rate against the SFU peak at the
    SM clock sampled during the timed region."""
    n = w.visible_pairs()
    mhz = clocks.get("sm_mhz") or clocks.get("sm_max_mhz")
    if not mhz or not sms:
        return {"exp2_per_step": n, "frac": None}
    peak = EX2_PER_CLK_PER_SM * sms * mhz * 1e6
    rate = n / (ms * 1e-3)
    return {"exp2_per_step": n, "achieved_per_s": round(rate, 0),
            "peak_per_s": round(peak, 0), "frac": round(rate / peak, 4),
            "peak_source": "%d ex2/clk/SM (measured) x %d SMs x %.0f MHz"
                           % (EX2_PER_CLK_PER_SM, sms, mhz)}


def dist_info():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def workload():
    from attention_attn_fwd_gb300.inputs import GQA_8K
    return GQA_8K


def max_over_ranks(values, device="cpu"):
    """Element-wise max of a list of floats over all ranks of the default
    process group (the values unchanged without one or with one rank).  The
    path shards into independent replicas, so timing is the slowest rank's
    and this is the only collective."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or \
            dist.get_world_size() == 1:
        return [float(x) for x in values]
    t = torch.tensor([float(x) for x in values], dtype=torch.float64,
                     device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(x) for x in t]


def whole_job_rate(units_per_rank, ms, world):
    """Units per second of the whole job: `world` replicas each process
    `units_per_rank` units in `ms` milliseconds (the max over ranks)."""
    return world * units_per_rank / (ms * 1e-3)


def config_dict(w, extra=None):
    d = {"workload": w.name, "B": w.B, "Hq": w.Hq, "Hkv": w.Hkv, "Sq": w.Sq,
         "Skv": w.Skv, "D": w.D, "causal": w.causal,
         "input_pos": w.input_pos, "scale": "1/sqrt(D)",
         "flops_per_step": w.flops(),
         "flops_convention": "4*B*Hq*Sq*Skv*D, halved for causal",
         "exact_visible_flops_per_step": w.exact_flops()}
    if extra:
        d.update(extra)
    return d


# ---------------------------------------------------------------- our arm
def run_ours(args):
    import torch
    import torch.distributed as dist

    import attention_attn_fwd_gb300 as attn
    from attention_attn_fwd_gb300.inputs import make_qkv

    ws, rank, local = dist_info()
    if ws > 1:
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", torch.cuda.current_device())
    w = workload()
    q, k, v = make_qkv(w, seed=0)
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    o = torch.empty_like(qd)
    lse = torch.empty((w.B, w.Hq, w.Sq), dtype=torch.float32, device=dev)
    flush = torch.empty(FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    dt = attn.ATTN_BF16 if w.dtype == "bf16" else attn.ATTN_F16

    def step(qp, kp, vp, op, lp):
        st = attn.attn_fwd(qp, kp, vp, op, lp, w.B, w.Hq, w.Hkv, w.Sq, w.Skv,
                           w.D, w.scale, int(w.causal), w.input_pos, dt,
                           stream.cuda_stream)
        if st != attn.ATTN_OK:
            raise RuntimeError("attn_fwd: " + attn.attn_status_string(st))

    ptrs = (qd.data_ptr(), kd.data_ptr(), vd.data_ptr(), o.data_ptr(),
            lse.data_ptr())
    for _ in range(args.warmup):
        flush.fill_(1.0)
        step(*ptrs)
    torch.cuda.synchronize()

    # ---- device-timed region: K launches, L2 flushed between them.
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    if ws > 1:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(dev.index) as clocks:
        t0 = time.perf_counter()
        for i in range(args.steps):
            flush.fill_(float(i))
            starts[i].record(stream)
            step(*ptrs)
            ends[i].record(stream)
        torch.cuda.synchronize()
        wall = time.perf_counter() - t0
    if ws > 1:
        dist.barrier()
    clk = clocks.summary()
    st, code = attn.attn_device_status()
    if st != attn.ATTN_OK:
        raise RuntimeError("device status %d code %#x" % (st, code))
    times_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    kernel_ms = sum(times_ms) / len(times_ms)

    # ---- end-to-end through the C ABI with host buffers: every step copies
    # its Q/K/V from pinned host memory and reads O and LSE back, inside the
    # timed region.  Copies and kernels run on three streams with double
    # buffers, so step i+1's upload and step i-1's download overlap step i.
    qh, kh, vh = q.pin_memory(), k.pin_memory(), v.pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in (qh, kh, vh))
    d2h = (o.numel() * o.element_size() + lse.numel() * lse.element_size())
    dev_bufs = [(qd, kd, vd, o, lse),
                (torch.empty_like(qd), torch.empty_like(kd),
                 torch.empty_like(vd), torch.empty_like(o),
                 torch.empty_like(lse))]
    host_out = [(torch.empty(o.shape, dtype=o.dtype).pin_memory(),
                 torch.empty(lse.shape, dtype=lse.dtype).pin_memory())
                for _ in range(2)]
    up, down = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev_up = [torch.cuda.Event() for _ in range(2)]
    ev_comp = [torch.cuda.Event() for _ in range(2)]
    ev_down = [torch.cuda.Event() for _ in range(2)]

    def e2e_steps(n):
        for i in range(n):
            s = i % 2
            qb, kb, vb, ob, lb = dev_bufs[s]
            if i >= 2:
                up.wait_event(ev_comp[s])       # inputs of step i-2 consumed
            with torch.cuda.stream(up):
                qb.copy_(qh, non_blocking=True)
                kb.copy_(kh, non_blocking=True)
                vb.copy_(vh, non_blocking=True)
                ev_up[s].record(up)
            stream.wait_event(ev_up[s])
            if i >= 2:
                stream.wait_event(ev_down[s])   # outputs of step i-2 read back
            step(qb.data_ptr(), kb.data_ptr(), vb.data_ptr(), ob.data_ptr(),
                 lb.data_ptr())
            ev_comp[s].record(stream)
            down.wait_event(ev_comp[s])
            with torch.cuda.stream(down):
                host_out[s][0].copy_(ob, non_blocking=True)
                host_out[s][1].copy_(lb, non_blocking=True)
                ev_down[s].record(down)

    e2e_steps(max(2, args.warmup))
    torch.cuda.synchronize()
    if ws > 1:
        dist.barrier()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(up)
    e2e_steps(args.steps)
    down.wait_event(ev_comp[(args.steps - 1) % 2])
    e1.record(down)
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1) / args.steps
    e2e_launches = args.steps

    # Max over ranks.
    kernel_ms, e2e_ms = max_over_ranks([kernel_ms, e2e_ms], dev)

    flops = w.flops()
    value = whole_job_rate(flops, kernel_ms, ws) / 1e12
    e2e_value = whole_job_rate(flops, e2e_ms, ws) / 1e12
    peak_tf, _, peak_src = peaks()
    achieved = flops / (kernel_ms * 1e-3) / 1e12  # one launch, one GPU
    traffic, traffic_src = measured_traffic()
    out = {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT,
        "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(kernel_ms, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": w.dtype,
        "data": "synthetic: Q/K/V ~ N(0,1) from a seeded CPU generator",
        "config": config_dict(w, {
            "l2": "flushed between timed steps (256 MiB write, untimed)",
            "parallelism": "replicas" if ws > 1 else "single GPU",
            "pct_of_dense_bf16_peak": round(100 * achieved / peak_tf, 2),
            "exact_visible_tflops": round(
                w.exact_flops() / (kernel_ms * 1e-3) / 1e12, 2),
            "ms_per_step_p50": round(statistics.median(times_ms), 4),
            "ms_per_step_max": round(max(times_ms), 4),
            "wall_s_timed_region": round(wall, 4),
            "exp2_roofline": exp2_roofline(
                w, kernel_ms, clk,
                torch.cuda.get_device_properties(dev).multi_processor_count)}),
        "roofline": {
            "bound": "tensor", "achieved": round(achieved, 2),
            "peak": peak_tf, "unit": "TFLOP/s",
            "frac": round(achieved / peak_tf, 4),
            "peak_source": "%s bf16 dense burst (cuBLAS)" % peak_src,
            "traffic": traffic,
            "traffic_source": traffic_src,
            "algorithmic_bytes": w.io_bytes()},
        "e2e": {"value": round(e2e_value, 2), "unit": UNIT,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": round(e2e_ms, 4),
                "pipelining": "3 streams (upload, compute, download), "
                              "double-buffered"},
        "gpu_launches": args.steps + e2e_launches,
        "clocks": clk,
    }
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        out["cpu_baseline"] = cpu_baseline(w, q, k, v, budget_s=args.cpu_s)
    if ws > 1:
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(out), flush=True)


# ------------------------------------------------------------- CPU oracle
def oracle_sample(w, q, k, v, heads):
    """Time the oracle on every row of the given query heads."""
    import numpy as np

    import oracle
    rows = np.array([(b, h, i) for b in range(w.B) for h in heads
                     for i in range(w.Sq)], dtype=np.int64)
    t0 = time.perf_counter()
    oracle.attention_rows(q, k, v, w.scale, w.causal, w.input_pos, rows)
    dt = time.perf_counter() - t0
    flops = w.flops() * len(heads) / w.Hq
    return flops, dt


def cpu_baseline(w, q, k, v, budget_s=15.0):
    import oracle
    heads, flops, secs = [], 0.0, 0.0
    h = 0
    while h < w.Hq and (secs < budget_s or not heads):
        f, dt = oracle_sample(w, q, k, v, [h])
        heads.append(h)
        flops += f
        secs += dt
        h += 1
    return {"value": round(flops / secs / 1e12, 6), "unit": UNIT,
            "cores": oracle.threads(), "kind": "oracle",
            "sample": "all %d rows of query heads %s (of %d), same inputs; "
                      "%.1f s" % (w.Sq, heads, w.Hq, secs)}


def run_reference(args):
    ws, rank, _ = dist_info()
    if rank != 0:
        return
    import oracle
    from attention_attn_fwd_gb300.inputs import make_qkv
    w = workload()
    q, k, v = make_qkv(w, seed=0)
    oracle.threads()  # build/load before timing
    for i in range(args.warmup):
        oracle_sample(w, q, k, v, [i % w.Hq])
    flops, secs = 0.0, 0.0
    for i in range(args.steps):
        f, dt = oracle_sample(w, q, k, v, [i % w.Hq])
        flops += f
        secs += dt
    value = flops / secs / 1e12
    out = {
        "metric": METRIC, "value": round(value, 6), "unit": UNIT,
        "impl": "reference", "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(1e3 * secs / args.steps, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64", "data": "synthetic: Q/K/V ~ N(0,1) from a seeded "
                                "CPU generator",
        "config": config_dict(w, {"sample_per_step": "all rows of one query "
                                                     "head"}),
        "cpu_baseline": {"value": round(value, 6), "unit": UNIT,
                         "cores": oracle.threads(), "kind": "oracle",
                         "sample": "each step: all %d rows of one query head"
                                   % w.Sq},
        "e2e": {"value": round(value, 6), "unit": UNIT,
                "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(out), flush=True)


# ------------------------------------------------------- split-KV decode
DECODE_SETS = 4
def run_decode(args, fp8=False):
    """Split-KV decode step: HBM-bound, reported in GB/s of algorithmic
    traffic (Q, K, V read once; O and LSE written once) against the measured
    copy bandwidth.  One kernel per step when the key ranges merge inside
    thread-block clusters (the automatic count here), else two (the forward
    kernel and the merge kernel).
    ``fp8``: the same step with E4M3 Q/K/V (half the K/V bytes) through
    attn_fwd_fp8, bf16 O.

    Steps rotate over DECODE_SETS independent input sets whose total is
    several times L2, so every step reads its K/V from HBM.  (A flush write
    before each step would leave ~L2-sized dirty lines that the step itself
    then has to write back, which charges the flush's traffic to an
    HBM-bound kernel.)"""
    import torch

    import attention_attn_fwd_gb300 as attn
    from attention_attn_fwd_gb300.inputs import DECODE, make_qkv

    ws, rank, local = dist_info()
    if ws > 1:
        torch.cuda.set_device(local)
    dev = torch.device("cuda", torch.cuda.current_device())
    w = DECODE.with_(name=DECODE.name.replace("bf16", "e4m3"),
                     dtype="e4m3") if fp8 else DECODE
    sets = []
    for i in range(DECODE_SETS):
        q, k, v = (t.to(dev) for t in make_qkv(w, seed=i))
        o = torch.empty(q.shape, dtype=w.out_dtype, device=dev)
        lse = torch.empty((w.B, w.Hq, w.Sq), dtype=torch.float32, device=dev)
        sets.append((q, k, v, o, lse))
    stream = torch.cuda.current_stream(dev)
    dt = attn.ATTN_E4M3 if fp8 else attn.ATTN_BF16
    splits, ws_bytes = attn.attn_splitkv_plan(w.B, w.Hq, w.Hkv, w.Sq, w.Skv,
                                              w.D, 1, w.input_pos, dt,
                                              args.splits)
    work = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    # Kernels per step: the forward kernel, plus the merge kernel unless
    # the key ranges merge inside clusters.
    kernels = 2 if attn.attn_dispatch(
        w.B, w.Hq, w.Hkv, w.Sq, w.Skv, w.D, 1, w.input_pos, dt,
        num_splits=splits)["merge"] == 2 else 1

    def step(i):
        q, k, v, o, lse = sets[i % DECODE_SETS]
        if fp8:
            st = attn.attn_fwd_fp8(
                q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                lse.data_ptr(), w.B, w.Hq, w.Hkv, w.Sq, w.Skv, w.D, w.scale,
                1.0, 1.0, 1.0, 1, w.input_pos, 0, splits, work.data_ptr(),
                ws_bytes, stream.cuda_stream)
        else:
            st = attn.attn_fwd_splitkv(
                q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                lse.data_ptr(), w.B, w.Hq, w.Hkv, w.Sq, w.Skv, w.D, w.scale,
                1, w.input_pos, dt, splits, work.data_ptr(), ws_bytes,
                stream.cuda_stream)
        if st != attn.ATTN_OK:
            raise RuntimeError("decode step: " + attn.attn_status_string(st))

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    with ClockSampler(dev.index) as clocks:
        for i in range(args.steps):
            starts[i].record(stream)
            step(args.warmup + i)
            ends[i].record(stream)
        torch.cuda.synchronize()
    # The same steps launched back to back, one event pair around them all:
    # the rate a loop of decode steps sees, without the event and launch
    # latency each isolated step above carries.
    b2b_a = torch.cuda.Event(enable_timing=True)
    b2b_b = torch.cuda.Event(enable_timing=True)
    b2b_a.record(stream)
    for i in range(args.steps):
        step(args.warmup + i)
    b2b_b.record(stream)
    torch.cuda.synchronize()
    st, code = attn.attn_device_status()
    if st != attn.ATTN_OK:
        raise RuntimeError("device status %d code %#x" % (st, code))
    ms = sum(s_.elapsed_time(e_) for s_, e_ in zip(starts, ends)) / args.steps
    gbs = w.io_bytes() / (ms * 1e-3) / 1e9
    ms_b2b = b2b_a.elapsed_time(b2b_b) / args.steps
    gbs_b2b = w.io_bytes() / (ms_b2b * 1e-3) / 1e9
    _, hbm, src = peaks()
    out = {
        "metric": "attention decode (split-KV) GB/s of algorithmic traffic"
                  + (", FP8 inputs" if fp8 else ""),
        "value": round(gbs, 1), "unit": "GB/s", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(ms, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": w.dtype,
        "data": "synthetic: Q/K/V ~ N(0,1) from a seeded CPU generator",
        "config": config_dict(w, {
            "num_splits": splits, "workspace_bytes": ws_bytes,
            "l2": "inputs larger than L2: %d rotating input sets, %.0f MB"
                  % (DECODE_SETS, DECODE_SETS * w.io_bytes() / 1e6),
            "algorithmic_bytes_per_step": w.io_bytes(),
            "tokens_per_s": round(w.B / (ms * 1e-3), 1),
            "back_to_back": {
                "note": "the same steps launched back to back between one "
                        "event pair (value: each step between its own "
                        "events)",
                "ms_per_step": round(ms_b2b, 5), "GB/s": round(gbs_b2b, 1),
                "frac": round(gbs_b2b / hbm, 4)},
            "tflops_formula": round(w.flops() / (ms * 1e-3) / 1e12, 2)}),
        "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": hbm,
                     "unit": "GB/s", "frac": round(gbs / hbm, 4),
                     "peak_source": "%s copy bandwidth" % src,
                     "traffic": None},
        "gpu_launches": args.steps * kernels,
        "clocks": clocks.summary(),
    }
    if rank == 0:
        print(json.dumps(out), flush=True)


# ------------------------------------------------------- sliding window
def run_window(args):
    """Causal GQA 32k prefill with a 4096-key sliding window: tensor-bound,
    reported in TFLOPS of the exactly visible query-key pairs (4*D FLOPs
    each; the causal-halved formula does not describe a window) against the
    measured dense bf16 peak.  L2 flushed between timed steps."""
    import torch

    import attention_attn_fwd_gb300 as attn
    from attention_attn_fwd_gb300.inputs import WINDOW_32K, make_qkv

    ws, rank, local = dist_info()
    if ws > 1:
        torch.cuda.set_device(local)
    dev = torch.device("cuda", torch.cuda.current_device())
    w = WINDOW_32K
    q, k, v = (t.to(dev) for t in make_qkv(w, seed=0))
    o = torch.empty_like(q)
    lse = torch.empty((w.B, w.Hq, w.Sq), dtype=torch.float32, device=dev)
    flush = torch.empty(FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    dt = attn.ATTN_BF16

    def step():
        st = attn.attn_fwd_window(
            q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
            lse.data_ptr(), w.B, w.Hq, w.Hkv, w.Sq, w.Skv, w.D, w.scale, 1,
            w.input_pos, w.window, dt, stream.cuda_stream)
        if st != attn.ATTN_OK:
            raise RuntimeError("attn_fwd_window: " +
                               attn.attn_status_string(st))

    for _ in range(args.warmup):
        flush.fill_(1.0)
        step()
    torch.cuda.synchronize()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    with ClockSampler(dev.index) as clocks:
        for i in range(args.steps):
            flush.fill_(float(i))
            starts[i].record(stream)
            step()
            ends[i].record(stream)
        torch.cuda.synchronize()
    st, code = attn.attn_device_status()
    if st != attn.ATTN_OK:
        raise RuntimeError("device status %d code %#x" % (st, code))
    ms = sum(s_.elapsed_time(e_) for s_, e_ in zip(starts, ends)) / args.steps
    flops = w.exact_flops()
    tflops = flops / (ms * 1e-3) / 1e12
    peak, _, src = peaks()
    out = {
        "metric": "attention fwd TFLOPS, causal sliding window (exact "
                  "visible FLOPs)",
        "value": round(tflops, 1), "unit": "TFLOPS", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(ms, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": w.dtype,
        "data": "synthetic: Q/K/V ~ N(0,1) from a seeded CPU generator",
        "config": config_dict(w, {
            "window": w.window,
            "l2": "flushed between timed steps (256 MiB write, untimed)"}),
        "roofline": {"bound": "tensor", "achieved": round(tflops, 1),
                     "peak": peak, "unit": "TFLOP/s",
                     "frac": round(tflops / peak, 4),
                     "peak_source": "%s bf16 dense burst (cuBLAS)" % src,
                     "traffic": None},
        "gpu_launches": args.steps,
        "clocks": clocks.summary(),
    }
    if rank == 0:
        print(json.dumps(out), flush=True)


# ------------------------------------------------------ per-config table
def run_table(args):
    """Every named forward workload (the small case, causal MHA 4k, causal
    GQA 8k, the KV-cache prefill chunk, the B4 H16 non-causal sweep) timed
    the same way as the headline line: L2 flushed between steps, CUDA events
    around each launch, medians and 95th percentiles.  One JSON line whose
    `table` lists the configurations; `value` repeats the GQA 8k median."""
    import torch

    import attention_attn_fwd_gb300 as attn
    from attention_attn_fwd_gb300.inputs import ALL, GQA_8K, make_qkv

    ws, rank, local = dist_info()
    if ws > 1:
        torch.cuda.set_device(local)
    dev = torch.device("cuda", torch.cuda.current_device())
    flush = torch.empty(FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    peak, _, src = peaks()
    rows, headline = [], None
    with ClockSampler(dev.index) as clocks:
        for w in ALL:
            q, k, v = (t.to(dev) for t in make_qkv(w, seed=0))
            o = torch.empty_like(q)
            lse = torch.empty((w.B, w.Hq, w.Sq), dtype=torch.float32,
                              device=dev)
            dt = attn.ATTN_BF16 if w.dtype == "bf16" else attn.ATTN_F16

            def step():
                st = attn.attn_fwd(
                    q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                    lse.data_ptr(), w.B, w.Hq, w.Hkv, w.Sq, w.Skv, w.D,
                    w.scale, int(w.causal), w.input_pos, dt,
                    stream.cuda_stream)
                if st != attn.ATTN_OK:
                    raise RuntimeError("attn_fwd: " +
                                       attn.attn_status_string(st))

            for _ in range(args.warmup):
                flush.fill_(1.0)
                step()
            torch.cuda.synchronize()
            ev = [(torch.cuda.Event(enable_timing=True),
                   torch.cuda.Event(enable_timing=True))
                  for _ in range(args.steps)]
            for i, (a_, b_) in enumerate(ev):
                flush.fill_(float(i))
                a_.record(stream)
                step()
                b_.record(stream)
            torch.cuda.synchronize()
            t = sorted(a_.elapsed_time(b_) for a_, b_ in ev)
            p50, p95 = t[len(t) // 2], t[min(len(t) - 1, int(0.95 * len(t)))]
            tf = w.flops() / (p50 * 1e-3) / 1e12
            rows.append({
                "workload": w.name, "ms_p50": round(p50, 5),
                "ms_p95": round(p95, 5), "tflops": round(tf, 1),
                "tflops_exact": round(w.exact_flops() / (p50 * 1e-3) / 1e12,
                                      1),
                "pct_of_peak": round(100.0 * tf / peak, 2)})
            if w.name == GQA_8K.name:
                headline = tf
            del q, k, v, o, lse
    st, code = attn.attn_device_status()
    if st != attn.ATTN_OK:
        raise RuntimeError("device status %d code %#x" % (st, code))
    out = {
        "metric": "attention fwd TFLOPS per configuration (median launch, "
                  "causal-halved FLOPs)",
        "value": round(headline, 1), "unit": "TFLOPS", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16 / f16 (per row)",
        "data": "synthetic: Q/K/V ~ N(0,1) from a seeded CPU generator",
        "config": {"workload": "all named forward workloads",
                   "l2": "flushed between timed steps (256 MiB write, "
                         "untimed)"},
        "roofline": {"bound": "tensor", "peak": peak, "unit": "TFLOP/s",
                     "peak_source": "%s bf16 dense burst (cuBLAS)" % src},
        "table": rows,
        "gpu_launches": args.steps * len(rows),
        "clocks": clocks.summary(),
    }
    if rank == 0:
        print(json.dumps(out), flush=True)


# ------------------------------------------------- split-KV, long key ranges
def run_splitkv_long(args):
    """Chunks of a few hundred query rows against long KV caches, through
    attn_fwd_splitkv at the count attn_splitkv_plan picks and through the
    one-pass attn_fwd, L2 flushed before each call, CUDA events around
    each (the split call's events enclose its forward and merge kernels).
    Each row's roofline bound is the larger of streaming Q, K, V and O once
    at the measured copy bandwidth and its exact visible FLOPs at the
    measured bf16 peak; `value` is the summed split time (lower is better),
    `roofline` the summed bounds over it."""
    import torch

    import attention_attn_fwd_gb300 as attn
    from attention_attn_fwd_gb300.inputs import LONG_KEY_CHUNKS, make_qkv

    ws, rank, local = dist_info()
    if ws > 1:
        torch.cuda.set_device(local)
    dev = torch.device("cuda", torch.cuda.current_device())
    flush = torch.empty(FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    peak, hbm, src = peaks()
    rows, launches, t_total, b_total = [], 0, 0.0, 0.0
    with ClockSampler(dev.index) as clocks:
        for w in LONG_KEY_CHUNKS:
            q, k, v = (t.to(dev) for t in make_qkv(w, seed=0))
            o = torch.empty_like(q)
            lse = torch.empty((w.B, w.Hq, w.Sq), dtype=torch.float32,
                              device=dev)
            dt = attn.ATTN_BF16
            splits, ws_bytes = attn.attn_splitkv_plan(
                w.B, w.Hq, w.Hkv, w.Sq, w.Skv, w.D, 1, w.input_pos, dt, 0)
            work = torch.empty(max(ws_bytes, 1), dtype=torch.uint8,
                               device=dev)
            kernels = 2 if attn.attn_dispatch(
                w.B, w.Hq, w.Hkv, w.Sq, w.Skv, w.D, 1, w.input_pos, dt,
                num_splits=splits)["merge"] == 2 else 1
            args_ = (q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                     lse.data_ptr(), w.B, w.Hq, w.Hkv, w.Sq, w.Skv, w.D,
                     w.scale, 1, w.input_pos, dt)

            def split_step():
                st = attn.attn_fwd_splitkv(*args_, splits, work.data_ptr(),
                                           ws_bytes, stream.cuda_stream)
                if st != attn.ATTN_OK:
                    raise RuntimeError("attn_fwd_splitkv: " +
                                       attn.attn_status_string(st))

            def one_pass():
                st = attn.attn_fwd(*args_, stream.cuda_stream)
                if st != attn.ATTN_OK:
                    raise RuntimeError("attn_fwd: " +
                                       attn.attn_status_string(st))

            med = {}
            for name, fn in (("split", split_step), ("one_pass", one_pass)):
                for _ in range(args.warmup):
                    flush.fill_(1.0)
                    fn()
                torch.cuda.synchronize()
                ev = [(torch.cuda.Event(enable_timing=True),
                       torch.cuda.Event(enable_timing=True))
                      for _ in range(args.steps)]
                for i, (a_, b_) in enumerate(ev):
                    flush.fill_(float(i))
                    a_.record(stream)
                    fn()
                    b_.record(stream)
                torch.cuda.synchronize()
                t = sorted(a_.elapsed_time(b_) for a_, b_ in ev)
                med[name] = t[len(t) // 2]
            io_bytes = w.io_bytes()
            hbm_us = io_bytes / (hbm * 1e9) * 1e6
            tensor_us = w.exact_flops() / (peak * 1e12) * 1e6
            bound_us = max(hbm_us, tensor_us)
            us = 1000 * med["split"]
            t_total += us
            b_total += bound_us
            launches += args.steps * (kernels + 1)
            rows.append({
                "workload": w.name, "num_splits": splits,
                "kernels_per_call": kernels,
                "us_split": round(us, 2),
                "us_one_pass": round(1000 * med["one_pass"], 2),
                "speedup": round(med["one_pass"] / med["split"], 2),
                "bound": "hbm" if hbm_us >= tensor_us else "tensor",
                "bound_us": round(bound_us, 2),
                "frac": round(bound_us / us, 4),
                "GB/s": round(io_bytes / (us * 1e-6) / 1e9, 1),
                "tflops_exact": round(w.exact_flops() / (us * 1e-6) / 1e12,
                                      1)})
            del q, k, v, o, lse, work
    st, code = attn.attn_device_status()
    if st != attn.ATTN_OK:
        raise RuntimeError("device status %d code %#x" % (st, code))
    out = {
        "metric": "split-KV time summed over long-key chunks (median call "
                  "at the planned range count)",
        "value": round(t_total, 2), "unit": "us", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup,
        "higher_is_better": False, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic: Q/K/V ~ N(0,1) from a seeded CPU generator",
        "config": {"workload": "long-key chunks (%s)" % ", ".join(
                       w.name for w in LONG_KEY_CHUNKS),
                   "l2": "flushed before each call (256 MiB write, "
                         "untimed)"},
        "roofline": {"bound": "per row (hbm or tensor)",
                     "achieved_us": round(t_total, 2),
                     "bound_us": round(b_total, 2),
                     "frac": round(b_total / t_total, 4),
                     "peak_source": "%s copy bandwidth and bf16 dense burst"
                                    % src,
                     "traffic": None},
        "table": rows,
        "gpu_launches": launches,
        "clocks": clocks.summary(),
    }
    if rank == 0:
        print(json.dumps(out), flush=True)


# ------------------------------------------------------------ FP8 forward
def run_fp8(args):
    """The headline GQA 8k causal forward with E4M3 Q/K/V (descale 1) and a
    bf16 O through attn_fwd_fp8; TFLOPS with the causal-halved FLOPs,
    against the dense FP8 peak taken as the measured bf16 burst peak x 2
    (the nominal FP8 / bf16 ratio, 4.5 / 2.25 PFLOP/s).  L2 flushed between
    timed steps (the FP8 inputs, ~50 MB, would fit in it)."""
    import torch

    import attention_attn_fwd_gb300 as attn
    from attention_attn_fwd_gb300.inputs import GQA_8K_FP8, make_qkv

    ws, rank, local = dist_info()
    if ws > 1:
        torch.cuda.set_device(local)
    dev = torch.device("cuda", torch.cuda.current_device())
    w = GQA_8K_FP8
    q, k, v = (t.to(dev) for t in make_qkv(w, seed=0))
    o = torch.empty(q.shape, dtype=w.out_dtype, device=dev)
    lse = torch.empty((w.B, w.Hq, w.Sq), dtype=torch.float32, device=dev)
    flush = torch.empty(FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        st = attn.attn_fwd_fp8(
            q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
            lse.data_ptr(), w.B, w.Hq, w.Hkv, w.Sq, w.Skv, w.D, w.scale, 1.0,
            1.0, 1.0, 1, w.input_pos, 0, 0, 0, 0, stream.cuda_stream)
        if st != attn.ATTN_OK:
            raise RuntimeError("attn_fwd_fp8: " + attn.attn_status_string(st))

    for _ in range(args.warmup):
        flush.fill_(1.0)
        step()
    torch.cuda.synchronize()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    with ClockSampler(dev.index) as clocks:
        for i in range(args.steps):
            flush.fill_(float(i))
            starts[i].record(stream)
            step()
            ends[i].record(stream)
        torch.cuda.synchronize()
    st, code = attn.attn_device_status()
    if st != attn.ATTN_OK:
        raise RuntimeError("device status %d code %#x" % (st, code))
    ms = sum(s_.elapsed_time(e_) for s_, e_ in zip(starts, ends)) / args.steps
    tflops = w.flops() / (ms * 1e-3) / 1e12
    bf16_peak, _, src = peaks()
    peak = 2.0 * bf16_peak
    out = {
        "metric": "attention fwd TFLOPS on 1 GB300 (causal-halved FLOPs), "
                  "FP8 E4M3 inputs",
        "value": round(tflops, 1), "unit": "TFLOPS", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(ms, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "e4m3",
        "data": "synthetic: Q/K/V ~ N(0,1) from a seeded CPU generator, "
                "rounded to E4M3",
        "config": config_dict(w, {
            "out_dtype": "bf16",
            "l2": "flushed between timed steps (256 MiB write, untimed)"}),
        "roofline": {"bound": "tensor", "achieved": round(tflops, 1),
                     "peak": round(peak, 1), "unit": "TFLOP/s",
                     "frac": round(tflops / peak, 4),
                     "peak_source": "%s bf16 dense burst (cuBLAS) x 2, the "
                                    "nominal FP8/bf16 ratio" % src,
                     "traffic": None},
        "gpu_launches": args.steps,
        "clocks": clocks.summary(),
    }
    if rank == 0:
        print(json.dumps(out), flush=True)


# -------------------------------------------------------------- backward
def run_bwd(args):
    """Backward pass (dQ, dK, dV) of the GQA 8k causal workload: the row
    pass, the dK/dV kernel and the dQ kernel of one attn_bwd call per step,
    inputs (Q, K, V, O, LSE, dO) resident, L2 flushed between steps.
    FLOPs: 2.5x the forward's causal-halved count (five tile products per
    visible score where the forward has two; this implementation computes
    seven, recomputing S and dP in both kernels, which is not counted)."""
    import torch

    import attention_attn_fwd_gb300 as attn
    from attention_attn_fwd_gb300.inputs import GQA_8K, make_do, make_qkv

    ws, rank, local = dist_info()
    if ws > 1:
        torch.cuda.set_device(local)
    dev = torch.device("cuda", torch.cuda.current_device())
    w = GQA_8K
    q, k, v = (t.to(dev) for t in make_qkv(w, seed=0))
    do = make_do(w, seed=0).to(dev)
    o, lse = attn.fwd(q, k, v, scale=w.scale, causal=True)
    dq, dk, dv = (torch.empty_like(t) for t in (q, k, v))
    ws_bytes = attn.attn_bwd_workspace_bytes(w.B, w.Hq, w.Sq)
    work = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    flush = torch.empty(FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    dt = attn.ATTN_BF16

    def step():
        st = attn.attn_bwd(q.data_ptr(), k.data_ptr(), v.data_ptr(),
                           o.data_ptr(), lse.data_ptr(), do.data_ptr(),
                           dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), w.B,
                           w.Hq, w.Hkv, w.Sq, w.Skv, w.D, w.scale, 1, 0, 0,
                           dt, work.data_ptr(), ws_bytes, stream.cuda_stream)
        if st != attn.ATTN_OK:
            raise RuntimeError("attn_bwd: " + attn.attn_status_string(st))

    for _ in range(args.warmup):
        flush.fill_(1.0)
        step()
    torch.cuda.synchronize()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    with ClockSampler(dev.index) as clocks:
        for i in range(args.steps):
            flush.fill_(float(i))
            starts[i].record(stream)
            step()
            ends[i].record(stream)
        torch.cuda.synchronize()
    st, code = attn.attn_device_status()
    if st != attn.ATTN_OK:
        raise RuntimeError("device status %d code %#x" % (st, code))
    ms = sum(s_.elapsed_time(e_) for s_, e_ in zip(starts, ends)) / args.steps
    flops = 2.5 * w.flops()
    tflops = flops / (ms * 1e-3) / 1e12
    peak, _, src = peaks()
    out = {
        "metric": "attention bwd TFLOPS (2.5x forward causal-halved FLOPs)",
        "value": round(tflops, 1), "unit": "TFLOPS", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(ms, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": w.dtype,
        "data": "synthetic: Q/K/V/dO ~ N(0,1) from seeded CPU generators",
        "config": config_dict(w, {
            "pass": "backward (dQ, dK, dV)",
            "bwd_flops_per_step": flops,
            "kernels_per_step": 3,
            "l2": "flushed between timed steps (256 MiB write, untimed)"}),
        "roofline": {"bound": "tensor", "achieved": round(tflops, 1),
                     "peak": peak, "unit": "TFLOP/s",
                     "frac": round(tflops / peak, 4),
                     "peak_source": "%s bf16 dense burst (cuBLAS)" % src,
                     "traffic": None},
        "gpu_launches": 3 * args.steps,
        "clocks": clocks.summary(),
    }
    if rank == 0:
        print(json.dumps(out), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--cpu-s", type=float, default=15.0,
                    help="CPU-oracle baseline budget in seconds")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--workload",
                    choices=["gqa8k", "decode", "window", "bwd", "fp8",
                             "decode_fp8", "table", "splitkv_long"],
                    default="gqa8k",
                    help="gqa8k: the headline causal GQA forward (default); "
                         "decode: the split-KV decode step; window: causal "
                         "GQA 32k with a 4096-key sliding window; bwd: the "
                         "backward pass of gqa8k; fp8: gqa8k with E4M3 "
                         "inputs; decode_fp8: decode with E4M3 inputs; "
                         "table: every named forward workload, one row each; "
                         "splitkv_long: split-KV against one pass on chunks "
                         "of few query rows over long key ranges")
    ap.add_argument("--splits", type=int, default=0,
                    help="split count for --workload decode (0: automatic)")
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "ours":
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        run_reference(args)
    elif args.workload == "decode":
        run_decode(args)
    elif args.workload == "decode_fp8":
        run_decode(args, fp8=True)
    elif args.workload == "fp8":
        run_fp8(args)
    elif args.workload == "window":
        run_window(args)
    elif args.workload == "bwd":
        run_bwd(args)
    elif args.workload == "splitkv_long":
        run_splitkv_long(args)
    elif args.workload == "table":
        run_table(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
