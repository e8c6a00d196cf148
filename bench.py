"""Benchmark of the multi-head attention forward pass on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config I | --workload NAME]
                    [--impl ours|reference]

One step is one whole forward pass (the QKV projection with head split, the
fused attention kernel and the output projection) over one batch of seeded
synthetic inputs already resident in HBM, timed as a whole with CUDA events
around the three launches; the per-kernel split comes from as many further
steps with events between the kernels (an event between two kernels keeps
the second from starting its prologue under the first one's tail). L2 is flushed
between timed steps, outside the timed events: a 512 MiB buffer is written and
read back, so L2 holds none of the inputs and no dirty line of the flush. With
N > 1 (torchrun) every rank runs an independent replica on its own GPU
(replicas only: the forward pass has no exchange step), the time is the max
over ranks and the value counts the work of all ranks.

Prints one JSON line. Counting: attention core 4 * n_q * n_k * d_h per (batch
item, head), halved under a causal mask; projections 2 * rows * d_in * width.
With a padding mask the effective count (valid rows and keys) is reported.

--impl reference times the oracle (plain fp64 numpy on the host cores) on a
bounded sample of the same workload: one (batch item, head) unit per step.
"""

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MHA forward TFLOP/s and fraction of GB300 bf16 dense peak, 1 GPU"
FALLBACK_PEAKS = {"bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "hbm_gbs": 6800.0}
L2_FLUSH_BYTES = 512 << 20


class L2Flush:
    """Replaces the contents of L2 between timed steps: a 512 MiB buffer is
    written and then read back, outside the timed events. Afterwards no input
    of the step is in L2, and L2 holds only clean lines of the flush buffer,
    so the timed step does not pay for writing back the flush's own data."""

    def __init__(self, dev):
        import torch
        self.buf = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
        self.acc = torch.empty((), dtype=torch.float32, device=dev)

    def fill_(self, v):
        import torch
        self.buf.fill_(v)
        torch.sum(self.buf, dim=0, out=self.acc)
CLOCK_WINDOW_S = 1.0


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--config", type=int, default=3,
                    help="workload index (0..4); the JSON line is for this one (default: 3, "
                         "the largest: B=2, T=8192, d_model=2048, h=16, d_h=128, causal + "
                         "padding)")
    ap.add_argument("--workload", default=None,
                    help="time this named workload instead of --config (any name of "
                         "head_scaled_dot_gb300.workloads: the five, the general head sizes, "
                         "the long-key ones)")
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-others", action="store_true",
                    help="skip the per-workload table of the other bf16 workloads")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true",
                    help="skip the oracle timing (for profiler runs)")
    ap.add_argument("--no-clocks", action="store_true",
                    help="skip the clock-sampling window (for profiler runs)")
    return ap.parse_args()


def chosen_workload(args):
    """The workload of the JSON line: --workload by name, else --config."""
    from head_scaled_dot_gb300 import workloads
    if args.workload:
        named = {w.name: w for w in workloads.WORKLOADS + [workloads.GENERAL_DIMS,
                                                           workloads.SMALL_DIMS,
                                                           workloads.SIMT_DIMS]
                 + workloads.LONG_KEYS}
        if args.workload not in named:
            raise SystemExit("unknown workload %r; one of: %s" % (args.workload,
                                                                 ", ".join(sorted(named))))
        return named[args.workload]
    return workloads.WORKLOADS[args.config]


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        d = json.load(open(path))
        return {k: float(d[k]) for k in FALLBACK_PEAKS}, "measured"
    except Exception:
        return dict(FALLBACK_PEAKS), "fallback"


# FP32 lanes per SM (four schedulers x 32) and flop per FMA: the peak of the
# CUDA-core kernels is SMs x 128 x 2 x the maximum SM clock.
FP32_LANES_PER_SM = 128


def alu_peak_tflops(dev, sm_max_mhz):
    """fp32 FMA peak of the device at the given SM clock, in TFLOP/s."""
    import torch
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    return sms * FP32_LANES_PER_SM * 2 * sm_max_mhz * 1e6 / 1e12


def sm_max_mhz():
    """Maximum SM clock: the measured-peaks record, else the GB300 maximum."""
    try:
        return float(json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))["sm_max_mhz"])
    except Exception:
        return 2070.0


def dist_setup(n):
    import torch
    import torch.distributed as dist
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1 and not dist.is_initialized():
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend=backend)
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x, world, device):
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


class ClockSampler:
    """nvidia-smi clock and throttle-reason samples while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.proc = None
        self.gpu = gpu_index
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(gpu_index), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for name, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(name)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm)}


def source_hash(path):
    return hashlib.sha256(open(path, "rb").read()).hexdigest()[:16]


def stored_traffic(kernel, workload_name):
    """Per-launch DRAM bytes from a committed ncu summary, or None when the
    kernel source changed since the counters were taken."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        d = json.load(open(path))[kernel][workload_name]
    except Exception:
        return None
    src = os.path.join(ROOT, "head_scaled_dot_gb300", "csrc", d["source"])
    if not os.path.exists(src) or source_hash(src) != d["source_sha256_16"]:
        return None
    return d["dram_bytes_per_launch"]


def to_device(inp, dev):
    import torch
    return {k: (v.to(dev) if torch.is_tensor(v) and k != "valid_len" else v)
            for k, v in inp.items()}


def measure_workload(w, steps, warmup, dev, world, e2e=True, sample_clocks=True):
    """Times `steps` forward passes of workload w. Returns a dict of results."""
    import torch

    from head_scaled_dot_gb300 import mha, workcount, workloads

    inp = workloads.make_inputs(w)
    lens = None if inp["valid_len"] is None else [int(x) for x in inp["valid_len"]]
    t = to_device(inp, dev)
    lib = mha.load()
    B, n_q, n_k = w.B, w.n_q, w.n_k
    dt = workloads.torch_dtype(w.dtype)
    nbytes = mha.workspace_size(B, n_q, n_k, w.d_model, w.h, w.d_h, w.d_vh, w.d_o, w.dtype)
    ws = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    Y = torch.empty((B, n_q, w.d_o), dtype=dt, device=dev)
    flush = L2Flush(dev)
    stream = torch.cuda.current_stream(dev)
    sp = mha._stream(stream)
    import ctypes
    P = ctypes.c_void_p
    L = mha.workspace_layout(B, n_q, n_k, w.h, w.d_h, w.d_vh, w.dtype)
    base = ws.data_ptr()
    err, Qp, Kp, Vp, Zp = base, base + L["q"], base + L["k"], base + L["v"], base + L["z"]
    lens_arg, keep = mha._lens(lens, B)
    DT, MK = mha.DTYPES[w.dtype], mha.MASKS[w.mask]
    # the scratch of the automatic split over the keys, after Z (as mha_forward
    # lays it out); workloads with few query tiles run the attention step split
    es = 2 if w.dtype == "bf16" else 4
    split_off = L["z"] + (B * n_q * w.h * w.d_vh * es + 1023) // 1024 * 1024
    split_bytes = L["total"] - split_off
    X_kv_p = None if t["X_kv"] is None else P(t["X_kv"].data_ptr())

    def step(ev):
        # the three kernels mha_forward enqueues (it also resets the 4-byte
        # error word first); with four events, also between them (an event
        # between two kernels keeps the second from starting its prologue
        # under the first one's tail, so whole steps are timed with two)
        split = len(ev) == 4
        ev[0].record(stream)
        rc = lib.mha_qkv_projection(P(t["X_q"].data_ptr()), X_kv_p, P(t["W_Q"].data_ptr()),
                                    P(t["W_K"].data_ptr()), P(t["W_V"].data_ptr()), P(Qp), P(Kp),
                                    P(Vp), B, n_q, n_k, w.d_model, w.h, w.d_h, w.d_vh, MK,
                                    lens_arg, DT, P(err), sp)
        if split:
            ev[1].record(stream)
        if split_bytes > 0:
            rc |= lib.mha_attention_split(P(Qp), P(Kp), P(Vp), P(Zp), B, n_q, n_k, w.h, w.d_h,
                                          w.d_vh, float(w.c), MK, lens_arg, 0 if w.cross else 1,
                                          0, DT, P(base + split_off), split_bytes, P(err), sp)
        else:
            rc |= lib.mha_attention(P(Qp), P(Kp), P(Vp), P(Zp), B, n_q, n_k, w.h, w.d_h,
                                    w.d_vh, float(w.c), MK, lens_arg, 0 if w.cross else 1, DT,
                                    P(err), sp)
        if split:
            ev[2].record(stream)
        rc |= lib.mha_output_projection(P(Zp), P(t["W_O"].data_ptr()), P(Y.data_ptr()), B, n_q,
                                        w.h, w.d_vh, w.d_o, None if w.cross else lens_arg, DT,
                                        P(err), sp)
        ev[-1].record(stream)
        if rc != 0:
            raise RuntimeError("launch failed with status %d" % rc)

    mk = lambda n=4: [torch.cuda.Event(enable_timing=True) for _ in range(n)]
    torch.cuda.synchronize(dev)
    ws[:4].zero_()
    for _ in range(warmup):
        flush.fill_(1.0)
        step(mk())
    torch.cuda.synchronize(dev)
    events = [mk(2) for _ in range(steps)]
    barrier(world)
    torch.cuda.synchronize(dev)
    # nvidia-smi samples every 200 ms, far longer than the timed steps: it
    # runs over a loaded window of identical untimed steps (about
    # CLOCK_WINDOW_S) that ends where the timed steps begin, so its samples
    # see the clocks of this workload under load
    clocks = ClockSampler(dev.index if dev.index is not None else 0) if sample_clocks else None
    if clocks is not None:
        spare = mk(2)
        t_end = time.perf_counter() + CLOCK_WINDOW_S
        while time.perf_counter() < t_end:
            for _ in range(8):
                flush.fill_(1.0)
                step(spare)
            spare[-1].synchronize()
    launches0 = mha.launch_count()
    for ev in events:
        flush.fill_(1.0)  # L2 flush, outside the timed events
        step(ev)
    torch.cuda.synchronize(dev)
    barrier(world)
    launches = mha.launch_count() - launches0
    # the per-kernel split, from as many further steps timed kernel by kernel
    split_events = [mk() for _ in range(steps)]
    for ev in split_events:
        flush.fill_(1.0)
        step(ev)
    torch.cuda.synchronize(dev)
    clk = clocks.stop() if clocks is not None else None
    if clk is not None:
        clk["window_s"] = CLOCK_WINDOW_S
    status = mha.get_device_error(P(err), stream)
    if status != 0:
        raise RuntimeError("device error word: %d" % status)
    per = {"qkv": [], "attention": [], "out": [], "step": []}
    for ev in events:
        per["step"].append(ev[0].elapsed_time(ev[1]))
    for ev in split_events:
        per["qkv"].append(ev[0].elapsed_time(ev[1]))
        per["attention"].append(ev[1].elapsed_time(ev[2]))
        per["out"].append(ev[2].elapsed_time(ev[3]))
    total_ms = sum(per["step"])
    fl = workcount.flops(w, lens)
    res = {"inputs": inp, "lens": lens, "flops": fl, "total_ms": total_ms, "per": per,
           "launches": launches, "clocks": clk, "Y": Y, "ws": ws}

    if e2e:
        res["e2e"] = measure_e2e_pipelined(w, inp, t, steps, warmup, dev, world, ws)
        res["e2e_serial"] = measure_e2e(w, inp, t, steps, warmup, dev, world, ws, flush)
    return res


def measure_e2e(w, inp, t, steps, warmup, dev, world, ws, flush):
    """The public call (mha.forward) with pinned host inputs copied in and the
    result copied out inside the timed region of every step."""
    import torch

    from head_scaled_dot_gb300 import mha
    hX = inp["X_q"].pin_memory()
    hXkv = None if inp["X_kv"] is None else inp["X_kv"].pin_memory()
    dX = torch.empty_like(t["X_q"])
    dXkv = None if hXkv is None else torch.empty_like(t["X_kv"])
    Y = torch.empty((w.B, w.n_q, w.d_o), dtype=t["X_q"].dtype, device=dev)
    hY = torch.empty(Y.shape, dtype=Y.dtype).pin_memory()
    stream = torch.cuda.current_stream(dev)

    def one(ev0, ev1):
        ev0.record(stream)
        dX.copy_(hX, non_blocking=True)
        if dXkv is not None:
            dXkv.copy_(hXkv, non_blocking=True)
        mha.forward(dX, dXkv, t["W_Q"], t["W_K"], t["W_V"], t["W_O"], w.h, w.d_h, w.d_vh, w.c,
                    w.mask, inp["valid_len"], out=Y, workspace=ws, check=False)
        hY.copy_(Y, non_blocking=True)
        ev1.record(stream)
        ev1.synchronize()  # the caller reads the result on the host

    for _ in range(warmup):
        flush.fill_(1.0)
        one(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
    barrier(world)
    tot = 0.0
    for _ in range(steps):
        flush.fill_(1.0)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        one(e0, e1)
        tot += e0.elapsed_time(e1)
    barrier(world)
    h2d = hX.numel() * hX.element_size() + (0 if hXkv is None else hXkv.numel() * hXkv.element_size())
    d2h = hY.numel() * hY.element_size()
    return {"ms": tot, "h2d": h2d, "d2h": d2h}


def measure_e2e_pipelined(w, inp, t, steps, warmup, dev, world, ws):
    """The public call (mha.forward) on a stream of batches: every step copies
    its input in from pinned host memory and its result out to pinned host
    memory, on copy streams of their own. Step i + 1's input copy is issued
    as soon as step i is enqueued, so that it and step i - 1's output copy
    run while step i computes (two device input and output buffers, events
    between the streams). The caller reads each result on the host once its
    copy is done. Timed from the first input copy to the last output copy."""
    import torch

    from head_scaled_dot_gb300 import mha
    hX = inp["X_q"].pin_memory()
    hXkv = None if inp["X_kv"] is None else inp["X_kv"].pin_memory()
    dX = [torch.empty_like(t["X_q"]) for _ in range(2)]
    dXkv = [None if hXkv is None else torch.empty_like(t["X_kv"]) for _ in range(2)]
    Y = [torch.empty((w.B, w.n_q, w.d_o), dtype=t["X_q"].dtype, device=dev) for _ in range(2)]
    hY = [torch.empty(Y[0].shape, dtype=Y[0].dtype).pin_memory() for _ in range(2)]
    cs = torch.cuda.current_stream(dev)
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev = lambda: torch.cuda.Event()
    in_ready, comp_done, out_done = [ev(), ev()], [ev(), ev()], [ev(), ev()]

    def run(n):
        first = torch.cuda.Event(enable_timing=True)
        last = torch.cuda.Event(enable_timing=True)

        def copy_in(i):
            b = i % 2
            with torch.cuda.stream(s_in):
                if i >= 2:
                    s_in.wait_event(comp_done[b])  # step i - 2 no longer reads dX[b]
                if i == 0:
                    first.record(s_in)
                dX[b].copy_(hX, non_blocking=True)
                if hXkv is not None:
                    dXkv[b].copy_(hXkv, non_blocking=True)
                in_ready[b].record(s_in)

        copy_in(0)
        for i in range(n):
            b = i % 2
            cs.wait_event(in_ready[b])
            if i >= 2:
                cs.wait_event(out_done[b])  # step i - 2's result is copied out of Y[b]
            mha.forward(dX[b], dXkv[b], t["W_Q"], t["W_K"], t["W_V"], t["W_O"], w.h, w.d_h,
                        w.d_vh, w.c, w.mask, inp["valid_len"], out=Y[b], workspace=ws,
                        stream=cs, check=False)
            comp_done[b].record(cs)
            with torch.cuda.stream(s_out):
                s_out.wait_event(comp_done[b])
                hY[b].copy_(Y[b], non_blocking=True)
                out_done[b].record(s_out)
                if i == n - 1:
                    last.record(s_out)
            if i + 1 < n:
                copy_in(i + 1)  # the next batch's input, while step i computes
            if i >= 1:
                out_done[(i - 1) % 2].synchronize()  # the caller reads step i - 1's result
        last.synchronize()
        return first.elapsed_time(last)

    run(max(warmup, 2))
    barrier(world)
    tot = run(steps)
    barrier(world)
    h2d = hX.numel() * hX.element_size() + (0 if hXkv is None else hXkv.numel() * hXkv.element_size())
    d2h = hY[0].numel() * hY[0].element_size()
    return {"ms": tot, "h2d": h2d, "d2h": d2h}


def decode_bytes(w, lens):
    """Algorithmic bytes of one decode launch: the valid part of K and V read
    once, Q read, Z written (the partial summaries are not counted)."""
    es = 2 if w.dtype == "bf16" else 4
    kv = sum(lens) * w.h * (w.d_h + w.d_vh) * es
    return kv + w.B * w.h * w.n_q * (w.d_h + w.d_vh) * es


def measure_decode(w, steps, warmup, dev, pk):
    """Times mha_attention_decode on the decode workload: inputs resident in
    HBM, L2 flushed between timed launches (outside the events)."""
    import torch

    from head_scaled_dot_gb300 import mha, workloads
    inp = workloads.make_decode_inputs(w)
    Q, K, V = (inp[k].to(dev) for k in ("Q", "K", "V"))
    lens = inp["cache_len"]
    Z = torch.empty((w.B, w.n_q, w.h * w.d_vh), dtype=Q.dtype, device=dev)
    ws = torch.empty(mha.decode_workspace_size(w.B, w.n_q, w.n_k, w.h, w.d_vh),
                     dtype=torch.uint8, device=dev)
    flush = L2Flush(dev)
    stream = torch.cuda.current_stream(dev)

    def one():
        mha.attention_decode(Q, K, V, w.c, lens, w.causal_tail, out=Z, workspace=ws,
                             stream=stream)

    for _ in range(warmup):
        flush.fill_(1.0)
        one()
    torch.cuda.synchronize(dev)
    tot = 0.0
    for _ in range(steps):
        flush.fill_(1.0)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        one()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        tot += e0.elapsed_time(e1)
    ms = tot / steps
    nbytes = decode_bytes(w, lens)
    gbs = nbytes / (ms * 1e-3) / 1e9
    return {"ms_per_launch": ms, "bytes_per_launch": nbytes,
            "roofline": {"kernel": "decode (split summaries + merge)", "bound": "hbm",
                         "achieved": gbs, "peak": pk["hbm_gbs"], "unit": "GB/s",
                         "frac": gbs / pk["hbm_gbs"],
                         # DRAM bytes of the streaming kernel (the call's dominant one)
                         "traffic": stored_traffic("decode", w.name)},
            "config": {"B": w.B, "h": w.h, "n_q": w.n_q, "n_k": w.n_k, "d_h": w.d_h,
                       "d_vh": w.d_vh, "cache_len": lens, "causal_tail": w.causal_tail}}


def oracle_sample(w, inp, lens, unit):
    """Runs the oracle as it stands on one (batch item, head) unit of the
    workload: the head's projections, its dense attention and its share of
    the output projection. Returns (seconds, flops)."""
    import oracle
    from head_scaled_dot_gb300 import workcount
    b, i = unit
    f = lambda x: None if x is None else x.double().numpy()
    X_q = f(inp["X_q"][b:b + 1])
    X_kv = None if inp["X_kv"] is None else f(inp["X_kv"][b:b + 1])
    cq = slice(i * w.d_h, (i + 1) * w.d_h)
    cv = slice(i * w.d_vh, (i + 1) * w.d_vh)
    L = None if lens is None else [lens[b]]
    t0 = time.perf_counter()
    oracle.mha_forward(X_q, X_kv, f(inp["W_Q"][:, cq]), f(inp["W_K"][:, cq]),
                       f(inp["W_V"][:, cv]), f(inp["W_O"][cv, :]), 1, w.d_h, w.d_vh, w.c,
                       oracle.MASK_NAMES[w.mask], L)
    dt = time.perf_counter() - t0
    fl = workcount.flops(w.with_(B=1, h=1), L)["total"]
    return dt, fl


def blas_threads():
    try:
        from threadpoolctl import threadpool_info
        n = [d.get("num_threads") for d in threadpool_info() if d.get("user_api") == "blas"]
        if n and n[0]:
            return int(n[0])
    except Exception:
        pass
    for k in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
        if os.environ.get(k, "").isdigit():
            return int(os.environ[k])
    return os.cpu_count()


def cpu_baseline(w, inp, lens, budget_s=12.0):
    """The oracle on (batch item, head) units of the workload, in order and
    again from the first when all are done, until about budget_s seconds of
    CPU work have been timed."""
    units = [(b, i) for b in range(w.B) for i in range(w.h)]
    secs = fl = 0.0
    done = 0
    while secs < budget_s:
        dt, f = oracle_sample(w, inp, lens, units[done % len(units)])
        secs += dt
        fl += f
        done += 1
    return {"value": fl / secs / 1e12, "unit": "TFLOP/s", "cores": blas_threads(),
            "kind": "oracle",
            "sample": "%d (batch item, head) units of %s (%.2f passes over its %d), "
                      "fp64 numpy, %.1f s" % (done, w.name, done / len(units), len(units), secs)}


def workload_config(w, lens):
    """The keys naming a workload in the JSON line (both arms)."""
    from head_scaled_dot_gb300 import workcount
    return {"workload": w.name, "B": w.B, "n_q": w.n_q, "n_k": w.n_k, "d_model": w.d_model,
            "h": w.h, "d_h": w.d_h, "d_vh": w.d_vh, "d_o": w.d_o, "mask": w.mask,
            "cross": w.cross, "seed": w.seed, "valid_len": lens,
            "gflop_per_step": workcount.flops(w, lens)["total"] / 1e9}


def run_reference(args):
    import torch
    rank, world, _ = dist_setup(args.gpus)
    if rank != 0:
        return
    from head_scaled_dot_gb300 import workloads
    w = chosen_workload(args)
    inp = workloads.make_inputs(w)
    lens = None if inp["valid_len"] is None else [int(x) for x in inp["valid_len"]]
    units = [(b, i) for b in range(w.B) for i in range(w.h)]
    for k in range(args.warmup):
        oracle_sample(w, inp, lens, units[k % len(units)])
    secs = fl = 0.0
    for k in range(args.steps):
        dt, f = oracle_sample(w, inp, lens, units[k % len(units)])
        secs += dt
        fl += f
    value = fl / secs / 1e12
    cores = blas_threads()
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * secs / args.steps, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": dict(workload_config(w, lens),
                           step="one (batch item, head) unit of the workload per step"),
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                             "sample": "one (batch item, head) unit of %s per step, %d steps"
                                       % (w.name, args.steps)},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def kernel_rows(res, pk):
    """Per kernel: the mean time of its launches (ms, the figure the rates
    use), their median and best, the rate on the effective count and its
    fraction of the measured bf16 peak (burst: the kernels are timed one by
    one; and sustained, for reference)."""
    fl = res["flops"]
    rows = {}
    for name, key in (("qkv_projection", "qkv"), ("attention", "attention"),
                      ("output_projection", "out")):
        t = res["per"][key]
        ms = sum(t) / len(t)
        tf = fl[key] / (ms * 1e-3) / 1e12
        rows[name] = {"ms": ms, "ms_median": statistics.median(t), "ms_best": min(t),
                      "tflops": tf, "frac_of_bf16_peak": tf / pk["bf16_tflops"],
                      "frac_of_bf16_peak_sustained": tf / pk["bf16_tflops_sustained"]}
    return rows


KERNEL_FILES = {"attention": "attn_tc.cu", "qkv_projection": "gemm_tc.cu",
                "output_projection": "gemm_tc.cu"}


def roofline(w, krows, pk, pk_kind, dev):
    """Roofline of the workload's dominant kernel (the largest time): the
    achieved TFLOP/s (effective count) over the measured bf16 peak, or, on
    the fp32 path (CUDA cores), over the derived fp32 FMA peak; DRAM bytes per
    launch from a committed ncu capture of the same kernel source."""
    dom = max(krows, key=lambda k: krows[k]["ms"])
    ach = krows[dom]["tflops"]
    roof = {"kernel": dom, "bound": "tensor", "achieved": ach, "peak": pk["bf16_tflops"],
            "unit": "TFLOP/s", "frac": ach / pk["bf16_tflops"], "peak_kind": pk_kind + " burst",
            "ms_per_launch": krows[dom]["ms"], "traffic": stored_traffic(dom, w.name)}
    attn_cuda_cores = w.dtype == "f32" or not all(32 <= d <= 128 and d % 8 == 0
                                                  for d in (w.d_h, w.d_vh))
    if w.dtype == "f32" or (dom == "attention" and attn_cuda_cores):
        # the fp32 path, and attention of head sizes off the tensor cores, run
        # on the CUDA cores
        alu = alu_peak_tflops(dev, sm_max_mhz())
        roof.update(bound="alu", peak=alu, frac=ach / alu,
                    peak_kind="derived: SMs x 128 FP32 lanes x 2 flop x max SM clock")
    elif dom == "attention" and w.n_q <= 128:
        # few query rows: 4 n_q d_h flop per key against 2 (d_h + d_vh) bytes of
        # K and V is below the ridge, so the bound is reading Q, K, V and
        # writing Z once
        nbytes = w.B * w.h * (w.n_q + w.n_k) * (w.d_h + w.d_vh) * 2
        gbs = nbytes / (krows[dom]["ms"] * 1e-3) / 1e9
        roof.update(bound="hbm", achieved=gbs, peak=pk["hbm_gbs"], unit="GB/s",
                    frac=gbs / pk["hbm_gbs"], peak_kind=pk_kind + " copy bandwidth",
                    bytes_per_launch=nbytes, attention_tflops=ach)
    return roof


def run_ours(args):
    import torch
    rank, world, local = dist_setup(args.gpus)
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    from head_scaled_dot_gb300 import mha, workloads
    mha.load()
    pk, pk_kind = peaks()
    w = chosen_workload(args)
    res = measure_workload(w, args.steps, args.warmup, dev, world, e2e=not args.no_e2e,
                           sample_clocks=not args.no_clocks)
    total_ms = max_over_ranks(res["total_ms"], world, dev)
    fl = res["flops"]["total"]
    value = world * fl * args.steps / (total_ms * 1e-3) / 1e12
    krows = kernel_rows(res, pk)
    roof = roofline(w, krows, pk, pk_kind, dev)
    others = {}
    if not args.no_others and rank == 0:
        for j, wj in enumerate(workloads.WORKLOADS):
            if wj.name == w.name or wj.dtype != "bf16":
                continue
            r = measure_workload(wj, max(3, args.steps // 2), 3, dev, 1, e2e=False,
                                 sample_clocks=False)
            kr = kernel_rows(r, pk)
            others[wj.name] = {"tflops": r["flops"]["total"] * len(r["per"]["step"])
                               / (r["total_ms"] * 1e-3) / 1e12,
                               "ms_per_step": r["total_ms"] / len(r["per"]["step"]),
                               "kernels": kr, "roofline": roofline(wj, kr, pk, pk_kind, dev)}
            del r
        # general head sizes: d_h = 96 (bf16 heads of 72..128 run in the
        # 128-wide tensor-core kernels), d_h = 32 (heads of 32..64 in the
        # 64-wide ones), d_h = 24 (the CUDA-core kernel, against the fp32 FMA
        # peak); the flop count uses the head size itself
        for gw in (workloads.GENERAL_DIMS, workloads.SMALL_DIMS, workloads.SIMT_DIMS):
            r = measure_workload(gw, max(3, args.steps // 2), 3, dev, 1, e2e=False,
                                 sample_clocks=False)
            kr = kernel_rows(r, pk)
            on_tc = gw.dtype == "bf16" and all(32 <= d <= 128 and d % 8 == 0
                                               for d in (gw.d_h, gw.d_vh))
            if on_tc:
                groof = {"kernel": "attention (tensor cores, head padded to %d)"
                                   % (64 if max(gw.d_h, gw.d_vh) <= 64 else 128),
                         "bound": "tensor", "peak": pk["bf16_tflops"],
                         "peak_kind": pk_kind + " burst"}
            else:
                groof = {"kernel": "attention (CUDA cores)", "bound": "alu",
                         "peak": alu_peak_tflops(dev, sm_max_mhz()),
                         "peak_kind": "derived: SMs x 128 FP32 lanes x 2 flop x max SM clock"}
            groof.update(achieved=kr["attention"]["tflops"], unit="TFLOP/s",
                         frac=kr["attention"]["tflops"] / groof["peak"],
                         ms_per_launch=kr["attention"]["ms"],
                         traffic=stored_traffic("attention", gw.name))
            others[gw.name] = {"tflops": r["flops"]["total"] * len(r["per"]["step"])
                               / (r["total_ms"] * 1e-3) / 1e12,
                               "ms_per_step": r["total_ms"] / len(r["per"]["step"]),
                               "kernels": kr, "roofline": groof}
            del r
        # few query rows against many keys: the attention step splits the keys
        # over thread blocks and merges the summaries
        for lw in workloads.LONG_KEYS:
            r = measure_workload(lw, max(3, args.steps // 2), 3, dev, 1, e2e=False,
                                 sample_clocks=False)
            kr = kernel_rows(r, pk)
            # 4 n_q d_h flop per key over 2 (d_h + d_vh) bytes of K and V: with
            # n_q <= 128 below the ridge (peak flop / copy bandwidth), so the
            # bound is reading Q, K, V and writing Z once
            es = 2
            nbytes = lw.B * lw.h * (lw.n_q * (lw.d_h + lw.d_vh) + lw.n_k * (lw.d_h + lw.d_vh)) * es
            gbs = nbytes / (kr["attention"]["ms"] * 1e-3) / 1e9
            lroof = {"kernel": "attention (keys split over thread blocks, summaries merged)",
                     "bound": "hbm", "achieved": gbs, "peak": pk["hbm_gbs"], "unit": "GB/s",
                     "frac": gbs / pk["hbm_gbs"], "bytes_per_launch": nbytes,
                     "ms_per_launch": kr["attention"]["ms"],
                     "attention_tflops": kr["attention"]["tflops"],
                     "traffic": stored_traffic("attention", lw.name)}
            others[lw.name] = {"tflops": r["flops"]["total"] * len(r["per"]["step"])
                               / (r["total_ms"] * 1e-3) / 1e12,
                               "ms_per_step": r["total_ms"] / len(r["per"]["step"]),
                               "kernels": kr, "roofline": lroof}
            del r
        dw = workloads.DECODE
        others[dw.name] = measure_decode(dw, max(3, args.steps), 3, dev, pk)
    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        cpu = cpu_baseline(w, res["inputs"], res["lens"])
    e2e = None
    if "e2e" in res:
        e = res["e2e"]
        e_ms = max_over_ranks(e["ms"], world, dev)
        es = res["e2e_serial"]
        es_ms = max_over_ranks(es["ms"], world, dev)
        e2e = {"value": world * fl * args.steps / (e_ms * 1e-3) / 1e12, "unit": "TFLOP/s",
               "h2d_bytes_per_step": e["h2d"], "d2h_bytes_per_step": e["d2h"],
               "how": "mha.forward on a stream of batches: each step's input copied in from "
                      "pinned host memory and its result copied out (both inside the timed "
                      "region), on copy streams that overlap the neighbouring steps' forward",
               "ms_per_step": e_ms / args.steps,
               "serial": {"value": world * fl * args.steps / (es_ms * 1e-3) / 1e12,
                          "ms_per_step": es_ms / args.steps,
                          "how": "copy in, forward, copy out, host read, one step at a time "
                                 "(L2 flushed before each step)"}}
    # with padding the primary count above is the effective one (valid rows
    # and keys only); the nominal count takes every row and key of the shapes
    nominal = None
    if res["lens"] is not None:
        from head_scaled_dot_gb300 import workcount
        nf = workcount.flops(w, None)["total"]
        nominal = {"gflop_per_step": nf / 1e9,
                   "dense_equivalent_tflops": world * nf * args.steps / (total_ms * 1e-3) / 1e12,
                   "note": "dense count: all n_q rows and n_k keys of every batch item. The "
                           "padded rows and keys are not computed, so this rate is not "
                           "achieved throughput (value, on the effective count, is)"}
    if rank != 0:
        return
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": total_ms / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": w.dtype,
        "data": "synthetic",
        "config": dict(workload_config(w, res["lens"]),
                       l2="flushed between timed steps (512 MiB written, then read back: clean lines only)",
                       clocks="nvidia-smi every 200 ms over a 1 s window of identical untimed "
                              "steps that ends where the timed steps begin",
                       parallelism="replicas" if world > 1 else "single GPU"),
        "frac_of_bf16_peak": value / world / pk["bf16_tflops"],
        "frac_of_bf16_peak_sustained": value / world / pk["bf16_tflops_sustained"],
        "step_ms_median": statistics.median(res["per"]["step"]),
        "step_ms_best": min(res["per"]["step"]),
        "nominal": nominal,
        "roofline": roof,
        "kernels": krows,
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": res["launches"],
        "clocks": res["clocks"],
        "other_workloads": others,
    }
    print(json.dumps(line), flush=True)


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)
    if int(os.environ.get("WORLD_SIZE", "1")) > 1:
        import torch.distributed as dist
        if dist.is_initialized():
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
