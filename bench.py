"""Benchmark: INT8-KV absorbed-MLA decode on the DeepSeek-V3-shaped workload.

One step = one decode step of the whole path for a batch of 32 sequences with
8192 cached tokens each: quantize-append of the step's new latent row (and
its RoPE key) into the INT8 cache, then decode attention over the INT8 cache
(partial scores, softmax, P.V, split-K combine).  Calibration and the
per-head scales run once before the timed region (the pages fix the
quantization parameters after calibration); they are timed separately and
reported under "calibration".

Prints one JSON line.  ``--impl reference`` times the CPU oracle on a bounded
sample of the same workload instead.
"""
import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "INT8-KV decode attn tokens/s and KV GB/s read (% of GB300 HBM peak), 1 GPU"
B, H, DL, DR, T = 32, 128, 512, 64, 8192
SOFTMAX_SCALE = 1.0 / math.sqrt(192.0)
WORKLOAD = f"dsv3-mla b{B} h{H} dl{DL} int8 dr{DR} bf16 ctx{T}"


def peaks():
    try:
        return json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))
    except Exception:
        return {}


def kv_bytes_per_step():
    # algorithmic KV bytes read per decode step: int8 latent + bf16 RoPE key per cached token
    return B * T * (DL + 2 * DR)


def flops_per_step():
    # QK over latent + RoPE (2*H*(DL+DR)) and P.V over the latent (2*H*DL), per cached token
    return B * T * 2 * H * (DL + DR + DL)


class ClockSampler:
    """Samples nvidia-smi clocks and throttle reasons around the timed region.

    Started before the timed region (and confirmed producing samples), stopped
    after it; samples whose timestamps fall within 50 ms of the region are kept.
    """

    Q = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.samples = []
        self._proc = None
        self.t0 = self.t1 = None

    def __enter__(self):
        try:
            self._proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", "10"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self._t = threading.Thread(target=self._read, daemon=True)
            self._t.start()
            deadline = time.time() + 3.0
            while not self.samples and time.time() < deadline:
                time.sleep(0.01)
        except Exception:
            self._proc = None
        return self

    def _read(self):
        for line in self._proc.stdout:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) >= 8:
                self.samples.append((time.time(), parts[1:]))

    def mark_start(self):
        self.t0 = time.time()

    def mark_end(self):
        self.t1 = time.time()
        time.sleep(0.05)

    def __exit__(self, *a):
        if self._proc is not None:
            self._proc.terminate()
            try:
                self._proc.wait(timeout=5)
            except Exception:
                self._proc.kill()

    def summary(self):
        if self.t0 is None or self.t1 is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        win = [s for t, s in self.samples if self.t0 - 0.05 <= t <= self.t1 + 0.05]
        if not win:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        num = lambda x: float(x) if x.replace(".", "", 1).isdigit() else None
        sm = [num(s[0]) for s in win if num(s[0]) is not None]
        mx = [num(s[1]) for s in win if num(s[1]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for s in win for i in range(4) if s[3 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(win),
                "window_ms": round((self.t1 - self.t0) * 1e3, 1)}


def recorded_traffic():
    """DRAM bytes per launch of mla_decode_kernel from the committed ncu record,
    or None when the kernel source has changed since that capture."""
    import hashlib
    try:
        rec = json.load(open(os.path.join(ROOT, "profiles", "traffic.json")))["mla_decode_kernel"]
        src = open(os.path.join(ROOT, rec["source"]), "rb").read()
        if hashlib.sha256(src).hexdigest() != rec["sha256"]:
            return None
        return rec["dram_bytes_per_launch"]
    except Exception:
        return None


def bench_config():
    """The workload both arms report (same keys)."""
    return {"workload": WORKLOAD, "batch": B, "heads": H, "latent": DL, "rope": DR, "context": T,
            "step": "quantize-append of the new token + MLA decode (+ split-K combine)",
            "l2": "inputs larger than L2: 167.8 MB of KV per step, two cache copies rotated"}


def calib_batch_law(gen, dev, shape=(4, H, 2048, 192), nu=3):
    """A calibration batch of the calibration-at-scale workload's law, drawn on the
    GPU: Student-t with nu = 3 (a normal over the root of a chi-square of three
    squared normals / 3), each head scaled by its own log-uniform sigma in [0.1, 10]."""
    import torch
    z = torch.randn(shape, generator=gen, device=dev)
    chi2 = sum(torch.randn(shape, generator=gen, device=dev) ** 2 for _ in range(nu))
    sig = torch.exp(torch.empty(shape[1], device=dev).uniform_(math.log(0.1), math.log(10.0), generator=gen))
    return (z * torch.rsqrt(chi2 / nu) * sig[None, :, None, None]).to(torch.bfloat16)


# ------------------------------------------------------------------ CPU oracle arm
class OracleSample:
    """The CPU oracle on whole decode sequences of the workload's shape (1 query
    token x 128 heads over 8192 cached tokens).  Four seeded sequences are drawn
    once and reused (the oracle's cost does not depend on the values)."""

    N_DISTINCT = 4

    def __init__(self):
        import workloads as W
        from oracle import fa3_oracle as O
        self.O = O
        w = W.mla_dsv3(B=self.N_DISTINCT, T=T)
        self.w = w
        self.inp = W.mla_inputs(w, with_calib=False)
        rng = np.random.default_rng(1)
        self.q_scale = rng.uniform(0.02, 0.04, H).astype(np.float32)
        self.kv_scale = np.float32(np.abs(self.inp.ckv).max() / 127)
        self.ckv8 = O.quantize(self.inp.ckv, self.kv_scale)

    def one(self, i):
        b = i % self.N_DISTINCT
        return self.O.mla_decode(self.inp.q[b:b + 1], self.ckv8[b:b + 1], self.inp.krope[b:b + 1], self.q_scale,
                                 float(self.kv_scale), self.inp.lens[b:b + 1], self.w.softmax_scale)

    def run(self, n_seq, threads):
        """Decodes n_seq sequences, `threads` at a time (numpy releases the GIL in its
        matmuls); returns the elapsed seconds."""
        from concurrent.futures import ThreadPoolExecutor
        t0 = time.perf_counter()
        if threads <= 1:
            for i in range(n_seq):
                self.one(i)
        else:
            with ThreadPoolExecutor(max_workers=threads) as ex:
                list(ex.map(self.one, range(n_seq)))
        return time.perf_counter() - t0


def _blas_limit(n):
    """Limits numpy's BLAS threads to n where threadpoolctl is installed."""
    try:
        from threadpoolctl import threadpool_limits
        return threadpool_limits(n), True
    except Exception:
        import contextlib
        return contextlib.nullcontext(), False


def cpu_baseline(seconds=8.0):
    """The oracle timed on the host cores, single-threaded and on every core."""
    cores = len(os.sched_getaffinity(0))
    smp = OracleSample()
    smp.run(1, 1)                                                     # warm
    lim, limited = _blas_limit(1)
    with lim:
        n1, el1 = 0, 0.0
        while el1 < seconds / 2 and n1 < 16:
            el1 += smp.run(1, 1)
            n1 += 1
    nall, elall = 0, 0.0
    while elall < seconds / 2 and nall < 8 * B:
        elall += smp.run(B, cores)
        nall += B
    single = {"value": n1 / el1, "unit": "tokens/s", "cores": 1,
              "sample": f"{n1} sequences one after another in {el1:.1f} s"
                        + ("" if limited else " (numpy's BLAS threads not limited: threadpoolctl absent; the "
                                              "int64 latent matmul, most of the work, is single-threaded)")}
    return {"value": nall / elall, "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "sample": f"{nall} whole decode sequences of the workload's shape (1 token x 128 heads x 8192 ctx) in "
                      f"{elall:.1f} s, {cores} sequences at a time on {cores} threads, numpy",
            "single_thread": single}


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    cores = len(os.sched_getaffinity(0))
    smp = OracleSample()
    # a step is the workload's 32 sequences, fewer if W + K whole steps would take
    # more than about two minutes; the line states how many were timed per step
    par = min(B, cores)
    t1 = smp.run(par, cores) / par                                   # seconds per sequence, all cores busy
    n_seq = B
    while n_seq > 1 and (args.warmup + args.steps) * max(n_seq, par) * t1 * 1.2 > 120.0:
        n_seq //= 2
    for _ in range(args.warmup):
        smp.run(n_seq, cores)
    el = [smp.run(n_seq, cores) for _ in range(args.steps)]
    total = sum(el)
    rate = n_seq * args.steps / total
    line = {
        "impl": "reference", "metric": METRIC, "value": rate, "unit": "tokens/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / args.steps,
        "sequences_per_step": n_seq,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "i8 codes, f64 arithmetic",
        "data": "synthetic", "config": bench_config(),
        "cpu_baseline": {"value": rate, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                         "sample": f"each step decodes {n_seq} whole sequences of the workload's shape (1 query "
                                   f"token x 128 heads over 8192 cached tokens), {cores} at a time on {cores} "
                                   f"threads, numpy; ms_per_step is the measured time of such a step"},
        "e2e": {"value": rate, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def slowest_rank_ms(ms_local, world, device):
    """The largest of the ranks' times (every rank's units are counted against it)."""
    if world <= 1:
        return float(ms_local)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(ms_local)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(units_per_rank, ms_slowest, world):
    """Units per second of the whole job: all ranks' units over the slowest rank's time."""
    return units_per_rank * world / (ms_slowest / 1e3)


# ------------------------------------------------------------------ GPU arm
def run_gpu(args):
    import torch
    import torch.distributed as dist

    import __graft_entry__ as G
    from int8_head_kv_gb300 import fa3 as F

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    G.build()
    stream = torch.cuda.current_stream()

    gen = torch.Generator(device=dev)
    gen.manual_seed(1234 + rank)
    # ---- synthetic activations (bf16), the workload's laws: N(0,1) queries, latent N(0, sigma) + 0.1% x20
    sig_kv = float(np.exp(np.random.default_rng(rank).uniform(math.log(0.1), math.log(10.0))))

    def latent(shape):
        x = torch.randn(shape, generator=gen, device=dev) * sig_kv
        m = torch.rand(shape, generator=gen, device=dev) < 1e-3
        return torch.where(m, x * 20, x).to(torch.bfloat16)

    # ---- calibration of the per-head query scale and the latent scale (timed separately)
    calib_q = [torch.randn(32, H, 1, DL, generator=gen, device=dev).to(torch.bfloat16) for _ in range(3)]
    calib_kv = [latent((1, 1, T, DL)) for _ in range(3)]
    qmn = torch.full((H,), float("inf"), device=dev); qmx = torch.full((H,), float("-inf"), device=dev)
    kmn = torch.full((1,), float("inf"), device=dev); kmx = torch.full((1,), float("-inf"), device=dev)
    # big calibration batch (B=4, H=128, S=2048, D=192 bf16) for the calibration throughput figure
    cal_big = calib_batch_law(gen, dev)
    cmn = torch.full((H,), float("inf"), device=dev); cmx = torch.full((H,), float("-inf"), device=dev)
    for _ in range(3):
        F.calibrate_perhead(cal_big, 0.9999, cmn, cmx)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    n_cal = 10
    for _ in range(n_cal):
        F.calibrate_perhead(cal_big, 0.9999, cmn, cmx)
    e1.record(stream)
    torch.cuda.synchronize()
    cal_ms = e0.elapsed_time(e1) / n_cal
    # the same call replayed from a CUDA graph: its three kernels without the host's per-call work
    cws = torch.zeros(F.calibrate_workspace_size(H), dtype=torch.uint8, device=dev)
    cst = torch.cuda.Stream()
    torch.cuda.synchronize()
    with torch.cuda.stream(cst):
        F.calibrate_perhead(cal_big, 0.9999, cmn, cmx, workspace=cws, stream=cst)
    cst.synchronize()
    cgraph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(cgraph, stream=cst):
        for _ in range(n_cal):
            F.calibrate_perhead(cal_big, 0.9999, cmn, cmx, workspace=cws, stream=cst)
    cgraph.replay()
    torch.cuda.synchronize()
    e0.record()
    for _ in range(3):
        cgraph.replay()
    e1.record()
    torch.cuda.synchronize()
    cal_graph_ms = e0.elapsed_time(e1) / (3 * n_cal)
    del cgraph, cws
    for x in calib_q:
        F.calibrate_perhead(x, 0.9999, qmn, qmx)
    for x in calib_kv:
        F.calibrate_perhead(x, 0.9999, kmn, kmx)
    q_scale = F.qparams(qmn, qmx)
    kv_scale = F.qparams(kmn, kmx)
    del cal_big

    # ---- the other attention calls at their workloads' shapes (reported beside the step)
    def timed(fn, n, rounds=3):
        # median over `rounds` timed batches of n calls (one batch swings with the host's timing)
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        per = []
        for _ in range(rounds):
            a, z = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            for _ in range(n):
                fn()
            z.record(stream)
            torch.cuda.synchronize()
            per.append(a.elapsed_time(z) / n)
        return sorted(per)[len(per) // 2]

    def i8(shape):
        return torch.randint(-127, 128, shape, dtype=torch.int8, device=dev, generator=gen)

    gB, gHq, gHkv, gD, gT = 16, 64, 8, 128, 4096
    # two cache copies used in turn: 2 x 134 MB, more than L2 holds
    gkv = [(i8((gB, gT, gHkv, gD)), i8((gB, gT, gHkv, gD))) for _ in range(2)]
    gq = i8((gB, gHq, gD))
    gs1, gs2 = torch.full((gHq,), 0.01, device=dev), torch.full((gHkv,), 0.01, device=dev)
    glens = torch.full((gB,), gT, dtype=torch.int32, device=dev)
    gstep = [0]

    def gqa_call():
        gk, gv = gkv[gstep[0] & 1]
        gstep[0] += 1
        F.decode_attn_gqa(gq, gk, gv, gs1, gs2, gs2, glens, 1 / math.sqrt(128))

    gqa_ms = timed(gqa_call, 50)
    # the same calls replayed from a CUDA graph, as a serving loop issues them: the
    # GPU time of a call without the host's per-call work
    gout = torch.empty(gB, gHq, gD, dtype=torch.bfloat16, device=dev)
    gws = torch.zeros(max(16, F.gqa_workspace_size(gB, gHq, gHkv, gD, gT)), dtype=torch.uint8, device=dev)
    gst = torch.cuda.Stream()
    torch.cuda.synchronize()
    with torch.cuda.stream(gst):
        for i in range(3):
            F.decode_attn_gqa(gq, gkv[i & 1][0], gkv[i & 1][1], gs1, gs2, gs2, glens, 1 / math.sqrt(128),
                              out=gout, workspace=gws, stream=gst)
    gst.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=gst):
        for i in range(20):
            F.decode_attn_gqa(gq, gkv[i & 1][0], gkv[i & 1][1], gs1, gs2, gs2, glens, 1 / math.sqrt(128),
                              out=gout, workspace=gws, stream=gst)
    graph.replay()
    torch.cuda.synchronize()
    ga, gz = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ga.record()
    for _ in range(5):
        graph.replay()
    gz.record()
    torch.cuda.synchronize()
    gqa_graph_ms = ga.elapsed_time(gz) / 100
    del graph, gkv
    pS = 4096
    pq, pk, pv = i8((1, pS, gHq, gD)), i8((1, pS, gHkv, gD)), i8((1, pS, gHkv, gD))
    pl = torch.full((1,), pS, dtype=torch.int32, device=dev)
    pout = torch.empty(1, pS, gHq, gD, dtype=torch.bfloat16, device=dev)
    pre_ms = timed(lambda: F.prefill_attn_gqa(pq, pk, pv, gs1, gs2, gs2, pl, pl, 1 / math.sqrt(128), out=pout), 5)
    pre_flop = gHq * (pS * (pS + 1) // 2) * 4 * gD
    del pq, pk, pv, pout

    # ---- two independent INT8 caches (rotated per step so consecutive steps share no data)
    NC = 2
    caches, ropes, qs = [], [], []
    zero_pos = torch.zeros(B, dtype=torch.int32, device=dev)
    for _ in range(NC):
        c8 = torch.empty(B, T, 1, DL, dtype=torch.int8, device=dev)
        kr = torch.empty(B, T, DR, dtype=torch.bfloat16, device=dev)
        for b0 in range(0, B, 8):
            F.quantize_append(latent((8, T, 1, DL)), kv_scale, c8[b0:b0 + 8], zero_pos[:8],
                              torch.randn(8, T, DR, generator=gen, device=dev).to(torch.bfloat16), kr[b0:b0 + 8])
        caches.append(c8)
        ropes.append(kr)
        qs.append(torch.randn(B, H, DL + DR, generator=gen, device=dev).to(torch.bfloat16))
    new_kv = [latent((B, 1, 1, DL)) for _ in range(NC)]
    new_rope = [torch.randn(B, 1, DR, generator=gen, device=dev).to(torch.bfloat16) for _ in range(NC)]
    pos = torch.full((B,), T - 1, dtype=torch.int32, device=dev)     # the step's token is the last one
    lens = torch.full((B,), T, dtype=torch.int32, device=dev)
    out = torch.empty(B, H, DL, dtype=torch.float32, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    ws = torch.empty(F.mla_workspace_size(B, H, DL, T), dtype=torch.uint8, device=dev)

    def step(i, ev=None, kev=None):
        c = i % NC
        F.quantize_append(new_kv[c], kv_scale, caches[c], pos, new_rope[c], ropes[c], err)
        if ev is not None:
            ev[0].record(stream)                     # the whole decode call
        if kev is not None:
            F.set_kernel_timing(kev[0], kev[1])      # its main kernel, recorded by the library
        F.decode_attn_mla(qs[c], caches[c][:, :, 0], ropes[c], q_scale, kv_scale, lens, SOFTMAX_SCALE, out=out,
                          workspace=ws, dev_err=err)
        if ev is not None:
            ev[1].record(stream)

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    if int(err.item()) != 0:
        raise RuntimeError(f"device error word {int(err.item())}")

    mla_ev = [tuple(torch.cuda.Event(enable_timing=True) for _ in range(2)) for _ in range(args.steps)]
    kern_ev = [tuple(torch.cuda.Event(enable_timing=True) for _ in range(2)) for _ in range(args.steps)]
    for evs in mla_ev + kern_ev:                        # create the CUDA events before the timed region
        for e in evs:
            e.record(stream)
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()
        clk.mark_start()
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0.record(stream)
        for i in range(args.steps):
            step(i)
        t1.record(stream)
        torch.cuda.synchronize()
        # Second pass of the same steps with events around the decode call and its main
        # kernel: an event between two kernels stops their programmatic launch overlap,
        # so the step time above is taken without them.
        for i in range(args.steps):
            step(i, mla_ev[i], kern_ev[i])
        torch.cuda.synchronize()
        clk.mark_end()
        if world > 1:
            dist.barrier()
    ms_total = slowest_rank_ms(t0.elapsed_time(t1), world, dev)
    F.set_kernel_timing(None, None)
    ms_step = ms_total / args.steps
    mla_ms = statistics.mean(ev[0].elapsed_time(ev[1]) for ev in mla_ev)
    kern_ms = statistics.mean(ev[0].elapsed_time(ev[1]) for ev in kern_ev)

    # ---- end to end through the public API with host buffers (pinned), copies inside the timed region
    hq = qs[0].cpu().pin_memory()
    hkv = new_kv[0].cpu().pin_memory()
    hrope = new_rope[0].cpu().pin_memory()
    hlens = lens.cpu().pin_memory()
    hpos = pos.cpu().pin_memory()
    hout = torch.empty(B, H, DL, dtype=torch.float32).pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in (hq, hkv, hrope, hlens, hpos))
    d2h = hout.numel() * hout.element_size()
    # Serving-style loop: two sets of device buffers; step i+1's inputs are copied in
    # on one copy stream and step i-1's output copied out on another while step i
    # computes on the main stream (events order every reuse of a buffer).
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    NBUF = 2
    dins = [(torch.empty_like(qs[0]), torch.empty_like(new_kv[0]), torch.empty_like(new_rope[0]),
             torch.empty_like(lens), torch.empty_like(pos)) for _ in range(NBUF)]
    douts = [torch.empty_like(out) for _ in range(NBUF)]
    houts = [hout] + [torch.empty_like(hout).pin_memory() for _ in range(NBUF - 1)]
    ev_in = [torch.cuda.Event() for _ in range(NBUF)]
    ev_used = [torch.cuda.Event() for _ in range(NBUF)]
    ev_comp = [torch.cuda.Event() for _ in range(NBUF)]
    ev_copied = [torch.cuda.Event() for _ in range(NBUF)]

    def e2e_step(i):
        c, k = i % NC, i % NBUF
        dq, dkv, drope, dl, dp = dins[k]
        s_in.wait_event(ev_used[k])                  # step i-2 has consumed these input buffers
        with torch.cuda.stream(s_in):
            dq.copy_(hq, non_blocking=True); dkv.copy_(hkv, non_blocking=True); drope.copy_(hrope, non_blocking=True)
            dl.copy_(hlens, non_blocking=True); dp.copy_(hpos, non_blocking=True)
        ev_in[k].record(s_in)
        stream.wait_event(ev_in[k])
        stream.wait_event(ev_copied[k])              # step i-2's output has left this buffer
        F.quantize_append(dkv, kv_scale, caches[c], dp, drope, ropes[c], err)
        F.decode_attn_mla(dq, caches[c][:, :, 0], ropes[c], q_scale, kv_scale, dl, SOFTMAX_SCALE, out=douts[k],
                          workspace=ws, dev_err=err)
        ev_used[k].record(stream)
        ev_comp[k].record(stream)
        s_out.wait_event(ev_comp[k])
        with torch.cuda.stream(s_out):
            houts[k].copy_(douts[k], non_blocking=True)
        ev_copied[k].record(s_out)

    def e2e_run(n):
        s_in.wait_stream(stream)
        s_out.wait_stream(stream)
        for i in range(n):
            e2e_step(i)
        stream.wait_stream(s_out)                    # the last output is on the host

    e2e_run(args.warmup)
    torch.cuda.synchronize()
    a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a0.record(stream)
    e2e_run(args.steps)
    a1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = slowest_rank_ms(a0.elapsed_time(a1), world, dev) / args.steps
    if int(err.item()) != 0:
        raise RuntimeError(f"device error word {int(err.item())}")

    pk = peaks()
    hbm = pk.get("hbm_gbs", 6800.0)
    bf16 = pk.get("bf16_tflops", 1900.0)
    tokens = B * world
    value = whole_job_rate(B, ms_step, world)
    kv_gbs = kv_bytes_per_step() / (mla_ms / 1e3) / 1e9           # whole decode call
    k_tflops = flops_per_step() / (kern_ms / 1e3) / 1e12          # main kernel alone
    k_gbs = kv_bytes_per_step() / (kern_ms / 1e3) / 1e9
    traffic = recorded_traffic()
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu:
        cpu = cpu_baseline(seconds=args.cpu_seconds)
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "i8 KV codes; f16 tensor-core MMA (exact integer latent partials); f32 softmax/accum",
        "data": "synthetic",
        "config": bench_config(),
        "kv_gbs": kv_gbs, "kv_hbm_frac_of_measured": kv_gbs / hbm,
        "roofline": {"bound": "tensor", "achieved": k_tflops, "peak": bf16, "unit": "TFLOP/s",
                     "frac": k_tflops / bf16, "traffic": traffic,
                     "kernel": "mla_decode_kernel", "ms_per_launch": kern_ms,
                     "algorithmic": f"{flops_per_step() / 1e9:.2f} GFLOP per launch (2*B*T*H*(2*Dl+Dr))",
                     "timing": "CUDA events recorded by the library around the kernel (fa3_set_kernel_timing), "
                               "on the launching stream, in a second timed pass of the same steps (the "
                               "step time is taken without any events between the kernels, which would "
                               "stop their programmatic launch overlap)",
                     "peak_source": "measured bf16 dense burst (MEASURED_PEAKS.json), of measured; f16 runs at "
                                    "the bf16 rate",
                     "frac_of_sustained": k_tflops / pk.get("bf16_tflops_sustained", bf16)},
        "hbm_roofline": {"kernel": "mla_decode_kernel", "achieved": k_gbs, "peak": hbm, "unit": "GB/s",
                         "frac": k_gbs / hbm},
        "decode_call": {"ms": mla_ms, "kv_gbs": kv_gbs, "tflops": flops_per_step() / (mla_ms / 1e3) / 1e12,
                        "kernels": "query pre-pass + mla_decode_kernel + split-K combine",
                        "timing": "CUDA events around the call, second timed pass"},
        "gqa_decode": {"workload": "llama70b-gqa b16 hq64 hkv8 d128 ctx4096, int8 q/k/v (one call: decode + combine; "
                                   "two cache copies used in turn)",
                       "us_per_call": gqa_ms * 1e3, "kv_gbs": gB * gT * gHkv * gD * 2 / (gqa_ms / 1e3) / 1e9,
                       "hbm_frac_of_measured": gB * gT * gHkv * gD * 2 / (gqa_ms / 1e3) / 1e9 / hbm,
                       "us_per_call_graph": gqa_graph_ms * 1e3,
                       "hbm_frac_of_measured_graph": gB * gT * gHkv * gD * 2 / (gqa_graph_ms / 1e3) / 1e9 / hbm},
        "prefill": {"workload": "llama70b-prefill b1 s4096 t4096 hq64 hkv8 d128 causal, int8 q/k/v",
                    "us_per_call": pre_ms * 1e3, "tflops": pre_flop / (pre_ms / 1e3) / 1e12,
                    "frac_of_measured_bf16": pre_flop / (pre_ms / 1e3) / 1e12 / bf16},
        "calibration": {"workload": "B=4 H=128 S=2048 D=192 bf16, ratio 0.9999, Student-t nu=3 x per-head "
                                    "log-uniform [0.1, 10] sigma", "ms_per_batch": cal_ms,
                        "gbs": 4 * H * 2048 * 192 * 2 / (cal_ms / 1e3) / 1e9,
                        "ms_per_batch_graph": cal_graph_ms,
                        "hbm_frac_of_measured_graph": 4 * H * 2048 * 192 * 2 / (cal_graph_ms / 1e3) / 1e9 / hbm},
        "cpu_baseline": cpu,
        "e2e": {"value": tokens / (e2e_ms / 1e3), "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h,
                "loop": "public API calls; each step copies its inputs from pinned host memory and its output "
                        "back, on two copy streams that overlap the neighbouring steps' compute"},
        "gpu_launches": 4 * args.steps,   # per step: quantize-append, query pre-pass, decode, combine
        "clocks": clk.summary(),
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def run_kernel(args):
    """Runs one kernel alone (for ncu captures): prints its mean time per call."""
    import torch
    import __graft_entry__ as G
    from int8_head_kv_gb300 import fa3 as F
    G.build()
    dev = torch.device("cuda")
    g = torch.Generator(device=dev)
    g.manual_seed(0)
    k = args.kernel
    if k == "mla":
        ckv = torch.randint(-127, 128, (B, T, DL), dtype=torch.int8, device=dev, generator=g)
        kr = torch.randn(B, T, DR, device=dev, generator=g).to(torch.bfloat16)
        q = torch.randn(B, H, DL + DR, device=dev, generator=g).to(torch.bfloat16)
        qs, kvs = torch.full((H,), 0.03, device=dev), torch.full((1,), 0.02, device=dev)
        lens = torch.full((B,), T, dtype=torch.int32, device=dev)
        out = torch.empty(B, H, DL, device=dev)
        ws = torch.empty(F.mla_workspace_size(B, H, DL, T), dtype=torch.uint8, device=dev)
        fn = lambda: F.decode_attn_mla(q, ckv, kr, qs, kvs, lens, SOFTMAX_SCALE, out=out, workspace=ws)
        unit = ("KV GB/s", kv_bytes_per_step())
    elif k == "mla_paged":
        # the same workload in a pool of 64-token pages stored in shuffled order
        ckv = torch.randint(-127, 128, (B, T, DL), dtype=torch.int8, device=dev, generator=g)
        kr = torch.randn(B, T, DR, device=dev, generator=g).to(torch.bfloat16)
        q = torch.randn(B, H, DL + DR, device=dev, generator=g).to(torch.bfloat16)
        qs, kvs = torch.full((H,), 0.03, device=dev), torch.full((1,), 0.02, device=dev)
        lens = torch.full((B,), T, dtype=torch.int32, device=dev)
        P, mp = 64, T // 64
        perm = torch.randperm(B * mp, device=dev, generator=g)
        ckv_pool = torch.empty(B * mp, P, DL, dtype=torch.int8, device=dev)
        kr_pool = torch.empty(B * mp, P, DR, dtype=torch.bfloat16, device=dev)
        ckv_pool[perm] = ckv.reshape(B * mp, P, DL)
        kr_pool[perm] = kr.reshape(B * mp, P, DR)
        del ckv, kr
        bt = perm.reshape(B, mp).to(torch.int32).contiguous()
        out = torch.empty(B, H, DL, device=dev)
        ws = torch.empty(F.mla_workspace_size(B, H, DL, T), dtype=torch.uint8, device=dev)
        fn = lambda: F.decode_attn_mla_paged(q, ckv_pool, kr_pool, qs, kvs, lens, bt, SOFTMAX_SCALE, out=out,
                                             workspace=ws)
        unit = ("KV GB/s", kv_bytes_per_step())
    elif k == "gqa_paged":
        Bq, Hq, Hkv, D, Tq, P = 16, 64, 8, 128, 4096, 16
        mp = Tq // P
        kp = torch.randint(-127, 128, (Bq * mp, P, Hkv, D), dtype=torch.int8, device=dev, generator=g)
        vp = torch.randint(-127, 128, (Bq * mp, P, Hkv, D), dtype=torch.int8, device=dev, generator=g)
        q8 = torch.randint(-127, 128, (Bq, Hq, D), dtype=torch.int8, device=dev, generator=g)
        s1, s2 = torch.full((Hq,), 0.01, device=dev), torch.full((Hkv,), 0.01, device=dev)
        lens = torch.full((Bq,), Tq, dtype=torch.int32, device=dev)
        bt = torch.randperm(Bq * mp, device=dev, generator=g).reshape(Bq, mp).to(torch.int32).contiguous()
        fn = lambda: F.decode_attn_gqa_paged(q8, kp, vp, s1, s2, s2, lens, bt, 1 / math.sqrt(128))
        unit = ("KV GB/s", Bq * Tq * Hkv * D * 2)
    elif k == "gqa":
        Bq, Hq, Hkv, D, Tq = 16, 64, 8, 128, 4096
        # two cache copies used in turn (2 x 134 MB: more than L2 holds)
        kvs = [(torch.randint(-127, 128, (Bq, Tq, Hkv, D), dtype=torch.int8, device=dev, generator=g),
                torch.randint(-127, 128, (Bq, Tq, Hkv, D), dtype=torch.int8, device=dev, generator=g))
               for _ in range(2)]
        q8 = torch.randint(-127, 128, (Bq, Hq, D), dtype=torch.int8, device=dev, generator=g)
        s1, s2 = torch.full((Hq,), 0.01, device=dev), torch.full((Hkv,), 0.01, device=dev)
        lens = torch.full((Bq,), Tq, dtype=torch.int32, device=dev)
        step = [0]

        def fn():
            kc, vc = kvs[step[0] & 1]
            step[0] += 1
            F.decode_attn_gqa(q8, kc, vc, s1, s2, s2, lens, 1 / math.sqrt(128))
        unit = ("KV GB/s", Bq * Tq * Hkv * D * 2)
    elif k == "prefill":
        # Llama-3.1-70B-shaped causal prefill: S = T new rows per sequence, 64 / 8 heads
        Bp, S_, Hq, Hkv, D = args.prefill_batch, args.prefill_len, 64, 8, 128
        q8 = torch.randint(-127, 128, (Bp, S_, Hq, D), dtype=torch.int8, device=dev, generator=g)
        kc = torch.randint(-127, 128, (Bp, S_, Hkv, D), dtype=torch.int8, device=dev, generator=g)
        vc = torch.randint(-127, 128, (Bp, S_, Hkv, D), dtype=torch.int8, device=dev, generator=g)
        s1, s2 = torch.full((Hq,), 0.003, device=dev), torch.full((Hkv,), 0.003, device=dev)
        ql = torch.full((Bp,), S_, dtype=torch.int32, device=dev)
        out = torch.empty(Bp, S_, Hq, D, dtype=torch.bfloat16, device=dev)
        fn = lambda: F.prefill_attn_gqa(q8, kc, vc, s1, s2, s2, ql, ql, 1 / math.sqrt(128), out=out)
        # causal: row i sees i + 1 keys; 2 contractions of 2*D flop per (row, head, key)
        unit = ("TFLOP/s", Bp * Hq * (S_ * (S_ + 1) // 2) * 4 * D / 1e3)
    elif k == "calib":
        x = calib_batch_law(g, dev)
        mn, mx = torch.full((H,), float("inf"), device=dev), torch.full((H,), float("-inf"), device=dev)
        fn = lambda: F.calibrate_perhead(x, 0.9999, mn, mx)
        unit = ("GB/s", x.numel() * 2)
    else:
        kv = torch.randn(32, args.t_new, 1, 512, device=dev, generator=g).to(torch.bfloat16)
        cache = torch.zeros(32, max(1024, args.t_new), 1, 512, dtype=torch.int8, device=dev)
        pos = torch.zeros(32, dtype=torch.int32, device=dev)
        # the scale the Recall-Window calibration gives for these values
        mn, mx = torch.full((1,), float("inf"), device=dev), torch.full((1,), float("-inf"), device=dev)
        F.calibrate_perhead(kv.transpose(1, 2).contiguous(), 0.9999, mn, mx)
        sc = F.qparams(mn, mx)
        fn = lambda: F.quantize_append(kv, sc, cache, pos)
        k = f"append t_new={args.t_new}"
        unit = ("GB/s", kv.numel() * 3)
    for _ in range(args.warmup):
        fn()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(args.steps):
        fn()
    e1.record()
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / args.steps
    print(json.dumps({"kernel": k, "us_per_call": ms * 1e3, unit[0]: unit[1] / (ms / 1e3) / 1e9}), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--prefill-len", type=int, default=4096, help="S = T for --kernel prefill")
    ap.add_argument("--prefill-batch", type=int, default=2, help="sequences for --kernel prefill")
    ap.add_argument("--kernel", choices=["mla", "mla_paged", "gqa", "gqa_paged", "calib", "append", "prefill"],
                    help="run one kernel alone (for profiling) instead of the benchmark step")
    ap.add_argument("--t-new", type=int, default=64, help="new tokens per sequence for --kernel append")
    args = ap.parse_args()
    if args.kernel:
        run_kernel(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
