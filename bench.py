#!/usr/bin/env python
"""KDA forward benchmark on GB300: prefill tokens/s (headline), % of roofline,
and decode steps/s.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

A step is one ``kda_chunk_fwd`` call over the whole workload (default: the
B=4 H=32 T=8192 d=128 bf16 prefill), inputs resident in HBM.  Each rank runs
its own copy of the workload (units are independent: weak scaling, no
collective on the data path); the barrier and the max over ranks bracket the
timed region.  Rank 0 prints one JSON line.

``--impl reference`` times the fp64 CPU oracle on the host cores instead (a
bounded sample of the same workload per step); it is the only other place that
runs ``oracle/``.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

SMI_FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
KERNEL_SRC = {"tc": "linear_attention_fwd_gb300/csrc/kda_chunk_tc.cu",
              "simt": "linear_attention_fwd_gb300/csrc/kda_chunk_simt.cu",
              "decode": "linear_attention_fwd_gb300/csrc/kda_decode.cu",
              "two_pass": "linear_attention_fwd_gb300/csrc/kda_chunk_state.cu"}
KERNEL_NAME = {"tc": "kda_chunk_tc_kernel", "simt": "kda_chunk_simt_kernel",
               "decode": "kda_recurrent_step_kernel",
               "two_pass": "kda_chunk_prep_kernel+kda_chunk_state_kernel"}
# kernels one prefill step launches: the two-pass path scans the chunk counts, then runs
# its chunk-parallel pass and its state pass
LAUNCHES_PER_STEP = {"tc": 1, "simt": 1, "two_pass": 3}


# ----------------------------------------------------------------------------- helpers
def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def rank_ops(ws, device):
    """The timing contract's cross-rank steps for an initialised process group (any backend):
    a barrier, and the maximum of a per-rank value over all ranks."""
    import torch
    import torch.distributed as dist

    def barrier():
        if ws > 1:
            dist.barrier()

    def max_over_ranks(x):
        if ws == 1:
            return x
        t = torch.tensor([x], dtype=torch.float64, device=device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        return float(t.item())

    return barrier, max_over_ranks


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return dict(hbm=float(d["hbm_gbs"]), bf16=float(d["bf16_tflops"]),
                    bf16_sust=float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                    src="measured")
    return dict(hbm=6800.0, bf16=1900.0, bf16_sust=1700.0, src="fallback")


PEAK_NOTE = ("copy bandwidth measured by the driver (a torch copy, read + write bytes): a "
             "lower bound on what the memory system delivers, so a streaming kernel can read "
             "slightly above 1.0")


def hbm_roofline(bytes_launch, ms, P, **extra):
    """Roofline entry against the measured HBM copy peak; a fraction above 1 is flagged."""
    ach = bytes_launch / (ms / 1e3) / 1e9
    r = {"bound": "hbm", "achieved": ach, "peak": P["hbm"], "unit": "GB/s", "frac": ach / P["hbm"],
         "peak_source": P["src"], "algorithmic_bytes_per_launch": bytes_launch}
    if ach > P["hbm"]:
        r["above_copy_peak"] = True
        r["peak_note"] = PEAK_NOTE
    r.update(extra)
    return r


def sha256(path):
    with open(os.path.join(ROOT, path), "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()


def recorded_traffic(kernel, workload):
    """DRAM bytes per launch from a committed ncu summary, if the kernel source
    is unchanged since the counters were taken; else None."""
    p = os.path.join(ROOT, "profiles", "dram_traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    e = d.get(f"{kernel}:{workload}")
    if not e or e.get("source_sha256") != sha256(KERNEL_SRC[kernel]):
        return None
    return float(e["bytes_per_launch"])


class ClockSampler:
    """nvidia-smi samples of SM clock / throttle reasons while the timed region runs."""

    def __init__(self, gpu_index: int, period_ms: int = 100):
        self.rows, self.proc, self.th = [], None, None
        self.cmd = ["nvidia-smi", f"--query-gpu={SMI_FIELDS}", "--format=csv,noheader,nounits",
                    "-i", str(gpu_index), "-lms", str(period_ms)]

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(self.cmd, stdout=subprocess.PIPE,
                                         stderr=subprocess.DEVNULL, text=True)
        except (FileNotFoundError, OSError):
            self.proc = None
            return self
        self.th = threading.Thread(target=self._read, daemon=True)
        self.th.start()
        time.sleep(0.3)
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.rows.append([x.strip() for x in line.split(",")])

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            if self.th is not None:
                self.th.join(timeout=5)

    def summary(self):
        if self.proc is None:
            return None
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in self.rows:
            if len(r) < 9:
                continue
            try:
                sm.append(float(r[1])); mx.append(float(r[2]))
            except ValueError:
                continue
            for n, v in zip(names, r[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm)}


def algorithmic_bytes(tokens, heads, dk, dv, es, num_seqs, state_in):
    """q, k, g (dk each), v, o (dv each), beta per token per head, plus the fp32
    final state written (and the initial state read, when given)."""
    per_tok = (3 * dk + 2 * dv + 1) * es
    state = num_seqs * heads * dk * dv * 4 * (2 if state_in else 1)
    return tokens * heads * per_tok + state


def chunk_flops(tokens, heads, dk, dv, C=64):
    """Tensor work of the chunk form per token per head: W S, Qbar S, Kp^T U
    (2 dk dv each) + A, M (lower halves, C dk) + T(beta K), T(beta V) (C dk,
    C dv) + M U (C dv), i.e. 6 dk dv + C (4 dk + 3 dv) at C = 64."""
    return tokens * heads * (6 * dk * dv + C * (4 * dk + 3 * dv))


# ----------------------------------------------------------------------------- oracle timing
def oracle_rate(inp, budget_s):
    """fp64 oracle throughput on a bounded sample of whole (sequence, head)
    units, run in parallel batches of one unit per host thread until about
    ``budget_s`` seconds of oracle time have passed (input conversion is not
    timed).  Returns (tokens/s scaled to all heads, threads, description, s)."""
    import itertools
    from concurrent.futures import ThreadPoolExecutor

    import oracle
    q = inp["q"]
    B, T, H, dk = q.shape
    cu = inp.get("cu_seqlens")
    if cu is None:
        lens = [T] * B
    else:
        c = cu.cpu().tolist()
        lens = [b - a for a, b in zip(c[:-1], c[1:])]
    starts = [0] + list(itertools.accumulate(lens))
    threads = oracle.default_threads()
    units = [(n, h) for h in range(H) for n in range(len(lens))]
    s0 = inp.get("initial_state")

    def unit_args(n, h):
        if cu is None:
            sel = lambda t: t[n:n + 1, :, h:h + 1]
        else:
            sel = lambda t: t[:, starts[n]:starts[n + 1], h:h + 1]
        return ([oracle._f64(sel(inp[x])) for x in ("q", "k", "v", "g")]
                + [oracle._f64(sel(inp["beta"].unsqueeze(-1))[..., 0])]
                + [None if s0 is None else oracle._f64(s0[n:n + 1, h:h + 1])])

    elapsed, done, used = 0.0, 0, 0
    with ThreadPoolExecutor(max_workers=threads) as ex:
        while used < len(units) and elapsed < budget_s:
            batch = units[used:used + threads]
            args = [unit_args(n, h) for n, h in batch]
            tb = time.perf_counter()
            list(ex.map(lambda a: oracle.forward(*a, threads=1), args))
            elapsed += time.perf_counter() - tb
            done += sum(lens[n] for n, _ in batch)
            used += len(batch)
    desc = (f"{used} of {len(units)} whole (sequence, head) units, {done} token-heads, "
            f"one unit per thread, scaled to H={H}")
    return done / H / elapsed, threads, desc, elapsed


# ----------------------------------------------------------------------------- main arms
def run_reference(args):
    ws, rank, _ = dist_env()
    if rank != 0:
        return 0
    import torch
    from linear_attention_fwd_gb300 import inputs
    w = inputs.WORKLOADS[args.workload]
    inp = inputs.make_workload(args.workload, device="cpu") if w.kind == "prefill" else None
    threads = None
    rates = []
    for i in range(args.warmup + args.steps):
        r, threads, desc, _ = oracle_rate(inp, budget_s=args.ref_step_s)
        if i >= args.warmup:
            rates.append(r)
    value = statistics.median(rates)
    line = {
        "impl": "reference", "metric": "KDA prefill tokens/s at H=32, d=128 on 1 GB300", "value": value,
        "unit": "tokens/s", "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": None, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64", "data": "synthetic",
        "config": {"workload": args.workload, "note": w.note},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": threads, "kind": "oracle",
                         "sample": desc},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def run_ours(args):
    import torch
    import torch.distributed as dist
    from linear_attention_fwd_gb300 import build as kbuild
    kbuild.build()
    from linear_attention_fwd_gb300 import inputs, kda

    ws, rank, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if ws > 1:
        dist.init_process_group("nccl", device_id=dev)
    barrier, max_over_ranks = rank_ops(ws, dev)

    P = peaks()
    w = inputs.WORKLOADS[args.workload]
    inp = inputs.make_workload(args.workload, device=dev)
    q, v = inp["q"], inp["v"]
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    N = B if inp["cu_seqlens"] is None else inp["cu_seqlens"].numel() - 1
    tokens = B * T
    kernel = args.kernel if args.kernel != "auto" else kda.kda_chunk_fwd_selected_impl(q, v, inp["cu_seqlens"])
    out = torch.empty((B, T, H, dv), dtype=q.dtype, device=dev)
    fs = torch.empty((N, H, dk, dv), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()
    # the two-pass path's workspace (per-chunk matrices), allocated once outside the timed region
    wsp = {}
    if kernel == "two_pass":
        wsp["workspace"] = torch.empty(kda.kda_chunk_fwd_workspace_bytes(q, v, inp["cu_seqlens"]),
                                       dtype=torch.uint8, device=dev)

    def step():
        kda.kda_chunk_fwd(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"],
                          inp["initial_state"], inp["cu_seqlens"], out=out, final_state=fs,
                          impl=kernel, stream=stream, **wsp)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    barrier()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    t_beg, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk:
        t_beg.record(stream)
        for a, b in ev:
            a.record(stream)
            step()
            b.record(stream)
        t_end.record(stream)
        torch.cuda.synchronize()
    barrier()
    ms_total = max_over_ranks(t_beg.elapsed_time(t_end))
    per_launch_ms = statistics.mean(a.elapsed_time(b) for a, b in ev)
    ms_step = ms_total / args.steps
    value = ws * tokens * args.steps / (ms_total / 1e3)

    es = q.element_size()
    bytes_launch = algorithmic_bytes(tokens, H, dk, dv, es, N, inp["initial_state"] is not None)
    achieved = bytes_launch / (per_launch_ms / 1e3) / 1e9
    traffic = recorded_traffic(kernel, args.workload)
    flops = chunk_flops(tokens, H, dk, dv)
    roofline = hbm_roofline(bytes_launch, per_launch_ms, P, traffic=traffic,
                            kernel=KERNEL_NAME[kernel],
                            tensor_tflops=flops / (per_launch_ms / 1e3) / 1e12,
                            tensor_frac_of_bf16_peak=flops / (per_launch_ms / 1e3) / 1e12 / P["bf16"])
    roofline["peak_note"] = PEAK_NOTE
    clocks = clk.summary()

    # ---- end to end through the public API with host buffers (pinned), copies timed: every
    # step copies its inputs host -> device, runs kda_chunk_fwd and copies its output and
    # final state device -> host. Steps are pipelined the way a serving loop runs them: step
    # k+1's inputs are copied (copy stream, second buffer set) while step k computes and
    # returns its results (compute stream).
    e2e = None
    if not args.no_e2e:
        names = ("q", "k", "v", "g", "beta")
        host = {n: inp[n].cpu().pin_memory() for n in names}
        s0h = None if inp["initial_state"] is None else inp["initial_state"].cpu().pin_memory()
        out_h = torch.empty(out.shape, dtype=out.dtype).pin_memory()
        fs_h = torch.empty(fs.shape, dtype=fs.dtype).pin_memory()
        h2d = sum(t.numel() * t.element_size() for t in host.values()) + \
            (0 if s0h is None else s0h.numel() * 4)
        d2h = out_h.numel() * out_h.element_size() + fs_h.numel() * 4
        dbuf = [{n: torch.empty_like(inp[n]) for n in names} for _ in range(2)]
        s0d = [None if s0h is None else torch.empty_like(inp["initial_state"]) for _ in range(2)]
        s_copy = torch.cuda.Stream()
        ev_in = [torch.cuda.Event() for _ in range(2)]
        ev_free = [torch.cuda.Event() for _ in range(2)]
        for e in ev_free:
            e.record(stream)

        def e2e_step(k):
            sl = k % 2
            s_copy.wait_event(ev_free[sl])   # the kernel two steps back has read this buffer set
            with torch.cuda.stream(s_copy):
                for n in names:
                    dbuf[sl][n].copy_(host[n], non_blocking=True)
                if s0h is not None:
                    s0d[sl].copy_(s0h, non_blocking=True)
            ev_in[sl].record(s_copy)
            stream.wait_event(ev_in[sl])
            with torch.cuda.stream(stream):
                kda.kda_chunk_fwd(dbuf[sl]["q"], dbuf[sl]["k"], dbuf[sl]["v"], dbuf[sl]["g"],
                                  dbuf[sl]["beta"], s0d[sl], inp["cu_seqlens"], out=out,
                                  final_state=fs, impl=kernel, stream=stream, **wsp)
                ev_free[sl].record(stream)
                out_h.copy_(out, non_blocking=True)
                fs_h.copy_(fs, non_blocking=True)

        e2e_steps = max(3, min(args.steps, 10))
        for k in range(2):
            e2e_step(k)
        torch.cuda.synchronize()
        barrier()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        s_copy.wait_event(a)
        for k in range(e2e_steps):
            e2e_step(k)
        b.record(stream)
        torch.cuda.synchronize()
        ms = max_over_ranks(a.elapsed_time(b))
        # the host link's own ceiling, measured beside the leg: one plain copy of a step's
        # input bytes from pinned host memory, and one of its output bytes back
        hb = torch.empty(h2d, dtype=torch.uint8).pin_memory()
        db = torch.empty(h2d, dtype=torch.uint8, device=dev)
        link = {}
        for name, dst, src, nb in (("h2d", db, hb, h2d), ("d2h", hb[:d2h], db[:d2h], d2h)):
            ms_c = _time_ms(lambda: dst.copy_(src, non_blocking=True), stream, reps=3, warm=1)
            link[name + "_copy_gbs"] = nb / (ms_c / 1e3) / 1e9
        del hb, db
        e2e = {"value": ws * tokens * e2e_steps / (ms / 1e3), "unit": "tokens/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "ms_per_step": ms / e2e_steps, "steps": e2e_steps,
               "overlap": "step k+1's host-to-device copies run while step k computes and "
                          "copies back (two input buffer sets, copy and compute streams)",
               "link": dict(link, bound_ms_per_step=max(h2d / link["h2d_copy_gbs"],
                                                        d2h / link["d2h_copy_gbs"]) / 1e6,
                            note="one pinned copy of a step's input (output) bytes; the "
                                 "step's copies cannot run faster than the larger of the two")}
        del host, dbuf, out_h, fs_h

    # ---- decode steps/s (fp32 state streamed in place)
    decode = None
    if not args.no_decode:
        decode = bench_decode(args, kda, inputs, dev, stream, P, barrier, max_over_ranks, ws)

    # ---- the widened rows (output gate, state checkpoints, multi-token decode), same workload
    extras = None
    if not args.no_extras and kernel == "tc":
        extras = bench_extras(kda, inputs, inp, out, fs, stream, P, bytes_launch, tokens, H, dk, dv, es, N)

    # ---- CPU baseline: the oracle on the host cores, bounded sample (rank 0, N = 1 only)
    cpu = None
    if not args.no_cpu_baseline and ws == 1 and rank == 0:
        rate, cores, desc, el = oracle_rate(inp, budget_s=args.cpu_budget)
        cpu = {"value": rate, "unit": "tokens/s", "cores": cores, "kind": "oracle",
               "sample": desc + f", {el:.1f} s"}

    if rank == 0:
        line = {
            "metric": "KDA prefill tokens/s at H=32, d=128 on 1 GB300",
            "value": value, "unit": "tokens/s", "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16" if kernel in ("tc", "two_pass") else "f32",
            "data": "synthetic",
            "config": {"workload": args.workload, "batch": B, "seq_len": T, "heads": H,
                       "dk": dk, "dv": dv, "num_seqs": N, "io_dtype": str(q.dtype).split(".")[-1],
                       "kernel": kernel, "parallelism": f"replicas x{ws} (independent units)",
                       "ctas": (kda.kda_chunk_fwd_auto_ctas(
                           kda.chunk_dims(q, inp["v"], inp.get("cu_seqlens")),
                           inp.get("cu_seqlens") is not None,
                           torch.cuda.get_device_properties(dev).multi_processor_count)
                           if kernel == "tc" else N * H),
                       "schedule": ("balanced: each CTA an equal share of the (sequence, head, "
                                    "chunk) items" if kernel == "tc" and inp.get("cu_seqlens") is None
                                    else "one CTA per (sequence, head) or uniform segments"),
                       "l2": f"inputs larger than L2 ({bytes_launch / 1e9:.2f} GB per step)",
                       "note": w.note},
            "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e,
            "gpu_launches": args.steps * LAUNCHES_PER_STEP[kernel], "clocks": clocks, "decode": decode,
            "extras": extras,
        }
        print(json.dumps(line), flush=True)
    if ws > 1:
        dist.destroy_process_group()
    return 0


def _time_ms(fn, stream, reps=5, warm=2):
    import torch
    for _ in range(warm):
        fn()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(reps):
        fn()
    b.record(stream)
    torch.cuda.synchronize()
    return a.elapsed_time(b) / reps


def bench_extras(kda, inputs, inp, out, fs, stream, P, bytes_launch, tokens, H, dk, dv, es, N):
    """The output gate fused into the store, state checkpoints every 512 tokens, and 4 decode
    tokens per call with the state on chip -- each against its own algorithmic bytes."""
    import torch
    gen = torch.Generator(device=out.device).manual_seed(5)
    z = torch.randn(inp["v"].shape, generator=gen, device=out.device).to(inp["v"].dtype)
    w = torch.ones(dv, device=out.device)
    ms = _time_ms(lambda: kda.kda_chunk_fwd_gated(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], z, w,
                                                   1e-6, inp["initial_state"], inp["cu_seqlens"],
                                                   out=out, final_state=fs, stream=stream), stream)
    gb = bytes_launch + tokens * H * dv * es
    gated = {"ms_per_step": ms, "tokens_per_s": tokens / (ms / 1e3), "roofline": hbm_roofline(gb, ms, P)}
    del z
    off = kda.checkpoint_offsets(inp["q"], inp["cu_seqlens"], 512)
    slots = int(off[-1].item())
    ck = torch.empty((max(slots, 1), H, dk, dv), dtype=torch.float32, device=out.device)
    ms = _time_ms(lambda: kda.kda_chunk_fwd_checkpointed(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"],
                                                          inp["initial_state"], inp["cu_seqlens"],
                                                          interval=512, out=out, final_state=fs,
                                                          checkpoints=ck, offsets=off, stream=stream), stream)
    cb = bytes_launch + slots * H * dk * dv * 4
    ckpt = {"interval": 512, "checkpoints": slots, "ms_per_step": ms, "tokens_per_s": tokens / (ms / 1e3),
            "roofline": hbm_roofline(cb, ms, P)}
    del ck
    wd = inputs.WORKLOADS["decode_n256_h64"]
    T = 4
    st = inputs.make_decode_state(num_slots=wd.batch, heads=wd.heads, dk=wd.dk, dv=wd.dv,
                                  device=out.device, seed=7)
    ins = inputs.make_decode_inputs(steps=T, rows=wd.batch, heads=wd.heads, dk=wd.dk, dv=wd.dv,
                                    dtype=wd.dtype, device=out.device, seed=8)
    a = {k: ins[k].transpose(0, 1).contiguous() for k in ins}
    dout = torch.empty((wd.batch, T, wd.heads, wd.dv), dtype=wd.dtype, device=out.device)
    ms = _time_ms(lambda: kda.kda_recurrent_steps(a["q"], a["k"], a["v"], a["g"], a["beta"], st,
                                                   out=dout, stream=stream), stream, reps=20)
    db = wd.batch * wd.heads * (2 * wd.dk * wd.dv * 4 + T * ((3 * wd.dk + 2 * wd.dv + 1) * 2))
    steps4 = {"workload": "decode_n256_h64", "tokens_per_row": T, "ms_per_call": ms,
              "row_tokens_per_s": wd.batch * T / (ms / 1e3), "roofline": hbm_roofline(db, ms, P)}
    del st, ins, a, dout
    # the other supported shapes at B=4 H=32 T=8192: fp32 inputs (the 1e-4 mode) on the SIMT
    # kernel, and bf16 with d = 64 on the tensor-core kernel (64-wide heads padded to 128 by the
    # TMA's zero fill) beside the SIMT kernel it ran on before
    other = {}
    for name, dtype, d, impl in (("fp32_d128", torch.float32, 128, "simt"), ("bf16_d64", torch.bfloat16, 64, "tc"),
                                 ("bf16_d64_simt", torch.bfloat16, 64, "simt")):
        x = inputs.make_prefill(batch=4, seqlen=8192, heads=32, dk=d, dv=d, dtype=dtype,
                                device=out.device, seed=9)
        o2 = torch.empty_like(x["v"])
        f2 = torch.empty((4, 32, d, d), dtype=torch.float32, device=out.device)
        ms = _time_ms(lambda: kda.kda_chunk_fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], None, None,
                                                 out=o2, final_state=f2, impl=impl, stream=stream),
                      stream, reps=2 if impl == "simt" else 5, warm=1)
        nb = algorithmic_bytes(4 * 8192, 32, d, d, x["q"].element_size(), 4, False)
        other[name] = {"kernel": KERNEL_NAME[impl], "ms_per_step": ms,
                       "tokens_per_s": 4 * 8192 / (ms / 1e3), "roofline": hbm_roofline(nb, ms, P)}
        del x, o2, f2
    # q and k L2-normalised inside the call (kda_chunk_fwd_qknorm) on raw N(0, 1) q and k of the
    # same shape: the same bytes as the plain call
    B_, T_ = inp["q"].shape[:2]
    x = inputs.make_prefill(batch=B_, seqlen=T_, heads=H, dk=dk, dv=dv, dtype=inp["q"].dtype,
                            device=out.device, seed=10, raw_qk=True,
                            init_state=inp["initial_state"] is not None) if inp["cu_seqlens"] is None else None
    qkn = None
    if x is not None:
        ms = _time_ms(lambda: kda.kda_chunk_fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], x["initial_state"], None,
                                                 out=out, final_state=fs, qk_eps=1e-6, stream=stream), stream)
        qkn = {"ms_per_step": ms, "tokens_per_s": tokens / (ms / 1e3),
               "roofline": hbm_roofline(bytes_launch, ms, P)}
        del x
    return {"gated": gated, "checkpointed": ckpt, "decode_steps": steps4, "other_shapes": other,
            "qk_l2norm": qkn}


def bench_decode(args, kda, inputs, dev, stream, P, barrier, max_over_ranks, ws):
    import torch
    w = inputs.WORKLOADS["decode_n256_h64"]
    steps = args.decode_steps
    inp = inputs.make_workload("decode_n256_h64", device=dev, decode_steps=steps)
    st = inp["state"]
    out = torch.empty((w.batch, w.heads, w.dv), dtype=w.dtype, device=dev)
    for s in range(3):
        kda.kda_recurrent_step(inp["q"][s], inp["k"][s], inp["v"][s], inp["g"][s], inp["beta"][s],
                               st, out=out, stream=stream)
    torch.cuda.synchronize()
    barrier()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for s in range(steps):
        kda.kda_recurrent_step(inp["q"][s], inp["k"][s], inp["v"][s], inp["g"][s], inp["beta"][s],
                               st, out=out, stream=stream)
    b.record(stream)
    torch.cuda.synchronize()
    ms = max_over_ranks(a.elapsed_time(b))
    per = ms / steps / 1e3
    rows_heads = w.batch * w.heads
    bytes_step = rows_heads * (2 * w.dk * w.dv * 4 + (3 * w.dk + 2 * w.dv + 1) * 2)
    del inp
    return {"workload": "decode_n256_h64", "steps": steps, "value": ws * steps / (ms / 1e3),
            "unit": "steps/s", "ms_per_step": ms / steps,
            "roofline": hbm_roofline(bytes_step, per * 1e3, P, kernel=KERNEL_NAME["decode"],
                                     traffic=recorded_traffic("decode", "decode_n256_h64")),
            "gpu_launches": steps}


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="prefill_b4_h32_t8192")
    ap.add_argument("--kernel", default="auto", choices=["auto", "simt", "tc", "two_pass"])
    ap.add_argument("--decode-steps", type=int, default=1000)
    ap.add_argument("--cpu-budget", type=float, default=12.0,
                    help="seconds of oracle work for the CPU baseline sample")
    ap.add_argument("--ref-step-s", type=float, default=4.0,
                    help="seconds of oracle work per --impl reference step")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-decode", action="store_true")
    ap.add_argument("--no-extras", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    args = ap.parse_args()
    if args.warmup < 3:
        print("warning: fewer than 3 warm-up steps", file=sys.stderr)
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
