"""Benchmark of the rolling FP8 attention cache on one GB300 (or N replicas).

Workload (the production-shaped call): one layer's ring of 5,788 slots,
10 heads of 128, bf16 inputs; one step = one 757-token frame write (RoPE +
E4M3 quantisation into the ring) + attention of the frame's 757 queries over
all 5,788 slots.  The pages report 5,788 slots with 757 new per call
("Where the Time Went", Runway Characters serving post); 10 heads of 128 is
the assumed 4-way split of 40 heads.  Inputs are synthetic: K, V ~ N(0,1)
times a per-head standard deviation drawn log-uniform in [0.25, 4]; Q ~ N(0,1).

L2: steps rotate over 16 independent rings (and 16 input frames), so each
step's ring, inputs and partials were last touched 15 steps earlier, after
more than 126 MB of other traffic: every step starts L2-cold.

Timing: every step is one CUDA graph replay (one ring's write + attention,
with the delta rotation in front every 42nd write of a ring).  W warm-up
steps, then exactly K steps between CUDA events on the launching stream,
with a barrier and device synchronisation on both sides.  Per-kernel
durations come from graphs of 16 back-to-back calls (one per ring).
The metric is time-like (microseconds per write + attention).

``--impl reference`` times the CPU oracle (float64 NumPy, the test oracle)
on this host's cores on a bounded sample of each step (see ``cpu_sample``).
Replicas only across GPUs: each rank runs its own rings; no collective is
on the data path.
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

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "µs per 757-token cache write + 5788-slot FP8 attn; GB/s & TFLOP/s vs GB300 peak"
WORKLOAD = ("production-shaped call: 757-token write + 757-query attention over a wrapped 5,788-slot "
            "ring, 10 heads x 128 (E4M3 cache, bf16 in, fp32 out)")
H, D, C, N_NEW, N_Q, MAX_POS = 10, 128, 5788, 757, 757, 40960
RINGS = 16
RESET_PERIOD = 42   # the pages reset positions once per 42 steps (Do It Once, at Write Time)
# algorithmic work per step
WRITE_BYTES = 2 * N_NEW * H * D * 2 + 2 * N_NEW * H * D + N_NEW * 4  # bf16 in, e4m3 out, slot_pos
ATTN_FLOPS = 4.0 * H * N_Q * C * D                                   # QK^T and PV
ATTN_BYTES = 2 * H * C * D + N_Q * H * D * 2 + N_Q * H * D * 4       # cache, q, fp32 out
DELTA_BYTES = 2 * H * C * D + 2 * C * 4                              # key cache read + write, positions
LAYERS = 60         # one ring per layer: the batched write / reset of a whole step
CALLS_PER_STEP = 240  # attention calls per step (4 passes x 60 blocks): where the old upkeep ran
# the original upkeep per call with a full window: copy the shifted bf16 window
# (read + write), read it again to rotate and quantise, write the FP8 cache
LEGACY_BYTES = 3 * 2 * C * H * D * 2 + 2 * C * H * D
# extra measurements after the headline step (bench --legs)
EXTRA_LEGS = ("batched", "legacy", "project", "full_step", "stress")
H2D_BYTES = 3 * N_NEW * H * D * 2
D2H_BYTES = N_Q * H * D * 4


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as fh:
            p = json.load(fh)
        return dict(hbm=float(p["hbm_gbs"]), bf16=float(p["bf16_tflops"]),
                    bf16_sus=float(p.get("bf16_tflops_sustained", p["bf16_tflops"])),
                    src="measured")
    except Exception:
        return dict(hbm=6800.0, bf16=1900.0, bf16_sus=1700.0, src="fallback")


def attention_traffic():
    """DRAM bytes per attention launch from the committed ncu summary, if it
    was taken on the current attention source; else None."""
    src = os.path.join(ROOT, "ring_kv_cache_gb300", "csrc", "kvring_attn.cu")
    prof = os.path.join(ROOT, "profiles", "attention_prod_traffic.json")
    try:
        sha = hashlib.sha256(open(src, "rb").read()).hexdigest()
        p = json.load(open(prof))
        if p.get("kvring_attn_cu_sha256") == sha:
            return float(p["dram_bytes_per_launch"])
    except Exception:
        pass
    return None


class ClockSampler:
    """Samples SM clocks and throttle reasons with nvidia-smi while running."""

    FIELDS = ("clocks.sm,clocks.max.sm,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
            time.sleep(0.15)
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc:
            time.sleep(0.06)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=2)
            except Exception:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                mx = float(parts[1])
            except ValueError:
                continue
            for nm, val in zip(names, parts[3:7]):
                if val.lower() == "active":
                    reasons.add(nm)
        return {"sm_mhz": float(np.median(sm)) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------------------
def gpu_arm(args, rank, world):
    import torch
    import ring_kv_cache_gb300 as kv
    from workloads import PROD, prod_session, to_torch_bf16

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    stream = torch.cuda.Stream(dev)
    rings = []
    frames = []
    with torch.cuda.stream(stream):
        for i in range(RINGS):
            sk, sv, fr = prod_session(seed=2 + 1000 * rank + i, frames=9)
            ring = kv.KvRing(H, D, C, N_NEW, MAX_POS, 10000.0, max_kv_splits=16, stream=stream)
            t = [(to_torch_bf16(q).to(dev), to_torch_bf16(k).to(dev), to_torch_bf16(v).to(dev))
                 for q, k, v in fr]
            ring.calibrate(t[0][1], t[0][2], stream=stream)
            for q, k, v in t[:8]:          # 6,056 tokens: the ring has wrapped
                ring.write(k, v, stream=stream)
            rings.append(ring)
            frames.append(t[8])
        outs = [torch.empty((N_Q, H, D), dtype=torch.float32, device=dev) for _ in range(RINGS)]
    torch.cuda.synchronize(dev)

    writes = [8] * RINGS          # frames already written per ring

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()

    def capture(fn):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            fn()
        return g

    def do_step(r, reset):
        q, k, v = frames[r]
        if reset:
            # positions reset every 42 steps: one delta rotation of the window
            rings[r].delta_rotate(kv.TO_OLDEST, stream=stream)
        rings[r].write(k, v, stream=stream)
        rings[r].attention(q, out=outs[r], stream=stream)

    # eager warm-up (every kernel has run once before capture)
    for i in range(max(args.warmup, RINGS)):
        r = i % RINGS
        do_step(r, writes[r] % RESET_PERIOD == 0)
        writes[r] += 1
    torch.cuda.synchronize(dev)

    # The K timed steps (write + attention of one ring each, a delta rotation
    # in front where a ring's window is due) are captured once into one CUDA
    # graph, so consecutive steps overlap where the kernels allow it: a write
    # is a programmatic dependent of the preceding attention and waits only
    # before it touches its ring.  The timed region is one replay.
    resets = [0]

    def steps(n):
        for i in range(n):
            r = i % RINGS
            rst = writes[r] % RESET_PERIOD == 0
            resets[0] += int(rst)
            do_step(r, rst)
            writes[r] += 1

    g_warm = capture(lambda: steps(args.warmup))
    g_warm.replay()
    torch.cuda.synchronize(dev)
    resets[0] = 0
    g_timed = capture(lambda: steps(args.steps))

    # timed region: exactly K steps, events around the whole region on the stream
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize(dev)
    with ClockSampler(dev.index) as clk:
        with torch.cuda.stream(stream):
            start.record(stream)
            g_timed.replay()
            stop.record(stream)
        torch.cuda.synchronize(dev)
    barrier()
    total_ms = start.elapsed_time(stop)
    timed_resets = resets[0]

    # Per-kernel durations: graphs of 16 back-to-back calls on the 16 rings
    # (each call L2-cold), timed with events around the replays.
    def timed(g, reps):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            e0.record(stream)
            for _ in range(reps):
                g.replay()
            e1.record(stream)
        torch.cuda.synchronize(dev)
        return e0.elapsed_time(e1)

    g_attn = capture(lambda: [rings[r].attention(frames[r][0], out=outs[r], stream=stream) for r in range(RINGS)])
    g_write = capture(lambda: [rings[r].write(frames[r][1], frames[r][2], stream=stream) for r in range(RINGS)])
    g_delta = capture(lambda: [rings[r].delta_rotate(kv.TO_OLDEST, stream=stream) for r in range(RINGS)])
    timed(g_attn, 2)
    a_reps = 8
    a_us = timed(g_attn, a_reps) * 1e3 / (a_reps * RINGS)
    d_ms = timed(g_delta, 1)                      # every window restarts at 0
    w_reps = RESET_PERIOD - 1
    w_us = timed(g_write, w_reps) * 1e3 / (w_reps * RINGS)
    d_ms += timed(g_delta, 1)                     # delta = 41 frames of positions
    d_us = d_ms * 1e3 / (2 * RINGS)
    # The fixed cost of each, with no data: the write's grid, launch mode,
    # wait, state read, completion ticket and state publication
    # (kvring_debug_write_floor), and the delta rotation's full grid with a
    # delta of 0 (no rows move).  Same graphs of 16 back-to-back calls.
    g_wfloor = capture(lambda: [rings[r].write_floor(N_NEW, stream=stream) for r in range(RINGS)])
    g_dfloor = capture(lambda: [rings[r].delta_rotate(0, stream=stream) for r in range(RINGS)])
    timed(g_wfloor, 1)
    wf_us = timed(g_wfloor, 8) * 1e3 / (8 * RINGS)
    df_us = timed(g_dfloor, 4) * 1e3 / (4 * RINGS)
    for r in range(RINGS):
        writes[r] = 1   # every window was just reset: the next reset is 41 writes away

    # end to end through the public API with pinned host buffers.  Three
    # streams, as a streaming deployment runs them: step i's inputs upload
    # (H2D) while step i-1 computes and step i-2's output downloads (D2H).
    # Events order every reuse: an input buffer set is overwritten only after
    # the compute that read it, a ring's output only after its download.
    # The K steps are captured once into a CUDA graph (copies, kernels and
    # cross-stream events; Python submission would otherwise set the pace)
    # and the timed region is one replay: every step's copies and kernels
    # lie inside it.
    NB = 2
    hin = [[torch.empty((N_NEW, H, D), dtype=torch.bfloat16).pin_memory() for _ in range(3)] for _ in range(NB)]
    hout = [torch.empty((N_Q, H, D), dtype=torch.float32).pin_memory() for _ in range(NB)]
    for b_ in range(NB):
        for j, x in enumerate(frames[b_ % RINGS]):
            hin[b_][j].copy_(x.cpu())
    din = [[torch.empty((N_Q, H, D), dtype=torch.bfloat16, device=dev) for _ in range(3)] for _ in range(NB)]
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)

    def e2e_steps(n):
        ev_in = [torch.cuda.Event() for _ in range(n)]
        ev_used = [torch.cuda.Event() for _ in range(n)]   # compute done with step i's inputs
        ev_out = [torch.cuda.Event() for _ in range(n)]    # step i's output downloaded
        last_out = {}                                       # ring -> step of its last download
        for i in range(n):
            r, b_ = i % RINGS, i % NB
            if i >= NB:
                s_in.wait_event(ev_used[i - NB])
            with torch.cuda.stream(s_in):
                for j in range(3):
                    din[b_][j].copy_(hin[b_][j], non_blocking=True)
                ev_in[i].record(s_in)
            stream.wait_event(ev_in[i])
            if r in last_out:
                stream.wait_event(ev_out[last_out[r]])
            if writes[r] % RESET_PERIOD == 0:
                rings[r].delta_rotate(kv.TO_OLDEST, stream=stream)
            writes[r] += 1
            rings[r].write(din[b_][1], din[b_][2], stream=stream)
            rings[r].attention(din[b_][0], out=outs[r], stream=stream)
            ev_used[i].record(stream)
            s_out.wait_event(ev_used[i])
            with torch.cuda.stream(s_out):
                hout[b_].copy_(outs[r], non_blocking=True)
                ev_out[i].record(s_out)
            last_out[r] = i

    def capture_e2e(n):
        gr = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gr, stream=stream):
            s_in.wait_stream(stream)
            s_out.wait_stream(stream)
            e2e_steps(n)
            stream.wait_stream(s_in)
            stream.wait_stream(s_out)
        return gr

    with torch.cuda.stream(stream):
        e2e_steps(max(args.warmup, NB))          # eager warm-up through the same calls
        torch.cuda.synchronize(dev)
        g_e2e = capture_e2e(args.steps)
        g_e2e.replay()                           # untimed replay
        torch.cuda.synchronize(dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        barrier()
        e0.record(stream)
        g_e2e.replay()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        barrier()
    e2e_ms = e0.elapsed_time(e1)

    # The same step's copies alone (no kernels), each direction on its own
    # stream and buffers as above, K steps as one graph replay: what the
    # host link alone allows per step.
    def copies_alone(s_cp, body):
        gr = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gr, stream=s_cp):
            for i in range(args.steps):
                body(i)
        with torch.cuda.stream(s_cp):
            gr.replay()
        torch.cuda.synchronize(dev)
        c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        # a graph replays on the current stream: make it the one the events
        # are recorded on, so they bracket the copies
        with torch.cuda.stream(s_cp):
            c0.record(s_cp)
            gr.replay()
            c1.record(s_cp)
        torch.cuda.synchronize(dev)
        return c0.elapsed_time(c1) * 1e3 / args.steps

    def h2d(i):
        for j in range(3):
            din[i % NB][j].copy_(hin[i % NB][j], non_blocking=True)

    def d2h(i):
        hout[i % NB].copy_(outs[i % RINGS], non_blocking=True)

    def both(i):          # both directions at once: H2D here, D2H forked to its stream
        if i == 0:
            s_out.wait_stream(s_in)
            with torch.cuda.stream(s_out):
                for j in range(args.steps):
                    d2h(j)
        h2d(i)
        if i == args.steps - 1:
            s_in.wait_stream(s_out)

    copy_us = {"h2d": copies_alone(s_in, h2d), "d2h": copies_alone(s_out, d2h), "both": copies_alone(s_in, both)}

    # precision levels used on the timed workload (for the issued-FLOP count)
    levels = []
    for r in rings:
        lv = r.levels().cpu().numpy()[: (N_Q + 127) // 128]
        levels.append(lv)
    levels = np.concatenate(levels).ravel()
    errs = [int(r.export()["state"][kv.STATE["error"]].item()) for r in rings]
    leg_errors = {}
    batched = run_leg(args.legs, "batched", lambda: batched_upkeep(args, dev, stream), leg_errors)
    legacy_us = run_leg(args.legs, "legacy", lambda: legacy_upkeep_us(dev, stream), leg_errors)
    proj = run_leg(args.legs, "project", lambda: project_write_us(dev, stream), leg_errors)
    del g_warm, g_timed, g_attn, g_write, g_delta, g_wfloor, g_dfloor, g_e2e
    full_step = run_leg(args.legs, "full_step", lambda: full_step_60_layers(dev, stream), leg_errors)
    stress = run_leg(args.legs, "stress", lambda: stress_40_heads(dev, stream), leg_errors)
    return dict(total_ms=total_ms, leg_errors=leg_errors, w_us=w_us, a_us=a_us, d_us=d_us, wf_us=wf_us, df_us=df_us,
                full_step=full_step, stress=stress, e2e_ms=e2e_ms, copy_us=copy_us,
                clocks=clk.summary(),
                batched=batched, legacy_us=legacy_us, proj=proj,
                resets=timed_resets,
                levels=levels, device_errors=int(np.bitwise_or.reduce(errs)))


def run_leg(legs, name, fn, errors):
    """Runs one extra measurement if it was asked for.  The headline step is
    measured before any of them, so a leg that raises is reported under
    `leg_errors` in the JSON line (and on stderr) instead of ending the run."""
    if name not in legs:
        return None
    try:
        return fn()
    except Exception as e:  # noqa: BLE001 -- any failure of a leg is reported, not fatal
        errors[name] = f"{type(e).__name__}: {e}"[:300]
        print(f"bench: leg {name} failed: {errors[name]}", file=sys.stderr)
        return None


def batched_upkeep(args, dev, stream):
    """The per-step upkeep of a whole model at once: one launch writes a
    757-token frame into each of 60 layer rings (349 MB), one launch resets
    all 60 windows (892 MB).  Inputs are N(0,1) bf16 drawn on the device; each
    call moves more than the L2 holds, so every replay is L2-cold."""
    import torch
    import ring_kv_cache_gb300 as kv
    with torch.cuda.stream(stream):
        g = torch.Generator(device=dev)
        g.manual_seed(7)
        rings = [kv.KvRing(H, D, C, N_NEW, MAX_POS, 10000.0, max_kv_splits=1, stream=stream)
                 for _ in range(LAYERS)]
        ks = [torch.randn((N_NEW, H, D), generator=g, device=dev).bfloat16() for _ in range(LAYERS)]
        vs = [torch.randn((N_NEW, H, D), generator=g, device=dev).bfloat16() for _ in range(LAYERS)]
        for r, k, v in zip(rings, ks, vs):
            r.calibrate(k, v, stream=stream)
        for _ in range(8):                      # fill and wrap every window
            kv.write_frames_many(rings, ks, vs, stream=stream)
        torch.cuda.synchronize(dev)

        def graph(fn):
            gr = torch.cuda.CUDAGraph()
            with torch.cuda.graph(gr, stream=stream):
                fn()
            return gr

        g_w = graph(lambda: kv.write_frames_many(rings, ks, vs, stream=stream))
        g_d = graph(lambda: kv.delta_rotate_many(rings, 100, stream=stream))

        def timed(gr, reps):
            gr.replay()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(reps):
                gr.replay()
            e1.record(stream)
            torch.cuda.synchronize(dev)
            return e0.elapsed_time(e1) * 1e3 / reps

        w_us = timed(g_w, 10)
        d_us = timed(g_d, 4)
    del rings, ks, vs
    torch.cuda.empty_cache()
    return dict(write_us=w_us, delta_us=d_us)


def full_step_60_layers(dev, stream):
    """The full denoising step on one GPU: 60 layer rings of the production
    shape, per step one 757-token write per layer (the cache upkeep) and 4
    passes x 60 attention calls of 757 queries ("Where the Time Went": 4
    passes through 60 blocks, 240 attention calls per step).  Upkeep,
    attention and the whole step are each one CUDA graph, replayed; the 60
    writes are also timed as one batched launch.  Inputs: per layer sigma_k,
    sigma_v log-uniform in [0.25, 4] (seed 3), N(0,1) draws of a seeded CUDA
    generator; 14.8 MB of cache per layer, so every call is L2-cold."""
    import torch
    import ring_kv_cache_gb300 as kv
    from workloads import cuda_frame, cuda_generator, log_uniform
    rng = np.random.default_rng(3)
    with torch.cuda.stream(stream):
        gen = cuda_generator(3, device=dev)
        rings, frames = [], []
        for _ in range(LAYERS):
            sk, sv = log_uniform(rng, H, 0.25, 4.0), log_uniform(rng, H, 0.25, 4.0)
            fr = [cuda_frame(gen, H, D, N_NEW, sk, sv, device=dev) for _ in range(2)]
            ring = kv.KvRing(H, D, C, N_NEW, MAX_POS, 10000.0, max_kv_splits=8, stream=stream)
            ring.calibrate(fr[0][1], fr[0][2], stream=stream)
            for i in range(8):                     # 6,056 tokens: wrapped
                ring.write(fr[i % 2][1], fr[i % 2][2], stream=stream)
            rings.append(ring)
            frames.append(fr)
        outs = [torch.empty((N_Q, H, D), dtype=torch.float32, device=dev) for _ in range(4 * LAYERS)]
    torch.cuda.synchronize(dev)

    def upkeep():
        for l in range(LAYERS):
            rings[l].write(frames[l][0][1], frames[l][0][2], stream=stream)

    def upkeep_batched():
        kv.write_frames_many(rings, [f[0][1] for f in frames], [f[0][2] for f in frames], stream=stream)

    def attention():
        for p in range(4):
            for l in range(LAYERS):
                rings[l].attention(frames[l][p % 2][0], out=outs[4 * l + p], stream=stream)

    def graph(fn):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            fn()
        return g

    def timed(g, reps):
        with torch.cuda.stream(stream):
            g.replay()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(reps):
                g.replay()
            e1.record(stream)
        torch.cuda.synchronize(dev)
        return e0.elapsed_time(e1) * 1e3 / reps

    g_up, g_upb, g_at = graph(upkeep), graph(upkeep_batched), graph(attention)
    g_step = graph(lambda: (upkeep(), attention()))
    res = dict(upkeep_us=timed(g_up, 5), upkeep_batched_us=timed(g_upb, 5),
               attention_us=timed(g_at, 3), step_us=timed(g_step, 3))
    del g_up, g_upb, g_at, g_step, rings, frames, outs
    torch.cuda.empty_cache()
    return res


def stress_40_heads(dev, stream):
    """The stress workload's call: the whole unsharded head set (40 heads x
    128) over a wrapped 5,788-slot ring, keys and values Student-t (3 degrees
    of freedom) with per-head scales log-uniform in [0.1, 10] (seed 5), a
    first frame of the seeded prompt length, then 757-token frames.  Four
    rings round-robin (59 MB of cache each), one attention call of 757
    queries (89.7 GFLOP) or one write (23.3 MB) per ring, as graphs of four
    calls; the precision levels the rule chose are reported."""
    import torch
    import ring_kv_cache_gb300 as kv
    from workloads import cuda_frame, cuda_generator, log_uniform, stress_prompt_length
    HS, NR = 40, 4
    rng = np.random.default_rng(5)
    n0 = stress_prompt_length(5)
    with torch.cuda.stream(stream):
        gen = cuda_generator(5, device=dev)
        rings, frames = [], []
        for _ in range(NR):
            sk, sv = log_uniform(rng, HS, 0.1, 10.0), log_uniform(rng, HS, 0.1, 10.0)
            q0, k0, v0 = cuda_frame(gen, HS, D, n0, sk, sv, dist="student_t3", device=dev)
            ring = kv.KvRing(HS, D, C, 2000, MAX_POS, 10000.0, max_kv_splits=8, stream=stream)
            ring.calibrate(k0, v0, stream=stream)
            ring.write(k0, v0, stream=stream)
            fr = [cuda_frame(gen, HS, D, N_NEW, sk, sv, dist="student_t3", device=dev) for _ in range(2)]
            for i in range(8):
                ring.write(fr[i % 2][1], fr[i % 2][2], stream=stream)
            rings.append(ring)
            frames.append(fr)
        outs = [torch.empty((N_Q, HS, D), dtype=torch.float32, device=dev) for _ in range(NR)]
    torch.cuda.synchronize(dev)

    def graph(fn):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            fn()
        return g

    def timed(g, reps):
        with torch.cuda.stream(stream):
            g.replay()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(reps):
                g.replay()
            e1.record(stream)
        torch.cuda.synchronize(dev)
        return e0.elapsed_time(e1) * 1e3 / (reps * NR)

    g_at = graph(lambda: [rings[i].attention(frames[i][0][0], out=outs[i], stream=stream) for i in range(NR)])
    g_wr = graph(lambda: [rings[i].write(frames[i][1][1], frames[i][1][2], stream=stream) for i in range(NR)])
    a_us, w_us = timed(g_at, 4), timed(g_wr, 8)
    lv = np.concatenate([r.levels().cpu().numpy()[: (N_Q + 127) // 128].ravel() for r in rings])
    flops = 4.0 * HS * N_Q * C * D
    wbytes = 2 * N_NEW * HS * D * 2 + 2 * N_NEW * HS * D + N_NEW * 4
    q_terms = lv.astype(np.float64)
    pv = np.where(lv >= 4, 2.0, 1.0)            # PV MMAs per tile in f16 (two at level 4)
    issued = float(np.mean(q_terms + 2.0 * pv)) / 2.0
    del g_at, g_wr, rings, frames, outs
    torch.cuda.empty_cache()
    return dict(attention_us=a_us, attention_tflops=flops / (a_us * 1e-6) / 1e12, flops_per_call=flops,
                write_us=w_us, write_gbs=wbytes / (w_us * 1e-6) / 1e9, write_bytes=wbytes,
                levels={str(k): int((lv == k).sum()) for k in (1, 2, 3, 4)},
                issued_mma_over_algorithmic=issued, prompt_tokens=n0)


D_MODEL = 5120                       # 40 heads x 128 (the model's width; 10 heads per GPU)


def project_write_us(dev, stream):
    """kvring_project_write at the production shape: a 757-token frame's
    x [757, 5,120] times W [3,840, 5,120] (29.8 GFLOP), keys and values
    written into the ring in the epilogue, queries stored.  Four rings with
    their own weights round-robin (4 x 39 MB of weights), so each call's
    weights are L2-cold; a CUDA graph of the four calls, replayed."""
    import torch
    import ring_kv_cache_gb300 as kv
    with torch.cuda.stream(stream):
        g = torch.Generator(device=dev)
        g.manual_seed(13)
        rings = [kv.KvRing(H, D, C, N_NEW, MAX_POS, 10000.0, max_kv_splits=1, stream=stream) for _ in range(4)]
        ws = [(torch.randn((3 * H * D, D_MODEL), generator=g, device=dev) * 0.015).bfloat16() for _ in range(4)]
        xs = [torch.randn((N_NEW, D_MODEL), generator=g, device=dev).bfloat16() for _ in range(4)]
        for r, x, w in zip(rings, xs, ws):
            _, kvo = r.project_write(x, w, write=False, store_kv=True, stream=stream)
            r.calibrate(kvo[0], kvo[1], stream=stream)
        torch.cuda.synchronize(dev)
        qs = [torch.empty((N_NEW, H, D), dtype=torch.bfloat16, device=dev) for _ in range(4)]
        gr = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gr, stream=stream):
            for r, x, w, q in zip(rings, xs, ws, qs):
                r.project_write(x, w, q_out=q, stream=stream)
        gr.replay()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        reps = 8
        e0.record(stream)
        for _ in range(reps):
            gr.replay()
        e1.record(stream)
        torch.cuda.synchronize(dev)
    us = e0.elapsed_time(e1) * 1e3 / (reps * 4)
    flops = 2.0 * N_NEW * 3 * H * D * D_MODEL
    return us, flops


def legacy_upkeep_us(dev, stream):
    """The upkeep the ring replaced, per call with a full 5,788-slot window:
    window copy, RoPE of every cached key, window scales, re-quantisation of
    the whole cache (two kernels).  Four rings round-robin, so each call's
    104 MB is L2-cold; a CUDA graph of four calls, replayed."""
    import torch
    import ring_kv_cache_gb300 as kv
    with torch.cuda.stream(stream):
        g = torch.Generator(device=dev)
        g.manual_seed(11)
        rings = [kv.KvRing(H, D, C, N_NEW, MAX_POS, 10000.0, max_kv_splits=1, stream=stream) for _ in range(4)]
        wins = [kv.LegacyWindows(r) for r in rings]
        ks = [torch.randn((N_NEW, H, D), generator=g, device=dev).bfloat16() for _ in range(4)]
        vs = [torch.randn((N_NEW, H, D), generator=g, device=dev).bfloat16() for _ in range(4)]
        for _ in range(8):                       # fill every window
            for w, k, v in zip(wins, ks, vs):
                w.upkeep(k, v, stream=stream)
        torch.cuda.synchronize(dev)
        gr = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gr, stream=stream):
            for _ in range(2):                   # two calls per ring: the buffers alternate back
                for w, k, v in zip(wins, ks, vs):
                    w.upkeep(k, v, stream=stream)
        gr.replay()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        reps = 4
        e0.record(stream)
        for _ in range(reps):
            gr.replay()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        us = e0.elapsed_time(e1) * 1e3 / (reps * 8)
    del rings, wins, ks, vs
    torch.cuda.empty_cache()
    return us


def reduce_max(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device="cuda" if dist.get_backend() == "nccl" else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------------------
# The CPU oracle (float64 NumPy, the test oracle) timed on this host, one
# sample recipe for both the default run's cpu_baseline and the reference
# arm.  A full step on the oracle takes seconds, so each sample is bounded
# and extrapolated: a write of SAMPLE_TOKENS tokens scaled to 757 (its cost
# is linear in the tokens), and attention of SAMPLE_Q[0] and SAMPLE_Q[1]
# queries, fitted as a fixed part (dequantising the whole cache, paid once
# per call) plus a per-query part, then evaluated at 757 queries.
SAMPLE_TOKENS = 64
SAMPLE_Q = (8, 64)


def cpu_setup():
    from oracle import Ring
    from workloads import prod_session, f32_from_bf16
    sk, sv, fr = prod_session(seed=2, frames=9)
    orc = Ring(H, D, C, MAX_POS)
    orc.calibrate(f32_from_bf16(fr[0][1]), f32_from_bf16(fr[0][2]))
    for q, k, v in fr[:8]:
        orc.write(f32_from_bf16(k), f32_from_bf16(v))
    q, k, v = fr[8]
    st = orc, (f32_from_bf16(q), f32_from_bf16(k), f32_from_bf16(v))
    cpu_sample(st)          # untimed: the first attention call pays one-time costs
    return st


def cpu_sample(st):
    """One bounded sample of a step on the oracle; returns the extrapolated
    seconds of the full 757-token write, of the full 757-query attention, and
    the process CPU seconds and wall seconds the sample took."""
    from oracle.attention import attention_exact
    orc, (q, k, v) = st
    c0, w0 = os.times(), time.perf_counter()
    t0 = time.perf_counter()
    orc.write(k[:SAMPLE_TOKENS], v[:SAMPLE_TOKENS])
    t1 = time.perf_counter()
    ta = []
    for nq in SAMPLE_Q:
        ts = time.perf_counter()
        attention_exact(orc, q[:nq], np.arange(orc.next_pos - nq, orc.next_pos))
        ta.append(time.perf_counter() - ts)
    per_q = max((ta[1] - ta[0]) / (SAMPLE_Q[1] - SAMPLE_Q[0]), 0.0)
    fixed = max(ta[0] - per_q * SAMPLE_Q[0], 0.0)
    c1, w1 = os.times(), time.perf_counter()
    cpu = (c1.user - c0.user) + (c1.system - c0.system)
    return dict(write_s=(t1 - t0) * N_NEW / SAMPLE_TOKENS, attn_s=fixed + per_q * N_Q, attn_fixed_s=fixed,
                cpu_s=cpu, wall_s=w1 - w0)


def cpu_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


def blas_threads():
    """The BLAS thread count NumPy would use (the oracle's einsum and
    elementwise work do not go through BLAS, so it runs on one core)."""
    try:
        import threadpoolctl
        info = [x for x in threadpoolctl.threadpool_info() if x.get("user_api") == "blas"]
        if info:
            return int(info[0]["num_threads"])
    except Exception:
        pass
    for var in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS"):
        if os.environ.get(var, "").isdigit():
            return int(os.environ[var])
    return None


def sample_text(n):
    return (f"{n} samples; each writes {SAMPLE_TOKENS} tokens into the wrapped 5,788-slot ring "
            f"(10 heads x 128), scaled x757/{SAMPLE_TOKENS}, and attends {SAMPLE_Q[0]} and {SAMPLE_Q[1]} "
            f"queries, fitted as fixed + per-query cost and evaluated at 757 queries; mean")


def summarise_samples(xs):
    step = [x["write_s"] + x["attn_s"] for x in xs]
    cpu, wall = sum(x["cpu_s"] for x in xs), sum(x["wall_s"] for x in xs)
    return dict(step_us=float(np.mean(step)) * 1e6, write_us=float(np.mean([x["write_s"] for x in xs])) * 1e6,
                attention_us=float(np.mean([x["attn_s"] for x in xs])) * 1e6,
                attention_fixed_us=float(np.mean([x["attn_fixed_s"] for x in xs])) * 1e6,
                threads_used=max(1, int(round(cpu / wall))) if wall > 0 else 1)


def cpu_single_threaded_parts(st):
    """Measured whole, on one core: the full 757-token write, and the delta
    rotation of the full window (after an untimed rotation by 0, which leaves
    the codes as they are, so one-time set-up is not counted)."""
    orc, (q, k, v) = st
    t0 = time.perf_counter()
    orc.write(k, v)
    t1 = time.perf_counter()
    orc.delta_rotate(0)
    t2 = time.perf_counter()
    orc.delta_rotate()
    t3 = time.perf_counter()
    return dict(write_757_us=(t1 - t0) * 1e6, delta_full_window_us=(t3 - t2) * 1e6)


def cpu_baseline(budget_s: float = 12.0):
    st = cpu_setup()
    xs = []
    t_end = time.perf_counter() + budget_s
    while time.perf_counter() < t_end or not xs:
        xs.append(cpu_sample(st))
    sm = summarise_samples(xs)
    return {"value": sm["step_us"], "unit": "µs", "cores": sm["threads_used"], "kind": "oracle",
            "extrapolated": True, "sample": sample_text(len(xs)),
            "affinity_cores": cpu_cores(), "blas_threads": blas_threads(),
            "parts_us": {"write": sm["write_us"], "attention": sm["attention_us"],
                         "attention_fixed": sm["attention_fixed_us"]},
            "single_threaded": cpu_single_threaded_parts(st)}


def reference_arm(args, rank, world):
    if rank != 0:
        return
    st = cpu_setup()
    for _ in range(args.warmup):
        cpu_sample(st)
    xs = [cpu_sample(st) for _ in range(args.steps)]
    sm = summarise_samples(xs)
    us = sm["step_us"]
    line = {
        "metric": METRIC, "value": us, "unit": "µs", "n_gpus": args.gpus, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": us / 1000.0, "higher_is_better": False,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "impl": "reference", "extrapolated": True,
        "config": {"workload": WORKLOAD, "l2": "n/a (CPU)"},
        "cpu_baseline": {"value": us, "unit": "µs", "cores": sm["threads_used"], "kind": "oracle",
                         "extrapolated": True, "sample": sample_text(len(xs)) + " (one sample per step)",
                         "affinity_cores": cpu_cores(), "blas_threads": blas_threads(),
                         "parts_us": {"write": sm["write_us"], "attention": sm["attention_us"],
                                      "attention_fixed": sm["attention_fixed_us"]}},
        "e2e": {"value": us, "unit": "µs", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="kvring", choices=["kvring", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-batched", action="store_true", help="run none of the extra legs (same as --legs none)")
    ap.add_argument("--legs", default=",".join(EXTRA_LEGS),
                    help="extra measurements after the headline step, comma-separated from "
                         f"{','.join(EXTRA_LEGS)} (or 'none')")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    args.legs = set() if args.no_batched else {x for x in args.legs.split(",") if x in EXTRA_LEGS}

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if world > 1:
        import torch
        import torch.distributed as dist
        if args.impl == "kvring":
            torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", 0)))
        dist.init_process_group("nccl" if args.impl == "kvring" else "gloo")

    if args.impl == "reference":
        reference_arm(args, rank, world)
        if world > 1:
            import torch.distributed as dist
            dist.barrier()
            dist.destroy_process_group()
        return

    res = gpu_arm(args, rank, world)
    total_ms = reduce_max(res["total_ms"], world)
    e2e_ms = reduce_max(res["e2e_ms"], world)
    if rank != 0:
        return
    peaks = load_peaks()
    K = args.steps
    units = K * world
    us_per_unit = total_ms * 1e3 / units
    w_us, a_us, d_us = res["w_us"], res["a_us"], res["d_us"]
    fp8_peak = 2.0 * peaks["bf16"]            # FP8 dense = 2 x bf16 (nominal 4.5 / 2.25 PF)
    lv = res["levels"]
    # issued tensor work relative to the algorithmic 2 FP8 units (QK, PV) per
    # tile: one FP8 QK per query term (the level), and PV in f16 at half the
    # FP8 rate (two PV MMAs at level 4)
    issued = float(np.mean(lv + 2.0 * np.where(lv >= 4, 2.0, 1.0))) / 2.0
    attn_tflops = ATTN_FLOPS / (a_us * 1e-6) / 1e12
    write_gbs = WRITE_BYTES / (w_us * 1e-6) / 1e9
    traffic = attention_traffic()
    line = {
        "metric": METRIC,
        "value": us_per_unit,
        "unit": "µs",
        "n_gpus": world,
        "steps": K,
        "warmup": args.warmup,
        "ms_per_step": total_ms / K,
        "higher_is_better": False,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "e4m3",
        "data": "synthetic",
        "config": {
            "workload": WORKLOAD,
            "heads": H, "head_dim": D, "capacity": C, "tokens_per_write": N_NEW, "queries": N_Q,
            "l2": f"cold: {RINGS} rings and input frames round-robin, >126 MB between reuses",
            "launch": "the K timed steps (write + attention of one ring each) as one CUDA graph, one replay",
            "resets": f"one delta rotation per ring every {RESET_PERIOD} writes (positions reset "
                      f"period), inside the timed region: {res['resets']} in {K} steps",
            "parallelism": "replicas" if world > 1 else "1 GPU",
        },
        "roofline": {
            "bound": "tensor",
            "kernel": "k_attention (FP8 attention, tcgen05)",
            "achieved": attn_tflops,
            "peak": fp8_peak,
            "unit": "TFLOP/s",
            "frac": attn_tflops / fp8_peak,
            "traffic": traffic,
            "peak_source": f"{peaks['src']}: FP8 = 2 x bf16 burst {peaks['bf16']} TFLOP/s",
            "issued_mma_over_algorithmic": issued,
            "issued_frac": attn_tflops * issued / fp8_peak,
            "algorithmic_flops_per_launch": ATTN_FLOPS,
            "avg_launch_us": a_us,
            "precision_levels": {str(k): int((lv == k).sum()) for k in (1, 2, 3, 4)},
        },
        "kernels": {
            "write": {"avg_launch_us": w_us, "algorithmic_bytes": WRITE_BYTES, "GB/s": write_gbs,
                      "frac_hbm": write_gbs / peaks["hbm"], "peak_gbs": peaks["hbm"],
                      "floor_us": res["wf_us"],
                      "floor_note": "same grid, launch, wait, state read, ticket and publication, no data "
                                    "(kvring_debug_write_floor)"},
            "attention": {"avg_launch_us": a_us, "TFLOP/s": attn_tflops,
                          "cache_GB/s": ATTN_BYTES / (a_us * 1e-6) / 1e9,
                          "note": "one call = one attention kernel (query prologue fused)"},
            "delta_rotate": {"avg_launch_us": d_us, "algorithmic_bytes": DELTA_BYTES,
                             "GB/s": DELTA_BYTES / (d_us * 1e-6) / 1e9,
                             "frac_hbm": DELTA_BYTES / (d_us * 1e-6) / 1e9 / peaks["hbm"],
                             "floor_us": res["df_us"],
                             "floor_note": "the same launch with delta 0 (no rows move)"},
            **({} if res["full_step"] is None else {"full_step_60_layers": {
                **res["full_step"],
                "upkeep_GB/s": LAYERS * WRITE_BYTES / (res["full_step"]["upkeep_us"] * 1e-6) / 1e9,
                "attention_TFLOP/s": CALLS_PER_STEP * ATTN_FLOPS / (res["full_step"]["attention_us"] * 1e-6) / 1e12,
                "note": "60 layer rings; per step 60 writes (upkeep; also as one batched launch) and 4 x 60 "
                        "attention calls, each set one CUDA graph; step = both in one graph"}}),
            **({} if res["stress"] is None else {"stress_40_heads": {
                **res["stress"],
                "attention_frac_fp8": res["stress"]["attention_tflops"] / fp8_peak,
                "note": "40 heads x 128, Student-t (3 dof) keys and values, scales log-uniform in [0.1, 10]; "
                        "per call over a wrapped 5,788-slot ring, four rings round-robin"}}),
            "timing": "per-kernel: CUDA graphs of 16 back-to-back calls on 16 rings, events around replays "
                      "(a write or reset whose ring no kernel still in flight touches runs before its wait, "
                      "so such calls overlap the call before them)",
            **({} if res["proj"] is None else {
                "project_write": {
                    "avg_launch_us": res["proj"][0], "algorithmic_flops": res["proj"][1],
                    "TFLOP/s": res["proj"][1] / (res["proj"][0] * 1e-6) / 1e12,
                    "frac_bf16": res["proj"][1] / (res["proj"][0] * 1e-6) / 1e12 / peaks["bf16"],
                    "note": "kvring_project_write: 757 x 5,120 x 3,840 bf16 projection (fp32 sums) "
                            "with the ring write in its epilogue"}}),
            **({} if res["legacy_us"] is None else {
                "legacy_upkeep": {
                    "avg_call_us": res["legacy_us"], "algorithmic_bytes": LEGACY_BYTES,
                    "GB/s": LEGACY_BYTES / (res["legacy_us"] * 1e-6) / 1e9,
                    "frac_hbm": LEGACY_BYTES / (res["legacy_us"] * 1e-6) / 1e9 / peaks["hbm"],
                    "per_step_us": {
                        "legacy (upkeep in each of 240 attention calls)": CALLS_PER_STEP * res["legacy_us"],
                        "ring (one write per layer, 60 launches)": LAYERS * w_us,
                        **({} if res["batched"] is None else {
                            "ring (60 layers in one batched write)": res["batched"]["write_us"]}),
                    },
                    "note": "the original upkeep (window copy, RoPE of every key, re-quantisation) per call; "
                            "the pages' step went from 69.7 ms to 6.2 ms of upkeep on 4 H100s",
                }}),
            **({} if res["batched"] is None else {
                "write_batched_60_layers": {
                    "avg_launch_us": res["batched"]["write_us"], "algorithmic_bytes": LAYERS * WRITE_BYTES,
                    "GB/s": LAYERS * WRITE_BYTES / (res["batched"]["write_us"] * 1e-6) / 1e9,
                    "frac_hbm": LAYERS * WRITE_BYTES / (res["batched"]["write_us"] * 1e-6) / 1e9 / peaks["hbm"],
                    "note": "kvring_write_frames_many: one launch, a 757-token frame into each of 60 rings"},
                "delta_batched_60_layers": {
                    "avg_launch_us": res["batched"]["delta_us"], "algorithmic_bytes": LAYERS * DELTA_BYTES,
                    "GB/s": LAYERS * DELTA_BYTES / (res["batched"]["delta_us"] * 1e-6) / 1e9,
                    "frac_hbm": LAYERS * DELTA_BYTES / (res["batched"]["delta_us"] * 1e-6) / 1e9 / peaks["hbm"],
                    "note": "kvring_delta_rotate_many: one launch, 60 full windows rotated"},
            }),
        },
        "e2e": {"value": e2e_ms * 1e3 / units, "unit": "µs",
                "h2d_bytes_per_step": H2D_BYTES, "d2h_bytes_per_step": D2H_BYTES,
                "copies_alone_us_per_step": res["copy_us"],
                "note": "the step's pinned-memory copies timed alone (no kernels): each direction, and both at once"},
        "gpu_launches": 2 * K + res["resets"],   # per step: write + attention; a delta rotation per reset
        "clocks": res["clocks"],
        "device_errors": res["device_errors"],
    }
    errors = dict(res["leg_errors"])
    if not args.no_cpu_baseline:
        cpu = run_leg({"cpu_baseline"}, "cpu_baseline", cpu_baseline, errors)
        if cpu is not None:
            line["cpu_baseline"] = cpu
    if errors:
        line["leg_errors"] = errors
    print(json.dumps(line))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
