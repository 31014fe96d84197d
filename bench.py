#!/usr/bin/env python
"""Benchmark of the Qwen3-TTS 12 Hz frame loop on one GB300 (or N replicas).

A step is one talker step of the whole batch: the code predictor completes
the pending frame of every live row (2-token prefill + 14 steps, 15 draws),
the next talker input is assembled, the 28-layer talker runs and codebook 0
is selected.  Metric: 16-code frames per second (frames emitted by all rows).

Default workload: 0.6B-shaped model in bf16, batch 1, 128-row prompt, 64 text
rows then tts_pad, 100 greedy frames (the latency path).  --workload 3..7
select the 1.7B batch-1, the 0.6B batch-32 and batch-256, and the 1.7B
batch-32 and batch-256 workloads.  With one rank and a batch-1 workload the
line also carries "batches": workloads 4..7 (--batches) timed in the same run,
each over its whole request after 3 warm-up steps, with HBM and tensor-pipe
fractions, prefill time and time to the first frame (--no-batches skips
them); and "codec": one 325-frame window of the full-size codec decoder
(--no-codec skips it).

Prints ONE JSON line (rank 0).  --impl reference times the CPU oracle instead.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import synth  # noqa: E402

ROWSTATE_BYTES = 16 * 4 + 128 * 4     # per-row state read back at the end of every call


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=300)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", default="ours", choices=["ours", "reference"])
    p.add_argument("--workload", type=int, default=2)
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--step-path", default="auto", choices=["auto", "graph", "frame", "cluster"],
                   help="batch-1 step path (the library's default when auto)")
    p.add_argument("--cpu-frames", type=int, default=0, help="oracle frames timed for the CPU baseline (0: auto)")
    p.add_argument("--no-batches", action="store_true", help="skip the batch entries")
    p.add_argument("--no-codec", action="store_true", help="skip the codec-decoder entry")
    p.add_argument("--codec-only", action="store_true",
                   help="no benchmark line: three decodes of the full-size codec window (for ncu launch lists)")
    p.add_argument("--profile-case", action="store_true",
                   help="no benchmark: prefill and 6 steps of the workload with 4 talker layers and a "
                        "context of 320 (full-size launch shapes on a small device footprint, for ncu)")
    p.add_argument("--batches", type=lambda v: [int(x) for x in v.split(",") if x], default=[4, 5, 6, 7],
                   help="workloads of the batch entries (4, 5: batch 32 / 256 of the 0.6B shape; 6, 7: 1.7B)")
    p.add_argument("--batch-steps", type=int, default=0,
                   help="timed steps of each batch entry (0: the whole request after 3 warm-up steps)")
    return p.parse_args()


# ---------------------------------------------------------------- ranks
def job_totals(max_vals, sum_vals, device="cpu"):
    """Whole-job figures of an N-rank run: the maximum over ranks of each entry
    of max_vals (times) and the sum over ranks of each entry of sum_vals
    (frames).  Without an initialised process group (one rank) the values come
    back unchanged.  device: where the reduction tensors live (the rank's GPU
    for NCCL, "cpu" for gloo)."""
    max_vals, sum_vals = [float(v) for v in max_vals], [float(v) for v in sum_vals]
    try:
        import torch
        import torch.distributed as dist
    except ImportError:
        return max_vals, sum_vals
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return max_vals, sum_vals
    t_max = torch.tensor(max_vals or [0.0], dtype=torch.float64, device=device)
    t_sum = torch.tensor(sum_vals or [0.0], dtype=torch.float64, device=device)
    dist.all_reduce(t_max, op=dist.ReduceOp.MAX)
    dist.all_reduce(t_sum, op=dist.ReduceOp.SUM)
    return t_max.tolist()[:len(max_vals)], t_sum.tolist()[:len(sum_vals)]


def job_rate(frames_all: float, seconds_max: float) -> float:
    """Frames of all ranks over the slowest rank's time."""
    return frames_all / seconds_max if seconds_max > 0 else 0.0


# ---------------------------------------------------------------- byte model
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "traffic.txt")


def measured_traffic(workload: int):
    """DRAM bytes per launch of the step's dominant kernel from the committed ncu
    capture, or None when there is none for this workload or the kernel's
    sources changed since it was taken."""
    import hashlib
    try:
        lines = open(TRAFFIC_FILE).read().splitlines()
    except OSError:
        return None, None
    for ln in lines:
        if ln.startswith("#") or not ln.strip():
            continue
        kv = dict(tok.split("=", 1) for tok in ln.split())
        if int(kv.get("workload", -1)) != workload:
            continue
        h = hashlib.sha256()
        for f in kv["sources"].split(","):
            with open(os.path.join(ROOT, "speech_lm_decode_gb300", "csrc", f), "rb") as fh:
                h.update(fh.read())
        if h.hexdigest()[:16] != kv["sha"]:
            return None, kv["kernel"]
        return float(kv["bytes"]), kv["kernel"]
    return None, None


def row_flops(d) -> float:
    """Algorithmic multiply-add FLOPs of the projections for one row and one
    frame: the talker (1 token through 28 layers + codec head) and the
    predictor (16 token passes through its layers: the 2-token prefill and 14
    steps, 15 heads, and the input projection when the widths differ)."""
    qkv = (d.n_q_heads + 2 * d.n_kv_heads) * d.head_dim

    def layer(H, F):
        return qkv * H + H * d.n_q_heads * d.head_dim + 2 * F * H + H * F
    G1 = d.n_groups - 1
    talker = d.n_layers * layer(d.hidden, d.ffn) + d.codec_vocab * d.hidden
    passes = G1 + 1
    pred = passes * d.cp_layers * layer(d.cp_hidden, d.cp_ffn) + G1 * d.cp_vocab * d.cp_hidden
    if d.hidden != d.cp_hidden:
        pred += passes * d.cp_hidden * d.hidden
    return 2.0 * (talker + pred)


def step_bytes(wl, live_pos):
    """Algorithmic bytes of one step: every weight streamed once per use plus
    the KV cache read (and written) by attention.  live_pos: talker position of
    each live row's new token."""
    d = wl.dims
    wb = synth.weight_bytes(d, wl.dtype)
    e = 4 if wl.dtype == synth.F32 else 2
    G1 = d.n_groups - 1
    weights = (d.n_layers * wb["talker_layer"] + wb["codec_head"] + wb["final_norm"]
               + G1 * (d.cp_layers * wb["cp_layer"] + wb["cp_head"] + wb["cp_final_norm"] + wb["cp_proj"]))
    per_pos = d.n_kv_heads * d.head_dim * 2 * e          # K and V of one position, one layer
    kv = 0
    cp_positions = 3 + sum(s + 2 for s in range(1, G1))  # prefill reads 1+2 positions, step s reads s+2
    for p in live_pos:
        kv += d.n_layers * ((p + 1) + 1) * per_pos         # read 0..p, write p
        kv += d.cp_layers * (cp_positions + 16) * per_pos
        kv += (d.n_groups + 1) * d.hidden * e              # embedding gathers
    return weights, kv


# ---------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.path = os.path.join("/tmp", f"q3_clocks_{os.getpid()}.csv")

    def __enter__(self):
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"], stdout=self.f,
                                         stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.f.close()

    def summary(self):
        if not self.proc:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        os.unlink(self.path)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def peaks():
    try:
        return json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json"))), "measured"
    except OSError:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


# ---------------------------------------------------------------- codec decoder
def codec_flops(d) -> float:
    """Algorithmic FLOPs (2 per multiply-add) of decoding one frame: every
    weight use once (convolutions as their multiply-adds)."""
    D, F, F2, Dc = d.hidden, d.ffn, d.up_ffn, d.codebook_dim
    f = 2 * D * Dc + d.n_layers * (3 * D * D + D * D + 2 * F * D + D * F)
    n = 1
    for _ in range(d.n_up):
        f += n * 2 * D * D
        n *= 2
        f += n * 2 * F2 * D
    C = d.dac_channels
    f += n * C * 7 * D
    for s in d.strides:
        Co = C // 2
        f += n * s * Co * 2 * C
        n *= s
        C = Co
        f += 3 * n * (7 * C * C + C * C)
    f += n * 7 * C
    return 2.0 * f


def run_codec(args, pk, pk_kind):
    """One 325-frame window (a 300-frame chunk + 25 frames of context) of the
    full-size decoder, device-resident codes: median of timed decodes."""
    import torch
    import speech_lm_decode_gb300 as q3
    import synth.codec as sc
    d = sc.CODEC_FULL
    T = 325
    w = sc.make_codec_weights(d, synth.BF16, 3)
    dev = torch.device("cuda", 0)
    stream = torch.cuda.Stream(dev)
    dec = q3.Q3Codec(d, synth.BF16, q3.codec_to_device(w, dev), max_frames=T, stream=stream)
    codes = torch.from_numpy(sc.make_codes(d, T, 4)).to(dev)
    out = torch.empty(T * dec.spf, dtype=torch.float32, device=dev)
    for _ in range(3):
        dec.decode_window(codes, out=out)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    times = []
    clocks = ClockSampler(dev.index)
    with clocks:
        for _ in range(7):
            torch.cuda.synchronize(dev)
            ev0.record(stream)
            dec.decode_window(codes, out=out)
            ev1.record(stream)
            torch.cuda.synchronize(dev)
            times.append(ev0.elapsed_time(ev1))
    ms = statistics.median(times)
    fl = codec_flops(d) * T
    ach = fl / (ms / 1000.0) / 1e12
    res = {"workload": f"codec decoder, one {T}-frame window (300-frame chunk + 25 frames of context), bf16, "
                       f"{dec.spf} samples per frame",
           "ms_per_window": ms, "frames_per_s": T / (ms / 1000.0), "samples_per_s": T * dec.spf / (ms / 1000.0),
           "real_time_factor": (T * 0.08) / (ms / 1000.0),
           "tensor": {"achieved": ach, "peak": pk["bf16_tflops_sustained"], "unit": "TFLOP/s",
                      "frac": ach / pk["bf16_tflops_sustained"], "flops_per_window": fl,
                      "peak_kind": pk_kind + " (sustained)",
                      "note": "one bf16 product per weight use; the MMAs run the fp32 operand as bf16 high + low "
                              "parts, twice that work"},
           "gpu_launches_per_window": dec.kernel_count(), "clocks": clocks.summary()}
    dec.close()
    if not args.no_cpu_baseline:
        import oracle.codec as oc
        ora = oc.Decoder(d, w)
        t0 = time.perf_counter()
        ora.decode_window(sc.make_codes(d, 3, 4))
        dt = time.perf_counter() - t0
        res["cpu_baseline"] = {"value": 3 / dt, "unit": "frames/s", "cores": omp_threads(), "kind": "oracle",
                               "sample": f"a 3-frame window of the same decoder, {dt:.1f} s"}
    return res


# ---------------------------------------------------------------- oracle (CPU baseline / reference arm)
def oracle_rate(wl, w, inp, n_frames, warm_frames=0, timed_threads=0):
    """Oracle frames/s on row 0 of the workload: prefill and warm_frames steps
    (untimed), then n_frames timed steps (with timed_threads worker threads
    when > 0).  Returns (rate, timed frames, seconds, warm frames run)."""
    import oracle
    rows = [0]
    lens = [wl.prompt_lens[0]]
    po = inp["prompt_offsets"]
    to = inp["text_offsets"]
    T = wl.frames
    o = oracle.Oracle(wl.dims, wl.dtype, w, 1, wl.max_ctx, T, capture=False)
    o.prefill(inp["prompt"][po[0]:po[1]], np.array([0, lens[0]], np.int32), inp["text"][to[0]:to[1]],
              np.array([0, to[1] - to[0]], np.int32), inp["tts_pad"], [wl.rows[0]], rows)
    warm = max(0, min(warm_frames, T - 1))
    if warm:
        o.step(warm)
    warm_done = int(o.get("frames")[0])
    n = max(1, min(n_frames, T - warm))
    prev = oracle.set_threads(timed_threads) if timed_threads > 0 else 0
    t0 = time.perf_counter()
    o.step(n)
    dt = time.perf_counter() - t0
    if timed_threads > 0:
        oracle.set_threads(prev)
    done = int(o.get("frames")[0]) - warm_done
    return done / dt, done, dt, warm


def omp_threads():
    v = os.environ.get("OMP_NUM_THREADS")
    return int(v) if v else os.cpu_count()


def cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo)."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for ln in out.splitlines():
            if ln.lower().startswith("model name"):
                return ln.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        for ln in open("/proc/cpuinfo"):
            if ln.lower().startswith(("model name", "cpu part")):
                return ln.split(":", 1)[1].strip()
    except OSError:
        pass
    return "unknown"


# ---------------------------------------------------------------- our arm
def run_ours(args, wl, rank, world):
    import torch
    import speech_lm_decode_gb300 as q3
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    w = synth.make_weights(wl.dims, wl.dtype, wl.weight_seed)
    inp = synth.make_inputs(wl)
    dw = q3.to_device_weights(w, dev)
    stream = torch.cuda.Stream(dev)
    path = {"auto": q3.Q3_PATH_AUTO, "graph": q3.Q3_PATH_GRAPH, "frame": q3.Q3_PATH_FRAME,
            "cluster": q3.Q3_PATH_CLUSTER}[args.step_path]
    q = q3.Q3TTS(wl.dims, wl.dtype, dw, wl.batch, wl.max_ctx, max(max(wl.n_text), 1), stream=stream,
                 step_path=path)
    d_inp = {k: (torch.from_numpy(v).to(dev) if k in ("prompt", "text", "tts_pad") else v) for k, v in inp.items()}
    codes_dev = torch.empty((wl.batch, wl.frames, wl.dims.n_groups), dtype=torch.int32, device=dev)
    lens = np.array(wl.prompt_lens)

    def prefill():
        q.prefill(d_inp["prompt"], inp["prompt_offsets"], d_inp["text"], inp["text_offsets"], d_inp["tts_pad"],
                  wl.rows)

    def barrier():
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize(dev)

    prefill()
    steps_done = 0
    frames = np.zeros(wl.batch, np.int32)
    reasons = np.zeros(wl.batch, np.int32)
    if args.warmup:
        _, frames, reasons = q.step_frames(min(args.warmup, wl.frames), codes_out=codes_dev.view(-1))
        steps_done = min(args.warmup, wl.frames)
    kernels_per_step = q.step_kernel_count()
    step_path = q3.PATH_NAMES.get(q.step_path(wl.batch), "graph")
    rf = row_flops(wl.dims)
    flops_total = 0.0
    ctx_lo, ctx_hi = 1 << 30, 0
    remaining = args.steps
    total_ms = 0.0
    total_frames = 0
    wbytes_total = 0
    kvbytes_total = 0
    timed_steps = 0
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(dev.index)
    with clocks:
        while remaining > 0:
            budget = wl.frames - steps_done
            if budget <= 0 or np.all(reasons != q3.Q3_RUNNING):
                prefill()
                steps_done = 0
                frames = np.zeros(wl.batch, np.int32)
                reasons = np.zeros(wl.batch, np.int32)
                continue
            n = min(remaining, budget)
            live_before = reasons == q3.Q3_RUNNING
            f_before = frames.copy()
            barrier()
            ev0.record(stream)
            _, frames, reasons = q.step_frames(n, codes_out=codes_dev.view(-1)[: wl.batch * n * wl.dims.n_groups])
            ev1.record(stream)
            barrier()
            total_ms += ev0.elapsed_time(ev1)
            total_frames += int(np.sum(frames - f_before))
            # bytes: every step streams the weights; each row live at a step reads its cache
            for j in range(n):
                k = steps_done + j + 1
                live = [int(lens[r] + k - 1) for r in range(wl.batch)
                        if live_before[r] and (frames[r] > f_before[r] + j or (reasons[r] != q3.Q3_RUNNING and
                                                                               frames[r] == f_before[r] + j))]
                wb, kb = step_bytes(wl, live)
                wbytes_total += wb
                kvbytes_total += kb
                flops_total += rf * len(live)
                if live:
                    ctx_lo, ctx_hi = min(ctx_lo, min(live) + 1), max(ctx_hi, max(live) + 1)
            steps_done += n
            timed_steps += n
            remaining -= n
    # time to the first frame: the prefill (prompt through the talker, selection
    # 0), then one step (frame 0 through the predictor, selection 1); median of 3
    pre, ttff = [], []
    for _ in range(3):
        barrier()
        ev0.record(stream)
        prefill()
        ev1.record(stream)
        q.step_frames(1, codes_out=codes_dev.view(-1)[: wl.batch * wl.dims.n_groups])
        ev2 = torch.cuda.Event(enable_timing=True)
        ev2.record(stream)
        barrier()
        pre.append(ev0.elapsed_time(ev1))
        ttff.append(ev0.elapsed_time(ev2))
    prefill_ms, ttff_ms = statistics.median(pre), statistics.median(ttff)
    # time to the first audio at batch 1 (the pages' first-packet latency):
    # prefill, 4 steps (the first streamed decode comes after 4 frames), and
    # the full-size codec decoder on those 4 frames; median of 3
    ttfa_ms = None
    if wl.batch == 1 and not getattr(args, "no_codec", False) and wl.frames >= 4:
        import synth.codec as sc
        dcodec = sc.CODEC_FULL
        dec = q3.Q3Codec(dcodec, synth.BF16, q3.codec_to_device(sc.make_codec_weights(dcodec, synth.BF16, 3), dev),
                         max_frames=16, stream=stream)
        wav = torch.empty(4 * dec.spf, dtype=torch.float32, device=dev)
        first = codes_dev.view(-1)[: 4 * wl.dims.n_groups]
        ta = []
        for _ in range(3):
            barrier()
            ev0.record(stream)
            prefill()
            q.step_frames(4, codes_out=first)
            dec.decode_window(first.view(4, wl.dims.n_groups), out=wav, check=False)
            ev2 = torch.cuda.Event(enable_timing=True)
            ev2.record(stream)
            barrier()
            ta.append(ev0.elapsed_time(ev2))
        ttfa_ms = statistics.median(ta)
        dec.close()
    (max_ms,), (all_frames,) = job_totals([total_ms], [total_frames], dev)
    res = dict(ms=max_ms, frames=all_frames, local_frames=total_frames, steps=timed_steps,
               wbytes=wbytes_total, kvbytes=kvbytes_total, kernels_per_step=kernels_per_step,
               clocks=clocks.summary(), local_ms=total_ms, flops=flops_total, ctx=(ctx_lo, ctx_hi),
               step_path=step_path, prefill_ms=prefill_ms, ttff_ms=ttff_ms, ttfa_ms=ttfa_ms)

    # e2e: the whole request through the C ABI from pinned host buffers, one call per step,
    # codes read back to pinned host memory after every step
    if not getattr(args, "no_e2e", False):
        h_prompt = torch.from_numpy(inp["prompt"]).pin_memory()
        h_text = torch.from_numpy(inp["text"]).pin_memory()
        h_pad = torch.from_numpy(inp["tts_pad"]).pin_memory()
        h_codes = torch.empty((wl.batch, 1, wl.dims.n_groups), dtype=torch.int32).pin_memory()
        barrier()
        t0 = time.perf_counter()
        q.prefill(h_prompt, inp["prompt_offsets"], h_text, inp["text_offsets"], h_pad, wl.rows)
        nsteps = 0
        fr = np.zeros(wl.batch, np.int32)
        for _ in range(wl.frames):
            _, fr, rs = q.step_frames(1, codes_out=h_codes)
            nsteps += 1
            if np.all(rs != q3.Q3_RUNNING):
                break
        barrier()
        e2e_s = time.perf_counter() - t0
        in_bytes = inp["prompt"].nbytes + inp["text"].nbytes + inp["tts_pad"].nbytes
        # whole job: every rank's frames over the slowest rank's time
        (e2e_s,), (e2e_frames,) = job_totals([e2e_s], [int(fr.sum())], dev)
        res["e2e"] = dict(frames=e2e_frames, seconds=e2e_s, steps=nsteps,
                          h2d_per_step=in_bytes / nsteps,
                          d2h_per_step=wl.batch * wl.dims.n_groups * 4 + wl.batch * ROWSTATE_BYTES + 16)
    q.close()
    return res, w, inp


def profile_case(args):
    """The workload's launches at full width and batch on a small footprint:
    4 talker layers, a 320-position cache, a prefill and 6 steps."""
    import dataclasses
    import torch
    import speech_lm_decode_gb300 as q3
    wl = synth.workload(args.workload)
    wl = dataclasses.replace(wl, dims=dataclasses.replace(wl.dims, n_layers=4), frames=12,
                             max_ctx=max(wl.prompt_lens) + 64,
                             rows=[dataclasses.replace(r, max_frames=12) for r in wl.rows])
    dev = torch.device("cuda", 0)
    w = synth.make_weights(wl.dims, wl.dtype, wl.weight_seed)
    inp = synth.make_inputs(wl)
    q = q3.Q3TTS(wl.dims, wl.dtype, q3.to_device_weights(w, dev), wl.batch, wl.max_ctx, max(wl.n_text))
    d_inp = {k: (torch.from_numpy(v).to(dev) if k in ("prompt", "text", "tts_pad") else v) for k, v in inp.items()}
    q.prefill(d_inp["prompt"], inp["prompt_offsets"], d_inp["text"], inp["text_offsets"], d_inp["tts_pad"], wl.rows)
    _, frames, _ = q.step_frames(6)
    torch.cuda.synchronize()
    q.close()
    print("profile case done:", wl.name, "with 4 talker layers,", int(frames.sum()), "frames")


def main():
    args = parse()
    if args.profile_case:
        profile_case(args)
        return
    if args.codec_only:
        import torch
        import speech_lm_decode_gb300 as q3
        import synth.codec as sc
        dev = torch.device("cuda", 0)
        d = sc.CODEC_FULL
        dec = q3.Q3Codec(d, synth.BF16, q3.codec_to_device(sc.make_codec_weights(d, synth.BF16, 3), dev),
                         max_frames=325)
        codes = torch.from_numpy(sc.make_codes(d, 325, 4)).to(dev)
        out = torch.empty(325 * dec.spf, dtype=torch.float32, device=dev)
        for _ in range(3):
            dec.decode_window(codes, out=out)
        torch.cuda.synchronize()
        print("codec windows done:", dec.kernel_count(), "launches per window")
        dec.close()
        return
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    wl = synth.workload(args.workload)
    metric = "16-code frames/sec"
    unit = "frames/s"
    config = {"workload": f"config {args.workload}: {wl.name}", "batch": wl.batch,
              "prompt_rows": (wl.prompt_lens[0] if len(set(wl.prompt_lens)) == 1
                              else f"{min(wl.prompt_lens)}..{max(wl.prompt_lens)}"),
              "frames_per_request": wl.frames, "max_ctx": wl.max_ctx,
              "l2": "no flush: every step streams >3 GB of weights, far above the 129 MB L2"}

    if args.impl == "reference":
        if rank != 0:
            return
        w = synth.make_weights(wl.dims, wl.dtype, wl.weight_seed)
        inp = synth.make_inputs(wl)
        n = max(1, min(args.steps, 40))
        rate, done, dt, warm = oracle_rate(wl, w, inp, n, warm_frames=min(args.warmup, 8))
        sample = (f"row 0 of the workload, {done} frames after its prefill and {warm} warm-up frames (untimed), "
                  f"{dt:.1f} s")
        line = {"impl": "reference", "metric": metric, "value": rate, "unit": unit, "n_gpus": args.gpus,
                "steps": done, "warmup": warm, "ms_per_step": 1000.0 * dt / max(done, 1), "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded random init)",
                "config": config,
                "cpu_baseline": {"value": rate, "unit": unit, "cores": omp_threads(), "kind": "oracle",
                                 "cpu_model": cpu_model(), "sample": sample},
                "e2e": {"value": rate, "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        print(json.dumps(line))
        return

    import torch
    if world > 1:
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", 0)))
        torch.distributed.init_process_group("nccl")
    res, w, inp = run_ours(args, wl, rank, world)
    if rank != 0:
        if world > 1:
            torch.distributed.destroy_process_group()
        return
    pk, pk_kind = peaks()
    sec = res["ms"] / 1000.0
    value = job_rate(res["frames"], sec)
    bytes_total = res["wbytes"] + res["kvbytes"]
    achieved = bytes_total / (res["local_ms"] / 1000.0) / 1e9
    # the step's kernel, as the library reports the path it ran
    kernel_name = {"frame": "frame_kernel (one launch = the whole step; traffic from ncu, bytes per launch)",
                   "cluster": "cluster_step_kernel (one launch = the whole step)",
                   "graph": "frame step (all kernels of one talker step)"}[res["step_path"]]
    traffic, tk = measured_traffic(args.workload) if res["step_path"] == "frame" else (None, None)
    line = {"metric": metric, "value": value, "unit": unit, "n_gpus": world, "steps": res["steps"],
            "warmup": args.warmup, "ms_per_step": res["ms"] / max(res["steps"], 1), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16" if wl.dtype == synth.BF16 else "f32",
            "data": "synthetic (seeded random-init weights, N(0,1) prompts)", "config": config,
            "us_per_frame": 1e6 * sec / max(res["frames"], 1),
            "roofline": {"bound": "hbm", "kernel": kernel_name,
                         "achieved": achieved, "peak": pk["hbm_gbs"], "unit": "GB/s",
                         "frac": achieved / pk["hbm_gbs"], "peak_kind": pk_kind,
                         "traffic": traffic, "algorithmic_bytes_per_step": bytes_total / max(res["steps"], 1)},
            "step_path": res["step_path"],
            "prefill_ms": res["prefill_ms"], "time_to_first_frame_ms": res["ttff_ms"],
            "time_to_first_audio_ms": res["ttfa_ms"],
            "gpu_launches": res["kernels_per_step"] * res["steps"],
            "clocks": res["clocks"]}
    if "e2e" in res:
        e = res["e2e"]
        line["e2e"] = {"value": job_rate(e["frames"], e["seconds"]), "unit": unit,
                       "h2d_bytes_per_step": e["h2d_per_step"], "d2h_bytes_per_step": e["d2h_per_step"],
                       "note": "prefill from pinned host + one q3tts_step_frames(1) per step, codes to pinned host"}
    if not args.no_batches and world == 1 and wl.batch == 1:
        line["batches"] = []
        del w, inp
        for idx in args.batches:
            wlb = synth.workload(idx)
            ba = argparse.Namespace(**vars(args))
            ba.warmup, ba.no_e2e, ba.step_path = 3, True, "auto"
            ba.steps = args.batch_steps or (wlb.frames - ba.warmup)
            rb, _, _ = run_ours(ba, wlb, rank, world)
            sb = rb["ms"] / 1000.0
            bb = rb["wbytes"] + rb["kvbytes"]
            ach_hbm = bb / sb / 1e9
            ach_tc = rb["flops"] / sb / 1e12
            line["batches"].append({
                "workload": f"config {idx}: {wlb.name}", "batch": wlb.batch, "steps": rb["steps"],
                "ms_per_step": rb["ms"] / max(rb["steps"], 1), "frames_per_s": job_rate(rb["frames"], sb),
                "ctx_range": list(rb["ctx"]), "step_path": rb["step_path"],
                "prefill_ms": rb["prefill_ms"], "time_to_first_frame_ms": rb["ttff_ms"],
                "hbm": {"achieved": ach_hbm, "peak": pk["hbm_gbs"], "unit": "GB/s", "frac": ach_hbm / pk["hbm_gbs"],
                        "bytes_per_step": bb / max(rb["steps"], 1), "peak_kind": pk_kind},
                "tensor": {"achieved": ach_tc, "peak": pk["bf16_tflops_sustained"], "unit": "TFLOP/s",
                           "frac": ach_tc / pk["bf16_tflops_sustained"], "flops_per_step": rb["flops"] / max(rb["steps"], 1),
                           "peak_kind": pk_kind + " (sustained)",
                           "note": "algorithmic FLOPs (one bf16 product per weight); the MMAs run the fp32 "
                                   "operand as bf16 high + low parts, twice that work"},
                "bound": "hbm" if ach_hbm / pk["hbm_gbs"] >= ach_tc / pk["bf16_tflops_sustained"] else "tensor",
                "gpu_launches_per_step": rb["kernels_per_step"], "clocks": rb["clocks"]})
            import torch
            torch.cuda.empty_cache()
        w = synth.make_weights(wl.dims, wl.dtype, wl.weight_seed) if not args.no_cpu_baseline else None
        inp = synth.make_inputs(wl) if not args.no_cpu_baseline else None
    if not args.no_codec and world == 1 and wl.batch == 1:
        line["codec"] = run_codec(args, pk, pk_kind)
    if not args.no_cpu_baseline and world == 1:
        n = args.cpu_frames or (20 if wl.dims.hidden <= 1024 else 10)
        rate, done, dt, _ = oracle_rate(wl, w, inp, n)
        r1, n1, dt1, _ = oracle_rate(wl, w, inp, 2 if wl.dims.hidden <= 1024 else 1, timed_threads=1)
        line["cpu_baseline"] = {"value": rate, "unit": unit, "cores": omp_threads(), "kind": "oracle",
                                "cpu_model": cpu_model(),
                                "sample": f"row 0, {done} frames after prefill, {dt:.1f} s",
                                "single_thread": {"value": r1, "unit": unit, "sample": f"row 0, {n1} frames, {dt1:.1f} s"}}
    print(json.dumps(line))
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
