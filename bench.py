#!/usr/bin/env python
"""Throughput of the streaming codec decoder on one GB300 (or N replicas).

Workload (one "step"): 64 independent streams of the Qwen3-TTS-12Hz-shaped
decoder, 250 frames (20 s of 24 kHz audio) each, stream s starting at global
frame s mod 25 and decoded in ragged ticks of up to 25 frames per stream with
the 72-frame attention window and every conv context carried between ticks;
the streams are reset at the start of each step.  Synthetic codes (uniform,
seed + stream id) and random N(0, 1/fan_in) weights.

value: seconds of audio decoded per second, all GPUs, inputs resident in HBM.
e2e:   the same through codec_decode_chunk_host: every tick copies its codes
       from page-locked host memory and its audio back.
Also reported: per-kernel roofline of the dominant kernel (CUDA events around
every launch, inside the timed region), the first-audio latency (1 frame from
an empty state), SM clocks sampled during the timed region, and the CPU
oracle timed on the host cores on a bounded sample (cpu_baseline).

--impl reference times the CPU oracle itself on the same workload's unit.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time
from pathlib import Path

import numpy as np

ROOT = Path(__file__).resolve().parent
sys.path.insert(0, str(ROOT))

from streaming_tts_vocoder_gb300.synthetic import (CONFIGS, FRAME_RATE_HZ, make_codes, make_latents,  # noqa: E402
                                                   make_weights, pack_blob, qwen3_config, staggered_schedule,
                                                   tiny_config)

METRIC = "codec decode audio-sec/sec at 64 streams (x real time)"
UNIT = "audio-s/s"
PEAKS_FILE = ROOT / "MEASURED_PEAKS.json"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "sm_max_mhz": 2070.0}
SMS = 152
FP32_LANES_PER_SM = 128


DECODER_NAMES = {"qwen3": "Qwen3-TTS-12Hz-shaped", "tiny": "tiny", "mimi": "Mimi-shaped latent-input",
                 "tiny_mimi": "tiny latent-input"}


def peaks():
    try:
        p = json.loads(PEAKS_FILE.read_text())
        return p, "measured"
    except Exception:
        return FALLBACK_PEAKS, "fallback"


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--decoder", choices=["qwen3", "tiny", "mimi", "tiny_mimi"], default="qwen3",
                    help="mimi / tiny_mimi: the latent-input variant (codec_decode_latents)")
    ap.add_argument("--precision", choices=["fp32", "fp16x3", "fp16"], default="fp16x3")
    ap.add_argument("--weights", choices=["fp32", "q8"], default="fp32",
                    help="q8: create the codec from the int8-per-32 weight file (codec_create_q8)")
    ap.add_argument("--streams", type=int, default=64)
    ap.add_argument("--frames", type=int, default=250)
    ap.add_argument("--chunk", type=int, default=25)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu", action="store_true", help="skip the cpu_baseline oracle timing")
    ap.add_argument("--first-audio-runs", type=int, default=100)
    ap.add_argument("--no-streaming", action="store_true",
                    help="skip the streaming-schedule section (TTFA, gaps, carried vs recompute)")
    ap.add_argument("--schedule", action="store_true",
                    help="latency of streaming chunk schedules (time to first audio, per-chunk latency, "
                         "playback gaps) for carried-state and recompute decoding, instead of the throughput line")
    ap.add_argument("--profile-call", default=None, metavar="S,CH,REPS",
                    help="profiling aid: REPS fixed decode calls of S streams x CH frames (graphs off), no timing")
    ap.add_argument("--workload", choices=["decoder", "istft", "source", "vocos"], default="decoder",
                    help="istft: the streaming iSTFT head alone (Vocos-shaped: n_fft 1024, hop 256, 24 kHz), "
                         "--streams streams x 10 chunks of 94 frames; source: the harmonic sine source (8 "
                         "harmonics, F0 every 256 samples) and the analysis STFT (n_fft 16, hop 4) on the "
                         "same streams and chunk lengths")
    ap.add_argument("--layer-times", default=None, metavar="S,CH",
                    help="per-launch CUDA-event times of one decode call of S streams x CH frames from an empty "
                         "state (graphs off), labelled by layer, one JSON line")
    return ap.parse_args()


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def barrier(world: int) -> None:
    """Process-group barrier across the replicas (no-op for one process)."""
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    """The slowest replica's time: every rank gets the max over ranks."""
    if world > 1:
        import torch
        import torch.distributed as dist
        t = torch.tensor([float(x)], dtype=torch.float64)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        return float(t.item())
    return float(x)


def job_throughput(units_per_rank: float, ms_max: float, world: int) -> float:
    """Whole-job rate: every replica's units over the slowest replica's time."""
    return world * units_per_rank / (ms_max / 1e3)


def config_dict(args, precision):
    return {
        "workload": f"{args.streams} staggered streams x {args.frames} frames, ragged ticks of <= {args.chunk} frames, "
                    f"{DECODER_NAMES[args.decoder]} decoder",
        "decoder": args.decoder,
        "streams": args.streams,
        "frames_per_stream": args.frames,
        "chunk_frames": args.chunk,
        "stagger": f"stream s starts at frame s mod {args.chunk}",
        "precision": precision,
        "weights": getattr(args, "weights", "fp32"),
        "samples_per_frame": 1920,
        "l2": "inputs larger than L2: each tick writes and reads GBs of activations",
        "parallelism": "replicas (one independent decoder per GPU, no collective)",
    }


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during a region."""

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.file = None

    def start(self):
        try:
            self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index),
                 "--query-gpu=clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
                 "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                 "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=self.file, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.file.flush()
        self.file.seek(0)
        rows = [ln.strip().split(",") for ln in self.file.read().splitlines() if ln.strip()]
        os.unlink(self.file.name)
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            try:
                sm.append(float(r[0]))
                mx = float(r[1])
                for nm, v in zip(names, r[4:8]):
                    if v.strip().lower() == "active":
                        reasons.add(nm)
            except (ValueError, IndexError):
                continue
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


def traffic_for(kernel: str, src_digest: str):
    """DRAM bytes per launch of `kernel` from the committed ncu summary, if it
    was taken on the current kernel source."""
    f = ROOT / "profiles" / "traffic.json"
    try:
        d = json.loads(f.read_text())
        e = d.get(kernel)
        if e and e.get("source_sha256") == src_digest:
            return e.get("dram_bytes_per_launch")
    except Exception:
        pass
    return None


def kernel_source_digest(files):
    h = hashlib.sha256()
    for f in files:
        h.update((ROOT / "streaming_tts_vocoder_gb300" / "csrc" / f).read_bytes())
    return h.hexdigest()


def weight_bytes(cfg, precision):
    """Bytes of the non-codebook weights as the kernels store them: fp32 or
    the fp16 hi + lo planes (4 bytes per weight), or the hi plane alone
    (single-pass fp16, 2 bytes) for the tensor-core contractions."""
    from streaming_tts_vocoder_gb300.synthetic import weight_manifest
    n = sum(t.size for t in weight_manifest(cfg) if not t.name.startswith("cb."))
    return n * (2 if precision == "fp16" else 4)


def oracle_sample(cfg, blob, frames, seed=1000):
    """Time the CPU oracle decoding `frames` frames of one stream."""
    from oracle import oracle as O
    m = O.OracleModel(cfg, blob)
    s = m.stream()
    if cfg.latent_dim:
        x = make_latents(cfg, frames, seed)
        t0 = time.perf_counter()
        s.decode_latents(x)
    else:
        codes = make_codes(cfg, frames, seed)
        t0 = time.perf_counter()
        s.decode(codes)
    dt = time.perf_counter() - t0
    return frames / FRAME_RATE_HZ / dt, dt, O.max_threads()


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    cfg = CONFIGS[args.decoder]()
    blob = pack_blob(cfg, make_weights(cfg, 0))
    from oracle import oracle as O
    m = O.OracleModel(cfg, blob)
    frames = {"qwen3": 25, "mimi": 100}.get(args.decoder, 250)
    times = []
    for i in range(args.warmup + args.steps):
        s = m.stream()
        if cfg.latent_dim:
            x = make_latents(cfg, frames, 1000 + i)
            t0 = time.perf_counter()
            s.decode_latents(x)
        else:
            codes = make_codes(cfg, frames, 1000 + i)
            t0 = time.perf_counter()
            s.decode(codes)
        dt = time.perf_counter() - t0
        if i >= args.warmup:
            times.append(dt)
    total = sum(times)
    value = args.steps * frames / FRAME_RATE_HZ / total
    sample = f"one stream x {frames} frames of the workload per step (one {frames}-frame chunk from an empty state)"
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f32 storage, f64 accumulation", "data": "synthetic",
        "config": config_dict(args, "oracle"),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": O.max_threads(), "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def run_ours(args):
    import torch
    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("gloo", init_method="env://")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    from streaming_tts_vocoder_gb300 import codec as C

    cfg = CONFIGS[args.decoder]()
    prec = {"fp16x3": C.PRECISION_FP16X3, "fp16": C.PRECISION_FP16, "fp32": C.PRECISION_FP32}[args.precision]
    blob = pack_blob(cfg, make_weights(cfg, 0))
    S, F, CH = args.streams, args.frames, args.chunk
    latent = cfg.latent_dim > 0
    if args.weights == "q8":
        from streaming_tts_vocoder_gb300.weights_q8 import pack_q8
        cod = C.Codec(cfg, q8=pack_q8(cfg, blob), max_streams=S, max_chunk_frames=CH, max_batch_frames=S * CH,
                      precision=prec)
    else:
        cod = C.Codec(cfg, blob, max_streams=S, max_chunk_frames=CH, max_batch_frames=S * CH, precision=prec)
    st = cod.state()
    spf = cod.samples_per_frame

    # inputs resident in HBM: one codes (or latents) tensor per tick
    codes = [make_latents(cfg, F, 1000 + s) if latent else make_codes(cfg, F, 1000 + s) for s in range(S)]
    ticks = staggered_schedule(S, F, CH)
    tick_inputs = []
    h2d = d2h = 0
    for tick in ticks:
        if latent:
            arr = np.zeros((len(tick), CH, cfg.latent_dim), np.float32)
            for b, (s, a, n) in enumerate(tick):
                arr[b, :n] = codes[s][a:a + n]
        else:
            arr = np.zeros((len(tick), cfg.Q, CH), np.int32)
            for b, (s, a, n) in enumerate(tick):
                arr[b, :, :n] = codes[s][:, a:a + n]
        nf = [n for _, _, n in tick]
        ids = [s for s, _, _ in tick]
        tick_inputs.append((torch.from_numpy(arr).to(dev), nf, ids, torch.from_numpy(arr).pin_memory()))
        h2d += arr.nbytes
        d2h += sum(nf) * spf * 4
    audio = torch.empty(S, CH * spf, device=dev)
    audio_h = torch.empty(S, CH * spf).pin_memory()
    stream = torch.cuda.current_stream()
    audio_s_per_step = S * F / FRAME_RATE_HZ

    launches = [0]

    def decode(inp, nf, out, ids):
        if latent:
            st.decode_latents(inp, nf, out, stream_ids=ids, stream=stream)
        else:
            st.decode(inp, nf, out, stream_ids=ids, stream=stream)

    def step():
        st.reset(stream=stream)
        launches[0] += 1
        for inp_d, nf, ids, _ in tick_inputs:
            decode(inp_d, nf, audio, ids)
            launches[0] += st.last_launches

    lat_d = torch.empty(S, CH, cfg.latent_dim, device=dev) if latent else None

    def step_host():
        st.reset(stream=stream)
        for _, nf, ids, inp_h in tick_inputs:
            if latent:
                # the public call takes device buffers: copy the latents in, decode, copy the audio out
                d = lat_d[: inp_h.shape[0]]
                d.copy_(inp_h, non_blocking=True)
                decode(d, nf, audio, ids)
                for b, n in enumerate(nf):
                    audio_h[b, : n * spf].copy_(audio[b, : n * spf], non_blocking=True)
                stream.synchronize()
            else:
                st.decode_host(inp_h, nf, audio_h, stream_ids=ids, stream=stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()

    # timed region (device time, CUDA events on the launching stream)
    clocks = ClockSampler(local)
    clocks.start()
    launches[0] = 0
    barrier(world)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        step()
    e1.record(stream)
    torch.cuda.synchronize()
    ms = max_over_ranks(e0.elapsed_time(e1), world)
    barrier(world)
    clk = clocks.stop()
    gpu_launches = launches[0]
    value = job_throughput(args.steps * audio_s_per_step, ms, world)

    # the same steps again with a CUDA event pair around every launch (the
    # per-kernel times of the roofline; the library runs the resblock chains
    # one after the other while recording, so no two recorded launches overlap)
    st.profile_begin(max_records=200000)
    torch.cuda.synchronize()
    p0, p1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    p0.record(stream)
    for _ in range(args.steps):
        step()
    p1.record(stream)
    torch.cuda.synchronize()
    ms_profiled = p0.elapsed_time(p1)
    kstats = st.profile_end(stream=stream)

    # end to end through the host-buffer entry point
    e2e = None
    if not args.no_e2e:
        step_host()
        torch.cuda.synchronize()
        barrier(world)
        t0 = time.perf_counter()
        for _ in range(args.steps):
            step_host()
        torch.cuda.synchronize()
        wall = max_over_ranks(time.perf_counter() - t0, world)
        e2e = {"value": job_throughput(args.steps * audio_s_per_step, 1e3 * wall, world), "unit": UNIT,
               "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h)}

    # first-audio latency: 1 frame from an empty state
    fa = None
    if args.first_audio_runs > 0:
        if latent:
            one = torch.from_numpy(np.ascontiguousarray(codes[0][:1])).reshape(1, 1, cfg.latent_dim).to(dev)
        else:
            one = torch.from_numpy(np.ascontiguousarray(codes[0][:, :1])).reshape(1, cfg.Q, 1).to(dev)
        a1 = torch.empty(1, spf, device=dev)
        dev_us, wall_us = [], []
        for i in range(args.first_audio_runs + 5):
            st.reset([0], stream=stream)
            torch.cuda.synchronize()
            s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            t0 = time.perf_counter()
            s0.record(stream)
            decode(one, [1], a1, [0])
            s1.record(stream)
            s1.synchronize()
            t1 = time.perf_counter()
            if i >= 5:
                dev_us.append(1e3 * s0.elapsed_time(s1))
                wall_us.append(1e6 * (t1 - t0))
        fa = {"device_us_median": statistics.median(dev_us), "wall_us_median": statistics.median(wall_us),
              "runs": len(dev_us), "launches": st.last_launches}
        # a one-frame call must read every weight once: its roof is the weight bytes at the copy bandwidth
        # (4 bytes per weight in every mode: fp32, or the fp16 hi + lo planes; 2 in single-pass fp16)
        pk_fa, pk_fa_src = peaks()
        wbytes = weight_bytes(cfg, args.precision)
        fa_gbs = wbytes / (fa["device_us_median"] * 1e-6) / 1e9
        fa["roofline"] = {"bound": "hbm", "achieved": fa_gbs, "peak": pk_fa["hbm_gbs"], "unit": "GB/s",
                          "frac": fa_gbs / pk_fa["hbm_gbs"], "traffic": None,
                          "algorithmic_bytes": wbytes,
                          "note": f"every non-codebook weight read once ({pk_fa_src} copy bandwidth)",
                          "floor_us": wbytes / (pk_fa["hbm_gbs"] * 1e9) * 1e6}

    streaming = None
    if rank == 0 and not args.no_streaming and not latent:
        streaming = streaming_schedules(cfg, blob, prec, stream)

    # roofline of the dominant kernel
    pk, pk_src = peaks()
    dom = max(kstats.items(), key=lambda kv: kv[1]["ms"])
    name, ks = dom
    roof = None
    if ks["launches"]:
        per_launch_s = ks["ms"] / 1e3 / ks["launches"]
        if name == "gemm_tc":
            achieved = ks["flops"] / ks["launches"] / per_launch_s / 1e12
            peak = pk.get("bf16_tflops_sustained", pk["bf16_tflops"])
            roof = {"bound": "tensor", "unit": "TFLOP/s", "peak_note": f"{pk_src} sustained bf16 (fp16 same rate)"}
            src = ["tc_gemm.cu", "common.cuh"]
        elif name == "gemm_simt":
            achieved = ks["flops"] / ks["launches"] / per_launch_s / 1e12
            peak = SMS * FP32_LANES_PER_SM * 2 * pk.get("sm_max_mhz", 2070.0) * 1e6 / 1e12
            roof = {"bound": "alu", "unit": "TFLOP/s",
                    "peak_note": "fp32 FMA: 152 SMs x 128 lanes x 2 flop x max SM clock"}
            src = ["kernels_simt.cu", "common.cuh"]
        else:
            achieved = ks["bytes"] / ks["launches"] / per_launch_s / 1e9
            peak = pk["hbm_gbs"]
            roof = {"bound": "hbm", "unit": "GB/s", "peak_note": f"{pk_src} copy bandwidth"}
            src = ["kernels_simt.cu", "common.cuh"]
        roof.update({"kernel": name, "achieved": achieved, "peak": peak, "frac": achieved / peak,
                     "launches": ks["launches"], "traffic": traffic_for(name, kernel_source_digest(src))})
        if name == "gemm_tc":
            # the fp16x3 split issues three MMAs per useful one: the tensor pipe's share of its peak
            roof["issued_frac"] = (3.0 if args.precision == "fp16x3" else 1.0) * achieved / peak
    # per kernel kind: share of device time, and the algorithmic bytes (flops)
    # over its summed event time against the measured copy bandwidth (tensor peak)
    kernels = {}
    tot_ms = max(1e-9, sum(x["ms"] for x in kstats.values()))
    for k, v in kstats.items():
        if not v["launches"]:
            continue
        e = {"launches": v["launches"], "ms": round(v["ms"], 3), "share": round(v["ms"] / tot_ms, 4)}
        if v["ms"] > 0:
            gbs = v["bytes"] / (v["ms"] / 1e3) / 1e9
            e["gbs"] = round(gbs, 1)
            e["hbm_frac"] = round(gbs / pk["hbm_gbs"], 4)
            if k in ("gemm_tc", "gemm_simt"):
                e["tflops"] = round(v["flops"] / (v["ms"] / 1e3) / 1e12, 2)
        kernels[k] = e

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu:
        frames = {"qwen3": 40, "mimi": 100}.get(args.decoder, 400)
        v, dt, cores = oracle_sample(cfg, blob, frames)
        cpu = {"value": v, "unit": UNIT, "cores": cores, "kind": "oracle",
               "sample": f"one stream x {frames} frames of the workload's decoder from an empty state ({dt:.1f} s)"}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms / args.steps, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": {"fp32": "f32", "fp16x3": "fp16x3 (hi/lo split, f32 accumulate)",
                      "fp16": "fp16 (single pass, f32 accumulate; approximate)"}[args.precision],
            "data": "synthetic (uniform codes, random N(0,1/fan_in) weights)",
            "config": config_dict(args, args.precision),
            "roofline": roof, "kernels": kernels, "gpu_launches": gpu_launches,
            "profiled_pass": {"ms_per_step": ms_profiled / args.steps,
                              "note": "roofline and kernels come from a second timed pass of the same steps with an "
                                      "event pair around every launch and the resblock chains serialized"},
            "e2e": e2e, "first_audio": fa, "streaming": streaming, "clocks": clk, "cpu_baseline": cpu,
            "frames_per_s": world * args.steps * S * F / (ms / 1e3),
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def run_profile_call(args):
    """A fixed launch sequence for ncu: REPS identical calls of S streams x CH
    frames each, CUDA graphs off, so that launch i of a kernel is the same
    layer in every call."""
    S, CH, REPS = (int(v) for v in args.profile_call.split(","))
    import torch
    from streaming_tts_vocoder_gb300 import codec as C
    cfg = CONFIGS[args.decoder]()
    latent = bool(cfg.latent_dim)
    blob = pack_blob(cfg, make_weights(cfg, 0))
    prec = {"fp16x3": C.PRECISION_FP16X3, "fp16": C.PRECISION_FP16, "fp32": C.PRECISION_FP32}[args.precision]
    cod = C.Codec(cfg, blob, max_streams=S, max_chunk_frames=CH, max_batch_frames=S * CH, precision=prec)
    st = cod.state()
    st.set_graphs(False)
    dev = torch.device("cuda")
    mk = make_latents if latent else make_codes
    inp = torch.from_numpy(np.stack([mk(cfg, CH, 1000 + s) for s in range(S)])).to(dev)
    audio = torch.empty(S, CH * cod.samples_per_frame, device=dev)
    for _ in range(REPS):
        if latent:
            st.decode_latents(inp, [CH] * S, audio)
        else:
            st.decode(inp, [CH] * S, audio)
    torch.cuda.synchronize()
    print(json.dumps({"profile_call": [S, CH, REPS], "mean_abs": float(audio.abs().mean())}))
    return 0


def layer_labels(cfg):
    """Names of the decoder's launches in call order (an operand prep carries
    the name of the GEMM it feeds)."""
    names = ["history fill"] + (["latent fill", "latent front"] if cfg.latent_dim else ["codebook gather", "pre-conv"])
    for l in range(cfg.layers):
        names += [f"L{l} rmsnorm 1", f"L{l} qkv", f"L{l} attention", f"L{l} out-proj", f"L{l} rmsnorm 2",
                  f"L{l} mlp 1", f"L{l} mlp 2"]
    names += ["final rmsnorm"] + [f"latent up {u}" for u in range(len(cfg.up_channels))]
    for s in range(len(cfg.strides)):
        names.append(f"stage {s} convT")
        # each resblock's convs but the last, resblock by resblock; then the
        # last convs, which add into the MRF sum in resblock order
        for k in cfg.rb_kernels:
            for d in cfg.dilations[:-1]:
                names.append(f"stage {s} rb k{k} d{d}")
        for k in cfg.rb_kernels:
            names.append(f"stage {s} rb k{k} d{cfg.dilations[-1]}")
    return names + ["final conv", "history commit"]


def run_layer_times(args):
    """Per-launch CUDA-event times of one decode call (the third of three
    identical calls from an empty state, graphs off), labelled by layer."""
    S, CH = (int(v) for v in args.layer_times.split(","))
    import torch
    from streaming_tts_vocoder_gb300 import codec as C
    cfg = CONFIGS[args.decoder]()
    latent = bool(cfg.latent_dim)
    blob = pack_blob(cfg, make_weights(cfg, 0))
    prec = {"fp16x3": C.PRECISION_FP16X3, "fp16": C.PRECISION_FP16, "fp32": C.PRECISION_FP32}[args.precision]
    cod = C.Codec(cfg, blob, max_streams=S, max_chunk_frames=CH, max_batch_frames=S * CH, precision=prec)
    st = cod.state()
    st.set_graphs(False)
    dev = torch.device("cuda")
    mk = make_latents if latent else make_codes
    inp = torch.from_numpy(np.stack([mk(cfg, CH, 1000 + s) for s in range(S)])).to(dev)
    audio = torch.empty(S, CH * cod.samples_per_frame, device=dev)
    for _ in range(3):
        st.reset()
        torch.cuda.synchronize()
        st.profile_begin()
        if latent:
            st.decode_latents(inp, [CH] * S, audio)
        else:
            st.decode(inp, [CH] * S, audio)
        st.profile_end()
    names = iter(layer_labels(cfg))
    rows, cur = [], None
    for kind, ms, flops, nbytes in st.profile_launches():
        if kind == "operand_prep":
            cur = cur or next(names)
            name = cur
        else:
            name = cur or next(names)
            cur = None
        rows.append({"layer": name, "kernel": kind, "us": round(ms * 1e3, 2),
                     "tflops": round(flops / ms / 1e9, 1) if ms and flops else None,
                     "gbs": round(nbytes / ms / 1e6, 1) if ms and nbytes else None})
    print(json.dumps({"layer_times": [S, CH], "decoder": args.decoder, "precision": args.precision,
                      "total_us": round(sum(r["us"] for r in rows), 1), "launches": rows}))
    return 0


def run_istft(args):
    """Throughput of the streaming iSTFT head on one GPU: S streams, each 10
    chunks of 94 frames (about 1 s of audio per chunk at hop 256, 24 kHz),
    spectra resident in HBM; the roofline is the call's algorithmic bytes
    (spectra in, audio out, carried frames read and written) over its
    CUDA-event time against the measured copy bandwidth."""
    import torch
    from streaming_tts_vocoder_gb300 import codec as C
    from streaming_tts_vocoder_gb300.synthetic import make_istft_spec
    n_fft, hop, sr, CH, NCH = 1024, 256, 24000, 94, 10
    S = args.streams
    nb = n_fft // 2 + 1
    ist = C.Istft(n_fft, hop, mag_clip=100.0, max_streams=S, max_chunk_frames=CH)
    dev = torch.device("cuda")
    stream = torch.cuda.current_stream()
    spec = torch.from_numpy(np.stack([make_istft_spec(n_fft, CH * NCH, 2000 + s) for s in range(S)])).to(dev)
    chunks = [spec[:, c * CH:(c + 1) * CH].contiguous() for c in range(NCH)]
    audio = torch.empty(S, CH * hop, device=dev)
    flush = torch.empty(64 << 20, dtype=torch.float32, device=dev)     # 256 MB > L2, written between steps

    def step():
        ist.reset(stream=stream)
        for c in range(NCH):
            ist.decode(chunks[c], [CH] * S, audio, stream=stream)

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()
    clk = ClockSampler(torch.cuda.current_device())
    clk.start()
    total = 0.0
    for _ in range(args.steps):
        flush.zero_()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        step()
        e1.record(stream)
        e1.synchronize()
        total += e0.elapsed_time(e1)
    clocks = clk.stop()
    ms = total / args.steps
    audio_s = S * CH * NCH * hop / sr
    frames = S * CH * NCH
    taps = n_fft // hop
    alg = frames * (2 * nb * 4 + hop * 4) + NCH * S * 2 * (taps - 1) * n_fft * 4
    pk, pk_src = peaks()
    achieved = alg / (ms / 1e3) / 1e9
    cpu = None
    if not args.no_cpu:
        from oracle import istft as O
        sample = make_istft_spec(n_fft, CH, 2000).astype(np.float64)
        t0 = time.perf_counter()
        reps = 0
        while time.perf_counter() - t0 < 5.0:
            O.IstftStream(n_fft, hop, 100.0).decode(sample)
            reps += 1
        dt = time.perf_counter() - t0
        cpu = {"value": reps * CH * hop / sr / dt, "unit": "audio-s/s", "cores": 1, "kind": "oracle",
               "sample": f"one stream x {CH} frames, repeated for {dt:.1f} s"}
    print(json.dumps({
        "metric": "iSTFT head audio-sec/sec", "value": audio_s / (ms / 1e3), "unit": "audio-s/s", "n_gpus": 1,
        "steps": args.steps, "warmup": max(3, args.warmup), "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic (seeded log-magnitudes and phases)",
        "config": {"workload": f"{S} streams x {NCH} chunks of {CH} frames, Vocos-shaped iSTFT head",
                   "n_fft": n_fft, "hop": hop, "sample_rate": sr, "l2": "a 256 MB buffer is written before each step"},
        "frames_per_s": frames / (ms / 1e3),
        "roofline": {"bound": "hbm", "kernel": "istft call (frame, overlap-add, commit kernels)",
                     "achieved": achieved, "peak": pk["hbm_gbs"], "unit": "GB/s", "frac": achieved / pk["hbm_gbs"],
                     "traffic": None, "peak_note": f"{pk_src} copy bandwidth",
                     "algorithmic_bytes_per_frame": alg / frames},
        "gpu_launches": args.steps * NCH * 3 + args.steps, "clocks": clocks, "cpu_baseline": cpu}))
    return 0


def run_vocos(args):
    """Throughput of the streaming Vocos-style generator + iSTFT head (24 kHz
    shape: 100 mels, width 512, MLP 1536, 8 blocks, n_fft 1024, hop 256): S
    streams, each 10 chunks of 94 frames (about 1 s of audio), mel frames
    resident in HBM.  The roofline is the pointwise GEMMs' useful flops over
    their share of the call, against the sustained tensor peak; the whole
    call's algorithmic flops per audio second are reported beside it."""
    import torch
    from streaming_tts_vocoder_gb300 import codec as C
    from streaming_tts_vocoder_gb300.synthetic import make_mels, make_vocos_weights, pack_vocos_blob, vocos_config
    cfg = vocos_config()
    S, CH, NCH = args.streams, 94, 10
    prec = {"fp16x3": C.PRECISION_FP16X3, "fp16": C.PRECISION_FP16, "fp32": C.PRECISION_FP32}[args.precision]
    W = make_vocos_weights(cfg, 0)
    voc = C.Vocos(cfg, pack_vocos_blob(cfg, W), max_streams=S, max_chunk_frames=CH, max_batch_frames=S * CH,
                  precision=prec)
    dev = torch.device("cuda")
    stream = torch.cuda.current_stream()
    mel = torch.from_numpy(np.stack([make_mels(cfg, CH * NCH, 3000 + s) for s in range(S)])).to(dev)
    chunks = [mel[:, c * CH:(c + 1) * CH].contiguous() for c in range(NCH)]
    audio = torch.empty(S, CH * cfg.hop, device=dev)

    def step():
        voc.reset(stream=stream)
        for c in range(NCH):
            voc.decode(chunks[c], [CH] * S, audio, stream=stream)

    clk = ClockSampler(torch.cuda.current_device())
    clk.start()
    ms = timed_steps(step, args.steps, max(3, args.warmup), stream)
    clocks = clk.stop()
    sr = 24000
    frames = S * CH * NCH
    audio_s = frames * cfg.hop / sr
    d, F, H = cfg.d, cfg.ffn, cfg.n_fft + 2
    flops_frame = 2.0 * (cfg.k * cfg.n_mels * d + cfg.layers * 2 * d * F + d * H)
    cpu = None
    if not args.no_cpu:
        from oracle import vocos as OV
        sample = make_mels(cfg, 8, 3000)
        t0 = time.perf_counter()
        OV.decode_full(cfg, W, sample)
        dt = time.perf_counter() - t0
        cpu = {"value": 8 * cfg.hop / sr / dt, "unit": "audio-s/s", "cores": 1, "kind": "oracle",
               "sample": f"one stream x 8 frames from an empty state ({dt:.1f} s)"}
    pk, pk_src = peaks()
    achieved = flops_frame * frames / (ms / 1e3) / 1e12
    print(json.dumps({
        "metric": "Vocos-style generator + iSTFT head audio-sec/sec", "value": audio_s / (ms / 1e3),
        "unit": "audio-s/s", "n_gpus": 1, "steps": args.steps, "warmup": max(3, args.warmup), "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": {"fp32": "f32", "fp16x3": "fp16x3 (pointwise layers), f32 elsewhere", "fp16": "fp16"}[args.precision],
        "data": "synthetic (seeded log-mel frames, random weights)",
        "config": {"workload": f"{S} streams x {NCH} chunks of {CH} frames, 24 kHz Vocos shape (100 mels, "
                               f"d 512, MLP 1536, 8 blocks, n_fft 1024, hop 256)",
                   "l2": "a 256 MB buffer is written before each step"},
        "frames_per_s": frames / (ms / 1e3),
        "roofline": {"bound": "tensor", "kernel": "whole call (algorithmic flops over call time)",
                     "achieved": achieved, "peak": pk.get("bf16_tflops_sustained", pk["bf16_tflops"]),
                     "unit": "TFLOP/s", "frac": achieved / pk.get("bf16_tflops_sustained", pk["bf16_tflops"]),
                     "traffic": None, "peak_note": f"{pk_src} sustained bf16",
                     "algorithmic_flops_per_frame": flops_frame},
        "gpu_launches": None, "clocks": clocks, "cpu_baseline": cpu}))
    return 0


def timed_steps(step, steps, warmup, stream):
    """Mean CUDA-event ms of `step` over `steps` runs after `warmup` runs, with
    a 256 MB buffer written before each timed run (larger than L2)."""
    import torch
    flush = torch.empty(64 << 20, dtype=torch.float32, device="cuda")
    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    total = 0.0
    for _ in range(steps):
        flush.zero_()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        step()
        e1.record(stream)
        e1.synchronize()
        total += e0.elapsed_time(e1)
    return total / steps


def run_source(args):
    """Throughput of the excitation ops on one GPU: S streams x 10 chunks of 94
    F0 frames (upp 256 at 24 kHz: about 1 s of audio per chunk) through the
    8-harmonic sine source, and the same amount of 24 kHz signal through the
    analysis STFT (n_fft 16, hop 4: HiFT-sized).  Rooflines: each op's
    algorithmic bytes (inputs read, outputs written, carried state) over its
    CUDA-event time against the measured copy bandwidth."""
    import torch
    from streaming_tts_vocoder_gb300 import codec as C
    from streaming_tts_vocoder_gb300.synthetic import make_f0
    S, CH, NCH, upp, sr, H, n_fft, hop = args.streams, 94, 10, 256, 24000, 8, 16, 4
    dev = torch.device("cuda")
    stream = torch.cuda.current_stream()
    src = C.SineSource(upp, float(sr), H, amplitude=0.1, max_streams=S, max_chunk_frames=CH)
    f0 = torch.from_numpy(np.stack([make_f0(CH * NCH, 3000 + s) for s in range(S)])).to(dev)
    f0c = [f0[:, c * CH:(c + 1) * CH].contiguous() for c in range(NCH)]
    exc = torch.empty(S, CH * upp, H, device=dev)

    def sine_step():
        src.reset(stream=stream)
        for c in range(NCH):
            src.decode(f0c[c], [CH] * S, exc, stream=stream)

    hops = CH * upp // hop                       # the same audio per chunk through the STFT
    st = C.Stft(n_fft, hop, max_streams=S, max_chunk_frames=hops)
    gen = torch.Generator(device="cpu").manual_seed(5)
    xc = [torch.randn(S, hops, hop, generator=gen).to(dev) for _ in range(NCH)]
    nb = n_fft // 2 + 1
    spec = torch.empty(S, hops, 2 * nb, device=dev)

    def stft_step():
        st.reset(stream=stream)
        for c in range(NCH):
            st.decode(xc[c], [hops] * S, spec, stream=stream)

    warm = max(3, args.warmup)
    clk = ClockSampler(torch.cuda.current_device())
    clk.start()
    ms_sine = timed_steps(sine_step, args.steps, warm, stream)
    ms_stft = timed_steps(stft_step, args.steps, warm, stream)
    clocks = clk.stop()
    audio_s = S * CH * NCH * upp / sr
    pk, pk_src = peaks()
    b_sine = S * NCH * (CH * 4 + CH * upp * H * 4)
    b_stft = S * NCH * (hops * hop * 4 + hops * 2 * nb * 4 + 2 * (n_fft - hop) * 4)
    roof = lambda b, ms, name: {"bound": "hbm", "kernel": name, "achieved": b / (ms / 1e3) / 1e9,
                                "peak": pk["hbm_gbs"], "unit": "GB/s", "frac": b / (ms / 1e3) / 1e9 / pk["hbm_gbs"],
                                "traffic": None, "peak_note": f"{pk_src} copy bandwidth"}
    print(json.dumps({
        "metric": "harmonic sine source audio-sec/sec", "value": audio_s / (ms_sine / 1e3), "unit": "audio-s/s",
        "n_gpus": 1, "steps": args.steps, "warmup": warm, "ms_per_step": ms_sine, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32 (u32 phase)", "data": "synthetic (seeded F0 contours)",
        "config": {"workload": f"{S} streams x {NCH} chunks of {CH} F0 frames, {H} harmonics, {upp} samples per "
                               f"frame, {sr} Hz", "l2": "a 256 MB buffer is written before each step"},
        "roofline": roof(b_sine, ms_sine, "sine source call (scan, output kernels)"),
        "stft": {"value": audio_s / (ms_stft / 1e3), "unit": "audio-s/s", "ms_per_step": ms_stft,
                 "config": {"n_fft": n_fft, "hop": hop, "frames_per_chunk": hops},
                 "roofline": roof(b_stft, ms_stft, "stft call (frame, history kernels)")},
        "gpu_launches": args.steps * (1 + 2 * NCH) * 2, "clocks": clocks, "cpu_baseline": None}))
    return 0


def playback_gaps(lats_ms, frames, frame_ms):
    """Chunks decoded back to back (chunk i ready after the sum of the first
    i + 1 latencies) and played as soon as ready: the silence before each
    chunk after the first, in ms."""
    ready, queued_until, gaps = 0.0, None, []
    for lat, n in zip(lats_ms, frames):
        ready += lat
        if queued_until is None:
            queued_until = ready + n * frame_ms
        else:
            gaps.append(max(0.0, ready - queued_until))
            queued_until = max(queued_until, ready) + n * frame_ms
    return gaps


def streaming_schedules(cfg, blob, prec, stream, frames=250, ctx=72, producer_ms=8.0, reps=3):
    """Streaming latency of one stream under the orchestrator's chunk
    schedules (the library's codec_chunk_frames: 1 then 25, the ramp 4, 4, 8,
    16, 25, adaptive doubling from 1), in two decode modes: carried (the
    decoder keeps its conv histories and K/V window across calls) and
    recompute (codec_decode_recompute: each call re-decodes up to `ctx` frames
    of left context from an empty slot and keeps only the new audio).

    Each call's device latency is measured with CUDA events; the timeline is
    then laid out on the host for two producers: codes all available up front
    (the decode cost alone), and frames arriving every producer_ms (a talker at
    real-time factor producer_ms / 80 ms; the pages measure the whole server
    pipeline at 0.08-0.10).  A chunk's decode starts when its last frame has
    arrived and the previous decode is done.  Reported per schedule and mode:
    TTFA (first chunk ready), inter-chunk gap (time between consecutive chunks
    becoming ready; p95), playback stall total when playback starts on the
    first chunk, and the uninterrupted-playback latency max_i(ready_i - audio
    before chunk i), the earliest start that never stalls."""
    import torch
    from streaming_tts_vocoder_gb300 import codec as C
    cod = C.Codec(cfg, blob, max_streams=1, max_chunk_frames=ctx + 25, precision=prec)
    st = cod.state()
    dev = torch.device("cuda")
    codes = make_codes(cfg, frames, 1000)
    spf = cod.samples_per_frame
    frame_ms = 1e3 / FRAME_RATE_HZ
    scheds = {
        "1_then_25": C.chunk_schedule(C.SCHEDULE_FIXED, first=1, steady=25),
        "ramp_4_4_8_16_25": C.chunk_schedule(C.SCHEDULE_RAMP, steady=25, ramp=(4, 4, 8, 16)),
        "adaptive_from_1": C.chunk_schedule(C.SCHEDULE_ADAPTIVE, first=1, steady=25),
    }
    T_max = ctx + 25
    codes_d = torch.zeros(1, cfg.Q, T_max, dtype=torch.int32, device=dev)
    audio = torch.empty(1, T_max * spf, device=dev)
    out = {}
    for name, sch in scheds.items():
        sizes = C.schedule_chunks(sch, frames)
        for mode in ("carried", "recompute"):
            for _ in range(reps):                # earlier passes warm the graph cache; keep the last
                st.reset([0], stream=stream)
                torch.cuda.synchronize()
                t, lats = 0, []
                for n in sizes:
                    lo = max(0, t - ctx) if mode == "recompute" else t
                    seg = np.zeros((cfg.Q, T_max), np.int32)
                    seg[:, : t + n - lo] = codes[:, lo:t + n]
                    codes_d.copy_(torch.from_numpy(seg).reshape(1, cfg.Q, T_max))
                    torch.cuda.synchronize()
                    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                    e0.record(stream)
                    if mode == "recompute":
                        st.decode_recompute(codes_d, [t - lo], [n], audio, stream_ids=[0], stream=stream)
                    else:
                        st.decode(codes_d, [n], audio, stream_ids=[0], stream=stream)
                    e1.record(stream)
                    e1.synchronize()
                    lats.append(e0.elapsed_time(e1))
                    t += n
            entry = {"chunks": len(sizes), "decode_ms_total": float(sum(lats)),
                     "chunk_latency_ms_p50": float(np.percentile(lats, 50)),
                     "chunk_latency_ms_p95": float(np.percentile(lats, 95))}
            for prod, pms in (("up_front", 0.0), (f"producer_{pms_label(producer_ms)}", producer_ms)):
                entry[prod] = stream_timeline(lats, sizes, frame_ms, pms)
            out[f"{name}/{mode}"] = entry
    st.close()
    cod.close()
    return {"decoder": cfg.name, "frames": frames, "frame_ms": frame_ms, "recompute_context_frames": ctx,
            "producer_ms_per_frame": producer_ms, "schedules": out}


def pms_label(ms):
    return f"{ms:g}ms_per_frame"


def stream_timeline(lats_ms, frames, frame_ms, producer_ms):
    """Ready times of chunks decoded in order (decode i starts when its last
    frame has arrived and decode i - 1 is done) and the playback metrics."""
    ready, t_free, arrived = [], 0.0, 0
    for lat, n in zip(lats_ms, frames):
        arrived += n
        start = max(arrived * producer_ms, t_free)
        t_free = start + lat
        ready.append(t_free)
    before = np.concatenate([[0.0], np.cumsum(np.asarray(frames, float) * frame_ms)[:-1]])
    gaps = np.diff(ready) if len(ready) > 1 else np.zeros(0)
    stalls = playback_gaps(list(np.diff(np.concatenate([[0.0], ready]))), frames, frame_ms)
    return {"ttfa_ms": float(ready[0]),
            "inter_chunk_gap_ms_p95": float(np.percentile(gaps, 95)) if gaps.size else 0.0,
            "playback_stall_ms_total": float(sum(stalls)),
            "uninterrupted_playback_ms": float(np.max(np.asarray(ready) - before))}


def run_schedule(args):
    import torch
    from streaming_tts_vocoder_gb300 import codec as C
    cfg = qwen3_config() if args.decoder == "qwen3" else tiny_config()
    blob = pack_blob(cfg, make_weights(cfg, 0))
    prec = {"fp16x3": C.PRECISION_FP16X3, "fp16": C.PRECISION_FP16, "fp32": C.PRECISION_FP32}[args.precision]
    out = {"metric": "streaming chunk latency, one stream", "precision": args.precision}
    out.update(streaming_schedules(cfg, blob, prec, torch.cuda.current_stream()))
    print(json.dumps(out))
    return 0


def main():
    args = parse()
    if args.impl == "reference":
        return run_reference(args)
    if args.profile_call:
        return run_profile_call(args)
    if args.layer_times:
        return run_layer_times(args)
    if args.workload == "istft":
        return run_istft(args)
    if args.workload == "source":
        return run_source(args)
    if args.workload == "vocos":
        return run_vocos(args)
    if args.schedule:
        return run_schedule(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
