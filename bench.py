#!/usr/bin/env python3
"""Packed GDN prefill throughput on the 32 x 1,024 chat wave (tokens/s, % of roofline).

One step = one gdn_prefill_packed call over the whole wave: 32 prompts of 1,024 tokens
packed into one pass (32,768 tokens), H_k = 16, H_v = 32, d_k = d_v = 128, bf16 q/k/v/o,
fp32 gates and states, one prefix-cache checkpoint per prompt (position 768: the last
multiple of 256 moved back out of the last 16 tokens) plus the final states. Inputs are
synthetic and seeded (packed_linear_attention_gb300.inputs), resident in HBM before the
timed region; they are larger than L2 and L2 is also flushed between timed steps.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

Under torchrun (N > 1) every rank runs its own wave (independent prompts: weak scaling,
no collective on the data path); rank 0 prints one JSON line with the max-over-ranks time.
`--impl reference` times the CPU oracle (the only other implementation) on a bounded
sample of the same workload on this machine's host cores.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "GDN packed-prefill tokens/s at 32x1024 (1 GB300) + % of roofline"
UNIT = "tokens/s"
WORKLOAD = dict(workload="chat_wave_32x1024", prompts=32, prompt_len=1024, tokens=32768,
                num_k_heads=16, num_v_heads=32, head_dim=128, chunk=64,
                checkpoints="768 per prompt + final", io="bf16 qkv/o, fp32 gates+states",
                l2="inputs > L2 and L2 flushed between timed steps")


def algorithmic_bytes(T, Hk, Hv, d, n_seqs, n_ckpt, s_in=2, s_out=2, init=False):
    """Bytes the method must move: read q, k, v, a, beta (and initial states if given),
    write o, checkpoints and final states. Intermediates are not counted."""
    b = 2 * T * Hk * d * s_in + T * Hv * d * s_in + 2 * T * Hv * 4 + T * Hv * d * s_out
    if init:
        b += n_seqs * Hv * d * d * 4
    b += (n_ckpt + n_seqs) * Hv * d * d * 4
    return b


def algorithmic_flops(T, Hk, Hv, d, C=64):
    """Dense tensor-core flops of the chunked method per pass: per token and value head
    6 d^2 (three state products) + 6 C d (W, U and the intra-chunk output), plus
    K K^T and Q K^T (2 C d each) once per token and key head."""
    return T * Hv * (6 * d * d + 6 * C * d) + T * Hk * (4 * C * d)


# DRAM traffic of the prefill kernel per full-wave launch (the median of three launches),
# from an ncu capture of this workload (dram__bytes_read.sum + dram__bytes_write.sum; one
# pass on the 8-prompt case, so captured at full size: `ncu --metrics
# gpu__time_duration.sum,dram__bytes_read.sum,dram__bytes_write.sum --clock-control none
# -k regex:chunked_prefill -s 3 -c 3 python bench.py --steps 3 --warmup 3
# --no-cpu-baseline --no-e2e --no-secondary`). It is reported only while the kernel
# sources hash to the values it was measured on; any change to them reports null until
# re-measured.
MEASURED_TRAFFIC = {
    "sources": {
        "packed_linear_attention_gb300/csrc/gdn_chunked.cu":
            "05dc96bf04958dee87460f0491551d5acece8a6a2563109877897692fb3072a8",
        "packed_linear_attention_gb300/csrc/gdn_chunk_util.cuh":
            "79a2646b770efccd02ab41cc732b8ffe6c5c890479fc9c579353bcf415d15a2f",
        "packed_linear_attention_gb300/csrc/ptx_sm103.cuh":
            "762c9e7ef68fa3e883aaeb592d47ce09eed2b387cc7b6e46fa74fa53d9b1da60",
        "packed_linear_attention_gb300/csrc/gdn_tma.cu":
            "b97a465a15c3850359ec63c6925ea5d4f1962a058db1f247ccd5c0a9055e72f2",
    },
    "read_bytes": 545.9e6,
    "write_bytes": 356.8e6,
}


def measured_traffic():
    import hashlib
    for rel, digest in MEASURED_TRAFFIC["sources"].items():
        try:
            with open(os.path.join(ROOT, rel), "rb") as f:
                if hashlib.sha256(f.read()).hexdigest() != digest:
                    return None
        except OSError:
            return None
    return MEASURED_TRAFFIC["read_bytes"] + MEASURED_TRAFFIC["write_bytes"]


def load_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            pk = json.load(f)
        return float(pk["hbm_gbs"]), float(pk["bf16_tflops"]), "measured"
    except Exception:
        return 6800.0, 1900.0, "fallback"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every `period_ms` while running; each
    sample keeps the host time at which it arrived, so that a summary can be restricted to
    a window (the loaded part of the run)."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, period_ms: int = 20):
        self.gpu = gpu_index
        self.period_ms = period_ms
        self.proc = None
        self.lines: list[tuple[float, str]] = []
        self._t = None
        self.window = None  # (t0, t1) host monotonic times, set by the caller

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", str(self.period_ms)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self._t = threading.Thread(target=self._read, daemon=True)
            self._t.start()
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.monotonic(), line.strip()))

    def live(self) -> bool:
        """True once a sample has arrived (or when nvidia-smi could not be started)."""
        return self.proc is None or bool(self.lines)

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            if self._t:
                self._t.join(timeout=2)

    def summary(self):
        if not self.lines:
            return None
        lines = [ln for t, ln in self.lines
                 if self.window is None or self.window[0] <= t <= self.window[1]]
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for nm, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(nm)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm),
                "window": "the timed steps and an untimed tail of the same steps (>= 0.25 s), "
                          f"sampled every {self.period_ms} ms"}


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def reduce_max(x: float, world: int, device=None) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate(tokens_per_rank: int, ms_local: float, world: int, device=None):
    """Whole-job throughput under weak scaling: every rank prefills its own pack of
    `tokens_per_rank` tokens; the job takes as long as the slowest rank. Returns
    (max milliseconds over ranks, total tokens per second)."""
    ms = reduce_max(ms_local, world, device)
    return ms, tokens_per_rank * world / (ms / 1e3)


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ---- CPU oracle (baseline / reference arm) -------------------------------------------------

def oracle_rate(pack, n_prompts: int, n_heads: int, threads: int):
    """Time the fp64 oracle on `n_prompts` prompts x `n_heads` value heads of the wave;
    returns (full-layer tokens/s, seconds, sample description)."""
    from oracle import ref
    from packed_linear_attention_gb300 import inputs as I
    heads = list(range(n_heads))
    sub = I.sub_pack(pack, list(range(n_prompts)), heads)
    args = (sub.cu_seqlens, sub.as_f32("q"), sub.as_f32("k"), sub.as_f32("v"), sub.a, sub.beta,
            sub.init, sub.ckpt_cu, sub.ckpt_pos)
    t0 = time.perf_counter()
    ref.prefill_arrays(*args, scale=sub.scale, threads=threads)
    dt = time.perf_counter() - t0
    layer_tokens = sub.total_tokens * n_heads / pack.num_v_heads
    desc = (f"{n_prompts} prompt(s) x 1024 tokens x {n_heads}/{pack.num_v_heads} value heads "
            f"of the wave, fp64 token-by-token oracle, {threads} threads; tokens/s scaled to "
            f"all {pack.num_v_heads} heads")
    return layer_tokens / dt, dt, desc


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    from packed_linear_attention_gb300 import inputs as I
    pack = I.chat_wave()
    threads = os.cpu_count() or 1
    # each step: the oracle over the whole wave (every prompt and value head), spread over
    # all host cores, as the GPU arm's cpu_baseline leg runs it
    n_prompts, n_heads = pack.num_seqs, pack.num_v_heads
    for _ in range(args.warmup):
        oracle_rate(pack, n_prompts, n_heads, threads)
    times, desc = [], ""
    for _ in range(args.steps):
        _, dt, desc = oracle_rate(pack, n_prompts, n_heads, threads)
        times.append(dt)
    ms = 1e3 * sum(times) / len(times)
    value = pack.total_tokens / (ms / 1e3)
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64", "data": "synthetic", "config": WORKLOAD,
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle",
                         "sample": desc},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)
    return 0


# ---- GPU arm --------------------------------------------------------------------------------

def run_gpu(args):
    import torch

    from packed_linear_attention_gb300 import build, gdn
    from packed_linear_attention_gb300 import inputs as I

    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    else:
        torch.cuda.set_device(0)
    dev = torch.device("cuda", torch.cuda.current_device())
    build.build()
    # each rank: its own independent wave (a smaller wave only for profiling captures)
    pack = I.chat_wave(num_prompts=args.prompts, seed=rank)
    T, Hk, Hv, d, N = pack.total_tokens, 16, 32, 128, pack.num_seqs
    h = gdn.gdn_handle_create(dev.index, 256 << 20)
    buf = gdn.to_device(pack, device=dev)
    stream = torch.cuda.current_stream(dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)  # 256 MiB > 129 MB L2

    def step():
        gdn.prefill(h, buf, stream)

    for _ in range(max(args.warmup, 3)):
        step()
    torch.cuda.synchronize()
    assert gdn.gdn_read_device_status(buf.workspace) == 0

    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    with ClockSampler(dev.index) as clocks:
        # the same steps, untimed, until nvidia-smi delivers samples (at most 5 s)
        t_wait = time.monotonic()
        while not clocks.live() and time.monotonic() - t_wait < 5.0:
            for _ in range(16):
                flush.zero_()
                step()
            torch.cuda.synchronize()
        barrier(world)
        torch.cuda.synchronize()
        t_on = time.monotonic()
        for i in range(args.steps):
            flush.zero_()
            starts[i].record(stream)
            step()
            ends[i].record(stream)
        torch.cuda.synchronize()
        # an untimed tail of the same steps, so that a timed region shorter than the sampling
        # period still has samples taken under its load
        t_off = time.monotonic()
        while time.monotonic() - t_off < 0.25:
            for _ in range(16):
                flush.zero_()
                step()
            torch.cuda.synchronize()
        clocks.window = (t_on, time.monotonic())
    assert gdn.gdn_read_device_status(buf.workspace) == 0
    barrier(world)
    per = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    ms_local = sum(per) / len(per)
    ms, value = aggregate(T, ms_local, world, dev)

    # the chunked kernel's automatic schedule choice (asked of the library)
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    choice = gdn.gdn_chunked_schedule(pack.cu_seqlens, Hv, sms)
    schedule = ("chunked, throughput schedule" if choice == gdn.KERNEL_CHUNKED_THROUGHPUT
                else "chunked, pipelined schedule") + f" ({N * Hv} units on {sms} SMs)"

    # roofline of the step's prefill launches (the only kernels of the step)
    hbm_gbs, tflops, peak_src = load_peaks()
    B = algorithmic_bytes(T, Hk, Hv, d, N, pack.num_ckpts)
    F = algorithmic_flops(T, Hk, Hv, d)
    achieved = B / (ms_local / 1e3) / 1e9
    t_hbm = B / (hbm_gbs * 1e9)
    t_tc = F / (tflops * 1e12)
    traffic = measured_traffic() if args.prompts == 32 else None
    roof = {"bound": "hbm", "achieved": achieved, "peak": hbm_gbs, "unit": "GB/s",
            "frac": achieved / hbm_gbs, "traffic": traffic,
            "peak_source": f"{peak_src} (MEASURED_PEAKS.json hbm_gbs, burst copy)",
            "algorithmic_bytes": B, "algorithmic_flops": F,
            "t_roof_us": max(t_hbm, t_tc) * 1e6, "t_hbm_us": t_hbm * 1e6,
            "t_tensor_us": t_tc * 1e6, "kernel_us": ms_local * 1e3,
            "frac_of_roofline": max(t_hbm, t_tc) / (ms_local / 1e3)}

    # end to end through the public API with host buffers
    e2e = None if args.no_e2e else run_e2e(args, torch, gdn, h, buf, pack, stream, world, dev)
    secondary = None
    if not args.no_secondary and world == 1:
        until_d2h = run_until_ckpt_d2h(torch, gdn, h, buf, stream, flush)
        del buf
        secondary = run_secondary(torch, gdn, I, h, stream, flush, hbm_gbs)
        secondary["wave_until_ckpt_d2h"] = until_d2h

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        threads = os.cpu_count() or 1
        rate, dt, desc = oracle_rate(pack, args.cpu_prompts, 32, threads)
        cpu = {"value": rate, "unit": UNIT, "cores": threads, "kind": "oracle",
               "sample": desc + f" ({dt:.1f} s)"}

    gdn.gdn_handle_destroy(h)
    if rank == 0:
        print(json.dumps({
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16", "data": "synthetic",
            "config": dict(WORKLOAD, parallelism=f"replicas x{world}" if world > 1 else "1 GPU",
                           prompts=pack.num_seqs, tokens=T, schedule=schedule),
            "roofline": roof, "cpu_baseline": cpu, "e2e": e2e, "secondary": secondary,
            "gpu_launches": args.steps, "clocks": clocks.summary(),
        }), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def _time_events(torch, fn, stream, flush, steps=10, warmup=3):
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    tot = 0.0
    for _ in range(steps):
        flush.zero_()
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record(stream)
        fn()
        e.record(stream)
        e.synchronize()
        tot += s.elapsed_time(e)
    return tot / steps


def run_until_ckpt_d2h(torch, gdn, h, buf, stream, flush, steps=10):
    """The wave's prefill followed by the copy of its checkpoints into the handle's pinned
    pool (side stream), timed on the host from the launch until the copy has completed
    (inputs resident, L2 flushed first)."""
    nbytes = buf.ckpt.numel() * 4
    for _ in range(3):
        gdn.prefill(h, buf, stream)
        gdn.gdn_checkpoint_copy(h, buf.ckpt, nbytes, 0, stream)
        gdn.gdn_checkpoint_copy_wait(h)
    tot = 0.0
    for _ in range(steps):
        flush.zero_()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        gdn.prefill(h, buf, stream)
        gdn.gdn_checkpoint_copy(h, buf.ckpt, nbytes, 0, stream)
        gdn.gdn_checkpoint_copy_wait(h)
        tot += time.perf_counter() - t0
    us = tot / steps * 1e6
    # the same with the copies started per group of prompts as their checkpoints are stored
    for _ in range(3):
        gdn.prefill_snapshot(h, buf, 0, stream)
        gdn.gdn_checkpoint_copy_wait(h)
    tot = 0.0
    for _ in range(steps):
        flush.zero_()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        gdn.prefill_snapshot(h, buf, 0, stream)
        gdn.gdn_checkpoint_copy_wait(h)
        tot += time.perf_counter() - t0
    torch.cuda.synchronize()
    return {"us": us, "ckpt_bytes": nbytes, "timing": "host clock, launch to copy completion",
            "copy_after_pass_api": "gdn_prefill_packed + gdn_checkpoint_copy",
            "overlapped_us": tot / steps * 1e6,
            "overlapped_api": "gdn_prefill_packed_snapshot (copies start per group of prompts "
                              "once their checkpoints are stored)"}


def run_secondary(torch, gdn, I, h, stream, flush, hbm_gbs):
    """Other workloads of the same path, timed the same way (not the headline metric):
    the ragged prefix-cache pack, 4 x 8K prompts, and the one-token decode step of 32
    sequences (HBM-bound: every state byte read and written once)."""
    out = {}
    sms = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
    for name, pack in (("ragged_prefix_8", I.ragged_prefix()), ("long_4x8192", I.long_prompts())):
        buf = gdn.to_device(pack)
        ms = _time_events(torch, lambda: gdn.prefill(h, buf, stream), stream, flush)
        B = algorithmic_bytes(pack.total_tokens, 16, 32, 128, pack.num_seqs, pack.num_ckpts,
                              init=pack.init is not None)
        out[name] = {"tokens": pack.total_tokens, "us": ms * 1e3,
                     "schedule": "chunked, " + (
                         "throughput" if gdn.gdn_chunked_schedule(pack.cu_seqlens, 32, sms)
                         == gdn.KERNEL_CHUNKED_THROUGHPUT else "pipelined") +
                     " schedule (automatic choice)",
                     "tokens_per_s": pack.total_tokens / (ms / 1e3),
                     "achieved_gbs": B / (ms / 1e3) / 1e9, "frac_hbm": B / (ms / 1e3) / 1e9 / hbm_gbs}
        del buf
    # one 32K-token prompt: whole (32 units) and split into 3 and 4 parallel segments
    pack = I.single_long_prompt()
    buf = gdn.to_device(pack)
    ms = _time_events(torch, lambda: gdn.prefill(h, buf, stream), stream, flush, steps=5)
    B = algorithmic_bytes(pack.total_tokens, 16, 32, 128, 1, pack.num_ckpts)
    entry = {"tokens": pack.total_tokens, "whole_us": ms * 1e3}
    auto_seg = gdn.gdn_split_segment_auto(pack.cu_seqlens, 32, sms)
    for parts in (3, 4, "auto"):
        if parts == "auto":
            seg = auto_seg
            if seg == 0:
                continue
        else:
            seg = (pack.total_tokens + parts - 1) // parts  # rounded up to the chunk grid
            seg = (seg + 63) // 64 * 64
        nbytes = gdn.gdn_prefill_split_workspace_size(buf.cfg, buf.cu, buf.ckpt_cu,
                                                      buf.ckpt_pos, seg)
        ws = torch.empty(nbytes, dtype=torch.uint8, device=buf.o.device)
        ms_s = _time_events(torch, lambda: gdn.gdn_prefill_packed_split(
            h, buf.cfg, buf.cu, buf.q, buf.k, buf.v, buf.a, buf.beta, buf.init, buf.ckpt_cu,
            buf.ckpt_pos, buf.o, buf.ckpt, buf.final, seg, ws, nbytes, stream),
            stream, flush, steps=5)
        entry[f"split{parts}_us"] = ms_s * 1e3
        entry[f"split{parts}_segment"] = seg
        del ws
    entry["best_frac_hbm"] = B / (min(v for kk, v in entry.items() if kk.endswith("_us"))
                                  / 1e6) / 1e9 / hbm_gbs
    out["single_32k"] = entry
    del buf
    # decode: 32 sequences, states resumed from a pool
    ms_step = I.mixed_step()
    B = ms_step.dec_q.shape[0]
    cfg = gdn.make_config(16, 32, 128)
    up = lambda x: torch.from_numpy(x.view(np.int16)).cuda().view(torch.bfloat16)  # noqa: E731
    q, k, v = up(ms_step.dec_q), up(ms_step.dec_k), up(ms_step.dec_v)
    a = torch.from_numpy(ms_step.dec_a).cuda()
    beta = torch.from_numpy(ms_step.dec_beta).cuda()
    pool = torch.from_numpy(ms_step.dec_states).cuda()
    slots = torch.arange(B, dtype=torch.int32, device="cuda")
    o = torch.empty((B, 32, 128), dtype=torch.bfloat16, device="cuda")
    ms = _time_events(torch, lambda: gdn.gdn_decode_step(h, cfg, B, q, k, v, a, beta, pool, B,
                                                         slots, o, stream), stream, flush)
    dbytes = B * 32 * 128 * 128 * 4 * 2 + B * (2 * 16 * 128 * 2 + 2 * 32 * 128 * 2 + 2 * 32 * 4)
    out["decode_32seq"] = {"sequences": B, "us": ms * 1e3, "achieved_gbs": dbytes / (ms / 1e3) / 1e9,
                           "frac_hbm": dbytes / (ms / 1e3) / 1e9 / hbm_gbs}
    # a mixed step: the prompt slices under the 1,024-token budget and the 32 decode tokens,
    # (a) as a prefill plus a separate decode launch, (b) as one pack in one launch, every
    # state gathered from and written back to a pool slot (gdn_prefill_packed_pool)
    pre = ms_step.prefill
    pbuf = gdn.to_device(pre)
    ms_two = _time_events(torch, lambda: (gdn.prefill(h, pbuf, stream), gdn.gdn_decode_step(
        h, cfg, B, q, k, v, a, beta, pool, B, slots, o, stream)), stream, flush)
    both = I.mixed_one_pack(ms_step)
    obuf = gdn.to_device(both)
    nslots = both.num_seqs
    spool = torch.zeros((nslots, 32, 128, 128), dtype=torch.float32, device="cuda")
    spool[pre.num_seqs:] = torch.from_numpy(ms_step.dec_states).cuda()
    slot_idx = list(range(nslots))
    start_zero = [1] * pre.num_seqs + [0] * B
    ms_one = _time_events(torch, lambda: gdn.gdn_prefill_packed_pool(
        h, obuf.cfg, obuf.cu, obuf.q, obuf.k, obuf.v, obuf.a, obuf.beta, spool, nslots,
        slot_idx, start_zero, obuf.ckpt_cu, None, obuf.o, None, obuf.workspace,
        obuf.workspace_bytes, stream), stream, flush)
    launches = gdn.gdn_prefill_launch_count(h)
    sms = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
    out["mixed_step"] = {
        "prompt_tokens": pre.total_tokens, "decode_tokens": B,
        "prefill_plus_decode_us": ms_two * 1e3, "one_pack_us": ms_one * 1e3,
        "one_pack_api": "gdn_prefill_packed_pool (states gathered from pool slots)",
        "one_pack_launches": launches,
        "one_pack_schedule": "throughput" if gdn.gdn_chunked_schedule(
            both.cu_seqlens, 32, sms) == gdn.KERNEL_CHUNKED_THROUGHPUT else "pipelined"}
    del pbuf, obuf, spool
    return out


def run_e2e(args, torch, gdn, h, buf, pack, stream, world, dev):
    """Host-resident inputs and outputs through gdn_prefill_packed_host: per step, the pinned
    q, k, v, a, beta go in and o, the checkpoints and the final states come back, group by
    group of prompts, the copies of one group overlapping the prefill of its neighbours."""
    host = {}
    for name in ("q", "k", "v", "a", "beta"):
        host[name] = getattr(buf, name).cpu().pin_memory()
    o_host = torch.empty(buf.o.shape, dtype=buf.o.dtype).pin_memory()
    f_host = torch.empty(buf.final.shape, dtype=torch.float32).pin_memory()
    c_host = torch.empty(buf.ckpt.shape, dtype=torch.float32).pin_memory()
    has_ck = buf.ckpt.numel() > 0
    hb = gdn.prefill_buffers(host["q"], host["k"], host["v"], host["a"], host["beta"], None,
                             o_host, c_host if has_ck else None, f_host)
    db = gdn.prefill_buffers(buf.q, buf.k, buf.v, buf.a, buf.beta, None, buf.o,
                             buf.ckpt if has_ck else None, buf.final)
    h2d = sum(x.numel() * x.element_size() for x in host.values())
    d2h = (o_host.numel() * o_host.element_size() + f_host.numel() * 4
           + (c_host.numel() * 4 if has_ck else 0))

    ws_bytes = gdn.gdn_prefill_host_workspace_size(buf.cfg, buf.cu, buf.ckpt_cu, args.e2e_group)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)

    def step():
        gdn.gdn_prefill_packed_host(h, buf.cfg, buf.cu, buf.ckpt_cu,
                                    buf.ckpt_pos if has_ck else None, hb, db,
                                    args.e2e_group, ws, ws_bytes, stream)
        stream.synchronize()

    for _ in range(2):
        step()
    steps = max(3, min(args.steps, 10))
    barrier(world)
    t0 = time.perf_counter()
    for _ in range(steps):
        step()
    dt = (time.perf_counter() - t0) / steps
    dt = reduce_max(dt, world, dev)
    return {"value": pack.total_tokens * world / dt, "unit": UNIT, "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "ms_per_step": dt * 1e3, "steps": steps,
            "api": f"gdn_prefill_packed_host, groups of {args.e2e_group} prompts"}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="gdn", choices=["gdn", "reference"])
    ap.add_argument("--cpu-prompts", type=int, default=32,
                    help="prompts of the wave in the timed CPU-oracle sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--e2e-group", type=int, default=4,
                    help="prompts per copy/compute group of the host-memory e2e leg")
    ap.add_argument("--no-secondary", action="store_true",
                    help="skip the ragged, 8K-prompt and decode timings")
    ap.add_argument("--prompts", type=int, default=32,
                    help="prompts in the wave (32 for the metric; fewer only for profiling)")
    args = ap.parse_args()
    if args.impl == "reference":
        return run_reference(args)
    return run_gpu(args)


if __name__ == "__main__":
    sys.exit(main())
