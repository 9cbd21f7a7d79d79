"""Benchmark of the Inkling attention block on GB300.

One step = the whole hot path over one batch: the sconv of the new K/V rows into the paged
cache, then the attention.  Prefill: inkling_sconv_kv, then inkling_rel_attn_prefill.
Decode over a bf16 cache: one call, inkling_rel_attn_decode_sconv (the conv in the decode
kernel's prologue); the two separate calls are timed too (two_call_step).

Default line (python bench.py): the 64K full-causal prefill, B=1 x 65536 new tokens, 64
query / 8 KV heads, head dim 128, relative-bias table [64 x 8192], exactly --steps timed
steps.  The same JSON line then carries `workloads`: every workload measured in the same
run with its own roofline, end-to-end figure and clock record:
  1 tiny prefill, 2 sliding-window prefill, 3 64K prefill        (TFLOP/s)
  4 MTP decode, window 4096 / full / the two as one layer pair   (KV-read GB/s)
  5 1M-token decode, 1 and 9 tokens                              (KV-read GB/s)
  and the FP8 (E4M3) KV cache forms of 2, 4 and 5.
Prefill metric: attention TFLOP/s counting only allowed (query, key) pairs, 4*D flops per
pair per head (QK^T and PV).  Decode metric: K/V bytes inside the causal/window range
over the step time; with --kv fp8 / the _fp8 entries, the E4M3 bytes (half).
--workload N [--variant V] [--kv fp8] times one workload alone (no sweep unless --sweep).
--workload 6 is the conv on a dense stream (inkling_sconv on the sliding-window prefill's
attention output, 32768 tokens x 4096 channels), in GB/s of algorithmic bytes.

python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--workload 3]
Under torchrun (N > 1) every rank runs an independent replica (the path has no exchange
step); value = work of all ranks / max time over ranks.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

import workloads as W  # noqa: E402

METRIC = "prefill attn TFLOP/s and decode KV-read GB/s on 1 GB300; % of roofline"
L2_FLUSH_BYTES = 512 << 20
REF_TOTAL_S = 120.0  # oracle seconds for a whole --impl reference run
L2_NOTE = ("flushed between timed steps: 512 MB written, then read back (the read retires the "
           "write's dirty lines before the timed region, so the kernel is not charged for their "
           "write-back)")


def flush_l2(buf: torch.Tensor, sink: torch.Tensor) -> None:
    """Evict the previous step's data from L2 (write a buffer 4x the L2), then read the buffer
    so that L2 holds clean lines: a 129 MB dirty L2 costs the next kernel ~20-40 us of
    write-backs that are the flush's, not the kernel's."""
    buf.fill_(1.0)
    torch.sum(buf, dim=0, keepdim=True, out=sink)


def max_over_ranks(values, ws: int, device) -> list:
    """Per-rank timings -> their maximum over all ranks (every rank gets the result)."""
    t = torch.tensor(list(values), dtype=torch.float64, device=device)
    if ws > 1:
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return t.tolist()


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


# --------------------------------------------------------------- algorithmic work ----
def allowed_pairs(n: int, L: int, window: int) -> int:
    """Number of (query, key) pairs with 0 <= p - j (<= window-1) for queries at
    positions L-n .. L-1 (closed form per query, summed)."""
    total = 0
    for p in range(L - n, L):
        keys = p + 1 if window <= 0 else min(p + 1, window)
        total += keys
    return total


def attn_flops(spec: W.Spec) -> float:
    pairs = sum(allowed_pairs(n, L, spec.window) for n, L in zip(spec.q_lens, spec.seq_lens))
    return 4.0 * 128 * spec.hq * pairs


def decode_kv_bytes(spec: W.Spec) -> float:
    """K+V bytes of the keys any query of the step may see (union over the n new tokens),
    per KV head: 2 * 128 * 2 bytes per key."""
    total = 0
    for n, L in zip(spec.q_lens, spec.seq_lens):
        if n == 0:
            continue
        lo = 0 if spec.window <= 0 else max(0, L - n - spec.window + 1)
        total += (L - lo) * spec.hkv * 2 * 128 * 2
    return float(total)


def is_decode(n: int) -> bool:
    return n in (4, 5)


DENSE_Q_LENS = (8192,) * 4   # the sliding-window prefill's sequences
DENSE_C = 32 * 128           # its attention output width (Hq x head dim)


def dense_bytes(q_lens, C: int) -> float:
    """Raw rows read once + conv outputs written once + state rows read and written."""
    T = sum(q_lens)
    return float(2 * T * C * 2 + 2 * len(q_lens) * 3 * C * 2)


def workload_spec(n: int, variant=None) -> W.Spec:
    return W.config(n, variant=variant)


def workload_name(spec: W.Spec) -> str:
    return (f"{spec.name}: B={spec.batch} new={spec.max_q_len} L<={spec.max_seq_len} "
            f"Hq={spec.hq} Hkv={spec.hkv} D=128 window={spec.window} R={spec.r}")


# --------------------------------------------------------------------- clocks -------
class ClockSampler:
    """nvidia-smi clocks/throttle reasons sampled every 50 ms during the timed region."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.gpu = str(device_index)
        try:  # the physical GPU behind this process's device, whatever the visible-set order
            self.gpu = "GPU-" + str(torch.cuda.get_device_properties(device_index).uuid)
        except Exception:
            pass
        self.proc = None
        self.lines = []
        self.skip = 0

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
            # nvidia-smi takes a moment to start: begin timing once it is sampling
            t_end = time.time() + 3.0
            while not self.lines and time.time() < t_end and self.proc.poll() is None:
                time.sleep(0.01)
            self.skip = len(self.lines)
        except (FileNotFoundError, OSError):
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        # the samples taken while the timed region ran (the last one before it included)
        for line in self.lines[max(0, self.skip - 1):]:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax = float(parts[2])
            except ValueError:
                continue
            for nm, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": smax,
                "reasons": sorted(reasons), "samples": len(sm)}


# DRAM bytes (read + write) per launch of the dominant kernel, from one ncu capture of
# `python bench.py [--workload W --variant V] --steps 2 --warmup 3 --no-cpu-baseline` (see
# profiles/), keyed by (workload, variant) and by the SHA-256 of the kernel source it was
# taken on: when that source has changed since, the figure no longer applies and the line
# reports null.
TRAFFIC = {
    (2, None): ("prefill.cu", "8dd95e6094469a10dd713dcb5f27c753c376a317c5928be4a0492058e1ad8105",
                562.07e6),
    (3, None): ("prefill.cu", "8dd95e6094469a10dd713dcb5f27c753c376a317c5928be4a0492058e1ad8105",
                2405.9e6),
    # decode: captured on the small-context forms (swa_8k, n1_256k, n9_256k) and scaled to
    # the full workloads by their algorithmic K/V bytes (the same for swa and swa_8k, 4x
    # for the 1M-token decodes)
    (4, "swa"): ("decode.cu", "5c022f1d15b6f440fa1d162d679b9393382f7e18ed02446048c3048227780e4a", 563.8e6),
    (4, "swa_8k"): ("decode.cu", "5c022f1d15b6f440fa1d162d679b9393382f7e18ed02446048c3048227780e4a", 563.8e6),
    (5, "n1"): ("decode.cu", "5c022f1d15b6f440fa1d162d679b9393382f7e18ed02446048c3048227780e4a", 4316.8e6),
    (5, "n9"): ("decode.cu", "5c022f1d15b6f440fa1d162d679b9393382f7e18ed02446048c3048227780e4a", 4314.8e6),
    (5, "n1_256k"): ("decode.cu", "5c022f1d15b6f440fa1d162d679b9393382f7e18ed02446048c3048227780e4a", 1079.2e6),
    (5, "n9_256k"): ("decode.cu", "5c022f1d15b6f440fa1d162d679b9393382f7e18ed02446048c3048227780e4a", 1078.7e6),
}


def kernel_traffic(workload: int, variant=None, fp8: bool = False):
    if fp8:
        return None
    if workload == 5 and variant is None:
        variant = "n1"
    if workload == 4 and variant is None:
        variant = "swa"
    entry = TRAFFIC.get((workload, variant))
    if entry is None:
        return None
    import hashlib
    src, sha, nbytes = entry
    path = os.path.join(ROOT, "relative_position_gqa_gb300", "csrc", src)
    try:
        with open(path, "rb") as f:
            if hashlib.sha256(f.read()).hexdigest() != sha:
                return None
    except OSError:
        return None
    return nbytes


def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return json.load(f), "measured"
    except (OSError, ValueError):
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


# ------------------------------------------------------------------ our arm ---------
K_SCALE, V_SCALE = 0.0625, 0.0625  # FP8 cache scales of the benchmark
MIN_TIMED_S = 0.25  # a timed loop lasts at least this long (several clock samples)


class Bench:
    """Device state shared by every workload of one run (the L2 flush buffers)."""

    def __init__(self, dev):
        self.dev = dev
        self.flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
        self.flush_sink = torch.empty(1, dtype=torch.float32, device=dev)


def measure_attn(ink, bench: Bench, n: int, variant, fp8: bool, steps: int, warmup: int,
                 ws: int, e2e_chunks: int = 0, exact: bool = False) -> dict:
    """One workload: the step (conv + attention, no event between the launches), the
    attention alone, the conv alone, and the step end to end over page-locked host
    buffers.  Returns the timings (max over ranks), work and clock record.  Each timed
    loop runs `steps` steps (exact) or, for short steps, enough that it lasts
    MIN_TIMED_S."""
    dev = bench.dev
    spec = workload_spec(n, variant)
    decode = is_decode(n)
    rank = int(os.environ.get("RANK", "0"))
    g = W.make_case(spec, seed=n + 1000 * rank, device=dev)
    if fp8:
        g.k_cache = W.fp8_history(g.k_cache, K_SCALE)
        g.v_cache = W.fp8_history(g.v_cache, V_SCALE)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    out = torch.empty(spec.total_q, spec.hq, 128, dtype=torch.bfloat16, device=dev)
    state0 = g.state.clone()
    ws_bytes = 0
    workspace = None
    plan = None
    if decode:
        ws_bytes = ink.decode_workspace_size(spec.batch, spec.hq, spec.hkv, spec.max_q_len,
                                             spec.max_seq_len, spec.window)
        workspace = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device=dev)
        plan = ink.decode_plan(spec.batch, spec.hq, spec.hkv, spec.max_q_len, spec.max_seq_len,
                               spec.window)
    elif fp8:  # the widened bf16 pages of the FP8 prefill
        ws_bytes = ink.prefill_fp8_workspace_size(spec.batch, spec.hkv, g.block_table.shape[1],
                                                  spec.max_q_len, spec.max_seq_len, spec.window)
        workspace = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    def attn(q, o):
        if fp8 and not decode:
            ink.rel_attn_prefill_fp8(q, g.k_cache, g.v_cache, g.block_table, g.cu_q_lens,
                                     g.seq_lens, g.bias, k_scale=K_SCALE, v_scale=V_SCALE,
                                     scale=spec.scale, window=spec.window,
                                     max_q_len=spec.max_q_len, max_seq_len=spec.max_seq_len,
                                     out=o, workspace=workspace, dev_status=status)
        elif fp8:
            ink.rel_attn_decode_fp8(q, g.k_cache, g.v_cache, g.block_table, g.cu_q_lens,
                                    g.seq_lens, g.bias, k_scale=K_SCALE, v_scale=V_SCALE,
                                    scale=spec.scale, window=spec.window,
                                    max_q_len=spec.max_q_len, max_seq_len=spec.max_seq_len,
                                    out=o, workspace=workspace, dev_status=status)
        elif decode:
            ink.rel_attn_decode(q, g.k_cache, g.v_cache, g.block_table, g.cu_q_lens, g.seq_lens,
                                g.bias, scale=spec.scale, window=spec.window,
                                max_q_len=spec.max_q_len, max_seq_len=spec.max_seq_len, out=o,
                                workspace=workspace, dev_status=status)
        else:
            ink.rel_attn_prefill(q, g.k_cache, g.v_cache, g.block_table, g.cu_q_lens,
                                 g.seq_lens, g.bias, scale=spec.scale, window=spec.window,
                                 max_q_len=spec.max_q_len, out=o, dev_status=status)

    def sconv(kr, vr):
        if fp8:
            ink.sconv_kv_fp8(kr, vr, g.w_k, g.w_v, g.state, g.cu_q_lens, g.slot_mapping,
                             g.k_cache, g.v_cache, k_scale=K_SCALE, v_scale=V_SCALE,
                             max_q_len=spec.max_q_len, dev_status=status)
        else:
            ink.sconv_kv(kr, vr, g.w_k, g.w_v, g.state, g.cu_q_lens, g.slot_mapping, g.k_cache,
                         g.v_cache, max_q_len=spec.max_q_len, dev_status=status)

    def reset():
        g.state.copy_(state0)
        flush_l2(bench.flush, bench.flush_sink)

    # the decode step over a bf16 cache is one call: the conv of the new tokens fused into
    # the decode kernel's prologue (inkling_rel_attn_decode_sconv); otherwise the two calls
    fused_step = decode and not fp8

    def fused():
        ink.rel_attn_decode_sconv(g.q, g.k_raw, g.v_raw, g.w_k, g.w_v, g.state, g.k_cache,
                                  g.v_cache, g.block_table, g.cu_q_lens, g.seq_lens, g.bias,
                                  scale=spec.scale, window=spec.window, max_q_len=spec.max_q_len,
                                  max_seq_len=spec.max_seq_len, out=out, workspace=workspace,
                                  dev_status=status)

    def two_calls():
        sconv(g.k_raw, g.v_raw)
        attn(g.q, out)

    step_fn = fused if fused_step else two_calls

    def check():
        torch.cuda.synchronize()
        if int(status.item()) != 0:
            raise RuntimeError(f"{spec.name}: device status {ink.status_string(int(status.item()))}")

    def timed(fn, k):
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(k)]
        for i in range(k):
            reset()
            evs[i][0].record(stream)
            fn()
            evs[i][1].record(stream)
        return evs

    def mean_ms(evs):
        return sum(a.elapsed_time(b) for a, b in evs) / len(evs)

    # ---- warm-up, then the step count: at least `steps`, and enough that the timed loop
    # lasts MIN_TIMED_S, so that the clock sampler sees several samples
    for _ in range(warmup):
        reset()
        two_calls()
        if fused_step:
            reset()
            fused()
    check()
    probe = timed(step_fn, 3)
    check()
    est_ms = mean_ms(probe)
    k = steps
    if not exact:
        k = max(steps, min(5000, int(math.ceil(MIN_TIMED_S * 1e3 / max(est_ms + 0.1, 1e-3)))))
        k = int(max_over_ranks([k], ws, dev)[0])

    # ---- device-resident timing.  The step is timed with no event between its two
    # launches, so that the attention kernel's programmatic dependent launch overlaps the
    # conv's tail as it would in a model; the attention and the conv are then timed alone.
    if ws > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    with ClockSampler(dev.index if dev.index is not None else 0) as clocks:
        ev_step = timed(step_fn, k)
        torch.cuda.synchronize()
    ev_attn = []
    for i in range(k):
        reset()
        sconv(g.k_raw, g.v_raw)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        attn(g.q, out)
        b.record(stream)
        ev_attn.append((a, b))
    ev_sconv = timed(lambda: sconv(g.k_raw, g.v_raw), k)
    check()
    if ws > 1:
        torch.distributed.barrier()
    step_ms, attn_ms, sconv_ms = mean_ms(ev_step), mean_ms(ev_attn), mean_ms(ev_sconv)

    two_call_ms = None
    if fused_step:
        # the same step as the two separate calls (inkling_sconv_kv, then the decode)
        ev_two = timed(two_calls, k)
        check()
        two_call_ms = mean_ms(ev_two)

    rollback_us = None
    if n == 4 and not fp8:
        # after a verify step, keep a seeded random prefix of each sequence's 9 tokens
        gen = torch.Generator().manual_seed(4)
        accepted = torch.randint(0, 10, (spec.batch,), generator=gen, dtype=torch.int32).to(dev)
        rb = []
        for i in range(warmup + steps):
            reset()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            ink.sconv_state_rollback(state0, g.k_raw, g.v_raw, g.cu_q_lens, accepted, g.state,
                                     dev_status=status)
            b.record(stream)
            if i >= warmup:
                rb.append((a, b))
        check()
        rollback_us = round(1e3 * mean_ms(rb), 2)

    # ---- end to end through the public API with host buffers: the step entry points
    # (inkling_prefill_step_host / inkling_decode_step_host and their _fp8 forms) take
    # page-locked Q, raw K/V and output buffers and overlap the copies of one group of
    # sequences with the compute of another.
    host_in = [t.cpu().pin_memory() for t in (g.q, g.k_raw, g.v_raw)]
    dev_in = [torch.empty_like(t, device=dev) for t in host_in]
    host_out = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in host_in)
    d2h = host_out.numel() * host_out.element_size()
    cu_host = g.cu_q_lens.cpu()
    up, down = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    # prefill: sixteen groups (a long sequence is cut into pieces of whole query tiles, so
    # the 64K prefill overlaps its copies too; 4 / 8 / 16 groups measured 1412 / 1419 /
    # 1428 TFLOP/s end to end on it, 647 / 689 / 691 on the window prefill).  decode: one group (its copies are a few
    # MB, and cutting the batch gives each group its own tail of ragged lengths: two groups
    # measured 1.66 ms on the full MTP decode against 1.41 ms for one)
    chunks = e2e_chunks if e2e_chunks > 0 else (1 if decode else 16)
    e2e_path = (f"inkling_{'decode' if decode else 'prefill'}_step_host{'_fp8' if fp8 else ''}, "
                f"{chunks} groups" + ("" if decode else " (sequences cut into query-tile pieces)"))

    def host_step():
        step_args = (host_in[0], host_in[1], host_in[2], host_out, (*dev_in, out), cu_host,
                     g.w_k, g.w_v, g.state, g.cu_q_lens, g.slot_mapping, g.k_cache, g.v_cache,
                     g.block_table, g.seq_lens, g.bias)
        if fp8:
            kw = dict(k_scale=K_SCALE, v_scale=V_SCALE, scale=spec.scale, window=spec.window,
                      max_q_len=spec.max_q_len, max_seq_len=spec.max_seq_len,
                      workspace=workspace, h2d_stream=up, d2h_stream=down, chunks=chunks,
                      dev_status=status)
            if decode:
                ink.decode_step_host_fp8(*step_args, **kw)
            else:
                ink.prefill_step_host_fp8(*step_args, **kw)
        elif decode:
            ink.decode_step_host(*step_args, scale=spec.scale, window=spec.window,
                                 max_q_len=spec.max_q_len, max_seq_len=spec.max_seq_len,
                                 workspace=workspace, h2d_stream=up, d2h_stream=down,
                                 chunks=chunks, dev_status=status)
        else:
            ink.prefill_step_host(*step_args, scale=spec.scale, window=spec.window,
                                  max_q_len=spec.max_q_len, h2d_stream=up, d2h_stream=down,
                                  chunks=chunks, dev_status=status)

    for _ in range(warmup):
        reset()
        host_step()
    check()
    ev_e2e = timed(host_step, k)
    check()
    e2e_ms = mean_ms(ev_e2e)
    step_ms, attn_ms, e2e_ms, sconv_ms = max_over_ranks([step_ms, attn_ms, e2e_ms, sconv_ms],
                                                        ws, dev)
    if two_call_ms is not None:
        two_call_ms = max_over_ranks([two_call_ms], ws, dev)[0]

    peaks, peak_src = measured_peaks()
    if decode:
        work = decode_kv_bytes(spec) / (2 if fp8 else 1)
        unit, scale_u = "GB/s", 1e9
        peak = float(peaks["hbm_gbs"])
        roof = {"bound": "hbm", "unit": "GB/s", "peak_source": f"{peak_src} hbm_gbs",
                "kernel": "decode_kernel<true> (FP8 cache)" if fp8 else "decode_kernel (+combine)"}
    else:
        work = attn_flops(spec)
        unit, scale_u = "TFLOP/s", 1e12
        peak = float(peaks["bf16_tflops"])
        roof = {"bound": "tensor", "unit": "TFLOP/s",
                "peak_source": f"{peak_src} bf16_tflops (burst; kernel timed per launch)",
                "kernel": "widen_pages_kernel + prefill_kernel" if fp8 else "prefill_kernel"}
    achieved = work / (attn_ms * 1e-3) / scale_u
    roof.update({"achieved": round(achieved, 1), "peak": peak, "frac": round(achieved / peak, 4),
                 "traffic": kernel_traffic(n, variant, fp8)})
    launches_per_step = (1 if fused_step else 2) + (1 if (decode and plan["merge"]) or
                                                      (fp8 and not decode) else 0)
    entry = {
        "workload": workload_name(spec) + (" kv=e4m3" if fp8 else ""),
        "value": round(ws * work / (step_ms * 1e-3) / scale_u, 3), "unit": unit,
        "ms_per_step": round(step_ms, 4), "steps": k, "attn_ms": round(attn_ms, 4),
        "sconv_ms": round(sconv_ms, 4),
        "e2e": {"value": round(ws * work / (e2e_ms * 1e-3) / scale_u, 3), "unit": unit,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": round(e2e_ms, 4), "path": e2e_path},
        "roofline": roof,
        "clocks": clocks.summary(),
        "gpu_launches": k * launches_per_step,
        "dtype": ("bf16 (KV cache e4m3, f16 MMA)" if decode else
                  "bf16 (KV cache e4m3 widened to bf16)") if fp8 else "bf16",
        "_work": work, "_attn_ms": attn_ms, "_e2e_ms": e2e_ms, "_spec": spec,
    }
    if decode:
        entry["decode_plan"] = plan
    entry["step_path"] = ("inkling_rel_attn_decode_sconv (the conv in the decode kernel's "
                          "prologue)" if fused_step else
                          f"inkling_sconv_kv{'_fp8' if fp8 else ''} + "
                          f"inkling_rel_attn_{'decode' if decode else 'prefill'}{'_fp8' if fp8 else ''}")
    if two_call_ms is not None:
        entry["two_call_step"] = {"value": round(ws * work / (two_call_ms * 1e-3) / scale_u, 3),
                                  "unit": unit, "ms_per_step": round(two_call_ms, 4),
                                  "path": "inkling_sconv_kv + inkling_rel_attn_decode"}
    if rollback_us is not None:
        entry["rollback_us"] = rollback_us
    del g, out, workspace, host_in, dev_in, host_out
    torch.cuda.empty_cache()
    return entry


def combined_decode(swa: dict, full: dict) -> dict:
    """One sliding-window and one full MTP decode layer as one figure: both calls' K/V
    bytes over both calls' time (the two layer kinds alternate in the model)."""
    work = swa["_work"] + full["_work"]
    step_ms = swa["ms_per_step"] + full["ms_per_step"]
    attn_ms = swa["_attn_ms"] + full["_attn_ms"]
    e2e_ms = swa["_e2e_ms"] + full["_e2e_ms"]
    peak = swa["roofline"]["peak"]
    achieved = work / (attn_ms * 1e-3) / 1e9
    return {
        "workload": "mtp_decode: one window-4096 layer + one full layer (K/V bytes of both "
                    "calls over both calls' time)",
        "value": round(work / (step_ms * 1e-3) / 1e9, 3), "unit": "GB/s",
        "ms_per_step": round(step_ms, 4), "attn_ms": round(attn_ms, 4),
        "e2e": {"value": round(work / (e2e_ms * 1e-3) / 1e9, 3), "unit": "GB/s",
                "h2d_bytes_per_step": swa["e2e"]["h2d_bytes_per_step"] + full["e2e"]["h2d_bytes_per_step"],
                "d2h_bytes_per_step": swa["e2e"]["d2h_bytes_per_step"] + full["e2e"]["d2h_bytes_per_step"],
                "ms_per_step": round(e2e_ms, 4)},
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak,
                     "unit": "GB/s", "frac": round(achieved / peak, 4), "traffic": None,
                     "peak_source": swa["roofline"]["peak_source"],
                     "kernel": swa["roofline"]["kernel"]},
        "clocks": {"from": ["4_mtp_decode_swa", "4_mtp_decode_full"]},
    }


def public(entry: dict) -> dict:
    return {k: v for k, v in entry.items() if not k.startswith("_")}


# every workload of the sweep: (key, workload, variant, FP8 cache)
SWEEP = [
    ("1_tiny_prefill", 1, None, False),
    ("2_swa_prefill", 2, None, False),
    ("3_full_prefill_64k", 3, None, False),
    ("4_mtp_decode_swa", 4, "swa", False),
    ("4_mtp_decode_full", 4, "full", False),
    ("5_decode_1m_n1", 5, "n1", False),
    ("5_decode_1m_n9", 5, "n9", False),
    ("2_swa_prefill_fp8", 2, None, True),
    ("4_mtp_decode_swa_fp8", 4, "swa", True),
    ("4_mtp_decode_full_fp8", 4, "full", True),
    ("5_decode_1m_n1_fp8", 5, "n1", True),
    ("5_decode_1m_n9_fp8", 5, "n9", True),
]


def sweep_key(n: int, variant, fp8: bool):
    """The sweep's key for a workload (variant None is the sliding-window MTP decode and
    the one-token 1M decode, as in workloads.config)."""
    v = variant if variant is not None else {4: "swa", 5: "n1"}.get(n)
    for key, n2, v2, f2 in SWEEP:
        if n2 == n and v2 == v and f2 == fp8:
            return key
    return None


def line_config(spec: W.Spec, ws: int, fp8: bool) -> dict:
    return {"workload": workload_name(spec) + (" kv=e4m3" if fp8 else ""),
            "global_batch": spec.batch * ws, "seq_len": spec.max_seq_len,
            "parallelism": f"replicas x{ws}", "l2": L2_NOTE}


def run_ours(args, ws, rank, local):
    import relative_position_gqa_gb300 as ink
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    ink._lib.load()  # raises if the CUDA library is missing: no fallback
    bench = Bench(dev)
    fp8 = args.kv == "fp8"
    # the headline: exactly --steps timed steps
    main = measure_attn(ink, bench, args.workload, args.variant, fp8, args.steps, args.warmup,
                        ws, args.e2e_chunks, exact=True)
    if args.traffic is not None:
        main["roofline"]["traffic"] = args.traffic
    spec = main["_spec"]
    line = {
        "metric": METRIC, "value": main["value"], "unit": main["unit"], "n_gpus": ws,
        "steps": main["steps"], "warmup": args.warmup, "ms_per_step": main["ms_per_step"],
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": main["dtype"],
        "data": "synthetic (seeded N(0,1) Q/K/V, N(0,0.5) sconv taps, N(0,sd) bias)",
        "config": line_config(spec, ws, fp8),
        "detail": {"attn_ms": main["attn_ms"], "sconv_ms": main["sconv_ms"],
                   "step_path": main["step_path"],
                   **({"two_call_step": main["two_call_step"]} if "two_call_step" in main else {}),
                   **({"decode_plan": main["decode_plan"]} if "decode_plan" in main else {}),
                   **({"rollback_us": main["rollback_us"]} if "rollback_us" in main else {})},
        "e2e": main["e2e"],
        "gpu_launches": main["gpu_launches"],
        "roofline": main["roofline"],
        "clocks": main["clocks"],
    }
    if args.sweep:
        # every configuration in the same run: prefill TFLOP/s and decode KV-read GB/s,
        # each with its roofline, end-to-end figure and clock record
        results = {}
        main_key = sweep_key(args.workload, args.variant, fp8)
        for key, n, variant, f8 in SWEEP:
            if key == main_key:
                results[key] = main
                continue
            results[key] = measure_attn(ink, bench, n, variant, f8, args.steps, args.warmup, ws)
        results["4_mtp_decode_combined"] = combined_decode(results["4_mtp_decode_swa"],
                                                           results["4_mtp_decode_full"])
        results["4_mtp_decode_combined_fp8"] = combined_decode(
            results["4_mtp_decode_swa_fp8"], results["4_mtp_decode_full_fp8"])
        line["workloads"] = {k: public(v) for k, v in results.items()}
        line["gpu_launches_all"] = sum(v.get("gpu_launches", 0) for v in results.values())
    return line


def run_dense(args, ws, rank, local):
    """--workload 6: inkling_sconv on a dense [T, C] stream with its own state."""
    import relative_position_gqa_gb300 as ink
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    ink._lib.load()
    c = W.make_dense(DENSE_Q_LENS, DENSE_C, seed=6 + 1000 * rank, device=dev)
    T = sum(DENSE_Q_LENS)
    y = torch.empty_like(c.x)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    state0 = c.state.clone()
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    flush_sink = torch.empty(1, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()

    def step(x):
        ink.sconv(x, c.w, c.state, c.cu_q_lens, max_q_len=max(DENSE_Q_LENS), y=y,
                  dev_status=status)

    def reset():
        c.state.copy_(state0)
        flush_l2(flush, flush_sink)

    for _ in range(args.warmup):
        reset()
        step(c.x)
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    if ws > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clocks:
        for i in range(args.steps):
            reset()
            ev[i][0].record(stream)
            step(c.x)
            ev[i][1].record(stream)
        torch.cuda.synchronize()
    if int(status.item()) != 0:
        raise RuntimeError(f"device status {ink.status_string(int(status.item()))}")
    step_ms = sum(a.elapsed_time(b) for a, b in ev) / args.steps
    host_in = c.x.cpu().pin_memory()
    dev_in = torch.empty_like(host_in, device=dev)
    host_out = torch.empty(y.shape, dtype=y.dtype).pin_memory()
    e2e_ev = []
    for i in range(args.warmup + args.steps):
        reset()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        dev_in.copy_(host_in, non_blocking=True)
        step(dev_in)
        host_out.copy_(y, non_blocking=True)
        b.record(stream)
        if i >= args.warmup:
            e2e_ev.append((a, b))
    torch.cuda.synchronize()
    e2e_ms = sum(a.elapsed_time(b) for a, b in e2e_ev) / len(e2e_ev)
    step_ms, e2e_ms = max_over_ranks([step_ms, e2e_ms], ws, dev)
    peaks, peak_src = measured_peaks()
    work = dense_bytes(DENSE_Q_LENS, DENSE_C)
    achieved = work / (step_ms * 1e-3) / 1e9
    peak = float(peaks["hbm_gbs"])
    return {
        "metric": METRIC, "value": round(ws * achieved, 1), "unit": "GB/s", "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(step_ms, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) rows and state, N(0,0.5) taps)",
        "config": {"workload": f"attn_out_sconv: B=4 x 8192 tokens, C={DENSE_C}, window 4",
                   "global_batch": 4 * ws, "seq_len": 8192, "parallelism": f"replicas x{ws}",
                   "l2": L2_NOTE},
        "e2e": {"value": round(ws * work / (e2e_ms * 1e-3) / 1e9, 1), "unit": "GB/s",
                "h2d_bytes_per_step": host_in.numel() * 2, "d2h_bytes_per_step": host_out.numel() * 2},
        "gpu_launches": args.steps,
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "traffic": args.traffic,
                     "peak_source": f"{peak_src} hbm_gbs", "kernel": "sconv_kernel<false>"},
        "clocks": clocks.summary(),
    }


def dense_oracle_sample(seed: int):
    """The oracle's dense conv on one 8192-token sequence of the same width."""
    import oracle
    c = W.make_dense(DENSE_Q_LENS[:1], DENSE_C, seed=seed)
    t0 = time.perf_counter()
    oracle.sconv_dense(c.x, c.w, c.state.clone(), c.cu_q_lens)
    secs = time.perf_counter() - t0
    return dense_bytes(DENSE_Q_LENS[:1], DENSE_C), secs


# ------------------------------------------------------------- oracle (CPU) arm -----
def oracle_case(spec: W.Spec, seed: int):
    """The CPU input set the oracle is timed on: the whole workload when it is small and
    has no random cache history, else its last sequence alone."""
    small_enough = (not spec.history_random) and spec.total_q * spec.hq < 3_000_000
    if not small_enough:
        spec = W.Spec(**{**spec.__dict__, "batch": 1, "q_lens": [spec.q_lens[-1]],
                         "seq_lens": [spec.seq_lens[-1]]})
    return spec, W.make_case(spec, seed=seed, device="cpu")


def oracle_sample(spec: W.Spec, case, budget_s: float, seed: int):
    """Time the fp64 oracle on a bounded sample of the workload: the sconv of every new
    token of `case` plus attention for seeded random query rows until `budget_s` of
    attention time is used.  Returns (allowed pairs done, attention seconds, sconv
    seconds, rows, cores, spec)."""
    import oracle
    cores = oracle.host_cores()
    kc, vc, st = case.k_cache.clone(), case.v_cache.clone(), case.state.clone()
    t0 = time.perf_counter()
    oracle.sconv_kv(case.k_raw, case.v_raw, case.w_k, case.w_v, st, case.cu_q_lens,
                    case.slot_mapping, kc, vc)
    t_sconv = time.perf_counter() - t0
    # attention rows: grow the sample until the time budget is used
    T = spec.total_q
    rows, done_pairs, t_attn = [], 0, 0.0
    cu = case.cu_q_lens.tolist()
    sl = case.seq_lens.tolist()
    rng = torch.Generator().manual_seed(seed)
    batch = max(cores, 8)
    while t_attn < budget_s and len(rows) < T:
        pick = torch.randint(0, T, (batch,), generator=rng).tolist()
        t0 = time.perf_counter()
        oracle.rel_attn(case.q, kc, vc, case.block_table, case.cu_q_lens, case.seq_lens,
                        case.bias, scale=spec.scale, window=spec.window, rows=pick)
        t_attn += time.perf_counter() - t0
        for t in pick:
            b = max(i for i in range(len(cu) - 1) if cu[i] <= t)
            n, L = cu[b + 1] - cu[b], sl[b]
            p = L - n + (t - cu[b])
            done_pairs += (p + 1) if spec.window <= 0 else min(p + 1, spec.window)
        rows += pick
    return (done_pairs, t_attn, t_sconv, len(rows), cores, spec)


def run_reference_dense(args, ws):
    per = [dense_oracle_sample(seed=6 + i) for i in range(args.warmup + args.steps)][args.warmup:]
    work = sum(b for b, _ in per)
    secs = sum(t for _, t in per)
    value = work / secs / 1e9
    cores = 1  # the dense conv oracle is single-threaded
    desc = f"fp64 C oracle, one thread: one 8192-token sequence x {DENSE_C} channels per step"
    return {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(secs / len(per) * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": {"workload": f"attn_out_sconv: B=4 x 8192 tokens, C={DENSE_C}"},
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": cores, "kind": "oracle",
                         "sample": desc},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def run_reference(args, ws, rank):
    if args.workload == 6:
        return run_reference_dense(args, ws)
    spec = workload_spec(args.workload, args.variant)
    decode = is_decode(args.workload)
    per_step = []
    desc = None
    sspec, case = oracle_case(spec, seed=args.workload)
    # each step a bounded sample: about two minutes of oracle time for the whole run,
    # at most --ref-seconds a step
    per_step_s = max(0.2, min(args.ref_seconds, REF_TOTAL_S / (args.warmup + args.steps)))
    for i in range(args.warmup + args.steps):
        pairs, t_attn, t_sconv, nrows, cores, sspec = oracle_sample(
            sspec, case, budget_s=per_step_s, seed=args.workload + i)
        if i >= args.warmup:
            per_step.append((pairs, t_attn, nrows))
        desc = (f"fp64 C oracle on {cores} host threads: {nrows} random query rows x "
                f"{sspec.hq} heads of the workload (plus one sequence's sconv, "
                f"{t_sconv:.2f} s, not counted)")
    pairs = sum(p for p, _, _ in per_step)
    secs = sum(t for _, t, _ in per_step)
    if decode:
        # bytes of K/V the sampled rows read, per the same accounting as our arm
        work = pairs * 2 * 128 * 2 / (spec.hq // spec.hkv)
        unit = "GB/s"
        value = work / secs / 1e9
    else:
        work = 4.0 * 128 * pairs
        unit = "TFLOP/s"
        value = work / secs / 1e12
    ms = secs / len(per_step) * 1e3
    return {
        "impl": "reference", "metric": METRIC, "value": value, "unit": unit, "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": line_config(spec, ws, False),
        "cpu_baseline": {"value": value, "unit": unit, "cores": cores, "kind": "oracle",
                         "sample": desc},
        "e2e": {"value": value, "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", type=int, default=None, choices=[1, 2, 3, 4, 5, 6],
                    help="default: 3 (the 64K full prefill), with every other workload "
                         "measured in the same run (--sweep)")
    ap.add_argument("--sweep", action=argparse.BooleanOptionalAction, default=None,
                    help="measure every workload after the headline one (default: on when "
                         "--workload is not given)")
    ap.add_argument("--variant", default=None, help="mtp_decode: swa|full (swa_8k: contexts <= 8192); decode_1m: n1|n9 (n1_256k|n9_256k: quarter length)")
    ap.add_argument("--kv", choices=["bf16", "fp8"], default="bf16",
                    help="KV cache type for the decode workloads")
    ap.add_argument("--ref-seconds", type=float, default=6.0,
                    help="oracle seconds per reference step / for the cpu_baseline sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--e2e-chunks", type=int, default=0,
                    help="groups for the end-to-end host-buffer step (0: 16 for prefill, 1 for decode)")
    ap.add_argument("--traffic", type=float, default=None,
                    help="DRAM bytes per launch of the dominant kernel from an ncu capture")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    if args.sweep is None:
        args.sweep = args.workload is None and args.kv == "bf16" and args.variant is None
    if args.workload is None:
        args.workload = 3

    ws, rank, local = dist_env()
    if ws > 1:
        backend = "nccl" if args.impl == "ours" else "gloo"
        if args.impl == "ours":
            torch.cuda.set_device(local)
        torch.distributed.init_process_group(backend=backend)

    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args, ws, rank)), flush=True)
        if ws > 1:
            torch.distributed.destroy_process_group()
        return

    if args.workload == 6:
        line = run_dense(args, ws, rank, local)
        if rank == 0 and not args.no_cpu_baseline:
            b, t = dense_oracle_sample(seed=99)
            line["cpu_baseline"] = {"value": b / t / 1e9, "unit": "GB/s", "cores": 1,
                                    "kind": "oracle",
                                    "sample": f"one 8192-token sequence x {DENSE_C} channels, "
                                              f"fp64 C oracle, one thread, {t:.2f} s"}
        if rank == 0:
            print(json.dumps(line), flush=True)
        if ws > 1:
            torch.distributed.destroy_process_group()
        return

    line = run_ours(args, ws, rank, local)
    if rank == 0 and not args.no_cpu_baseline:
        spec = workload_spec(args.workload, args.variant)
        sspec, case = oracle_case(spec, seed=args.workload)
        pairs, t_attn, t_sconv, nrows, cores, sspec = oracle_sample(sspec, case,
                                                                    args.ref_seconds, seed=99)
        if is_decode(args.workload):
            v = pairs * 2 * 128 * 2 / (spec.hq // spec.hkv) / t_attn / 1e9
            unit = "GB/s"
        else:
            v = 4.0 * 128 * pairs / t_attn / 1e12
            unit = "TFLOP/s"
        line["cpu_baseline"] = {
            "value": v, "unit": unit, "cores": cores, "kind": "oracle",
            "sample": f"{nrows} random query rows x {sspec.hq} heads (all allowed keys each), "
                      f"fp64 C oracle, {t_attn:.1f} s"}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if ws > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
