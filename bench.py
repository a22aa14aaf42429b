"""Benchmark of the paged varlen rel-bias attention hot path on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

One step = one call of the whole hot path (device plan, decode and/or prefill
kernels, split-KV merge) over one batch of synthetic input already resident
in HBM.  The headline line is the decode batch (64 decodes, Lk ~ U{1024..32768},
H 32, Hkv 8, E 1024): `value` = algorithmic KV bytes read / step time (GB/s).
The chunked-prefill (TFLOP/s on unmasked pairs), long batch-1 decode and
continuous-batch workloads are measured in the same run and reported under
"workloads".  Inputs are larger than L2 (no flush needed).  `--impl reference`
times the fp64 CPU oracle on the host cores instead (rank 0 only).
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
import threading
import time
from typing import Optional

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "paged rel-bias attn: decode KV-read GB/s & prefill TFLOP/s (% of roofline)"
HEADLINE = "decode_batch"
SECONDARY = ["chunked_prefill", "long_decode", "continuous_batch"]
FP8_SCALES = (0.0625, 0.05)  # k_scale, v_scale of the E4M3 caches the bench builds
TIMED_KERNELS = ("prepass", "stage", "decode", "prefill", "combine")
HEADDIM = ("decode_batch_d64", "chunked_prefill_d64", "decode_batch_d256", "chunked_prefill_d256")
D = 128


# ---------------------------------------------------------------------------------- work model

def work_of(case):
    """Algorithmic work of one step: KV bytes of decode-shaped rows, flops of visible pairs.

    Decode: sum over decode requests of (#visible keys) * Hkv * D * 2 (K and V) * 2 bytes.
    Prefill: 4 * D * H * (#visible (q, k) pairs) over prefill requests.
    """
    G = case.H // case.Hkv
    D = getattr(case, "D", 128)
    kv_bytes = 0
    flops = 0
    pairs = 0
    for lq, lk in zip(case.q_lens, case.kv_lens):
        n_pairs = 0
        for i in range(lq):
            qa = i + lk - lq
            lo = max(0, qa - case.window_left) if case.window_left >= 0 else 0
            hi = lk - 1
            if case.causal:
                hi = min(hi, qa)
            if case.window_right >= 0:
                hi = min(hi, qa + case.window_right)
            n_pairs += max(0, hi - lo + 1)
        if lq * G <= 16:
            # each key of the union of visible ranges is read once for all heads
            qa0, qa1 = lk - lq, lk - 1
            lo = max(0, qa0 - case.window_left) if case.window_left >= 0 else 0
            hi = min(lk - 1, qa1) if case.causal else lk - 1
            if case.window_right >= 0:
                hi = min(hi, qa1 + case.window_right)
            kv_bytes += max(0, hi - lo + 1) * case.Hkv * D * 2 * 2
        else:
            pairs += n_pairs
            flops += 4 * D * case.H * n_pairs
    return kv_bytes, flops, pairs


def prefill_keys(case):
    """Cache keys of the prefill-shaped requests (more than 16 query rows per KV head), summed."""
    G = case.H // case.Hkv
    return sum(lk for lq, lk in zip(case.q_lens, case.kv_lens) if lq * G > 16)


def total_bytes(case, fp8=False):
    """Compulsory HBM bytes of one step: q in and out, the decode rows' visible K/V, every key of the prefill
    requests' K/V once, and the rel_logits band each row reads (E4M3 caches: one byte per K/V element)."""
    kv, _, _ = work_of(case)
    el = 1 if fp8 else 2
    b = case.q.numel() * 2 * 2  # q in, out
    b += prefill_keys(case) * case.Hkv * case.D * 2 * el
    if case.E > 0:
        b += _bias_bytes(case)
    return kv * el // 2 + b


def _bias_bytes(case):
    n = 0
    for lq, lk in zip(case.q_lens, case.kv_lens):
        # row i reads rd in [0, min(E, visible extent)) : count with a closed form per row
        for i in range(lq):
            qa = i + lk - lq
            hi_rd = qa  # keys j >= 0
            if case.window_left >= 0:
                hi_rd = min(hi_rd, case.window_left)
            n += max(0, min(case.E, hi_rd + 1))
    return n * case.H * 4


# ---------------------------------------------------------------------------------- helpers

def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            pk = json.load(f)
        return {"hbm_gbs": float(pk["hbm_gbs"]), "bf16_tflops": float(pk["bf16_tflops"]),
                "bf16_tflops_sustained": float(pk.get("bf16_tflops_sustained", pk["bf16_tflops"])),
                "source": "measured"}
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


KERNEL_SOURCES = {"ink_decode_kernel": "ink_decode.cu", "ink_prefill_kernel": "ink_prefill.cu",
                  "ink_prefill_pair_kernel": "ink_prefill.cu", "ink_generic_kernel": "ink_generic.cu",
                  "ink_stage_kernel": "ink_stage.cu",
                  "ink_combine_kernel": "ink_combine.cu", "ink_prepass_kernel": "ink_prepass.cu",
                  "ink_append_kernel": "ink_append.cu", "ink_append_fp8_kernel": "ink_append.cu"}


def kernel_source_hash(kernel):
    """Hash of what one kernel is compiled from: its own .cu file and the shared header."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "paged_varlen_attention_causal_gb300", "csrc")
    for name in ("ink_common.cuh", KERNEL_SOURCES[kernel]):
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def traffic_of(kernel, workload):
    """DRAM bytes per launch from the committed ncu summary, if taken on the kernel's current source."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    try:
        with open(path) as f:
            k = json.load(f)["kernels"][kernel]
        if k.get("source_hash") != kernel_source_hash(kernel):
            return None
        return k[workload]
    except Exception:
        return None


class _Nvml:
    """Read-only NVML queries through ctypes (SM clock, its maximum, clock-event reasons)."""

    SM = 1  # NVML_CLOCK_SM
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown", 0x40: "hw_thermal_slowdown",
               0x80: "hw_power_brake_slowdown"}

    def __init__(self, uuid: Optional[str], index: int):
        import ctypes
        self.c = ctypes
        self.lib = ctypes.CDLL("libnvidia-ml.so.1")
        if self.lib.nvmlInit_v2() != 0:
            raise OSError("nvmlInit failed")
        self.h = ctypes.c_void_p()
        rc = 1
        if uuid:
            rc = self.lib.nvmlDeviceGetHandleByUUID(ctypes.c_char_p(uuid.encode()), ctypes.byref(self.h))
        if rc != 0:
            rc = self.lib.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(index), ctypes.byref(self.h))
        if rc != 0:
            raise OSError("no NVML handle for the device")
        self.reason_fn = getattr(self.lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            self.lib.nvmlDeviceGetCurrentClocksThrottleReasons
        self.max_sm = self._clock(self.lib.nvmlDeviceGetMaxClockInfo)

    def _clock(self, fn) -> Optional[float]:
        v = self.c.c_uint(0)
        return float(v.value) if fn(self.h, self.c.c_int(self.SM), self.c.byref(v)) == 0 else None

    def sample(self):
        v = self.c.c_ulonglong(0)
        bits = v.value if self.reason_fn(self.h, self.c.byref(v)) == 0 else 0
        return self._clock(self.lib.nvmlDeviceGetClockInfo), [n for b, n in self.REASONS.items() if bits & b]

    def close(self):
        self.lib.nvmlShutdown()


def _device_uuid(index: int) -> Optional[str]:
    import torch
    u = getattr(torch.cuda.get_device_properties(index), "uuid", None)
    if u is None:
        return None
    u = str(u)
    return u if u.startswith("GPU-") else "GPU-" + u


def hold_stream(stream, ms: float = 20.0):
    """Queue a bounded spin kernel (torch's) ahead of a timed region, so that the host enqueues the region's
    launches while the GPU is still busy: a stall of the launching thread (the clock sampler's thread holding
    the interpreter lock, say) then leaves no idle gap between the timed kernels."""
    import torch

    with torch.cuda.stream(stream):
        torch.cuda._sleep(int(ms * 1e-3 * 2.1e9))  # cycles, at about the maximum SM clock


class ClockSampler:
    """SM clock and clock-event reasons sampled while the timed region runs.

    NVML is polled every 2 ms from a thread (the timed regions last milliseconds,
    shorter than nvidia-smi's start-up); nvidia-smi at 100 ms is the fallback.
    """

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index, period_s: float = 0.002):
        self.gpu = gpu_index
        self.period = period_s
        self.proc = None
        self.nvml = None
        self.lines = []
        self.sm, self.reasons = [], set()
        self.stop = threading.Event()
        self.t = None
        try:
            self.nvml = _Nvml(_device_uuid(gpu_index), gpu_index)
        except Exception:
            self.nvml = None

    def _poll(self):
        while True:
            clk, rs = self.nvml.sample()
            if clk is not None:
                self.sm.append(clk)
            self.reasons.update(rs)
            if self.stop.wait(self.period):
                return

    def __enter__(self):
        if self.nvml is not None:
            self.t = threading.Thread(target=self._poll, daemon=True)
            self.t.start()
            return self
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.nvml is not None:
            self.stop.set()
            self.t.join(timeout=5)
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        if self.nvml is not None:
            if not self.sm:
                return {"sm_mhz": None, "sm_max_mhz": self.nvml.max_sm, "reasons": sorted(self.reasons),
                        "samples": 0, "source": "nvml"}
            return {"sm_mhz": statistics.median(self.sm), "sm_max_mhz": self.nvml.max_sm,
                    "reasons": sorted(self.reasons), "samples": len(self.sm), "source": "nvml"}
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0, "source": "nvidia-smi"}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm), "source": "nvidia-smi"}


# ---------------------------------------------------------------------------------- ranks

def max_over_ranks(x: float, device=None) -> float:
    """Largest value of `x` over all ranks (the step time the job is charged); identity without a group."""
    import torch
    import torch.distributed as dist

    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(units_per_rank: float, world: int, ms_max: float) -> float:
    """Weak scaling: every rank processes the same work; value = all ranks' units / slowest rank's time."""
    return world * units_per_rank / (ms_max * 1e-3)


# ---------------------------------------------------------------------------------- our arm

def run_ours(args, rank, world, local_rank):
    import torch

    import paged_varlen_attention_causal_gb300 as ink
    from workloads import HEADDIM_WORKLOADS, PROFILE_WORKLOADS, WORKLOADS, build_case, fp8_kv, workload

    WORKLOADS = {**WORKLOADS, **PROFILE_WORKLOADS, **HEADDIM_WORKLOADS}
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    ink.build()
    ink.load()
    peaks = load_peaks()
    dist = None
    if world > 1:
        import torch.distributed as dist  # noqa: F811

    def barrier():
        if dist is not None:
            dist.barrier()

    def attend(case, q, block_table, cache_seqlens, cu_seqlens_q, rel_logits, out, lse, splits=0):
        """One call of the public API; an E4M3 cache (uint8) goes through the FP8 entry point.  The caller knows
        its batch, so the workspace is sized to stage the K/V of its prefill-shaped requests."""
        kw = dict(block_table=block_table, cache_seqlens=cache_seqlens, cu_seqlens_q=cu_seqlens_q,
                  max_seqlen_q=case.max_seqlen_q, softmax_scale=case.softmax_scale, causal=case.causal,
                  window_left=case.window_left, window_right=case.window_right, rel_extent=case.E,
                  rel_logits=rel_logits, num_splits=splits, out=out, lse=lse)
        if case.key_cache.dtype == torch.uint8:
            return ink.ink_rel_attn_varlen_fp8kv(q, case.key_cache, case.value_cache, k_scale=FP8_SCALES[0],
                                                 v_scale=FP8_SCALES[1], stage_kv_tokens=prefill_keys(case), **kw)
        return ink.ink_rel_attn_varlen(q, case.key_cache, case.value_cache, stage_kv_tokens=prefill_keys(case),
                                       **kw)

    def call(case, out, lse, splits=0):
        return attend(case, case.q, case.block_table, case.cache_seqlens, case.cu_seqlens_q, case.rel_logits, out,
                      lse, splits)

    def measure(name, steps, warmup, main_kernel, fp8=False):
        case = workload(name, device=dev)
        if fp8:  # the same workload over an E4M3 copy of its KV cache
            case.key_cache, case.value_cache = fp8_kv(case, *FP8_SCALES)
            torch.cuda.empty_cache()
        out = torch.empty_like(case.q)
        lse = torch.empty(case.T, case.H, dtype=torch.float32, device=dev)
        stream = torch.cuda.current_stream(dev)
        for _ in range(warmup):
            call(case, out, lse)
        torch.cuda.synchronize(dev)
        flags = ink.read_device_errors()
        if flags & ~ink.DEVERR["EMPTY_ROWS"]:
            raise RuntimeError(f"{name}: device error flags {flags:#x}")
        # the step time: `steps` calls back to back between two events, nothing recorded in between (an
        # event between two kernels would hold back the next kernel's programmatic early launch)
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        n0 = ink.launch_count()
        barrier()
        torch.cuda.synchronize(dev)
        with ClockSampler(local_rank) as clk:
            hold_stream(stream)
            start.record(stream)
            for k in range(steps):
                call(case, out, lse)
            end.record(stream)
            torch.cuda.synchronize(dev)
        barrier()
        launches = ink.launch_count() - n0
        ms = start.elapsed_time(end) / steps
        # then the same steps again with every kernel bracketed by its own pair of events on the launching
        # stream (the library's measurement hooks; this loop is the only thread calling it)
        kev = {kn: [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                    for _ in range(steps)] for kn in TIMED_KERNELS}
        for pairs_ in kev.values():  # torch creates the CUDA events on first record; the library needs real handles
            for a, b in pairs_:  # stop before start: a kernel the step does not launch reads as a negative time
                b.record(stream)
                a.record(stream)
        torch.cuda.synchronize(dev)
        for k in range(steps):
            for kn in TIMED_KERNELS:
                ink.set_timing_events(kn, kev[kn][k][0], kev[kn][k][1])
            call(case, out, lse)
        torch.cuda.synchronize(dev)
        for kn in TIMED_KERNELS:
            ink.set_timing_events(kn, None, None)

        def kernel_ms(kn):
            t = [a.elapsed_time(b) for a, b in kev[kn]]
            return sum(t) / steps if all(x > 0 for x in t) else 0.0

        per_kernel = {kn: kernel_ms(kn) for kn in TIMED_KERNELS}
        ms_max = max_over_ranks(ms, dev)
        kv, flops, pairs = work_of(case)
        if fp8:
            kv //= 2  # one byte per K / V element
        res = {"workload": name, "desc": WORKLOADS[name], "ms_per_step": ms_max, "kernel_ms": per_kernel[main_kernel],
               "per_kernel_ms": per_kernel, "kv_bytes": kv, "flops": flops, "launches": launches,
               "clocks": clk.summary(), "compulsory_bytes": total_bytes(case, fp8)}
        # end-to-end through the public API with host buffers: every step uploads its inputs from pinned
        # host memory and reads its out/lse back; step k + 1's upload runs while step k computes, and
        # the host waits for each step's result one step later (double-buffered on both sides)
        ref_out = out.to("cpu")  # every e2e step must reproduce the device-timed result bit for bit
        keys = ["q", "block_table", "cache_seqlens", "cu_seqlens_q"] + (["rel_logits"] if case.rel_logits is not None else [])
        pin = {k: getattr(case, k).to("cpu").pin_memory() for k in keys}
        h2d = sum(v.numel() * v.element_size() for v in pin.values())
        d2h = out.numel() * out.element_size() + lse.numel() * 4
        dev_in = [{k: getattr(case, k) for k in keys}, {k: getattr(case, k).clone() for k in keys}]
        dev_out = [(out, lse), (torch.empty_like(out), torch.empty_like(lse))]
        host_res = [(torch.empty(out.shape, dtype=out.dtype).pin_memory(), torch.empty(lse.shape).pin_memory())
                    for _ in range(2)]
        s_up = [torch.cuda.Stream(dev), torch.cuda.Stream(dev)]  # large inputs go up in two halves
        s_down = torch.cuda.Stream(dev)
        ev = lambda: torch.cuda.Event()
        up_done, comp_done, down_done = [ev(), ev()], [ev(), ev()], [ev(), ev()]

        def upload(b, after):
            if after is not None:  # the compute that last read buffer set b is done
                for su in s_up:
                    su.wait_event(after)
            for key, v in pin.items():
                dst = dev_in[b][key]
                n = v.numel()
                halves = [(0, n)] if n * v.element_size() < (256 << 20) else [(0, n // 2), (n // 2, n)]
                for i, (a, z) in enumerate(halves):
                    with torch.cuda.stream(s_up[i]):
                        dst.view(-1)[a:z].copy_(v.view(-1)[a:z], non_blocking=True)
            joined = ev()
            joined.record(s_up[1])
            s_up[0].wait_event(joined)
            up_done[b].record(s_up[0])

        def e2e_run(nsteps):
            upload(0, None)
            for k in range(nsteps):
                b = k % 2
                if k + 1 < nsteps:
                    upload(1 - b, comp_done[1 - b] if k >= 1 else None)
                stream.wait_event(up_done[b])
                if k >= 2:
                    stream.wait_event(down_done[b])  # its output buffers are read back already
                c = dev_in[b]
                attend(case, c["q"], c["block_table"], c["cache_seqlens"], c["cu_seqlens_q"], c.get("rel_logits"),
                       dev_out[b][0], dev_out[b][1])
                comp_done[b].record(stream)
                s_down.wait_event(comp_done[b])
                with torch.cuda.stream(s_down):
                    host_res[b][0].copy_(dev_out[b][0], non_blocking=True)
                    host_res[b][1].copy_(dev_out[b][1], non_blocking=True)
                down_done[b].record(s_down)
                if k >= 1:
                    down_done[1 - b].synchronize()  # the host has step k - 1's result
            down_done[(nsteps - 1) % 2].synchronize()

        e_steps = max(2, steps // 2)
        e2e_run(2)  # warm-up of the streams and events
        torch.cuda.synchronize(dev)
        barrier()
        t0 = time.perf_counter()
        e2e_run(e_steps)
        if not torch.equal(host_res[(e_steps - 1) % 2][0], ref_out):
            raise RuntimeError(f"{name}: the end-to-end result differs from the device-timed one")
        e2e_ms = (time.perf_counter() - t0) * 1e3 / e_steps
        res["e2e_ms"] = max_over_ranks(e2e_ms, dev)
        res["h2d_bytes"] = h2d
        res["d2h_bytes"] = d2h
        del case, out, lse, pin, dev_in, dev_out, host_res
        torch.cuda.empty_cache()
        return res

    def measure_append(steps, warmup, fp8=False):
        """KV append of one serving step: 4 x 8192 new tokens, Hkv 8, into 16-key pages (K and V); with fp8,
        quantized into an E4M3 cache."""
        case = build_case("kv_append", [8192] * 4, [8192] * 4, H=8, Hkv=8, E=0, seed=1100, device=dev)
        if fp8:
            case.key_cache = torch.zeros(case.key_cache.shape, dtype=torch.uint8, device=dev)
            case.value_cache = torch.zeros_like(case.key_cache)
            torch.cuda.empty_cache()

        def store():
            if fp8:
                ink.reshape_and_cache_fp8(key, value, case.key_cache, case.value_cache, slots,
                                          k_scale=FP8_SCALES[0], v_scale=FP8_SCALES[1])
            else:
                ink.reshape_and_cache(key, value, case.key_cache, case.value_cache, slots)

        g = torch.Generator(device=dev).manual_seed(1101)
        key = torch.randn(case.T, case.Hkv, 128, generator=g, device=dev).to(torch.bfloat16)
        value = torch.randn(case.T, case.Hkv, 128, generator=g, device=dev).to(torch.bfloat16)
        # slot of token j of request b: its logical position through the block table (all positions are new)
        pos = torch.arange(8192, device=dev)
        slots = torch.cat([case.block_table[b, pos // case.BS].long() * case.BS + pos % case.BS for b in range(4)])
        for _ in range(warmup):
            store()
        torch.cuda.synchronize(dev)
        kev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
        stream = torch.cuda.current_stream(dev)
        for a, b in kev:
            a.record(stream)
            b.record(stream)
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        n0 = ink.launch_count()
        barrier()
        torch.cuda.synchronize(dev)
        with ClockSampler(local_rank) as clk:
            hold_stream(stream)
            start.record(stream)
            for k in range(steps):
                ink.set_timing_events("append", kev[k][0], kev[k][1])
                store()
            end.record(stream)
            torch.cuda.synchronize(dev)
        ink.set_timing_events("append", None, None)
        barrier()
        ms = max_over_ranks(start.elapsed_time(end) / steps, dev)
        kms = sum(a.elapsed_time(b) for a, b in kev) / steps
        # K and V, read once (bf16) and written once (bf16, or one E4M3 byte per element)
        nbytes = 2 * case.T * case.Hkv * 128 * (2 + (1 if fp8 else 2))
        del case, key, value, slots
        torch.cuda.empty_cache()
        return {"ms_per_step": ms, "kernel_ms": kms, "bytes": nbytes, "launches": ink.launch_count() - n0,
                "clocks": clk.summary()}

    def measure_split_sweep(steps, warmup):
        """The long batch-1 decode (1,048,576 keys) timed at 16 / 32 / 64 / 128 splits and at the library's own
        choice (num_splits = 0): one step per call, CUDA events around the decode kernel and the whole step."""
        case = workload("long_decode", device=dev)
        out = torch.empty_like(case.q)
        lse = torch.empty(case.T, case.H, dtype=torch.float32, device=dev)
        stream = torch.cuda.current_stream(dev)
        kv, _, _ = work_of(case)
        res = {}
        for splits in (0, 16, 32, 64, 128):
            for _ in range(warmup):
                call(case, out, lse, splits)
            kev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                   for _ in range(steps)]
            for a, b in kev:
                a.record(stream)
                b.record(stream)
            start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            barrier()
            torch.cuda.synchronize(dev)
            hold_stream(stream)
            start.record(stream)
            for k in range(steps):  # the step time, nothing recorded between the kernels
                call(case, out, lse, splits)
            end.record(stream)
            torch.cuda.synchronize(dev)
            for k in range(steps):  # the decode kernel's own time
                ink.set_timing_events("decode", kev[k][0], kev[k][1])
                call(case, out, lse, splits)
            torch.cuda.synchronize(dev)
            ink.set_timing_events("decode", None, None)
            ms = max_over_ranks(start.elapsed_time(end) / steps, dev)
            kms = sum(a.elapsed_time(b) for a, b in kev) / steps
            key = "library" if splits == 0 else str(splits)
            res[key] = {"ms_per_step": round(ms, 4), "gbs": round(kv / (ms * 1e-3) / 1e9, 1),
                        "kernel_gbs": round(kv / (kms * 1e-3) / 1e9, 1)}
        res["library_splits"] = int(ink.num_splits(ink.Dims(case.T, case.B, case.H, case.Hkv, 128, case.num_blocks,
                                                            case.BS, case.block_table.shape[1]),
                                                   case.max_seqlen_q, max(case.kv_lens), -1, -1))
        del case, out, lse
        torch.cuda.empty_cache()
        return res

    def measure_graph(steps, warmup):
        """A small decode step (8 requests, Lk 4096, H 32, Hkv 8, E 1024) called through the API every step
        and replayed from one captured CUDA graph: the host cost per step that the graph removes."""
        case = build_case("graph_decode", [1] * 8, [4096] * 8, H=32, Hkv=8, E=1024, seed=1200, device=dev)
        out = torch.empty_like(case.q)
        lse = torch.empty(case.T, case.H, dtype=torch.float32, device=dev)
        dims = ink.Dims(case.T, case.B, case.H, case.Hkv, 128, case.num_blocks, case.BS,
                        case.block_table.shape[1])
        ws = torch.empty(ink.workspace_size(dims, case.max_seqlen_q, 0), dtype=torch.uint8, device=dev)

        def run():
            ink.ink_rel_attn_varlen(
                case.q, case.key_cache, case.value_cache, block_table=case.block_table,
                cache_seqlens=case.cache_seqlens, cu_seqlens_q=case.cu_seqlens_q, max_seqlen_q=case.max_seqlen_q,
                softmax_scale=case.softmax_scale, rel_extent=case.E, rel_logits=case.rel_logits, out=out, lse=lse,
                workspace=ws)

        side = torch.cuda.Stream(dev)
        side.wait_stream(torch.cuda.current_stream(dev))
        with torch.cuda.stream(side):
            for _ in range(3):
                run()
        torch.cuda.current_stream(dev).wait_stream(side)
        torch.cuda.synchronize(dev)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            run()
        torch.cuda.synchronize(dev)
        stream = torch.cuda.current_stream(dev)

        def timed(fn):
            for _ in range(warmup):
                fn()
            start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            barrier()
            torch.cuda.synchronize(dev)
            start.record(stream)  # no hold here: the host's own launch cost is part of what this compares
            for _ in range(steps):
                fn()
            end.record(stream)
            torch.cuda.synchronize(dev)
            return start.elapsed_time(end) / steps

        n0 = ink.launch_count()
        with ClockSampler(local_rank) as clk:  # both arms under the same sampler thread
            eager_ms = timed(run)
            per_step = (ink.launch_count() - n0) / (steps + warmup)
            want = out.clone()
            graph_ms = timed(graph.replay)
        if not torch.equal(out, want):
            raise RuntimeError("graph replay and direct call differ")
        kv, _, _ = work_of(case)
        del case, out, lse, ws, graph
        torch.cuda.empty_cache()
        return {"eager_ms": max_over_ranks(eager_ms, dev), "graph_ms": max_over_ranks(graph_ms, dev),
                "kv_bytes": kv, "launches_per_step": per_step, "clocks": clk.summary()}

    steps, warmup = args.steps, args.warmup
    headline = args.workload
    # head sizes 64 / 256: decodes run in the decode kernel, prefills in the head-size-generic kernel (timed
    # under the prefill's id)
    head_kernel = "prefill" if headline.startswith("chunked_prefill") else "decode"
    head = measure(headline, steps, warmup, head_kernel, fp8=args.kv_fp8)
    sec = {}
    skip = {x for x in args.skip.split(",") if x}
    if not args.headline_only:
        s2, w2 = max(3, steps // 2), max(3, warmup)
        jobs = [
            ("kv_append", lambda: measure_append(s2, w2)),
            ("kv_append_fp8", lambda: measure_append(s2, w2, fp8=True)),
            ("graph_decode", lambda: measure_graph(max(50, steps * 10), max(5, warmup))),
            ("long_decode_splits", lambda: measure_split_sweep(max(5, steps // 2), w2)),
            ("decode_batch_d64", lambda: measure("decode_batch_d64", s2, w2, "decode")),
            ("chunked_prefill_d64", lambda: measure("chunked_prefill_d64", s2, w2, "prefill")),
            ("decode_batch_d256", lambda: measure("decode_batch_d256", s2, w2, "decode")),
            ("chunked_prefill_d256", lambda: measure("chunked_prefill_d256", s2, w2, "prefill")),
            ("decode_batch_fp8", lambda: measure("decode_batch", s2, w2, "decode", fp8=True)),
            ("long_decode", lambda: measure("long_decode", s2, w2, "decode")),
            ("decode_batch", lambda: measure("decode_batch", s2, w2, "decode")),
            ("continuous_batch", lambda: measure("continuous_batch", s2, w2, "prefill")),
            ("chunked_prefill_fp8", lambda: measure("chunked_prefill", s2, w2, "prefill", fp8=True)),
            ("chunked_prefill", lambda: measure("chunked_prefill", s2, w2, "prefill")),
        ]
        for name, fn in jobs:  # this order is also the order of the "workloads" object: the prefill last
            if name in skip or name == headline + ("_fp8" if args.kv_fp8 else ""):
                continue
            try:
                sec[name] = fn()
            except Exception as exc:  # report, keep the headline line
                sec[name] = {"error": f"{type(exc).__name__}: {exc}"}

    def gbs(nbytes, ms):
        return nbytes / (ms * 1e-3) / 1e9

    def tfs(flops, ms):
        return flops / (ms * 1e-3) / 1e12

    def roof_decode(r, name, fp8=False, kernel="ink_decode_kernel"):
        ach = gbs(r["kv_bytes"], r["kernel_ms"])
        return {"bound": "hbm", "achieved": round(ach, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": round(ach / peaks["hbm_gbs"], 4), "frac_of_8000": round(ach / 8000.0, 4),
                "traffic": traffic_of(kernel, name),
                "peak_source": peaks["source"], "kernel": kernel + (" (E4M3 cache)" if fp8 else "")}

    # every prefill workload measured here has unsplit units, which run in the 2-SM pair kernel
    def roof_prefill(r, name, fp8=False, kernel="ink_prefill_pair_kernel"):
        ach = tfs(r["flops"], r["kernel_ms"])
        return {"bound": "tensor", "achieved": round(ach, 2), "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                "frac": round(ach / peaks["bf16_tflops"], 4), "traffic": traffic_of(kernel, name),
                "peak_source": peaks["source"], "kernel": kernel + (" (E4M3 cache, staged)" if fp8 else "")}

    def step_bound(r):
        """The step's own floor: its flops at the tensor peak or its compulsory bytes at the HBM peak."""
        t = max(r["flops"] / (peaks["bf16_tflops"] * 1e12), r["compulsory_bytes"] / (peaks["hbm_gbs"] * 1e9))
        return {"bound_ms": round(t * 1e3, 4), "frac": round(t * 1e3 / r["ms_per_step"], 4),
                "compulsory_bytes": r["compulsory_bytes"], "flops": r["flops"]}

    def kernels_of(r):
        return {k: round(v, 4) for k, v in r["per_kernel_ms"].items() if v > 0}

    def clk_of(r):
        c = r["clocks"]
        return {"sm_mhz": c["sm_mhz"], "sm_max_mhz": c["sm_max_mhz"], "reasons": c["reasons"]}

    if rank != 0:
        return
    fp8_head = args.kv_fp8
    hkw = {"kernel": "ink_generic_kernel"} if headline in HEADDIM and headline.startswith("chunked") else {}
    if headline.startswith("chunked_prefill"):
        unit = "TFLOP/s"
        value = job_throughput(head["flops"], world, head["ms_per_step"]) / 1e12
        e2e = job_throughput(head["flops"], world, head["e2e_ms"]) / 1e12
        roof = roof_prefill(head, headline + ("_fp8" if fp8_head else ""), fp8_head, **hkw)
    else:
        unit = "GB/s"
        value = job_throughput(head["kv_bytes"], world, head["ms_per_step"]) / 1e9
        e2e = job_throughput(head["kv_bytes"], world, head["e2e_ms"]) / 1e9
        roof = roof_decode(head, headline + ("_fp8" if fp8_head else ""), fp8_head, **hkw)
    cpu_secs = args.cpu_seconds_each
    workloads_out = {}
    for name, r in sec.items():
        if "error" in r:
            workloads_out[name] = r
            continue
        if name in ("kv_append", "kv_append_fp8"):
            fp8 = name == "kv_append_fp8"
            ach = gbs(r["bytes"], r["kernel_ms"])
            kern = "ink_append_fp8_kernel" if fp8 else "ink_append_kernel"
            workloads_out[name] = {
                "metric": "KV append GB/s (K and V read and written)", "ms_per_step": round(r["ms_per_step"], 4),
                "value": round(gbs(r["bytes"], r["ms_per_step"]), 1), "unit": "GB/s",
                "desc": "4 x 8192 new tokens, Hkv 8, 16-key pages" + (", into an E4M3 cache" if fp8 else ""),
                "gpu_launches": r["launches"], "clocks": clk_of(r),
                "roofline": {"bound": "hbm", "achieved": round(ach, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                             "frac": round(ach / peaks["hbm_gbs"], 4), "traffic": traffic_of(kern, name),
                             "peak_source": peaks["source"], "kernel": kern}}
            continue
        if name == "long_decode_splits":
            workloads_out[name] = {"metric": "long decode KV-read GB/s by split count (step, and decode kernel)",
                                   "unit": "GB/s", **r}
            continue
        if name == "graph_decode":
            workloads_out[name] = {
                "metric": "decode step time, direct API call vs CUDA graph replay (ms)",
                "desc": "8 decodes, Lk 4096, H 32, Hkv 8, E 1024 (KV 134 MB, not flushed)",
                "eager_ms": round(r["eager_ms"], 4), "graph_ms": round(r["graph_ms"], 4),
                "graph_kv_gbs": round(gbs(r["kv_bytes"], r["graph_ms"]), 1),
                "gpu_launches_per_step": r["launches_per_step"], "clocks": clk_of(r)}
            continue
        fp8 = name.endswith("_fp8")
        base = name[:-4] if fp8 else name
        kern = "ink_generic_kernel" if base in HEADDIM and base.startswith("chunked") else None
        kw = {"kernel": kern} if kern else {}
        entry = {"ms_per_step": round(r["ms_per_step"], 4), "kernel_ms": kernels_of(r),
                 "e2e_ms": round(r["e2e_ms"], 4), "gpu_launches": r["launches"], "clocks": clk_of(r)}
        if base.startswith("chunked_prefill"):
            entry.update({"metric": "prefill TFLOP/s (visible pairs)", "value": round(tfs(r["flops"], r["ms_per_step"]), 2),
                          "unit": "TFLOP/s", "roofline": roof_prefill(r, name, fp8, **kw), "step_roofline": step_bound(r)})
        elif base == "continuous_batch":
            entry.update({"metric": "decode KV-read GB/s + prefill TFLOP/s over the step",
                          "decode_gbs": round(gbs(r["kv_bytes"], r["ms_per_step"]), 1),
                          "prefill_tflops": round(tfs(r["flops"], r["ms_per_step"]), 2),
                          "step_roofline": step_bound(r),
                          "roofline": roof_prefill(r, name),
                          "roofline_decode": roof_decode({**r, "kernel_ms": r["per_kernel_ms"]["decode"]}, name)})
        else:
            entry.update({"metric": "decode KV-read GB/s" + (" (E4M3 cache bytes)" if fp8 else ""),
                          "value": round(gbs(r["kv_bytes"], r["ms_per_step"]), 1), "unit": "GB/s",
                          "roofline": roof_decode(r, name, fp8, **kw)})
        if not args.no_cpu_baseline:
            try:
                entry["cpu_baseline"] = cpu_baseline(base, cpu_secs, fp8=fp8, short=True)
            except Exception as exc:
                entry["cpu_baseline"] = {"error": f"{type(exc).__name__}: {exc}"}
        workloads_out[name] = entry
    cpu = None
    if not args.no_cpu_baseline:
        cpu = cpu_baseline(headline, args.cpu_seconds, fp8=fp8_head)
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": unit, "n_gpus": world, "steps": steps,
        "warmup": warmup, "ms_per_step": round(head["ms_per_step"], 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded; see workloads/)",
        "config": {"workload": headline, "desc": WORKLOADS[headline], "parallelism": f"replicas x{world}",
                   "kv_cache": "e4m3" if fp8_head else "bf16",
                   "l2": "inputs larger than L2 (no flush)"},
        "roofline": roof,
        "e2e": {"value": round(e2e, 2), "unit": unit, "h2d_bytes_per_step": head["h2d_bytes"],
                "d2h_bytes_per_step": head["d2h_bytes"], "ms_per_step": round(head["e2e_ms"], 4),
                "note": "q, rel_logits and metadata copied from pinned host memory and out/lse read back "
                        "every step (the next step's upload overlaps this step's compute); the paged KV cache is "
                        "resident state in HBM"},
        "gpu_launches": head["launches"],
        "kernel_ms": kernels_of(head),
        "clocks": head["clocks"],
        "cpu_baseline": cpu,
        "workloads": workloads_out,
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------------- oracle arm

def _row_pairs(case, lq, lk, i):
    """Visible keys of query row i of a request with lq queries and lk keys."""
    qa = i + lk - lq
    lo = max(0, qa - case.window_left) if case.window_left >= 0 else 0
    hi = lk - 1
    if case.causal:
        hi = min(hi, qa)
    if case.window_right >= 0:
        hi = min(hi, qa + case.window_right)
    return max(0, hi - lo + 1)


def cpu_baseline(name, seconds, fp8=False, short=False, case=None):
    """The fp64 oracle, as it stands, on the host cores over a bounded sample of the workload (about
    `seconds` of CPU work), in the GPU line's own units.

    Decode-shaped requests: whole requests (all heads), in order, pass after pass -> KV GB/s.
    Prefill-shaped requests: stratified rows -- batches of 64 (token, head) rows drawn uniformly from each
    prefill request in turn (seeded) -> TFLOP/s on the rows' visible pairs.  A mix gets half the time for
    each and also reports the step time those two rates imply.  fp8: the same workload over the E4M3
    cache the GPU line reads, through the oracle's FP8 entry.  `case`: the workload already built on the
    host (the reference arm times several samples of one build)."""
    import numpy as np

    import oracle
    from workloads import fp8_kv, workload

    if case is None:
        case = workload(name, device="cpu")
    oracle.build()
    threads = oracle.threads()
    kw = case.oracle_kwargs()
    G = case.H // case.Hkv
    kc, vc = case.key_cache, case.value_cache
    if fp8:
        kc, vc = fp8_kv(case, *FP8_SCALES)
    cu = case.cu_seqlens_q.tolist()
    dec = [b for b in range(case.B) if case.q_lens[b] * G <= 16 and case.q_lens[b] > 0]
    pre = [b for b in range(case.B) if case.q_lens[b] * G > 16]

    def run(rows):
        if fp8:
            oracle.attention_fp8kv(case.q, kc, vc, case.block_table, case.cache_seqlens, case.cu_seqlens_q,
                                   k_scale=FP8_SCALES[0], v_scale=FP8_SCALES[1], rows=rows, **kw)
        else:
            oracle.attention(case.q, kc, vc, case.block_table, case.cache_seqlens, case.cu_seqlens_q, rows=rows, **kw)

    budget = seconds / (2 if dec and pre else 1)
    el = 1 if fp8 else 2
    dec_bytes, dec_s, dec_reqs = 0, 0.0, 0
    if dec:
        t0 = time.perf_counter()
        while time.perf_counter() - t0 < budget:
            for b in dec:
                run(np.arange(cu[b] * case.H, cu[b + 1] * case.H, dtype=np.int64))
                lq, lk = case.q_lens[b], case.kv_lens[b]
                keys = max(_row_pairs(case, lq, lk, i) for i in range(lq))  # the union of the rows' ranges
                dec_bytes += keys * case.Hkv * case.D * 2 * el
                dec_reqs += 1
                if time.perf_counter() - t0 >= budget:
                    break
        dec_s = time.perf_counter() - t0
    pre_flops, pre_s, pre_rows = 0, 0.0, 0
    if pre:
        g = np.random.default_rng(17)
        t0 = time.perf_counter()
        k = 0
        while time.perf_counter() - t0 < budget:
            b = pre[k % len(pre)]
            k += 1
            lq, lk = case.q_lens[b], case.kv_lens[b]
            rows = np.unique(g.integers(cu[b] * case.H, cu[b + 1] * case.H, size=64)).astype(np.int64)
            run(rows)
            pre_flops += sum(4 * case.D * _row_pairs(case, lq, lk, int(r) // case.H - cu[b]) for r in rows)
            pre_rows += rows.size
        pre_s = time.perf_counter() - t0
    cpu_name = ""
    try:
        with open("/proc/cpuinfo") as f:
            for ln in f:
                if ln.lower().startswith(("model name", "cpu part")):
                    cpu_name = ln.split(":", 1)[1].strip()
                    break
    except Exception:
        pass
    res = {"kind": "oracle", "cores": threads}
    parts = []
    if dec:
        parts.append(f"{dec_reqs} whole decode requests ({dec_s:.1f} s)")
    if pre:
        parts.append(f"{pre_rows} stratified prefill rows ({pre_s:.1f} s)")
    res["sample"] = f"{name}{' (E4M3 cache)' if fp8 else ''}: " + ", ".join(parts)
    dec_rate = dec_bytes / dec_s if dec_s > 0 else 0.0
    pre_rate = pre_flops / pre_s if pre_s > 0 else 0.0
    if dec and pre:
        kv, flops, _ = work_of(case)
        step_s = kv * el / 2 / dec_rate + flops / pre_rate
        res.update({"value": round(step_s * 1e3, 3), "unit": "ms per step (extrapolated)",
                    "decode_gbs": round(dec_rate / 1e9, 6), "prefill_tflops": round(pre_rate / 1e12, 6)})
    elif pre:
        res.update({"value": round(pre_rate / 1e12, 6), "unit": "TFLOP/s"})
    else:
        res.update({"value": round(dec_rate / 1e9, 6), "unit": "GB/s"})
    if not short:
        res["seconds"] = round(dec_s + pre_s, 2)
        res["cpu"] = cpu_name
    return res


def run_reference(args, rank, world):
    if rank != 0:
        return
    from workloads import HEADDIM_WORKLOADS, PROFILE_WORKLOADS, WORKLOADS, workload

    WORKLOADS = {**WORKLOADS, **PROFILE_WORKLOADS, **HEADDIM_WORKLOADS}
    case = workload(args.workload, device="cpu")
    times = []
    val = None
    for k in range(args.warmup + args.steps):
        r = cpu_baseline(args.workload, args.cpu_seconds / max(1, args.steps), fp8=args.kv_fp8, case=case)
        if k >= args.warmup:
            times.append(r)
    vals = [r["value"] for r in times]
    val = statistics.median(vals)
    last = times[-1]
    line = {
        "impl": "reference", "metric": METRIC, "value": val, "unit": last["unit"], "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "higher_is_better": not last["unit"].startswith("ms"),
        "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded; see workloads/)",
        "config": {"workload": args.workload, "desc": WORKLOADS[args.workload], "parallelism": "host cores",
                   "kv_cache": "e4m3" if args.kv_fp8 else "bf16"},
        "cpu_baseline": {"value": val, "unit": last["unit"], "cores": last["cores"], "kind": "oracle",
                         "sample": last["sample"]},
        "e2e": {"value": val, "unit": last["unit"], "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------------- main

def free_port() -> int:
    import socket

    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as sk:
        sk.bind(("127.0.0.1", 0))
        return sk.getsockname()[1]


def relaunch_cmd(gpus: int, argv, port: int):
    """The command that runs this benchmark as `gpus` ranks on one node (rendezvous on 127.0.0.1)."""
    return [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", f"--nproc-per-node={gpus}",
            "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.abspath(__file__), *argv]


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=HEADLINE,
                    choices=["decode_batch", "chunked_prefill", "long_decode", "continuous_batch",
                             "decode_batch_quarter", "chunked_prefill_quarter", "decode_batch_d64",
                             "chunked_prefill_d64", "decode_batch_d256", "chunked_prefill_d256"])
    ap.add_argument("--headline-only", action="store_true")
    ap.add_argument("--kv-fp8", action="store_true",
                    help="run the headline workload over an E4M3 copy of its KV cache")
    ap.add_argument("--skip", default="", help="comma-separated secondary workloads to leave out")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=15.0, help="oracle time for the headline's cpu_baseline")
    ap.add_argument("--cpu-seconds-each", type=float, default=6.0,
                    help="oracle time for each other workload's cpu_baseline")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.gpus > 1 and "WORLD_SIZE" not in os.environ:
        # one process per GPU: start the ranks under torch.distributed.run and wait for them
        sys.exit(subprocess.call(relaunch_cmd(args.gpus, sys.argv[1:], free_port())))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if world != args.gpus and "WORLD_SIZE" in os.environ:
        raise SystemExit(f"--gpus {args.gpus} but WORLD_SIZE={world}")
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    if world > 1:
        import torch
        import torch.distributed as dist

        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl")
    run_ours(args, rank, world, local_rank)
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()


if __name__ == "__main__":
    main()
