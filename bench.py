#!/usr/bin/env python3
"""Benchmark of the attention-over-KV-cache hot path on GB300.

One step = one request on every layer of the workload: the prompt prefilled in
chunks (prefill_step per chunk: the chunk's store, then the attention; for q8_0 each
chunk adds its own positions to the layer's fp16 copy, copy_valid = pos0), the decode steps
(decode_step per token: the split pass stores the token and attends, then the
combine; the loop captured once in a CUDA graph), then the cache state serialised from the head-major cache
(kv_state_get) and restored into a layer-major cache (kv_state_set).

`value` is the whole request's throughput per attention layer: (prompt +
generated tokens) x layers / step time, summed over ranks.  The phases are
reported beside it (prefill tok/s, decode tok/s, state GB/s).  The roofline
object is for the dominant kernel, the prefill attention, whose algorithmic
work per chunk is 4 * H_q * D * sum_t (t + 1) flops (causal half only).

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
       python bench.py --impl reference ...   (the CPU oracle, bounded sample)
Multi-GPU (torchrun): every rank runs an independent replica (weak scaling).
"""

import argparse
import gc
import json
import os
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import seeded_inputs as si  # noqa: E402

METRIC = "prefill tok/s and decode tok/s per attention layer; % tensor/HBM roofline"
DEFAULT_WORKLOAD = "q8_0_58k"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


# --------------------------------------------------------------------------- helpers
def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


def prefill_flops(w, chunks=None):
    """Algorithmic flops of prefill attention: 4*H_q*D*(t+1) per query row t (QK^T and PV, causal)."""
    out = []
    for p, c in (chunks or w.chunks()):
        rows = c * p + c * (c + 1) // 2
        out.append(4.0 * w.n_head_q * w.head_dim * rows)
    return out


# DRAM traffic per launch from ncu captures (dram__bytes_read.sum + dram__bytes_write.sum), each valid
# only for the kernel sources it was taken on (first 16 hex digits of the SHA-256 of each listed file
# under csrc/); any change to one of them makes the bench report null for that kernel instead.
# Entries: kernel -> {"sources": {file: sha16}, workload: (bytes per call, what was captured)}.
TRAFFIC = {
    # the step's 29 prefill_step calls (the front kernel, the attention, the split merge), mean per call
    "prefill": {"sources": {"prefill.cu": "9b2cbe58ac7ea91d", "quant.cuh": "b2cae791609f3353"},
                "q8_0_58k": (415433030, "mean per call over the 29 prefill_step calls of one step (all three kernels)")},
    "append_chunk": {"sources": {"append.cu": "2302d1cd16863358", "quant.cuh": "b2cae791609f3353"},
                     "q8_0_58k": (8412364, "one 2048-token chunk append (writes still in L2 at the launch end)")},
    "append_prompt": {"sources": {"append.cu": "2302d1cd16863358", "quant.cuh": "b2cae791609f3353"},
                      "q8_0_58k": (330861952, "the 58,300-token prompt in one append")},
    "decode_attn": {"sources": {"decode.cu": "d280bfd9f3fbd2ec"},
                    "q8_0_58k": (128035097, "split pass + combine at position 58,555")},
    "decode_step": {"sources": {"decode.cu": "d280bfd9f3fbd2ec", "quant.cuh": "b2cae791609f3353"},
                    "q8_0_58k": (128019635, "split pass storing the token + combine at position 58,555")},
    "state_pack": {"sources": {"state.cu": "0b844f534c53c1b8"},
                   "q8_0_58k": (201804441, "pack of 58,556 tokens (the kernel writes the header)")},
    "state_unpack": {"sources": {"state.cu": "0b844f534c53c1b8"},
                     "q8_0_58k": (202305715, "unpack of 58,556 tokens")},
}


def _source_sha16(name):
    import hashlib
    src = os.path.join(ROOT, "decode_attention_kv_cache_gb300", "csrc", name)
    try:
        return hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
    except OSError:
        return None


def recorded_traffic(kernel, workload):
    """(bytes per call, note) from the ncu record, or (None, why) when there is none for the current
    sources."""
    rec = TRAFFIC.get(kernel)
    if rec is None or workload not in rec:
        return None, "no ncu record for this workload"
    for name, sha in rec["sources"].items():
        if _source_sha16(name) != sha:
            return None, "%s changed since the ncu capture" % name
    return rec[workload]


def prefill_split_keys(n_ctx):
    """Keys per prefill split as the library chooses them: about a fifth of the cache in steps of
    2048 keys, at least 4096, and at most 64 splits (in 256-key tiles)."""
    keys = max((n_ctx // 10 + 512) // 1024 * 2048, 4096)
    return max(keys, -(-n_ctx // (64 * 256)) * 256)


def cache_bytes_per_token(w):
    if w.cache == "q8_0":
        return 2 * w.n_head_kv * w.head_dim * 34 // 32
    return 2 * w.n_head_kv * w.head_dim * 2


class ClockSampler:
    """nvidia-smi samples (200 ms) during the timed region."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.idx = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.idx), "--query-gpu=" + self.FIELDS, "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except (OSError, ValueError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    smax.append(float(parts[2]))
                except ValueError:
                    continue
                for n, v in zip(names, parts[5:9]):
                    if v.lower() == "active":
                        reasons.add(n)
        os.unlink(self.path)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        busy = [s for s in sm if s > 0.5 * max(sm)] or sm
        return {"sm_mhz": float(np.median(busy)), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm)}


# --------------------------------------------------------------------------- distributed
def dist_init():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend=backend)
    return rank, world, local


def dist_barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def dist_max(x, world):
    if world <= 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if torch.cuda.is_available() and dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([float(x)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# --------------------------------------------------------------------------- GPU arm
class GpuRequest:
    """Inputs resident in HBM (and pinned host copies for the end-to-end run), two caches, output buffers.

    Multi-layer stacks draw their inputs on the device (seeded_inputs.layer_qkv_device) and reuse one
    prefill/decode output buffer for every layer (the layers of the attention-only stack share no data).
    """

    def __init__(self, kvc, w, device, seed_offset=0, device_inputs=None, host_copies=True, extra_rows=0,
                 inputs=None):
        import torch
        self.torch, self.kvc, self.w, self.dev = torch, kvc, w, device
        wl = w if seed_offset == 0 else si.Workload(**{**w.__dict__, "seed": w.seed + 1000 * seed_offset})
        self.wl = wl
        self.device_inputs = (w.n_layer > 1) if device_inputs is None else device_inputs
        n_rows = w.n_tokens + extra_rows
        self.host, self.dev_in = [], []
        for layer in range(w.n_layer):
            if inputs is not None:           # caller-provided device tensors (one tuple per layer)
                self.dev_in.append(inputs[layer])
            elif self.device_inputs:
                dq, dk, dv = si.layer_qkv_device(wl, layer, device, n_rows=n_rows)
                self.dev_in.append((dq, dk, dv))
                if host_copies:
                    self.host.append(tuple(t.cpu().pin_memory() for t in (dq, dk, dv)))
            else:
                q, k, v = si.layer_qkv(wl, layer, n_rows=n_rows)
                hq, hk, hv = (t.pin_memory() for t in (q, k, v))
                if host_copies:
                    self.host.append((hq, hk, hv))
                self.dev_in.append(tuple(t.to(device) for t in (hq, hk, hv)))
        self.src = kvc.KVCache(w.n_layer, w.n_ctx, w.n_head_kv, w.head_dim, w.cache, "head_major", device)
        self.dst = kvc.KVCache(w.n_layer, w.n_ctx, w.n_head_kv, w.head_dim, w.cache, "layer_major", device)
        n_out = w.n_layer if w.n_layer == 1 else 1
        self.out_p = torch.empty(n_out, w.n_prompt, w.n_head_q, w.head_dim, device=device)
        self.out_d = torch.empty(n_out, max(w.n_decode, 1), w.n_head_q, w.head_dim, device=device)
        self.scratch = torch.empty(self.src.scratch_bytes(w.n_head_q), dtype=torch.uint8, device=device)
        self.pscratch = self.src.prefill_scratch(w.n_head_q, w.chunk if w.chunk > 0 else w.n_prompt)
        self.state = torch.empty(self.src.state_size(w.n_tokens), dtype=torch.uint8, device=device)
        if host_copies:
            self.host_out_p = torch.empty(self.out_p.shape, dtype=torch.float32).pin_memory()
            self.host_out_d = torch.empty(self.out_d.shape, dtype=torch.float32).pin_memory()
            self.host_state = torch.empty(self.state.shape, dtype=torch.uint8).pin_memory()
        self.chunks = w.chunks()
        self.graphs = []
        self.flops = prefill_flops(w)

    def out_slot(self, layer):
        return layer if self.w.n_layer == 1 else 0

    def launches_per_step(self):
        """Kernels one step launches: per chunk two (prefill_step: the chunk's store, with its part of the
        fp16 copy for q8_0, then the attention) plus the split merge when the chunk's last row reaches past the
        first key split; per decode step the split pass (which stores the token) and the combine; the
        state pack and unpack."""
        w = self.w
        keys = prefill_split_keys(w.n_ctx)
        merges = sum(1 for p, c in self.chunks if p + c - 1 >= keys)
        return w.n_layer * (2 * len(self.chunks) + merges + 2 * w.n_decode) + 2

    def _decode_loop(self, layer):
        kvc, w = self.kvc, self.w
        q, k, v = self.dev_in[layer]
        for i in range(w.n_decode):
            pos = w.n_prompt + i
            kvc.decode_step(self.src, layer, pos, q[pos], k[pos], v[pos], out=self.out_d[self.out_slot(layer), i],
                            scratch=self.scratch)

    def attention_only(self):
        """Every chunk's prefill_step of every layer, back to back, as the step issues them (the
        roofline's timing of the attention with no event between two launches; each call also stores
        its chunk again, the same bytes, and for q8_0 writes the chunk's part of the fp16 copy the
        attention reads)."""
        kvc, w = self.kvc, self.w
        for layer in range(w.n_layer):
            q, k, v = self.dev_in[layer]
            for p, c in self.chunks:
                kvc.prefill_step(self.src, layer, p, q[p:p + c], k[p:p + c], v[p:p + c],
                                 out=self.out_p[self.out_slot(layer), p:p + c], scratch=self.pscratch, copy_valid=p)

    def capture(self):
        """Capture each layer's decode loop in a CUDA graph (after one eager run)."""
        torch = self.torch
        for layer in range(self.w.n_layer):
            self._decode_loop(layer)
        torch.cuda.synchronize()
        self.graphs = []
        for layer in range(self.w.n_layer):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                self._decode_loop(layer)
            self.graphs.append(g)
        torch.cuda.synchronize()

    def step(self, ev=None, on_layer=None):
        """One request on every layer.  ev: dict of event lists to record phase/launch times;
        on_layer(layer): called after each layer's prefill and decode (checks only, never timed)."""
        kvc, w, torch = self.kvc, self.w, self.torch
        E = torch.cuda.Event
        for layer in range(w.n_layer):
            q, k, v = self.dev_in[layer]
            if ev is not None:
                e0 = E(enable_timing=True); e0.record(); ev["prefill"].append([e0])
            for ci, (p, c) in enumerate(self.chunks):
                if ev is not None:
                    a = E(enable_timing=True); a.record()
                kvc.prefill_step(self.src, layer, p, q[p:p + c], k[p:p + c], v[p:p + c],
                                 out=self.out_p[self.out_slot(layer), p:p + c], scratch=self.pscratch, copy_valid=p)
                if ev is not None:
                    b = E(enable_timing=True); b.record(); ev["attn"].append((a, b, self.flops[ci]))
            if ev is not None:
                e1 = E(enable_timing=True); e1.record(); ev["prefill"][-1].append(e1)
            if w.n_decode:
                if self.graphs:
                    self.graphs[layer].replay()
                else:
                    self._decode_loop(layer)
            if ev is not None:
                e2 = E(enable_timing=True); e2.record(); ev["decode"].append((e1, e2))
            if on_layer is not None:
                on_layer(layer)
        if ev is not None:
            e3 = E(enable_timing=True); e3.record()
        kvc.kv_state_get(self.src, w.n_tokens, dst=self.state)
        n = kvc.kv_state_set(self.dst, self.state)
        assert n == w.n_tokens
        if ev is not None:
            e4 = E(enable_timing=True); e4.record(); ev["state"].append((e3, e4))

    def h2d(self):
        for (hq, hk, hv), (dq, dk, dv) in zip(self.host, self.dev_in):
            # host inputs hold exactly the request's rows

            dq.copy_(hq, non_blocking=True); dk.copy_(hk, non_blocking=True); dv.copy_(hv, non_blocking=True)

    def d2h(self):
        self.host_out_p.copy_(self.out_p, non_blocking=True)
        self.host_out_d.copy_(self.out_d, non_blocking=True)
        self.host_state.copy_(self.state, non_blocking=True)

    def io_bytes(self):
        h2d = sum(t.numel() * t.element_size() for trip in self.host for t in trip)
        d2h = sum(t.numel() * t.element_size() for t in (self.host_out_p, self.host_out_d, self.host_state))
        return h2d, d2h


def l2_flush(torch, buf):
    buf.add_(1)


def workload_config(w):
    """The bench line's config: the workload by name and shape (both arms print the same)."""
    return {"workload": w.name, "n_layer": w.n_layer, "n_head_q": w.n_head_q, "n_head_kv": w.n_head_kv,
            "head_dim": w.head_dim, "cache": w.cache, "in_dtype": w.in_dtype, "n_ctx": w.n_ctx,
            "n_prompt": w.n_prompt, "chunk": w.chunk, "n_decode": w.n_decode,
            "parallelism": "replicas (one independent layer stack per GPU)",
            "l2": "flushed (256 MiB write) before each timed step", "decode_loop": "CUDA graph"}


def run_gpu(args, rank, world, local):
    import torch
    import decode_attention_kv_cache_gb300 as kvc

    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    w = si.WORKLOADS[args.workload]
    req = GpuRequest(kvc, w, device, seed_offset=rank)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=device)  # 256 MiB > 129 MB L2
    req.step()
    if w.n_decode:
        req.capture()
    for _ in range(args.warmup):
        l2_flush(torch, flush)
        req.step()
    torch.cuda.synchronize()
    assert kvc.kvc_device_status() == 0

    # ---- timed region: K steps, L2 flushed before each (outside the step's events).  The steps
    # that give `value` carry events only at their boundaries, so every kernel follows the previous
    # one in the stream exactly as in use (an event between two launches would stand between a
    # kernel and its programmatic dependent); K more steps, with events around every phase and
    # every attention call, give the phase times and the roofline.
    ev = {"prefill": [], "attn": [], "decode": [], "state": []}
    steps = []
    clocks = ClockSampler(local)
    clocks.start()
    dist_barrier(world)
    torch.cuda.synchronize()
    # no garbage-collector pass on the host while it issues the timed steps (a pass that stalls the host
    # mid-step leaves the GPU idle inside the step's events)
    gc.collect()
    gc.disable()
    torch.cuda.nvtx.range_push("kvc_timed")
    for _ in range(args.steps):
        l2_flush(torch, flush)
        s0 = torch.cuda.Event(enable_timing=True); s0.record()
        req.step()
        s1 = torch.cuda.Event(enable_timing=True); s1.record()
        steps.append((s0, s1))
    torch.cuda.synchronize()
    torch.cuda.nvtx.range_pop()
    dist_barrier(world)
    for _ in range(args.steps):
        l2_flush(torch, flush)
        req.step(ev)
    chain = []
    for _ in range(args.steps):
        l2_flush(torch, flush)
        a = torch.cuda.Event(enable_timing=True); a.record()
        req.attention_only()
        b = torch.cuda.Event(enable_timing=True); b.record()
        chain.append((a, b))
    torch.cuda.synchronize()
    gc.enable()
    clk = clocks.stop()
    step_ms = [a.elapsed_time(b) for a, b in steps]
    total_ms = dist_max(sum(step_ms), world)
    attn_ms = sum(a.elapsed_time(b) for a, b, _ in ev["attn"])   # each call between its own events
    chain_ms = sum(a.elapsed_time(b) for a, b in chain)             # the calls back to back
    attn_flops = sum(f for _, _, f in ev["attn"])
    n_attn = len(ev["attn"])
    prefill_ms = sum(x[0].elapsed_time(x[1]) for x in ev["prefill"])
    decode_ms = sum(a.elapsed_time(b) for a, b in ev["decode"])
    state_ms = sum(a.elapsed_time(b) for a, b in ev["state"])
    K = args.steps
    tokens = (w.n_prompt + w.n_decode) * w.n_layer
    value = tokens * world * K / (total_ms / 1e3)

    # ---- end to end: host buffers, copies inside the timed region
    e2e = None
    if not args.no_e2e:
        e2e = end_to_end(kvc, torch, w, req, device, rank, world, K, flush, local)
    assert kvc.kvc_device_status() == 0

    peaks, peak_src = load_peaks()
    traffic, traffic_launch = recorded_traffic("prefill", w.name)
    achieved = attn_flops / (chain_ms / 1e3) / 1e12
    peak = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    roof = {"kernel": "prefill attention (prefill_step; tcgen05 f16 x f16 -> f32)", "bound": "tensor",
            "achieved": achieved, "peak": peak, "unit": "TFLOP/s", "frac": achieved / peak,
            "peak_source": "%s dense bf16 burst (f16 runs at the bf16 rate)" % peak_src,
            "traffic": traffic, "traffic_launch": traffic_launch, "launches": n_attn // K,
            "avg_launch_ms": chain_ms / n_attn,
            "timed": "the step's prefill_step calls back to back (each: the chunk's store, for q8_0 with "
                     "the chunk's part of the fp16 copy, the attention and the split merge; L2 flushed before "
                     "each pass), CUDA events at the ends of each pass",
            "achieved_calls_between_events": attn_flops / (attn_ms / 1e3) / 1e12,
            "algorithmic_flops_per_step": attn_flops / K}
    bt = cache_bytes_per_token(w)
    dec_bytes = sum(w.n_layer * ((w.n_prompt + i + 1) * bt + w.n_head_q * w.head_dim * (2 + 4)
                                 + 2 * w.n_head_kv * w.head_dim * 2 + bt) for i in range(w.n_decode))
    state_bytes = 2 * 2 * req.state.numel()
    phases = {
        "prefill_tok_s": w.n_prompt * w.n_layer * K / (prefill_ms / 1e3),
        "prefill_ms_per_step": prefill_ms / K,
        "prefill_attn_ms_per_step": attn_ms / K,
        "prefill_attn_back_to_back_ms_per_step": chain_ms / K,
        "decode_tok_s": (w.n_decode * w.n_layer * K / (decode_ms / 1e3)) if w.n_decode else None,
        "decode_ms_per_step": decode_ms / K,
        "decode_algorithmic_GB_s": (dec_bytes * K / (decode_ms / 1e3) / 1e9) if w.n_decode else None,
        "decode_l2": "warm: the steps run back to back in a CUDA graph, so part of the cache stays in L2 "
                     "between steps (the cold figure is kernels.decode_step)",
        "state_ms_per_step": state_ms / K,
        "state_algorithmic_GB_s": state_bytes * K / (state_ms / 1e3) / 1e9,
    }
    line = {
        "metric": METRIC, "value": value, "unit": "tok/s", "n_gpus": world, "steps": K, "warmup": args.warmup,
        "ms_per_step": total_ms / K, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f16xf16->f32 (tensor), f32 softmax; int8/f16 cache", "data": "synthetic (seeded N(0,1))",
        "config": workload_config(w),
        "phases": phases, "roofline": roof, "e2e": e2e, "gpu_launches": req.launches_per_step() * K,
        "timing": "value: K steps with events at the step boundaries only; phases: K more steps with "
                  "events around each phase and each attention call; roofline: K passes of the attention "
                  "calls alone",
        "clocks": clk,
    }
    if w.n_layer == 1:
        hbm = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
        gc.collect()
        gc.disable()
        try:
            line["kernels"] = kernel_rooflines(kvc, torch, w, req, flush, max(10, K), hbm, peak_src)
        finally:
            gc.enable()
    if w.chunk_sweep:
        line["chunk_sweep"] = chunk_sweep(kvc, torch, w, req, device, flush, max(3, K))
    if args.npl:
        line["batched_decode"] = batched_decode(kvc, torch, w, device, [int(x) for x in args.npl.split(",")])
    return line


def kernel_rooflines(kvc, torch, w, req, flush, reps, peak_gbs, peak_src):
    """HBM rooflines of the bandwidth-bound calls, each timed cold: L2 flushed (256 MiB write) before
    every one of `reps` calls, CUDA events on the current stream around the call alone.  Run on the
    filled cache of layer 0 after the timed steps; the appends rewrite the same tokens at the same
    positions, so the cache bytes do not change.  achieved = algorithmic bytes / mean call time:
      append      n * (2 * H_kv * D * input bytes read + B_tok written)
      decode_attn (p + 1) * B_tok of cache + the query (H_q * D * input bytes) + the output (H_q * D * 4)
      decode_step the same plus the append of the token at p
      state       n * B_tok read + the same written (+ the 32-byte header)
    (B_tok = cache bytes per token and layer; p = the decode position; n = tokens.)  `traffic` is the
    DRAM bytes ncu counted for the same call (all its kernels), or null when the kernels changed since."""
    E = torch.cuda.Event
    q, k, v = req.dev_in[0]
    bt = cache_bytes_per_token(w)
    inb = 4 if w.in_dtype == "f32" else 2
    H, Hq, D = w.n_head_kv, w.n_head_q, w.head_dim
    row_in = 2 * H * D * inb

    def obj(name, nbytes, fn, what):
        pairs = []
        fn()   # untimed: the first launch of a kernel also loads its module
        torch.cuda.synchronize()
        torch.cuda.nvtx.range_push("kvc_kernel_" + name)
        for _ in range(reps):
            l2_flush(torch, flush)
            a = E(enable_timing=True); a.record()
            fn()
            b = E(enable_timing=True); b.record()
            pairs.append((a, b))
        torch.cuda.synchronize()
        torch.cuda.nvtx.range_pop()
        ms = float(np.mean([a.elapsed_time(b) for a, b in pairs]))
        gbs = nbytes / (ms / 1e3) / 1e9
        tr, note = recorded_traffic(name, w.name)
        return {"bound": "hbm", "what": what, "algorithmic_bytes": nbytes, "ms": ms, "achieved": gbs,
                "peak": peak_gbs, "unit": "GB/s", "frac": gbs / peak_gbs, "peak_source": "%s HBM copy" % peak_src,
                "traffic": tr, "traffic_note": note, "timing": "cold: L2 flushed before each of %d calls" % reps}

    out = {}
    full = [(p, c) for p, c in req.chunks if c == w.chunk] or req.chunks
    p, c = full[len(full) // 2]
    out["append_chunk"] = obj("append_chunk", c * (row_in + bt),
                              lambda: kvc.kv_cache_append(req.src, 0, p, k[p:p + c], v[p:p + c]),
                              "kv_cache_append of one %d-token prompt chunk" % c)
    n = w.n_prompt
    out["append_prompt"] = obj("append_prompt", n * (row_in + bt),
                               lambda: kvc.kv_cache_append(req.src, 0, 0, k[:n], v[:n]),
                               "kv_cache_append of the whole %d-token prompt in one call" % n)
    if w.n_decode:
        pos = w.n_tokens - 1
        dec = (pos + 1) * bt + Hq * D * (inb + 4)
        out["decode_attn"] = obj("decode_attn", dec,
                                 lambda: kvc.decode_attn(req.src, 0, pos, q[pos], out=req.out_d[0, -1],
                                                         scratch=req.scratch),
                                 "decode_attn at position %d (split pass + combine)" % pos)

        out["decode_step"] = obj("decode_step", dec + row_in + bt,
                                 lambda: kvc.decode_step(req.src, 0, pos, q[pos], k[pos], v[pos], out=req.out_d[0, -1],
                                                         scratch=req.scratch),
                                 "decode_step at position %d: split pass storing the token + combine" % pos)
    sb = req.state.numel()
    out["state_pack"] = obj("state_pack", 2 * sb - 32,
                            lambda: kvc.kv_state_get(req.src, w.n_tokens, dst=req.state),
                            "kv_state_get of %d tokens (header + records)" % w.n_tokens)
    out["state_unpack"] = obj("state_unpack", 2 * sb - 32,
                              lambda: kvc.kv_state_set(req.dst, req.state),
                              "kv_state_set of %d tokens, including its one synchronous header read" % w.n_tokens)
    return out


def batched_decode(kvc, torch, w, device, npls, n_past=2048, n_gen=128):
    """Generation with npl sequences decoded together (decode_step_batch), the setup of a batched
    bench: each sequence holds an n_past-token prompt of this workload's shape in its own cache, then
    n_gen steps each store one token per sequence and decode all sequences in one call
    (decode_step_batch), in a CUDA graph.
    Reports generated tokens/s over all sequences and the algorithmic cache bytes read per second."""
    res = {}
    bt = cache_bytes_per_token(w)
    n_tok = n_past + n_gen
    seqs = []
    for i in range(max(npls)):
        ws = si.Workload(**{**w.__dict__, "name": "npl%d" % i, "n_layer": 1, "n_prompt": n_past, "n_decode": n_gen,
                            "n_ctx": n_tok, "seed": w.seed + 100 + i})
        q, k, v = si.layer_qkv_device(ws, 0, device, n_rows=n_tok)
        g = kvc.KVCache(1, n_tok, w.n_head_kv, w.head_dim, w.cache, "head_major", device)
        kvc.kv_cache_append(g, 0, 0, k[:n_past], v[:n_past])
        seqs.append((g, q, k, v))
    for npl in npls:
        caches = [s[0] for s in seqs[:npl]]
        qs = torch.stack([s[1][n_past:n_tok] for s in seqs[:npl]], dim=1)   # [step][seq][H_q][D]
        out = torch.empty(n_gen, npl, w.n_head_q, w.head_dim, device=device)
        scratch = torch.empty(npl * caches[0].scratch_bytes(w.n_head_q), dtype=torch.uint8, device=device)

        ks = torch.stack([s[2][n_past:n_tok] for s in seqs[:npl]], dim=1)   # [step][seq][H_kv][D]
        vs = torch.stack([s[3][n_past:n_tok] for s in seqs[:npl]], dim=1)

        def gen():
            for t in range(n_gen):
                pos = [n_past + t] * npl
                kvc.decode_step_batch(caches, 0, pos, qs[t], ks[t], vs[t], out=out[t], scratch=scratch)
        s = torch.cuda.Stream(device)
        with torch.cuda.stream(s):
            gen()
            torch.cuda.synchronize()
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph, stream=s):
                gen()
        graph.replay()
        torch.cuda.synchronize()
        a = torch.cuda.Event(enable_timing=True); b = torch.cuda.Event(enable_timing=True)
        a.record(); graph.replay(); b.record(); b.synchronize()
        ms = a.elapsed_time(b)
        cache_bytes = npl * sum((n_past + t + 1) * bt for t in range(n_gen))
        res[str(npl)] = {"tg_tok_s": npl * n_gen / (ms / 1e3), "us_per_step": ms * 1e3 / n_gen,
                         "algorithmic_GB_s": cache_bytes / (ms / 1e3) / 1e9}
        del graph
    res["setup"] = "npl sequences, %d-token prompts, %d generated tokens each, one decode_step_batch " \
                   "per step in a CUDA graph" % (n_past, n_gen)
    return res


def end_to_end(kvc, torch, w, req, device, rank, world, K, flush, local=0):
    """The same request through the public API with host buffers: every step copies its inputs in from
    pinned host memory and its outputs (prefill and decode attention, the state) back out, inside the
    timed region.  For a one-layer request two requests alternate, so that step i's input copy and
    step i-1's output copy run on their own streams while the other request computes (as a serving
    loop overlaps transfers with compute); the inputs copied in each step are larger than L2.  A
    layer stack (tens of GB of inputs) runs its steps one after another, L2 flushed before each."""
    h2d, d2h = req.io_bytes()
    tokens = (w.n_prompt + w.n_decode) * w.n_layer
    if w.n_layer > 1:
        for _ in range(2):
            req.h2d(); req.step(); req.d2h()
        torch.cuda.synchronize()
        dist_barrier(world)
        e_ms = []
        for _ in range(K):
            l2_flush(torch, flush)
            a = torch.cuda.Event(enable_timing=True); a.record()
            req.h2d(); req.step(); req.d2h()
            b = torch.cuda.Event(enable_timing=True); b.record()
            b.synchronize()
            e_ms.append(a.elapsed_time(b))
        e_total = dist_max(sum(e_ms), world)
        return {"value": tokens * world * K / (e_total / 1e3), "unit": "tok/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": e_total / K, "overlap": "none (steps in series)"}
    reqs = [req, GpuRequest(kvc, w, device, seed_offset=rank)]
    if w.n_decode:
        reqs[1].capture()
    main = torch.cuda.current_stream(device)
    s_in, s_out = torch.cuda.Stream(device), torch.cuda.Stream(device)
    E = torch.cuda.Event

    def run(n):
        done, out_done, inp = [], [], []
        start = E(enable_timing=True)
        start.record(main)
        s_in.wait_event(start)
        s_out.wait_event(start)

        def h2d(j):
            # step j's inputs, once its request's previous step (j - 2) no longer reads them
            if j >= 2:
                s_in.wait_event(done[j - 2])
            with torch.cuda.stream(s_in):
                reqs[j % 2].h2d()
            e = E(); e.record(s_in); inp.append(e)

        h2d(0)
        for i in range(n):
            r = reqs[i % 2]
            # the next step's inputs are queued before this step: the host may wait inside this step
            # (kv_state_set reads the stream header), and the copy then still runs beside its compute
            if i + 1 < n:
                h2d(i + 1)
            main.wait_event(inp[i])
            if i >= 2:
                main.wait_event(out_done[i - 2])      # request r's previous outputs are on the host
            r.step()
            d = E(); d.record(main); done.append(d)
            s_out.wait_event(d)
            with torch.cuda.stream(s_out):
                r.d2h()
            o = E(); o.record(s_out); out_done.append(o)
        main.wait_event(out_done[-1])
        main.wait_event(done[-1])
        stop = E(enable_timing=True)
        stop.record(main)
        stop.synchronize()
        return start.elapsed_time(stop)

    run(2)
    torch.cuda.synchronize()
    dist_barrier(world)
    clocks = ClockSampler(local)
    clocks.start()
    gc.collect()
    gc.disable()
    try:
        e_ms = run(K)
    finally:
        gc.enable()
    e_total = dist_max(e_ms, world)
    clk = clocks.stop()
    return {"value": tokens * world * K / (e_total / 1e3), "unit": "tok/s", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "ms_per_step": e_total / K, "clocks": clk,
            "overlap": "two requests alternate: copies in and out on their own streams beside compute",
            "l2": "each step copies in %d bytes of inputs (> L2)" % h2d}


def chunk_sweep(kvc, torch, w, req, device, flush, reps):
    """Prefill time (prefill_step calls, L2 flushed before each) of the same prompt under each
    chunking, and the fit T = b * chunks + a * tokens: b is this layer's fixed cost per chunk and a
    its cost per token, the two numbers the pipeline chunk rule takes as b/a."""
    import numpy as np
    ms = {}
    for chunk in w.chunk_sweep:
        ww = si.Workload(**{**w.__dict__, "chunk": chunk, "n_decode": 0})
        r = GpuRequest(kvc, ww, device, inputs=req.dev_in)
        r.step()
        ts = []
        for _ in range(reps):
            l2_flush(torch, flush)
            ev = {"prefill": [], "attn": [], "decode": [], "state": []}
            r.step(ev)
            torch.cuda.synchronize()
            ts.append(sum(x[0].elapsed_time(x[1]) for x in ev["prefill"]))
        ms[len(r.chunks)] = (chunk or w.n_prompt, min(ts))
        del r
    k = np.array(sorted(ms), dtype=np.float64)
    t = np.array([ms[int(x)][1] for x in k])
    b, c = np.polyfit(k, t, 1)
    a = c / w.n_prompt
    out = {"prefill_ms": {str(ms[int(x)][0]): ms[int(x)][1] for x in k},
           "fit": {"b_us_per_chunk": b * 1e3, "a_us_per_token": a * 1e3,
                   "b_over_a_tokens": (b / a) if a > 0 else None}}
    if a > 0 and b > 0:
        out["pipeline_chunk"] = {str(s): kvc.pipeline_chunk(w.n_prompt, 8192, s, b / a) for s in (2, 4, 8)}
    return out


# --------------------------------------------------------------------------- CPU oracle (baseline / reference arm)
def oracle_plan(w):
    """Sample sizes of the oracle legs, bounded so that one sample costs tens of seconds of CPU work:
    the oracle dequantises the attended context to float64 for every sampled chunk and decode step,
    which at a 58k-token context costs seconds per call."""
    if w.n_ctx > 32768:
        return dict(max_chunks=3, rows_per_chunk=16, decode_samples=2)
    return dict(max_chunks=16, rows_per_chunk=64, decode_samples=32)


class OracleRun:
    """One layer of a workload on the CPU oracle: inputs drawn and every token appended (timed) once;
    then bounded samples of the prefill and decode work, each extrapolated to the whole request."""

    def __init__(self, w):
        from oracle.cache import OracleCache
        self.w = w
        q, k, v = si.layer_qkv(w, 0)
        self.qf, kf, vf = (t.float().numpy() for t in (q, k, v))
        self.o = OracleCache(1, w.n_ctx, w.n_head_kv, w.head_dim, w.cache)
        self.chunks = w.chunks()
        t0 = time.perf_counter()
        for p, c in self.chunks:
            self.o.append(0, p, kf[p:p + c], vf[p:p + c])
        for p in range(w.n_prompt, w.n_tokens):
            self.o.append(0, p, kf[p:p + 1], vf[p:p + 1])
        self.t_append = time.perf_counter() - t0

    def sample(self, max_chunks, rows_per_chunk, decode_samples, sample_offset=0, first_chunk=0):
        """Time the oracle on a bounded sample; extrapolate to the whole request.

        Prefill: `max_chunks` evenly spaced chunks (shifted by first_chunk), each the cache
        dequantisation (scaled by cache length) and the attention of `rows_per_chunk` rows plus the
        chunk's first and last (scaled by the causal row work sum (t+1)).  Decode: `decode_samples`
        steps scaled by sum (pos+1).  The appends of every token (timed once) and the state pack and
        unpack are whole.  `sample_offset` picks another seeded set of rows.
        """
        from oracle import state as ostate
        from oracle.attention import attend
        from oracle.cache import OracleCache
        w, o, chunks = self.w, self.o, self.chunks
        t0 = time.perf_counter()
        n_pick = min(max_chunks, len(chunks))
        pick = np.linspace(0, len(chunks) - 1, n_pick).round().astype(int)
        pick = sorted(set(((pick + first_chunk) % len(chunks)).tolist()))
        rng = np.random.default_rng(w.seed + 7919 * sample_offset)
        t_deq = t_att = 0.0
        deq_units = att_units = 0.0
        for ci in pick:
            p, c = chunks[ci]
            t1 = time.perf_counter()
            kh, vh = o.dequantized(0, p + c)
            t2 = time.perf_counter()
            rows = np.unique(np.concatenate([[0, c - 1], rng.choice(c, size=min(rows_per_chunk, c), replace=False)]))
            attend(self.qf[p + rows], p + rows, kh, vh)
            t3 = time.perf_counter()
            t_deq += t2 - t1
            t_att += t3 - t2
            deq_units += p + c
            att_units += float(np.sum(p + rows + 1))
        full_deq_units = float(sum(p + c for p, c in chunks))
        full_att_units = float(w.n_prompt) * (w.n_prompt + 1) / 2
        t_prefill = t_deq * full_deq_units / deq_units + t_att * full_att_units / att_units
        t_decode = 0.0
        n_dec = 0
        if w.n_decode and decode_samples:
            steps = np.linspace(0, w.n_decode - 1, min(decode_samples, w.n_decode)).round().astype(int)
            steps = sorted(set(((steps + first_chunk) % w.n_decode).tolist()))
            n_dec = len(steps)
            t4 = time.perf_counter()
            units = 0.0
            for i in steps:
                pos = w.n_prompt + i
                o.decode(0, pos, self.qf[pos])
                units += pos + 1
            full = float(sum(w.n_prompt + i + 1 for i in range(w.n_decode)))
            t_decode = (time.perf_counter() - t4) * full / units
        t5 = time.perf_counter()
        blob = ostate.pack(o, w.n_tokens)
        o2 = OracleCache(1, w.n_ctx, w.n_head_kv, w.head_dim, w.cache)
        ostate.unpack(blob, o2)
        t_state = time.perf_counter() - t5
        total = self.t_append + t_prefill + t_decode + t_state
        return {"value": (w.n_prompt + w.n_decode) / total, "seconds_extrapolated": total,
                "seconds_measured": self.t_append + time.perf_counter() - t0,
                "parts_s": {"append": self.t_append, "prefill": t_prefill, "decode": t_decode, "state": t_state},
                "sample": "one layer; appends and state whole; prefill: %d of %d chunks, %d rows each, "
                          "dequantisation scaled by cache length, attention by causal row work; decode: %d of %d "
                          "steps scaled by key count" % (len(pick), len(chunks), rows_per_chunk + 2,
                                                         n_dec, w.n_decode)}


def oracle_sample(w, sample_offset=0, **plan):
    """The oracle on one bounded sample of the workload (oracle_plan's sizes unless given)."""
    return OracleRun(w).sample(sample_offset=sample_offset, **(plan or oracle_plan(w)))


def _oracle_env():
    env = dict(os.environ)
    for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS", "BLIS_NUM_THREADS"):
        env[k] = "1"
    env.pop("WORLD_SIZE", None)
    env.pop("RANK", None)
    return env


def _oracle_cmd(workload, offset):
    return [sys.executable, os.path.abspath(__file__), "--oracle-child", "--workload", workload,
            "--oracle-offset", str(offset)]


def _host_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def _mem_available_gb():
    try:
        with open("/proc/meminfo") as f:
            for line in f:
                if line.startswith("MemAvailable:"):
                    return int(line.split()[1]) / (1 << 20)
    except OSError:
        pass
    return None


def oracle_all_cores(workload, gb_per_process):
    """The oracle on every host core: one single-threaded oracle process per core (at most 16, and
    no more than the available memory holds at gb_per_process each), started together, each on its
    own seeded sample of the workload.  Independent requests share nothing, so the host's rate is the
    sum of the processes' rates, each measured while all of them run."""
    n = min(_host_cores(), 16)
    mem = _mem_available_gb()
    if mem is not None:
        n = max(1, min(n, int(mem // gb_per_process)))
    env = _oracle_env()
    procs = [subprocess.Popen(_oracle_cmd(workload, i + 1), stdout=subprocess.PIPE, stderr=subprocess.PIPE,
                              text=True, env=env) for i in range(n)]
    vals, err = [], None
    for p in procs:
        try:
            out, e = p.communicate(timeout=900)
        except subprocess.TimeoutExpired:
            p.kill()
            out, e = p.communicate()
        if p.returncode == 0:
            vals.append(json.loads(out.strip().splitlines()[-1])["value"])
        else:
            err = (e or "")[-400:]
    if len(vals) != n:
        return {"value": None, "unit": "tok/s", "cores": n, "kind": "oracle", "error": err}
    return {"value": float(sum(vals)), "unit": "tok/s", "cores": n, "kind": "oracle",
            "sample": "%d concurrent single-threaded oracle processes, each on its own seeded sample of the "
                      "workload (the single-thread sample); value = the sum of their rates" % n}


def cpu_baseline(workload):
    """The oracle in a child process restricted to one thread (so `cores` is exact), then on every
    host core (oracle_all_cores)."""
    r = subprocess.run(_oracle_cmd(workload, 0), capture_output=True, text=True, env=_oracle_env(), timeout=900)
    if r.returncode != 0:
        return {"value": None, "unit": "tok/s", "cores": 1, "kind": "oracle", "error": r.stderr[-400:]}
    d = json.loads(r.stdout.strip().splitlines()[-1])
    out = {"value": d["value"], "unit": "tok/s", "cores": 1, "kind": "oracle", "sample": d["sample"],
           "seconds_measured": d["seconds_measured"], "parts_s": d["parts_s"]}
    w = si.WORKLOADS[workload]
    if d["seconds_measured"] > 60:
        # the concurrent processes would take at least as long again: keep the bench within minutes
        out["all_cores"] = {"value": None, "skipped": "the single-thread sample took %.0f s" % d["seconds_measured"]}
        return out
    # float64 dequantised K and V of the whole context, plus the sampled rows' score matrices
    # (measured peaks: 2.0 GB for f16_17k, 5.4 GB for q8_0_58k)
    gb = 2.5 + 2 * w.n_ctx * w.n_head_kv * w.head_dim * 8 * 3 / 1e9
    try:
        out["all_cores"] = oracle_all_cores(workload, gb)
    except Exception as e:   # the single-thread figure stands on its own
        out["all_cores"] = {"value": None, "error": repr(e)[-400:]}
    return out


def run_reference(args, rank, world):
    """The reference arm: the CPU oracle on this host's cores.  The inputs are drawn and the cache
    filled once; each step then times a bounded sample (one chunk, rotating over the prompt, with two
    rows, and one decode step) extrapolated to the whole request, plus the appends and the state."""
    if rank != 0:
        return None
    for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        os.environ.setdefault(k, "1")
    w = si.WORKLOADS[args.workload]
    run = OracleRun(w)
    small = dict(max_chunks=1, rows_per_chunk=2, decode_samples=1)
    n_chunks = len(run.chunks)
    for i in range(args.warmup):
        run.sample(first_chunk=(7 * i) % n_chunks, **small)
    vals, secs = [], []
    samp = None
    for i in range(args.steps):
        d = run.sample(first_chunk=(7 * (args.warmup + i)) % n_chunks, **small)
        vals.append(d["value"])
        secs.append(d["seconds_extrapolated"])
        samp = d["sample"]
    value = float(np.mean(vals))
    return {"impl": "reference", "metric": METRIC, "value": value, "unit": "tok/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * float(np.mean(secs)),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64 (oracle)",
            "data": "synthetic (seeded N(0,1))",
            "config": workload_config(w),
            "cpu_baseline": {"value": value, "unit": "tok/s", "cores": 1, "kind": "oracle", "sample": samp},
            "e2e": {"value": value, "unit": "tok/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(si.WORKLOADS))
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--npl", default="", help="also time batched decode for these sequence counts, e.g. 1,2,4,8")
    ap.add_argument("--oracle-child", action="store_true", help=argparse.SUPPRESS)
    ap.add_argument("--oracle-offset", type=int, default=0, help=argparse.SUPPRESS)
    args = ap.parse_args()

    if args.oracle_child:
        print(json.dumps(oracle_sample(si.WORKLOADS[args.workload], sample_offset=args.oracle_offset)))
        return
    rank, world, local = dist_init()
    if args.impl == "reference":
        line = run_reference(args, rank, world)
        if line is not None:
            print(json.dumps(line), flush=True)
        return
    if args.warmup < 3:
        args.warmup = 3
    line = run_gpu(args, rank, world, local)
    if rank == 0:
        w = si.WORKLOADS[args.workload]
        if w.n_layer == 1 and not args.no_cpu_baseline:
            line["cpu_baseline"] = cpu_baseline(args.workload)
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
