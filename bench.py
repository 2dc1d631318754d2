"""Throughput of the nanochat-style GPT forward pass on one B300 (per rank).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config NAME] [--impl ours|reference]

Default workload: the largest model, d24 (24 layers, d_model 1536, 12 query
heads x 128, one KV head, MLP 6144, vocab 65536).  The headline leg is its
prefill of 8 rows x 2048 uniform-random tokens with all-position fp32 logits;
one step = one nc_prefill over the whole batch.  The "decode" leg times the
same model's decode workload: 128 rows, 2048-token prompt, 128 decode steps,
tokens/s over the decode steps (one step = one nc_decode_step for the batch).
With --config d12_prefill / d20_prefill the legs are that model's workloads.
Each leg carries its own roofline (dominant kernel class), end-to-end figure
through the public API with pinned host buffers, and fp64 CPU-oracle
baseline.  At N = 1 the d12 workloads are measured too (key "d12").

Prints ONE JSON line on rank 0.  Under torchrun every rank runs its own
replica of the workload on its own GPU (rows are independent, no collective);
value = tokens of all ranks / max-over-ranks time.

--impl reference times the fp64 CPU oracle on a bounded sample of the same
workload (rank 0 only).
"""
from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import os
import statistics
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import nc_inputs  # noqa: E402

METRIC = "prefill tokens/s and decode tokens/s at 1 B300; % of bf16 TC peak / HBM BW"
PEAKS_FALLBACK = {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}
DECODE_OF = {"d12_prefill": "d12_decode", "d20_prefill": "d20_decode", "d24_prefill": "d24_decode"}


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(PEAKS_FALLBACK), "fallback"


# --------------------------------------------------------------------------- #
# algorithmic work (numerators of every roofline fraction)
# --------------------------------------------------------------------------- #

def prefill_flops(s, B, T, last_only=False):
    """Algorithmic FLOPs of one prefill, per kernel class (2 per MAC; causal
    attention counts the T(T+1)/2 unmasked pairs, QK^T and PV)."""
    M = B * T
    d, hd, nh, F, V, L = s.d_model, s.head_dim, s.n_head, s.d_mlp, s.vocab, s.n_layer
    return {
        "qkv": 2.0 * M * d * (nh + 2 * s.n_kv_head) * hd * L,
        "attn": 4.0 * nh * hd * (T * (T + 1) / 2) * B * L,
        "oproj": 2.0 * M * nh * hd * d * L,
        "fc": 2.0 * M * d * F * L,
        "proj": 2.0 * M * F * d * L,
        "lm_head": 2.0 * (B if last_only else M) * d * V,
    }


def decode_bytes_by_class(s, B, ctx):
    """Algorithmic HBM bytes of one decode step at context length ctx (keys
    0..ctx-1 read, one new K/V row written), split by the kernel class that
    moves them: the projection weights once (QKV, O, FC, PROJ, unembedding;
    2 bytes each, 1 with FP8 weights), the K/V read (attention), the new K/V
    rows (QKV), the embedding rows and the fp32 logits."""
    d, hd, nh, F, V, L = s.d_model, s.head_dim, s.n_head, s.d_mlp, s.vocab, s.n_layer
    nkv = s.n_kv_head
    wb = 1.0 if s.dtype == "fp8" else 2.0
    return {
        "embed": B * d * 2.0,
        "qkv": wb * L * (nh + 2 * nkv) * hd * d + L * B * nkv * 2 * hd * 2.0,
        "attn": L * B * nkv * 2.0 * ctx * hd * 2,
        "oproj": wb * L * d * nh * hd,
        "fc": wb * L * F * d,
        "proj": wb * L * d * F,
        "lm_head": wb * V * d + B * V * 4.0,
    }


def decode_bytes(s, B, ctx):
    """Algorithmic HBM bytes of one decode step (sum over the classes)."""
    return sum(decode_bytes_by_class(s, B, ctx).values())


def weight_bytes(s):
    """Bytes of the model's weights in device memory: bf16, or FP8 projection
    matrices with a bf16 embedding table (a decode step gathers only B rows
    of the embedding; decode_bytes_by_class counts what it streams)."""
    if s.dtype == "fp8":
        return 2 * s.vocab * s.d_model + (nc_inputs.param_count(s) - s.vocab * s.d_model)
    return 2 * nc_inputs.param_count(s)


# --------------------------------------------------------------------------- #
# clocks during the timed region (read-only queries)
# --------------------------------------------------------------------------- #

class ClockSampler:
    """SM clock and clock-event reasons of this process's GPU, sampled every
    10 ms by a background thread while the timed region runs.  NVML is
    called through ctypes (libnvidia-ml); nvidia-smi at 50 ms is the
    fallback.  Read only: no GPU setting is changed."""
    NVML_CLOCK_SM = 1
    # clock-event reason bits of the NVML API
    REASON_BITS = (("sw_power_cap", 0x4), ("hw_slowdown", 0x8), ("sw_thermal_slowdown", 0x20),
                   ("hw_thermal_slowdown", 0x40), ("hw_power_brake", 0x80))

    def __init__(self, gpu_index, period_s=0.01):
        self.gpu, self.period = gpu_index, period_s
        self.sm, self.bits, self.mx = [], 0, None
        self.nvml = None
        self.smi, self.note = None, None

    def _uuid(self):
        import torch
        u = str(torch.cuda.get_device_properties(self.gpu).uuid)
        return u if u.startswith("GPU-") else "GPU-" + u

    def _open_nvml(self):
        L = ctypes.CDLL("libnvidia-ml.so.1")
        if L.nvmlInit_v2() != 0:
            raise OSError("nvmlInit_v2 failed")
        h = ctypes.c_void_p()
        if L.nvmlDeviceGetHandleByUUID(self._uuid().encode(), ctypes.byref(h)) != 0:
            if L.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(self.gpu), ctypes.byref(h)) != 0:
                raise OSError("no NVML handle for this device")
        self.reasons_fn = getattr(L, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            L.nvmlDeviceGetCurrentClocksThrottleReasons
        mx = ctypes.c_uint()
        if L.nvmlDeviceGetMaxClockInfo(h, self.NVML_CLOCK_SM, ctypes.byref(mx)) == 0:
            self.mx = float(mx.value)
        self.nvml, self.h = L, h

    def __enter__(self):
        try:
            self._open_nvml()
        except Exception as e:
            self.nvml, self.note = None, f"nvml: {type(e).__name__}: {e}"[:160]
            self._start_smi()
            return self
        self.stop = threading.Event()
        self.th = threading.Thread(target=self._loop, daemon=True)
        self.th.start()
        return self

    def _loop(self):
        L, h = self.nvml, self.h
        c, r = ctypes.c_uint(), ctypes.c_ulonglong()
        while not self.stop.is_set():
            if L.nvmlDeviceGetClockInfo(h, self.NVML_CLOCK_SM, ctypes.byref(c)) == 0:
                self.sm.append(float(c.value))
            if self.reasons_fn(h, ctypes.byref(r)) == 0:
                self.bits |= int(r.value)
            self.stop.wait(self.period)

    SMI_Q = ("clocks.sm,clocks.max.sm,clocks_event_reasons.hw_slowdown,"
             "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
             "clocks_event_reasons.sw_power_cap")

    def _start_smi(self):
        import subprocess
        import tempfile
        try:
            ident = self._uuid()
        except Exception:
            ident = str(self.gpu)
        self.smi_out = tempfile.TemporaryFile(mode="w+")
        try:
            self.smi = subprocess.Popen(["nvidia-smi", f"--id={ident}", f"--query-gpu={self.SMI_Q}",
                                         "--format=csv,noheader,nounits", "-lms", "50"],
                                        stdout=self.smi_out, stderr=subprocess.DEVNULL)
        except OSError as e:
            self.smi, self.note = None, (self.note or "") + f"; nvidia-smi: {e}"
            return
        t0 = time.time()                    # let the first sample land (at most 5 s)
        while time.time() - t0 < 5 and self.smi.poll() is None:
            self.smi_out.flush()
            if os.fstat(self.smi_out.fileno()).st_size > 0:
                break
            time.sleep(0.05)

    def _stop_smi(self):
        if self.smi is None:
            return
        self.smi.terminate()
        try:
            self.smi.wait(timeout=5)
        except Exception:
            self.smi.kill()
        self.smi_out.seek(0)
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        self.smi_reasons = set()
        for line in self.smi_out:
            p = [t.strip() for t in line.split(",")]
            if len(p) < 6:
                continue
            try:
                self.sm.append(float(p[0]))
                self.mx = float(p[1])
            except ValueError:
                continue
            for n, v in zip(names, p[2:6]):
                if v.lower() == "active":
                    self.smi_reasons.add(n)

    def __exit__(self, *a):
        self._stop_smi()
        if self.nvml is not None:
            self.stop.set()
            self.th.join(timeout=2)
            try:
                self.nvml.nvmlShutdown()
            except Exception:
                pass

    def summary(self):
        if not self.sm:
            return {"sm_mhz": None, "sm_max_mhz": self.mx, "reasons": [], "samples": 0, "note": self.note}
        if self.nvml is not None:
            reasons = sorted(n for n, bit in self.REASON_BITS if self.bits & bit)
            src = "nvml (ctypes) 10 ms"
        else:
            reasons, src = sorted(getattr(self, "smi_reasons", set())), "nvidia-smi 50 ms"
        out = {"sm_mhz": statistics.median(self.sm), "sm_max_mhz": self.mx, "reasons": reasons,
               "samples": len(self.sm), "source": src}
        if self.note:
            out["note"] = self.note
        return out


# --------------------------------------------------------------------------- #
# DRAM traffic of the dominant kernels, from ncu captures
# --------------------------------------------------------------------------- #

# profiles/traffic.json lists, per kernel class and workload, the DRAM bytes
# (read + write) of one launch measured by ncu and the SHA-256 prefix of the
# kernel's source file at capture time; a figure is used only while the
# source still hashes the same (otherwise the kernel changed and it is null).
KCLASS_SOURCE = {"lm_head": "k_gemm_tc.cuh", "qkv": "k_gemm_tc.cuh", "oproj": "k_gemm_tc.cuh",
                 "fc": "k_gemm_tc.cuh", "proj": "k_gemm_tc.cuh", "attn": "k_attn_tc.cuh",
                 "decode_attn": "k_attn_mma.cuh", "decode_gemm": "k_gemm_skinny.cuh"}


def source_sha256(name):
    path = os.path.join(ROOT, "dense_gpt_transformer_fwd_b300", "csrc", name)
    with open(path, "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:16]


def measured_traffic(kclass, workload):
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        rows = json.load(f).get("launches", [])
    for r in rows:
        if r.get("class") == kclass and r.get("workload") == workload:
            src = r.get("source")
            if src and os.path.exists(os.path.join(ROOT, "dense_gpt_transformer_fwd_b300", "csrc", src)) \
                    and source_sha256(src) == r.get("sha256"):
                return float(r["bytes_per_launch"])
    return None


# --------------------------------------------------------------------------- #
# the fp64 CPU oracle (reported baseline)
# --------------------------------------------------------------------------- #

def blas_threads():
    """Threads the oracle's BLAS uses (OpenBLAS defaults to every available core, up to 64)."""
    try:
        from threadpoolctl import threadpool_info
        return max([i.get("num_threads", 1) for i in threadpool_info()] or [1])
    except ImportError:
        env = os.environ.get("OPENBLAS_NUM_THREADS") or os.environ.get("OMP_NUM_THREADS")
        return int(env) if env else min(len(os.sched_getaffinity(0)), 64)


def oracle_baselines(w, wd, flat, prompt, nxt, decode_steps=8):
    """fp64 oracle on row 0: the prefill of its prompt (timed), then
    `decode_steps` decode steps continuing from that cache (timed apart).
    Returns the two cpu_baseline objects."""
    from oracle.gpt_oracle import OracleModel
    o = OracleModel(flat, w.shape)
    T = w.prompt_len
    t0 = time.perf_counter()
    o.prefill(prompt[:1, :T])
    dt = time.perf_counter() - t0
    threads = blas_threads()
    pre = {"value": round(T / dt, 2), "unit": "tokens/s", "cores": threads, "kind": "oracle",
           "sample": f"fp64 prefill of row 0 ({T} tokens, all-position logits) of {w.name}; {dt:.1f} s"}
    dec = None
    if wd is not None and nxt is not None:
        t0 = time.perf_counter()
        for t in range(decode_steps):
            o.decode(nxt[t][:1])
        dd = time.perf_counter() - t0
        dec = {"value": round(decode_steps / dd, 3), "unit": "tokens/s", "cores": threads,
               "kind": "oracle",
               "sample": (f"fp64 decode of row 0 for {decode_steps} steps at context {T + 1}..{T + decode_steps} "
                          f"(continuing the prefill above; {wd.name} decodes at context "
                          f"{wd.prompt_len + 1}..{wd.max_seq}); {dd:.1f} s")}
    return pre, dec


# --------------------------------------------------------------------------- #
# ranks
# --------------------------------------------------------------------------- #

def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("gloo")
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(world, v):
    if world == 1:
        return v
    import torch
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def reference_tokens_per_step(shape):
    """Prefix length the reference arm prefills per step: about 0.2 TFLOP of
    fp64 work (a few seconds on the host cores), whatever the model."""
    per_token = 2.0 * (shape.n_layer * nc_inputs.layer_param_count(shape) + shape.vocab * shape.d_model)
    t = int(2e11 / per_token)
    return max(32, min(512, 1 << (t.bit_length() - 1)))


def run_reference(args, world, rank):
    """The oracle, as it stands, on the host cores: each step is the prefill of
    row 0's first tokens of the benchmark workload (all-position logits)."""
    if rank != 0:
        return
    w = nc_inputs.WORKLOADS[args.config]
    flat = nc_inputs.gen_weights(w.shape, w.weight_seed)
    prompt, _ = _tokens(w)
    T = min(reference_tokens_per_step(w.shape), w.prompt_len)
    from oracle.gpt_oracle import OracleModel
    o = OracleModel(flat, w.shape)
    for _ in range(args.warmup):
        o.prefill(prompt[:1, :T])
    t0 = time.perf_counter()
    for _ in range(args.steps):
        o.prefill(prompt[:1, :T])
    dt = time.perf_counter() - t0
    value = args.steps * T / dt
    threads = blas_threads()
    sample = f"row 0, tokens 0..{T - 1} of {w.name} ({w.batch}x{w.prompt_len}), all-position logits"
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": dt * 1e3 / args.steps, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": w.name, "global_batch": w.batch, "seq_len": w.prompt_len},
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": threads, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def _tokens(w):
    prompt = nc_inputs.gen_tokens(w.shape.vocab, (w.batch, w.prompt_len), w.prompt_seed)
    nxt = (nc_inputs.gen_tokens(w.shape.vocab, (w.decode_steps, w.batch), w.decode_seed)
           if w.decode_steps else None)
    return prompt, nxt


# --------------------------------------------------------------------------- #
# GPU legs
# --------------------------------------------------------------------------- #

def bench_prefill(args, world, local, w, flat, prompt):
    import torch
    import dense_gpt_transformer_fwd_b300 as ncp
    B, T, V = w.batch, w.prompt_len, w.shape.vocab
    m = ncp.Model(w.shape, flat, max_batch=B, max_seq=T)
    tok = torch.from_numpy(prompt).to("cuda")
    logits = torch.empty((B * T, V), dtype=torch.float32, device="cuda")
    stream = torch.cuda.current_stream()

    def step():
        m.kv_reset()
        m.prefill(tok, out=logits)

    for _ in range(args.warmup):
        step()
    m.sync()
    barrier(world)
    torch.cuda.synchronize()
    l0 = m.launch_count
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk:
        ev0.record(stream)
        for _ in range(args.steps):
            step()
        ev1.record(stream)
        torch.cuda.synchronize()
    m.sync()
    launches = m.launch_count - l0
    ms = ev0.elapsed_time(ev1) / args.steps
    barrier(world)
    ms_max = max_over_ranks(world, ms)

    # per-kernel-class device time (events around each launch), separate pass
    m.profile_begin()
    for _ in range(args.steps):
        step()
    prof = m.profile_end()
    prof = {k: (t / args.steps, n // args.steps) for k, (t, n) in prof.items()}

    # end to end through the public API with host buffers (pinned)
    tok_h = torch.from_numpy(prompt).pin_memory()
    out_h = torch.empty((B * T, V), dtype=torch.float32, pin_memory=True)
    for _ in range(2):
        m.kv_reset()
        m.prefill(tok_h, out=out_h)
    torch.cuda.synchronize()
    barrier(world)
    e2e_steps = max(1, min(args.steps, 5))
    ev0.record(stream)
    t0 = time.perf_counter()
    for _ in range(e2e_steps):
        m.kv_reset()
        m.prefill(tok_h, out=out_h)
    ev1.record(stream)
    torch.cuda.synchronize()
    e2e_s = max_over_ranks(world, max(time.perf_counter() - t0, ev0.elapsed_time(ev1) / 1e3) / e2e_steps)
    m.sync()
    m.close()
    del logits, out_h
    torch.cuda.empty_cache()
    return {"ms": ms_max, "launches": launches, "prof": prof, "clocks": clk.summary(),
            "e2e_s": e2e_s, "h2d": B * T * 4, "d2h": B * T * V * 4}


def bench_decode(args, world, local, w, flat, prompt, nxt):
    """Decode leg: the workload's steps replayed from the captured graph into
    one logits buffer (timed), an eager pass with per-kernel-class events, and
    an end-to-end pass with pinned host token and logit buffers."""
    import torch
    import dense_gpt_transformer_fwd_b300 as ncp
    B, V = w.batch, w.shape.vocab
    steps = w.decode_steps
    m = ncp.Model(w.shape, flat, max_batch=B, max_seq=w.max_seq)
    tok = torch.from_numpy(prompt).to("cuda")
    nxt_d = torch.from_numpy(nxt).to("cuda")
    out = torch.empty((B, V), dtype=torch.float32, device="cuda")
    stream = torch.cuda.current_stream()
    # warm-up pass (prefill + a few steps: the graph is captured at the second)
    m.prefill(tok, last_only=True)
    for t in range(min(max(args.warmup, 3), steps)):
        m.decode_step(nxt_d[t], out=out)
    m.kv_reset()
    m.prefill(tok, last_only=True)
    m.sync()
    barrier(world)
    torch.cuda.synchronize()
    l0 = m.launch_count
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk:
        ev0.record(stream)
        for t in range(steps):
            m.decode_step(nxt_d[t], out=out)
        ev1.record(stream)
        torch.cuda.synchronize()
    m.sync()
    ms = ev0.elapsed_time(ev1) / steps
    launches = m.launch_count - l0
    barrier(world)
    ms_max = max_over_ranks(world, ms)

    # eager pass with events around every kernel: device time per class
    m.kv_reset()
    m.prefill(tok, last_only=True)
    m.profile_begin()
    for t in range(steps):
        m.decode_step(nxt_d[t], out=out)
    prof = m.profile_end()
    prof = {k: (t / steps, n // steps) for k, (t, n) in prof.items()}

    # end to end: pinned host tokens in, pinned host logits out, every step
    tok_h = torch.from_numpy(nxt).pin_memory()
    out_h = torch.empty((B, V), dtype=torch.float32, pin_memory=True)
    m.kv_reset()
    m.prefill(tok, last_only=True)
    for t in range(2):                                 # the host-buffer graph is captured here
        m.decode_step(tok_h[t], out=out_h)
    m.kv_reset()
    m.prefill(tok, last_only=True)
    torch.cuda.synchronize()
    barrier(world)
    t0 = time.perf_counter()
    for t in range(steps):
        m.decode_step(tok_h[t], out=out_h)
    torch.cuda.synchronize()
    e2e_s = max_over_ranks(world, (time.perf_counter() - t0) / steps)
    m.sync()
    m.close()
    torch.cuda.empty_cache()
    ctxs = [w.prompt_len + t + 1 for t in range(steps)]
    by_class = {k: float(np.mean([decode_bytes_by_class(w.shape, B, c)[k] for c in ctxs]))
                for k in decode_bytes_by_class(w.shape, B, ctxs[0])}
    return {"ms": ms_max, "launches": launches, "prof": prof, "bytes_by_class": by_class,
            "bytes": float(sum(by_class.values())), "clocks": clk.summary(), "e2e_s": e2e_s,
            "h2d": B * 4, "d2h": B * V * 4}


def class_table(prof, work, unit_scale):
    """Per kernel class: device ms per step, launches, share and the achieved
    rate (work per step / device time)."""
    total = sum(t for t, _ in prof.values()) or 1.0
    out = {}
    for k, (t, n) in prof.items():
        if t <= 0:
            continue
        e = {"ms": round(t, 4), "launches": n, "share": round(t / total, 4)}
        if k in work:
            e["rate"] = round(work[k] / (t / 1e3) / unit_scale, 1)
        out[k] = e
    return out


def prefill_leg(args, world, local, w, flat, prompt, peaks, peak_src):
    r = bench_prefill(args, world, local, w, flat, prompt)
    B, T = w.batch, w.prompt_len
    flops = prefill_flops(w.shape, B, T)
    prof = r["prof"]
    dom = max((k for k in prof if k in flops), key=lambda k: prof[k][0])
    peak = peaks["bf16_tflops"]
    ach = flops[dom] / (prof[dom][0] / 1e3) / 1e12
    roof = {"bound": "tensor", "kernel": dom, "achieved": round(ach, 1), "peak": peak,
            "unit": "TFLOP/s", "frac": round(ach / peak, 4),
            "traffic": measured_traffic(dom, w.name),
            "peak_source": f"{peak_src} bf16 dense (burst)",
            "frac_of_sustained": round(ach / peaks.get("bf16_tflops_sustained", peak), 4),
            "per_launch": f"{flops[dom] / max(prof[dom][1], 1) / 1e9:.1f} GFLOP per launch, "
                          f"{prof[dom][0] / max(prof[dom][1], 1) * 1e3:.1f} us per launch"}
    total = sum(flops.values())
    return r, {
        "value": round(world * B * T / (r["ms"] / 1e3), 1), "ms_per_step": round(r["ms"], 4),
        "gpu_launches": r["launches"], "gpu_launches_per_step": r["launches"] // args.steps,
        "e2e": {"value": round(world * B * T / r["e2e_s"], 1), "unit": "tokens/s",
                "h2d_bytes_per_step": r["h2d"], "d2h_bytes_per_step": r["d2h"]},
        "roofline": roof,
        "step_tflops": round(total / (r["ms"] / 1e3) / 1e12, 1),
        "step_frac_of_peak": round(total / (r["ms"] / 1e3) / 1e12 / peak, 4),
        "kernels": class_table(prof, flops, 1e12),
        "kernel_rate_unit": "TFLOP/s",
        "clocks": r["clocks"],
    }


def decode_leg(args, world, local, w, flat, prompt, nxt, peaks, peak_src):
    r = bench_decode(args, world, local, w, flat, prompt, nxt)
    prof, by = r["prof"], r["bytes_by_class"]
    dom = max((k for k in prof if k in by), key=lambda k: prof[k][0])
    hbm = peaks["hbm_gbs"]
    ach = by[dom] / (prof[dom][0] / 1e3) / 1e9
    gbs = r["bytes"] / (r["ms"] / 1e3) / 1e9
    tclass = "decode_attn" if dom == "attn" else "decode_gemm"
    roof = {"bound": "hbm", "kernel": dom, "achieved": round(ach, 1), "peak": hbm, "unit": "GB/s",
            "frac": round(ach / hbm, 4), "traffic": measured_traffic(tclass, w.name),
            "peak_source": f"{peak_src} HBM copy",
            "per_launch": f"{by[dom] / max(prof[dom][1], 1) / 1e6:.1f} MB per launch, "
                          f"{prof[dom][0] / max(prof[dom][1], 1) * 1e3:.1f} us per launch (eager pass)"}
    return r, {
        "workload": w.name,
        "value": round(world * w.batch / (r["ms"] / 1e3), 1), "unit": "tokens/s",
        "ms_per_step": round(r["ms"], 4), "steps": w.decode_steps,
        "gpu_launches": r["launches"], "gpu_launches_per_step": r["launches"] // w.decode_steps,
        "step_gbs": round(gbs, 1), "step_frac_of_hbm": round(gbs / hbm, 4),
        "step_frac_of_nominal_8tbs": round(gbs / 8000.0, 4),
        "e2e": {"value": round(world * w.batch / r["e2e_s"], 1), "unit": "tokens/s",
                "h2d_bytes_per_step": r["h2d"], "d2h_bytes_per_step": r["d2h"]},
        "roofline": roof,
        "kernels": class_table(prof, by, 1e9),
        "kernel_rate_unit": "GB/s",
        "config": {"global_batch": w.batch * world, "prompt_len": w.prompt_len,
                   "decode_steps": w.decode_steps,
                   "l2": f"working set > L2 (weights {weight_bytes(w.shape) / 1e9:.2f} GB, "
                         f"KV cache {r['bytes_by_class']['attn'] / 1e9:.2f} GB read per step)"},
        "clocks": r["clocks"],
    }


def run_case(args):
    """A plain run of the workload for profilers: warmup + steps iterations."""
    import torch
    import dense_gpt_transformer_fwd_b300 as ncp
    from dense_gpt_transformer_fwd_b300 import build
    build.build()
    w = nc_inputs.WORKLOADS[args.config]
    B, T = args.batch or w.batch, args.seq or w.prompt_len
    flat = nc_inputs.gen_weights(w.shape, w.weight_seed)
    prompt = nc_inputs.gen_tokens(w.shape.vocab, (B, T), w.prompt_seed)
    n = args.warmup + args.steps
    if args.case == "prefill":
        m = ncp.Model(w.shape, flat, max_batch=B, max_seq=T)
        tok = torch.from_numpy(prompt).cuda()
        out = torch.empty((B * T, w.shape.vocab), dtype=torch.float32, device="cuda")
        for _ in range(n):
            m.kv_reset()
            m.prefill(tok, out=out)
    else:
        steps = max(n, 1)
        nxt = nc_inputs.gen_tokens(w.shape.vocab, (steps, B), (w.decode_seed or 0) + 1)
        m = ncp.Model(w.shape, flat, max_batch=B, max_seq=T + steps)
        m.prefill(torch.from_numpy(prompt).cuda(), last_only=True)
        nd = torch.from_numpy(nxt).cuda()
        out = torch.empty((B, w.shape.vocab), dtype=torch.float32, device="cuda")
        for t in range(steps):
            m.decode_step(nd[t], out=out)
    m.sync()
    print(json.dumps({"case": args.case, "workload": w.name, "batch": B, "seq": T, "iterations": n,
                      "launches": m.launch_count}))
    m.close()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--config", default="d24_prefill", choices=sorted(nc_inputs.WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-decode", action="store_true", help="skip the decode leg")
    ap.add_argument("--no-extra", action="store_true", help="skip the d12 measurements")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--batch", type=int, default=None,
                    help="override the workload's batch (smaller cases for profiling)")
    ap.add_argument("--seq", type=int, default=None, help="override the workload's prompt length")
    ap.add_argument("--case", choices=["prefill", "decode"], default=None,
                    help="profiling case: run only --warmup + --steps iterations of the workload "
                         "(no timing passes, no oracle) and print one short line; for ncu captures")
    args = ap.parse_args()
    if args.case:
        run_case(args)
        return
    args.warmup = max(args.warmup, 3)
    world, rank, local = dist_setup()

    if args.impl == "reference":
        run_reference(args, world, rank)
        return

    import torch
    torch.cuda.set_device(local)
    from dense_gpt_transformer_fwd_b300 import build
    build.build()

    peaks, peak_src = load_peaks()
    w = nc_inputs.WORKLOADS[args.config]
    if args.batch or args.seq:
        from dataclasses import replace
        w = replace(w, name=f"{w.name}[batch={args.batch or w.batch},seq={args.seq or w.prompt_len}]",
                    batch=args.batch or w.batch, prompt_len=args.seq or w.prompt_len)
    flat = nc_inputs.gen_weights(w.shape, w.weight_seed)
    prompt, nxt = _tokens(w)
    line = {"metric": METRIC, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": w.shape.dtype, "data": "synthetic"}
    wd = pd = nd = None

    if w.decode_steps == 0:
        _, leg = prefill_leg(args, world, local, w, flat, prompt, peaks, peak_src)
        line.update(leg)
        line["config"] = {"workload": w.name, "global_batch": w.batch * world, "seq_len": w.prompt_len,
                          "parallelism": f"replicas{world}", "logits": "fp32, all positions",
                          "l2": f"working set > L2 (weights {weight_bytes(w.shape) / 1e9:.2f} GB, logits "
                                f"{w.batch * w.prompt_len * w.shape.vocab * 4 / 1e9:.1f} GB per step)"}
        if not args.no_decode and w.name in DECODE_OF:
            wd = nc_inputs.WORKLOADS[DECODE_OF[w.name]]
            pd, nd = _tokens(wd)
            _, line["decode"] = decode_leg(args, world, local, wd, flat, pd, nd, peaks, peak_src)
    else:
        wd, pd, nd = w, prompt, nxt
        _, leg = decode_leg(args, world, local, w, flat, prompt, nxt, peaks, peak_src)
        cfg = leg.pop("config")
        line.update({k: v for k, v in leg.items() if k not in ("workload", "unit")})
        line["config"] = {"workload": w.name, "seq_len": w.prompt_len, "parallelism": f"replicas{world}",
                          **cfg}

    if world == 1 and not args.no_extra and w.shape.name != "d12" and not (args.batch or args.seq):
        # the smallest bf16 model as extra keys (not the headline)
        extra = {}
        w12 = nc_inputs.WORKLOADS["d12_prefill"]
        f12 = nc_inputs.gen_weights(w12.shape, w12.weight_seed)
        p12, _ = _tokens(w12)
        _, e = prefill_leg(args, world, local, w12, f12, p12, peaks, peak_src)
        extra["prefill"] = {k: e[k] for k in ("value", "ms_per_step", "step_frac_of_peak", "roofline", "e2e")}
        w12d = nc_inputs.WORKLOADS["d12_decode"]
        p12d, n12d = _tokens(w12d)
        _, e = decode_leg(args, world, local, w12d, f12, p12d, n12d, peaks, peak_src)
        extra["decode"] = {k: e[k] for k in ("workload", "value", "ms_per_step", "step_gbs",
                                             "step_frac_of_hbm", "roofline", "e2e")}
        line["d12"] = extra
        if w.shape.name == "d24":
            # the same decode workload with FP8 projection weights
            w8 = nc_inputs.WORKLOADS["d24_decode_fp8"]
            f8 = nc_inputs.gen_weights(w8.shape, w8.weight_seed)
            p8, n8 = _tokens(w8)
            _, e = decode_leg(args, world, local, w8, f8, p8, n8, peaks, peak_src)
            line["decode_fp8"] = {k: e[k] for k in ("workload", "value", "ms_per_step", "step_gbs",
                                                    "step_frac_of_hbm", "roofline", "kernels", "e2e")}

    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        pre, dec = oracle_baselines(w, wd, flat, prompt if w.decode_steps == 0 else pd, nd)
        if w.decode_steps == 0:
            line["cpu_baseline"] = pre
            if dec is not None and "decode" in line:
                line["decode"]["cpu_baseline"] = dec
        else:
            line["cpu_baseline"] = dec
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
