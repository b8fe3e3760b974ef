#!/usr/bin/env python
"""Benchmark of the extend-attention hot path on one GB300 (or N replicas).

One step = one pass of the extend hot path over one batch of the
Llama-3-8B-shaped workload (16 sequences, Hq=32, Hkv=8, D=128, prefix lens
uniform[0,4096], extend lens uniform[1,1024], 262144-slot pool with permuted
slots, bf16 N(0,1), sm_scale 1/sqrt(128)):
  1. build_unified_kv_indices (prefix slots + extend slots -> unified list)
  2. extend_attention_fwd_unified (device scheduler, paged gather, QK^T,
     mask, online softmax, PV, split-KV combine)
Inputs are resident in HBM when the timed region starts; L2 is flushed
(a 512 MiB buffer is written, then read back so that L2 holds clean lines)
before every timed step, outside the timing.

value = algorithmic FLOPs of all ranks / max over ranks of the device time
(TFLOP/s); FLOPs = 2 (Lq + Lv) per visible (query head, key) pair.

--impl reference times the float64 CPU oracle instead (the reference arm of
this build), on a bounded row sample of the same workload per step.
"""
from __future__ import annotations

import argparse
import copy
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

from paged_kv_extend_gb300 import workloads as W  # noqa: E402

WORKLOAD = "llama3_8b"
L2_FLUSH_BYTES = 512 << 20


# ------------------------------------------------------------ work counters
def visible_pairs(spec: W.WorkloadSpec, prefix, extend, rows=None, qo_indptr=None):
    """Number of visible (query, key) pairs per query token (summed over the
    batch, or for the given token rows): causal over prefix + extend, cut by
    the sliding window."""
    total = 0
    win = spec.sliding_window
    per_token = []
    for p, e in zip(prefix, extend):
        if e == 0:
            continue
        qpos = torch.arange(p, p + e, dtype=torch.int64)
        n = qpos + 1
        if win > 0:
            n = torch.clamp(n, max=win + 1)
        per_token.append(n)
    if not per_token:
        return 0
    allv = torch.cat(per_token)
    if rows is None:
        return int(allv.sum())
    return int(allv[rows].sum())


def mask_visible_per_token(wl: W.Workload) -> torch.Tensor:
    """Visible keys per extend token under the workload's custom mask (the
    mask replaces the causal term; the window still applies)."""
    s = wl.spec
    out = []
    for b in range(wl.batch):
        E, P = wl.extend_lens[b], wl.prefix_lens[b]
        if E == 0:
            continue
        T = P + E
        m = wl.custom_mask[int(wl.mask_indptr[b]): int(wl.mask_indptr[b]) + E * T].view(E, T).bool()
        if s.sliding_window > 0:
            qpos = torch.arange(P, P + E).view(E, 1)
            m = m & (qpos - torch.arange(T).view(1, T) <= s.sliding_window)
        out.append(m.sum(dim=1))
    return torch.cat(out).to(torch.int64)


def extend_flops(wl: W.Workload) -> float:
    s = wl.spec
    if wl.custom_mask is not None:
        return 2.0 * (s.lq + s.lv) * s.hq * int(mask_visible_per_token(wl).sum())
    return 2.0 * (s.lq + s.lv) * s.hq * visible_pairs(s, wl.prefix_lens, wl.extend_lens)


def extend_bytes(wl: W.Workload, unified: bool, kv_elem_bytes: int = 2) -> float:
    """Algorithmic bytes: every visible K/V row once per (sequence, KV head),
    4 B per prefix index (8 B per unified index), Q read, O write, lse."""
    s = wl.spec
    kv_row = (s.lq if s.v_aliases_k else s.lq + s.lv) * kv_elem_bytes
    keys = 0
    for p, e in zip(wl.prefix_lens, wl.extend_lens):
        if e == 0:
            continue
        lo = 0 if s.sliding_window <= 0 else max(0, p - s.sliding_window)
        keys += p + e - lo
    idx = (8 if unified else 4) * sum(wl.prefix_lens) + (8 * sum(wl.extend_lens) if unified else 0)
    n = sum(wl.extend_lens)
    qo = n * s.hq * (s.lq + s.lv) * 2 + n * s.hq * 4
    return keys * s.hkv * kv_row + idx + qo


def decode_bytes(wl: W.Workload, kv_elem_bytes: int = 2) -> float:
    s = wl.spec
    kv_row = (s.lq if s.v_aliases_k else s.lq + s.lv) * kv_elem_bytes
    keys = 0
    for p in wl.prefix_lens:
        T = p + 1
        keys += T if s.sliding_window <= 0 else min(T, s.sliding_window + 1)
    return keys * s.hkv * kv_row + 4 * keys + wl.batch * s.hq * ((s.lq + s.lv) * 2 + 4)


# ------------------------------------------------------------------ peaks
def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), float(d["bf16_tflops_sustained"]), "measured"
    except Exception:
        return 6800.0, 1900.0, 1700.0, "fallback"


# ------------------------------------------------------------ clock sampler
class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled every 20 ms while the
    timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    @staticmethod
    def smi_id(gpu_index: int) -> str:
        """nvidia-smi's name for CUDA device ``gpu_index``: its UUID when
        nvidia-smi lists it (nvidia-smi ignores CUDA_VISIBLE_DEVICES, so the
        CUDA index can name another GPU), else the index itself."""
        try:
            uuid = "GPU-" + str(torch.cuda.get_device_properties(gpu_index).uuid)
            listed = subprocess.run(["nvidia-smi", "--query-gpu=uuid", "--format=csv,noheader"],
                                    capture_output=True, text=True, timeout=20).stdout.split()
            if uuid in listed:
                return uuid
        except Exception:
            pass
        return str(gpu_index)

    def __init__(self, gpu_index: int):
        self.samples = []
        self.window = None
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "20", "-i", self.smi_id(gpu_index)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.time(), line.strip()))

    def mark(self, t0, t1):
        self.window = (t0, t1)

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.05)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        t0, t1 = self.window or (0, 1e30)
        mhz, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        inside = [s for t, s in self.samples if t0 - 0.025 <= t <= t1 + 0.025]
        if not inside:  # timed region shorter than the sampling period
            inside = [s for _, s in self.samples][-3:]
        for s in inside:
            parts = [x.strip() for x in s.split(",")]
            if len(parts) < 9:
                continue
            try:
                mhz.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for nm, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(nm)
        if not mhz:
            return None
        return {"sm_mhz": statistics.median(mhz), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(mhz)}


# -------------------------------------------------------------- distributed
def dist_setup():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if ws > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend)
    return ws, rank, local


def barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, ws: int, dev) -> float:
    if ws == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ------------------------------------------------------------ reference arm
def oracle_sample_rows(wl, count, seed):
    g = torch.Generator().manual_seed(seed)
    total = wl.n_q_tokens * wl.spec.hq
    return torch.randperm(total, generator=g)[:min(count, total)].sort().values


def oracle_rate(wl, rows, k_ext, v_ext, kb, vb):
    """Run the oracle on the given (token*Hq + head) rows; return (seconds,
    flops)."""
    import oracle
    s = wl.spec
    t0 = time.perf_counter()
    oracle.extend_attention(wl.q, k_ext, v_ext, kb, vb, wl.qo_indptr, wl.kv_indptr,
                            wl.kv_indices, wl.sm_scale, s.logit_cap, s.sliding_window, rows=rows,
                            custom_mask=wl.custom_mask, mask_indptr=wl.mask_indptr,
                            sinks=None if wl.sinks is None else wl.sinks.double())
    dt = time.perf_counter() - t0
    tok = rows // s.hq
    if wl.custom_mask is not None:
        pairs = int(mask_visible_per_token(wl)[tok].sum())
    else:
        pairs = visible_pairs(s, wl.prefix_lens, wl.extend_lens, rows=tok)
    return dt, 2.0 * (s.lq + s.lv) * pairs


def calibrate_rows(wl, k_ext, v_ext, kb, vb, target_s):
    rows = oracle_sample_rows(wl, 256, seed=1)
    dt, fl = oracle_rate(wl, rows, k_ext, v_ext, kb, vb)
    per_row = dt / rows.numel()
    return max(64, min(wl.n_q_tokens * wl.spec.hq, int(target_s / max(per_row, 1e-9))))


def run_reference(args, ws, rank):
    if rank != 0:
        return 0
    import oracle
    oracle.build()
    name = args.workload if not W.SPECS[args.workload].decode else WORKLOAD
    wl = W.draw(W.SPECS[name])
    k_ext, v_ext = wl.extend_kv()
    kb, vb = wl.pool()
    # size each step so the whole run stays within about two minutes
    nrows = calibrate_rows(wl, k_ext, v_ext, kb, vb,
                           target_s=min(4.0, 120.0 / max(1, args.steps)))
    for w in range(args.warmup):
        oracle_rate(wl, oracle_sample_rows(wl, max(64, nrows // 8), seed=100 + w), k_ext, v_ext, kb, vb)
    tot_t = tot_f = 0.0
    for k in range(args.steps):
        dt, fl = oracle_rate(wl, oracle_sample_rows(wl, nrows, seed=1000 + k), k_ext, v_ext, kb, vb)
        tot_t += dt
        tot_f += fl
    value = tot_f / tot_t / 1e12
    cores = oracle.num_threads()
    sample = (f"{nrows} random (token, q-head) rows of the {name} workload per step "
              f"(of {wl.n_q_tokens * wl.spec.hq}); float64 oracle")
    line = {
        "impl": "reference", "metric": "extend-attn TFLOP/s", "value": value, "unit": "TFLOP/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": tot_t / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": config_dict(wl),
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


WORKLOAD_TEXT = {
    "llama3_8b": "batch=16 Hq=32 Hkv=8 D=128 prefix~U[0,4096] extend~U[1,1024] pool=2^18 slots "
                 "(permuted) bf16 N(0,1) sm_scale=1/sqrt(128)",
    "long_prefix": "batch=64 Hq=32 Hkv=8 D=128 prefix=8192 extend=16 pool=2^20 slots (permuted) "
                   "bf16 N(0,1) logit_cap=30",
    "mla": "batch=8 Hq=16 Hkv=1 Lq=576 (512+64 rope) Lv=512 (V aliases K) prefix=2048 extend=512 "
           "pool=65536 slots (permuted) bf16 N(0,0.5) sm_scale=1/sqrt(192)",
    "heavy_tail": "256 seqs Hq=28 Hkv=4 D=128 prefix,extend~lognormal(6,1.2) clipped [0,16384]/"
                  "[1,4096] sliding_window=4096 pool=2^22 slots (permuted) bf16 N(0,1)",
    "tiny": "batch=2 Hq=4 Hkv=2 D=64 prefix={16,0} extend={8,5} pool=64 slots sm_scale=1/8",
    "decode_gqa": "decode: batch=64 Hq=32 Hkv=8 D=128 T=8193 pool=2^20 slots (permuted)",
    "decode_mla": "decode: batch=64 Hq=16 Hkv=1 Lq=576 Lv=512 (V aliases K) T=4096 pool=2^20 slots",
    "spec_verify": "batch=64 Hq=32 Hkv=8 D=128 prefix~U[1024,4096] extend=64 draft-tree tokens "
                   "under a custom mask (prefix + ancestors + self) pool=2^20 slots (permuted)",
    "split_192": "batch=16 Hq=16 Hkv=16 Lq=192 (128+64 rope) Lv=128 prefix~U[0,4096] "
                 "extend~U[1,1024] pool=2^18 slots (permuted) bf16 N(0,1) sm_scale=1/sqrt(192)",
    "split_288": "batch=16 Hq=16 Hkv=4 Lq=288 (256+32 rope) Lv=256 prefix~U[0,4096] "
                 "extend~U[1,1024] pool=2^18 slots (permuted) bf16 N(0,1) sm_scale=1/sqrt(288)",
    "sinks_swa": "batch=16 Hq=64 Hkv=8 D=64 prefix~U[0,4096] extend~U[1,1024] sliding_window=128 "
                 "sink logit per head ~N(0,1.5) pool=2^18 slots (permuted)",
}


def config_dict(wl):
    s = wl.spec
    step = ("decode_attention_fwd" if s.decode else
            "build_unified_kv_indices + extend_attention_fwd_unified")
    return {"workload": f"{s.name}: {WORKLOAD_TEXT.get(s.name, '')}",
            "batch": s.batch, "q_tokens": wl.n_q_tokens,
            "kv_tokens": int(sum(wl.prefix_lens) + sum(wl.extend_lens)),
            "seed": s.seed, "l2": "flushed before every timed step (512 MiB write, then read back so the evicted lines are clean)",
            "step": step}


# ------------------------------------------------------------- our arm
class ExtendStep:
    """Device-resident inputs and the one-step call sequence (unified
    index build + unified extend attention)."""

    def __init__(self, wl: W.Workload, dev, fp8=None):
        from paged_kv_extend_gb300 import pkx
        self.pkx = pkx
        s = wl.spec
        self.wl = wl
        self.dev = dev
        self.kv_scales = {"k_scale": FP8_SCALE, "v_scale": FP8_SCALE} if fp8 is not None else {}
        self.kb, self.vb = (wl.pool(dev) if fp8 is None
                            else wl.pool_fp8(fp8, FP8_SCALE, FP8_SCALE, dev))
        self.q = wl.q.to(dev)
        self.prefix_indptr = wl.kv_indptr.to(dev)
        self.prefix_indices = wl.kv_indices.to(dev)
        self.extend_start = wl.extend_start_loc.to(dev)
        self.extend_lens = wl.extend_seq_lens.to(dev)
        self.extend_indices = wl.extend_kv_indices.to(dev)
        self.qo_indptr = wl.qo_indptr.to(dev)
        n = wl.n_q_tokens
        self.uptr = torch.empty(wl.batch + 1, dtype=torch.int32, device=dev)
        self.uidx = torch.empty(self.prefix_indices.numel() + self.extend_indices.numel(),
                                dtype=torch.int64, device=dev)
        self.plen = torch.empty(wl.batch, dtype=torch.int32, device=dev)
        self.o = torch.empty(n, s.hq, s.lv, dtype=torch.bfloat16, device=dev)
        self.lse = torch.empty(n, s.hq, dtype=torch.float32, device=dev)
        nbytes = pkx.extend_workspace_size(wl.batch, n, s.hq, s.hkv, s.lq, s.lv)
        self.ws = torch.empty(nbytes, dtype=torch.uint8, device=dev)
        self.custom_mask = wl.custom_mask.to(dev) if wl.custom_mask is not None else None
        self.mask_indptr = wl.mask_indptr.to(dev) if wl.mask_indptr is not None else None
        self.sinks = wl.sinks.to(dev).float() if wl.sinks is not None else None
        self.launches = 4  # index build, scheduler, attention, combine
        self.tokens = wl.n_q_tokens  # query (extend) tokens of one step
        self.flops = extend_flops(wl)
        self.bytes = extend_bytes(wl, unified=True, kv_elem_bytes=1 if fp8 is not None else 2)

    def inputs(self):
        ins = [self.q, self.prefix_indptr, self.prefix_indices, self.extend_start,
               self.extend_lens, self.extend_indices, self.qo_indptr]
        if self.custom_mask is not None:  # the draft tree changes every step
            ins += [self.custom_mask, self.mask_indptr]
        return ins

    def twin(self):
        """The same step over the same pool with its own input, output and
        workspace buffers (double buffering of the end-to-end loop)."""
        t = copy.copy(self)
        for name in ("q", "prefix_indptr", "prefix_indices", "extend_start", "extend_lens",
                     "extend_indices", "qo_indptr", "uptr", "uidx", "plen", "o", "lse", "ws",
                     "custom_mask", "mask_indptr"):
            if getattr(self, name) is not None:
                setattr(t, name, torch.empty_like(getattr(self, name)))
        return t

    def __call__(self):
        s = self.wl.spec
        self.pkx.build_unified_kv_indices(self.prefix_indptr, self.prefix_indices,
                                          self.extend_start, self.extend_lens,
                                          self.extend_indices, self.wl.batch,
                                          out=(self.uptr, self.uidx, self.plen))
        self.pkx.extend_attention_fwd_unified(
            self.q, self.o, self.kb, self.vb, self.qo_indptr, self.uptr, self.uidx, self.plen,
            self.wl.sm_scale, s.logit_cap, s.sliding_window, lse=self.lse, workspace=self.ws,
            custom_mask=self.custom_mask, mask_indptr=self.mask_indptr, sinks=self.sinks,
            **self.kv_scales)


class DecodeStep:
    """One decode step over a decode workload (one query per sequence)."""

    def __init__(self, wl: W.Workload, dev, fp8=None):
        from paged_kv_extend_gb300 import pkx
        self.pkx = pkx
        s = wl.spec
        self.wl = wl
        self.kv_scales = {"k_scale": FP8_SCALE, "v_scale": FP8_SCALE} if fp8 is not None else {}
        self.kb, self.vb = (wl.pool(dev) if fp8 is None
                            else wl.pool_fp8(fp8, FP8_SCALE, FP8_SCALE, dev))
        self.q = wl.q.to(dev)
        self.kvp, self.kvi = wl.kv_indptr.to(dev), wl.kv_indices.to(dev)
        self.o = torch.empty(s.batch, s.hq, s.lv, dtype=torch.bfloat16, device=dev)
        self.lse = torch.empty(s.batch, s.hq, dtype=torch.float32, device=dev)
        self.ws = torch.empty(pkx.decode_workspace_size(s.batch, s.hq, s.hkv, s.lq, s.lv),
                              dtype=torch.uint8, device=dev)
        self.launches = 3  # scheduler, attention, combine
        self.tokens = s.batch  # one new token per sequence
        self.flops = 2.0 * (s.lq + s.lv) * s.hq * sum(
            min(p + 1, s.sliding_window + 1) if s.sliding_window > 0 else p + 1
            for p in wl.prefix_lens)
        self.bytes = decode_bytes(wl, kv_elem_bytes=1 if fp8 is not None else 2)

    def inputs(self):
        return [self.q, self.kvp, self.kvi]

    def twin(self):
        t = copy.copy(self)
        for name in ("q", "kvp", "kvi", "o", "lse", "ws"):
            setattr(t, name, torch.empty_like(getattr(self, name)))
        return t

    def __call__(self):
        s = self.wl.spec
        self.pkx.decode_attention_fwd(self.q, self.o, self.kb, self.vb, self.kvp, self.kvi,
                                      self.wl.sm_scale, s.logit_cap, s.sliding_window,
                                      lse=self.lse, workspace=self.ws, **self.kv_scales)


# k_scale = v_scale of the fp8-pool measurements (N(0, 1) rows stay in range)
FP8_SCALE = 0.5


def make_step(name, dev, fp8=None):
    wl = W.draw(W.SPECS[name])
    return (DecodeStep if wl.spec.decode else ExtendStep)(wl, dev, fp8=fp8)


def flush_l2(flush):
    """Evict L2: write the 512 MiB buffer (about four times L2), then read it
    back, so that the lines left in L2 are clean ones of this buffer and the
    timed kernel pays for no write-back of the flush's own dirty lines."""
    flush.zero_()
    flush.view(torch.int64).sum()


def time_steps(step, steps, flush, dev, attn_events=False, pkx=None):
    """Per-step device time (ms) with CUDA events on the current stream, L2
    flushed before each step outside the events.  With ``attn_events`` a
    second loop of the same steps times the attention kernel alone (events
    recorded around it inside the library); the step times come from the
    first, uninstrumented loop, since an event between two kernels keeps the
    second from starting early."""
    def loop(instrumented):
        starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
        ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
        ab = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
        ae = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
        for e in ab + ae:
            e.record()
        torch.cuda.synchronize(dev)
        for k in range(steps):
            flush_l2(flush)
            if instrumented:
                pkx.set_attention_events(ab[k], ae[k])
            starts[k].record()
            step()
            ends[k].record()
        if instrumented:
            pkx.set_attention_events(None, None)
        torch.cuda.synchronize(dev)
        return ([s.elapsed_time(e) for s, e in zip(starts, ends)],
                [s.elapsed_time(e) for s, e in zip(ab, ae)])
    step_ms, _ = loop(False)
    attn_ms = loop(True)[1] if attn_events else None
    return step_ms, attn_ms


def measure_e2e(step: ExtendStep, steps, warmup, flush, dev):
    """Same metric through the public API with host buffers: every step
    copies its inputs (q, prefix indptr/indices, extend starts/lens/indices,
    qo_indptr) from pinned host memory, runs the step and reads o back into
    pinned host memory.  The KV pool is device-resident state (it is the
    cache), as in serving."""
    pin = lambda t: t.cpu().pin_memory()
    dev_in = step.inputs()
    host_in = [pin(t) for t in dev_in]
    host_o = torch.empty(step.o.shape, dtype=step.o.dtype).pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in host_in)
    d2h = host_o.numel() * host_o.element_size()

    def e2e_step():
        for h, d in zip(host_in, dev_in):
            d.copy_(h, non_blocking=True)
        step()
        host_o.copy_(step.o, non_blocking=True)

    for _ in range(warmup):
        e2e_step()
    ms, _ = time_steps(e2e_step, steps, flush, dev)
    return sum(ms) / len(ms), h2d, d2h


def measure_e2e_pipelined(step, steps, warmup, flush, dev):
    """The end-to-end loop as a server runs it: step i's inputs are copied
    host-to-device on one stream while step i-1 computes, and step i's o is
    copied back on another stream while step i+1 computes (two device
    buffer sets alternate).  Every step's own copies and the L2 flush before
    its compute are inside the timed region; time per step = total / steps."""
    pin = lambda t: t.cpu().pin_memory()
    pair = (step, step.twin())
    host_in = [pin(t) for t in step.inputs()]
    host_o = [torch.empty(st.o.shape, dtype=st.o.dtype).pin_memory() for st in pair]
    comp = torch.cuda.current_stream(dev)
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)

    def run(n):
        ev = lambda: torch.cuda.Event()
        h2d_done, comp_done, d2h_done = [ev() for _ in range(n)], [ev() for _ in range(n)], \
            [ev() for _ in range(n)]
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        t0.record(s_in)
        for i in range(n):
            st = pair[i & 1]
            with torch.cuda.stream(s_in):
                if i >= 2:
                    s_in.wait_event(comp_done[i - 2])  # this buffer set's inputs are free
                for h, d in zip(host_in, st.inputs()):
                    d.copy_(h, non_blocking=True)
                h2d_done[i].record(s_in)
            comp.wait_event(h2d_done[i])
            if i >= 2:
                comp.wait_event(d2h_done[i - 2])  # this buffer set's o has been read
            flush.zero_()
            st()
            comp_done[i].record(comp)
            with torch.cuda.stream(s_out):
                s_out.wait_event(comp_done[i])
                host_o[i & 1].copy_(st.o, non_blocking=True)
                d2h_done[i].record(s_out)
        s_out.wait_event(d2h_done[n - 1])
        t1.record(s_out)
        torch.cuda.synchronize(dev)
        return t0.elapsed_time(t1) / n

    run(max(warmup, 2))
    ms = run(steps)
    # the copies really carried the data: the last o read back equals the device o
    last = pair[(steps - 1) & 1]
    assert torch.equal(host_o[(steps - 1) & 1], last.o.cpu()), "pipelined e2e lost data"
    return ms


def e2e_entry(pipelined, serial, unit, h2d, d2h):
    """The end-to-end figure: the faster of the two host loops, named, with
    the other one beside it."""
    modes = {
        "pipelined": "step i's H2D and D2H run on copy streams while the neighbouring steps "
                     "compute (two device buffer sets); each step's copies and its L2 flush "
                     "are inside the timed region",
        "serial": "per step: H2D of the inputs, the step, D2H of o, in order on one stream "
                  "(L2 flushed before each step, outside the events)",
    }
    best = "pipelined" if pipelined >= serial else "serial"
    return {"value": max(pipelined, serial), "unit": unit, "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "mode": f"{best}: {modes[best]}",
            "pipelined_value": pipelined, "serial_value": serial}


def measure_component(name, dev, flush, steps, hbm_peak, bf16_peak, fp8=None):
    """One workload's step, device-timed, with the attention kernel's own
    time; TFLOP/s and GB/s of algorithmic work and the roofline fractions.
    fp8: the pool in that torch float8 dtype (k_scale = v_scale = 0.5)."""
    from paged_kv_extend_gb300 import pkx
    step = make_step(name, dev, fp8=fp8)
    for _ in range(3):
        step()
    ms, attn = time_steps(step, steps, flush, dev, attn_events=True, pkx=pkx)
    status = pkx.workspace_status(step.ws)
    m, a = sum(ms) / len(ms), sum(attn) / len(attn)
    pool = "" if fp8 is None else f" [pool {str(fp8).replace('torch.', '')}, scales {FP8_SCALE}]"
    out = {"workload": f"{name}: {WORKLOAD_TEXT.get(name, '')}{pool}", "ms": m, "attn_kernel_ms": a,
           "tokens/s": step.tokens / (m * 1e-3),
           "TFLOP/s": step.flops / (m * 1e-3) / 1e12,
           "attn_kernel_TFLOP/s": step.flops / (a * 1e-3) / 1e12,
           "GB/s": step.bytes / (m * 1e-3) / 1e9,
           "attn_kernel_GB/s": step.bytes / (a * 1e-3) / 1e9,
           "frac_of_bf16_peak": step.flops / (a * 1e-3) / 1e12 / bf16_peak,
           "frac_of_hbm": step.bytes / (a * 1e-3) / 1e9 / hbm_peak,
           "algorithmic_flops": step.flops, "algorithmic_bytes": step.bytes,
           "status": status}
    del step
    torch.cuda.empty_cache()
    return out


def time_launches(fn, steps, flush, dev):
    """Mean device time (ms) of ``fn`` with CUDA events on the current
    stream, L2 flushed before each launch outside the events."""
    for _ in range(3):
        fn()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    torch.cuda.synchronize(dev)
    for k in range(steps):
        flush_l2(flush)
        starts[k].record()
        fn()
        ends[k].record()
    torch.cuda.synchronize(dev)
    return sum(s.elapsed_time(e) for s, e in zip(starts, ends)) / steps


def measure_kv_ops(dev, flush, steps, hbm_peak):
    """The steps on either side of the attention call, each on its own:
    the KV write of a batch's extend tokens into the pool (set_kv_buffer)
    and the KV-index gather from the request-to-token table, for the
    default extend batch and for the long-prefix batch.  HBM GB/s of
    algorithmic bytes (every byte read or written once) and the fraction of
    the measured copy bandwidth."""
    from paged_kv_extend_gb300 import pkx
    out = {}
    for name in ("llama3_8b", "long_prefix"):
        wl = W.draw(W.SPECS[name])
        s = wl.spec
        kb, vb = wl.pool(dev)
        k_ext, v_ext = wl.extend_kv(dev)
        loc = wl.extend_kv_indices.to(dev, torch.int64)
        n = loc.numel()
        ms = time_launches(lambda: pkx.set_kv_buffer(kb, vb, loc, k_ext, v_ext), steps, flush, dev)
        nbytes = 2.0 * n * s.hkv * (s.lq + s.lv) * 2 + 8.0 * n
        out[f"set_kv_buffer/{name}"] = {
            "what": f"{n} extend tokens x {s.hkv} KV heads x (K {s.lq} + V {s.lv}) bf16 into "
                    f"a {s.num_slots}-slot pool at random slots",
            "ms": ms, "GB/s": nbytes / (ms * 1e-3) / 1e9,
            "frac_of_hbm": nbytes / (ms * 1e-3) / 1e9 / hbm_peak,
            "algorithmic_bytes": nbytes}
        del kb, vb, k_ext, v_ext
        table, rpi, seq = wl.req_to_token(seed=1)
        table, rpi, seq = table.to(dev), rpi.to(dev), seq.to(dev)
        total = int(sum(p + e for p, e in zip(wl.prefix_lens, wl.extend_lens)))
        kvp = torch.empty(wl.batch + 1, dtype=torch.int32, device=dev)
        kvi = torch.empty(total, dtype=torch.int32, device=dev)
        ms = time_launches(lambda: pkx.create_kv_indices(table, rpi, seq, None, kv_indptr=kvp,
                                                         kv_indices=kvi), steps, flush, dev)
        nbytes = 8.0 * total + 16.0 * wl.batch + 4.0 * (wl.batch + 1)
        out[f"create_kv_indices/{name}"] = {
            "what": f"{wl.batch} sequences, {total} indices gathered from a "
                    f"{tuple(table.shape)} request-to-token table",
            "ms": ms, "GB/s": nbytes / (ms * 1e-3) / 1e9,
            "frac_of_hbm": nbytes / (ms * 1e-3) / 1e9 / hbm_peak,
            "algorithmic_bytes": nbytes}
        del table, rpi, seq, kvp, kvi
        torch.cuda.empty_cache()
    # a page table of 16-slot pages for the decode batch (64 x 8193 keys)
    ps = 16
    wl = W.draw(W.SPECS["decode_gqa"])
    t = [p + 1 for p in wl.prefix_lens]
    n_pages = [(x + ps - 1) // ps for x in t]
    g = torch.Generator().manual_seed(5)
    page_ids = torch.randperm(wl.spec.num_slots // ps, generator=g)[: sum(n_pages)]
    ptr = torch.tensor([0] + list(torch.tensor(n_pages).cumsum(0)), dtype=torch.int32, device=dev)
    ids = page_ids.to(device=dev, dtype=torch.int32)
    last = torch.tensor([x - (n - 1) * ps for x, n in zip(t, n_pages)], dtype=torch.int32,
                        device=dev)
    tptr = torch.empty(wl.batch + 1, dtype=torch.int32, device=dev)
    tidx = torch.empty(sum(t), dtype=torch.int32, device=dev)
    ms = time_launches(lambda: pkx.expand_paged_kv_indices(ptr, ids, last, ps, token_indptr=tptr,
                                                           token_indices=tidx), steps, flush, dev)
    nbytes = 4.0 * sum(t) + 4.0 * sum(n_pages) + 8.0 * wl.batch + 4.0 * (wl.batch + 1)
    out["expand_paged_kv_indices/decode_gqa"] = {
        "what": f"{wl.batch} sequences, {sum(n_pages)} pages of {ps} -> {sum(t)} token slots",
        "ms": ms, "GB/s": nbytes / (ms * 1e-3) / 1e9,
        "frac_of_hbm": nbytes / (ms * 1e-3) / 1e9 / hbm_peak, "algorithmic_bytes": nbytes}
    return out


def measure_split(dev, flush, steps, bf16_peak, name="llama3_8b"):
    """The two-stage extend call against the ragged + paged + merge_state
    split the pages take for 4096 or more extend tokens, on the same batch
    (same algorithmic FLOPs; device time of the whole call)."""
    from paged_kv_extend_gb300 import pkx
    wl = W.draw(W.SPECS[name])
    s = wl.spec
    kb, vb = wl.pool(dev)
    k_ext, v_ext = wl.extend_kv(dev)
    q, qo = wl.q.to(dev), wl.qo_indptr.to(dev)
    kvp, kvi = wl.kv_indptr.to(dev), wl.kv_indices.to(dev)
    n = wl.n_q_tokens
    o = torch.empty(n, s.hq, s.lv, dtype=torch.bfloat16, device=dev)
    lse = torch.empty(n, s.hq, dtype=torch.float32, device=dev)
    ws2 = torch.empty(pkx.extend_workspace_size(wl.batch, n, s.hq, s.hkv, s.lq, s.lv),
                      dtype=torch.uint8, device=dev)
    wsr = torch.empty(pkx.ragged_paged_workspace_size(wl.batch, n, s.hq, s.hkv, s.lq, s.lv),
                      dtype=torch.uint8, device=dev)
    args = (q, k_ext, v_ext, o, kb, vb, qo, kvp, kvi, wl.sm_scale, s.logit_cap, s.sliding_window)
    flops = extend_flops(wl)
    out = {}
    for label, fn, w in (("two_stage", pkx.extend_attention_fwd, ws2),
                         ("ragged_paged", pkx.extend_attention_fwd_ragged_paged, wsr)):
        ms = time_launches(lambda: fn(*args, lse=lse, workspace=w), steps, flush, dev)
        if pkx.workspace_status(w) != 0:
            raise SystemExit(f"{label}: device status {pkx.workspace_status(w)}")
        out[f"{label}/{name}"] = {
            "what": ("one extend call (scheduler, attention, combine)" if label == "two_stage"
                     else "ragged pass over the extend keys + paged pass over the prefix "
                          "keys + merge_state"),
            "ms": ms, "TFLOP/s": flops / (ms * 1e-3) / 1e12,
            "frac_of_bf16_peak": flops / (ms * 1e-3) / 1e12 / bf16_peak,
            "algorithmic_flops": flops}
    del kb, vb, k_ext, v_ext, ws2, wsr
    torch.cuda.empty_cache()
    return out


def measure_fused_write(dev, flush, steps, bf16_peak, name="llama3_8b"):
    """The two-stage extend call with the KV write fused in (the new tokens'
    K/V rows stored into the pool by the attention kernel's otherwise idle
    warps) against the standalone KV write followed by the two-stage call,
    on the same batch: device time of the whole sequence."""
    from paged_kv_extend_gb300 import pkx
    wl = W.draw(W.SPECS[name])
    s = wl.spec
    kb, vb = wl.pool(dev)
    k_ext, v_ext = wl.extend_kv(dev)
    q, qo = wl.q.to(dev), wl.qo_indptr.to(dev)
    kvp, kvi = wl.kv_indptr.to(dev), wl.kv_indices.to(dev)
    loc = wl.extend_kv_indices.to(dev, torch.int64)
    n = wl.n_q_tokens
    o = torch.empty(n, s.hq, s.lv, dtype=torch.bfloat16, device=dev)
    lse = torch.empty(n, s.hq, dtype=torch.float32, device=dev)
    ws2 = torch.empty(pkx.extend_workspace_size(wl.batch, n, s.hq, s.hkv, s.lq, s.lv),
                      dtype=torch.uint8, device=dev)
    args = (q, k_ext, v_ext, o, kb, vb, qo, kvp, kvi, wl.sm_scale, s.logit_cap, s.sliding_window)
    flops = extend_flops(wl)

    def standalone():
        pkx.set_kv_buffer(kb, vb, loc, k_ext, v_ext)
        pkx.extend_attention_fwd(*args, lse=lse, workspace=ws2)

    def fused():
        pkx.extend_attention_fwd(*args, lse=lse, workspace=ws2, cache_loc=loc)

    out = {}
    for label, fn in (("write_then_extend", standalone), ("fused_write_extend", fused)):
        ms = time_launches(fn, steps, flush, dev)
        if pkx.workspace_status(ws2) != 0:
            raise SystemExit(f"{label}: device status {pkx.workspace_status(ws2)}")
        out[f"{label}/{name}"] = {
            "what": ("set_kv_buffer of the extend rows, then the two-stage call"
                     if label == "write_then_extend" else
                     "the two-stage call with cache_loc (KV write inside the attention kernel)"),
            "ms": ms, "TFLOP/s": flops / (ms * 1e-3) / 1e12,
            "frac_of_bf16_peak": flops / (ms * 1e-3) / 1e12 / bf16_peak,
            "algorithmic_flops": flops}
    del kb, vb, k_ext, v_ext, ws2
    torch.cuda.empty_cache()
    return out


def run_ours(args, ws, rank, local):
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU (the CUDA library has no CPU path)")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    from paged_kv_extend_gb300 import build as pkx_build
    from paged_kv_extend_gb300 import pkx
    if rank == 0:
        pkx_build.build()
    barrier(ws)
    pkx.load_library()
    hbm_peak, bf16_peak, bf16_sus, peak_src = load_peaks()

    step = make_step(args.workload, dev)
    wl = step.wl
    flops = step.flops
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    if pkx.workspace_status(step.ws) != 0:
        raise SystemExit(f"device status {pkx.workspace_status(step.ws)} after warm-up")

    clocks = ClockSampler(local) if rank == 0 else None
    time.sleep(0.2)
    barrier(ws)
    torch.cuda.synchronize(dev)
    t0 = time.time()
    step_ms, attn_ms = time_steps(step, args.steps, flush, dev, attn_events=True, pkx=pkx)
    t1 = time.time()
    barrier(ws)
    if clocks:
        clocks.mark(t0, t1)
    clock_info = clocks.stop() if clocks else None

    ms = sum(step_ms) / len(step_ms)
    ms_max = max_over_ranks(ms, ws, dev)
    attn_avg = sum(attn_ms) / len(attn_ms)
    value = flops * ws / (ms_max * 1e-3) / 1e12
    achieved = flops / (attn_avg * 1e-3) / 1e12

    e2e_serial_ms, h2d, d2h = measure_e2e(step, args.steps, 2, flush, dev)
    e2e_serial_ms = max_over_ranks(e2e_serial_ms, ws, dev)
    e2e_ms = measure_e2e_pipelined(step, args.steps, 2, flush, dev)
    e2e_ms = max_over_ranks(e2e_ms, ws, dev)

    components = {"attn_kernel_share_of_step": attn_avg / ms}
    if not args.no_components:
        names = (args.components.split(",") if args.components
                 else ["long_prefix", "mla", "heavy_tail", "decode_gqa", "decode_mla",
                       "split_192", "split_288", "kv_ops", "split", "fused_write",
                       "decode_gqa_fp8", "llama3_8b_fp8", "mla_fp8", "decode_mla_fp8"])
        if args.all_workloads:
            names = ["long_prefix", "mla", "heavy_tail", "decode_gqa", "decode_mla", "kv_ops",
                     "split", "decode_gqa_fp8", "long_prefix_fp8", "llama3_8b_fp8", "mla_fp8",
                     "decode_mla_fp8"]
        for name in names:
            if name == args.workload:
                continue
            if name.endswith("_fp8"):
                components[name] = measure_component(name[:-4], dev, flush,
                                                     max(5, min(args.steps, 20)), hbm_peak,
                                                     bf16_peak, fp8=torch.float8_e4m3fn)
                continue
            if name == "split":
                components.update(measure_split(dev, flush, max(5, min(args.steps, 20)),
                                                bf16_peak))
                continue
            if name == "fused_write":
                components.update(measure_fused_write(dev, flush, max(5, min(args.steps, 20)),
                                                      bf16_peak))
                continue
            if name == "kv_ops":
                components.update(measure_kv_ops(dev, flush, max(5, min(args.steps, 50)),
                                                 hbm_peak))
                continue
            components[name] = measure_component(name, dev, flush, max(5, min(args.steps, 20)),
                                                 hbm_peak, bf16_peak)

    cpu = None
    if rank == 0 and ws == 1 and not args.no_cpu_baseline and not wl.spec.decode:
        import oracle
        oracle.build()
        k_ext, v_ext = wl.extend_kv()
        kb, vb = wl.pool()
        nrows = calibrate_rows(wl, k_ext, v_ext, kb, vb, target_s=10.0)
        rows = oracle_sample_rows(wl, nrows, seed=4242)
        dt, fl = oracle_rate(wl, rows, k_ext, v_ext, kb, vb)
        cpu = {"value": fl / dt / 1e12, "unit": "TFLOP/s", "cores": oracle.num_threads(),
               "kind": "oracle",
               "sample": f"{nrows} random (token, q-head) rows of {wl.n_q_tokens * wl.spec.hq}, "
                         f"{dt:.1f} s of float64 CPU work"}

    traffic = None
    prof = os.path.join(ROOT, "profiles", f"attn_kernel_{args.workload}.md")
    if os.path.exists(prof):
        import hashlib
        src = b"".join(open(os.path.join(ROOT, "paged_kv_extend_gb300", "csrc", f), "rb").read()
                       for f in ("attention.cu", "ptx.cuh"))
        h = hashlib.sha1(src).hexdigest()[:12]
        for line in open(prof):
            if line.startswith("traffic_bytes_per_launch:"):
                parts = line.split()
                # sha1: the kernel sources the counters belong to; a later
                # source whose change leaves this kernel's code as it was is
                # listed after it, with the reason in the profile
                if len(parts) >= 4 and h in parts[3:]:
                    traffic = float(parts[1])

    if wl.spec.decode:
        metric, unit = "decode-shape HBM GB/s", "GB/s"
        value = step.bytes * ws / (ms_max * 1e-3) / 1e9
        roof = {"bound": "hbm", "achieved": step.bytes / (attn_avg * 1e-3) / 1e9,
                "peak": hbm_peak, "unit": "GB/s",
                "frac": step.bytes / (attn_avg * 1e-3) / 1e9 / hbm_peak, "traffic": traffic,
                "peak_source": f"hbm_gbs copy bandwidth, of {peak_src}",
                "kernel": "attn_kernel (decode)", "algorithmic_bytes_per_launch": step.bytes}
        e2e_value = step.bytes * ws / (e2e_ms * 1e-3) / 1e9
        e2e_serial = step.bytes * ws / (e2e_serial_ms * 1e-3) / 1e9
    else:
        metric, unit = "extend-attn TFLOP/s", "TFLOP/s"
        roof = {"bound": "tensor", "achieved": achieved, "peak": bf16_peak,
                "unit": "TFLOP/s", "frac": achieved / bf16_peak, "traffic": traffic,
                "peak_source": f"bf16_tflops burst, of {peak_src}",
                "kernel": "mla_pair_kernel<unified>" if wl.spec.lq == 576 else "attn_kernel<unified>",
                "algorithmic_flops_per_launch": flops,
                "algorithmic_bytes_per_launch": step.bytes}
        e2e_value = flops * ws / (e2e_ms * 1e-3) / 1e12
        e2e_serial = flops * ws / (e2e_serial_ms * 1e-3) / 1e12
    line = {
        "metric": metric, "value": value, "unit": unit, "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_max,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic", "config": config_dict(wl),
        "roofline": roof,
        "cpu_baseline": cpu,
        "e2e": e2e_entry(e2e_value, e2e_serial, unit, h2d, d2h),
        "tokens_per_s": step.tokens * ws / (ms_max * 1e-3),
        "gpu_launches": step.launches * args.steps,
        "clocks": clock_info,
        "components": components,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-components", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--components", default="",
                    help="comma-separated components to measure besides the step (workload "
                         "names, a workload name + _fp8 for an e4m3 pool, kv_ops, split; "
                         "default decode_gqa,mla,kv_ops,split,decode_gqa_fp8)")
    ap.add_argument("--workload", default=WORKLOAD, choices=sorted(W.SPECS),
                    help="workload of the timed step (default: the Llama-3-8B-shaped layer)")
    ap.add_argument("--all-workloads", action="store_true",
                    help="also measure every other workload as a component")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    ws, rank, local = dist_setup()
    if args.impl == "reference":
        rc = run_reference(args, ws, rank)
    else:
        rc = run_ours(args, ws, rank, local)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return rc


if __name__ == "__main__":
    sys.exit(main())
