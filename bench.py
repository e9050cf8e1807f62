#!/usr/bin/env python
"""Throughput of fused attention forward + backward on one GB300.

A step is one pass of the whole hot path over one batch: segment metadata,
forward (O, LSE), backward preprocess, dK/dV pass (+ atomic dQ) and the dQ
conversion, all through the C ABI on device-resident inputs.  The headline
workload is the packed THD GQA configuration (2 rows x 8192 tokens, segments of
U[64,2048] tokens, 5 % padding, Hq=32, Hkv=8, D=128, packed QKV, causal).

Metric: algorithmic TFLOP/s (exact unmasked-pair count, five-GEMM backward
convention) and the fraction of the measured bf16 dense tensor peak.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

With N > 1 (torchrun) every rank runs an independent replica of the workload
(the path needs no exchange); timings are the max over ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "fused attn fwd+bwd TFLOP/s (BF16, causal-adj) and % of tensor-core peak, 1 GB300"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
WORKLOAD_DESC = {
    "thd_gqa": "packed THD GQA: 2 rows x 8192 tokens, segments U[64,2048] (last truncated), "
               "5% padding tail, Hq=32, Hkv=8, D=128, packed QKV (3HD), causal within segments",
    "bshd": "dense BSHD: B=4, S=2048, Hq=Hkv=16, D=128, separate Q/K/V, causal",
    "cross_bias": "cross-attention: B=2, Sq=4096, Skv=8192, Hq=Hkv=16, d_qk=192, d_v=128, "
                  "independent Q/KV segments U[128,4096], bias [1,16,4096,8192] with dBias",
    "long_kv": "long context: B=1, S=32768, Hq=64, Hkv=8, D=128, packed KV (HD_2HD), causal",
    "tiny": "tiny: B=2, S=128, H=2, D=64, two segments + padding per row, causal",
}


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1500)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="thd_gqa")
    ap.add_argument("--dq-mode", default="deterministic", choices=["atomic", "deterministic"])
    ap.add_argument("--force-general", action="store_true",
                    help="run the general (per-token) metadata path even where the fast "
                         "path applies, to measure what not taking it costs")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-other-workloads", action="store_true",
                    help="skip the other named workloads measured after the headline one")
    ap.add_argument("--no-extras", action="store_true",
                    help="skip the deterministic-mode and per-pass side measurements")
    return ap.parse_args()


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return FALLBACK_PEAKS, "fallback"


# kernel sources behind each roofline entry: a recorded DRAM traffic figure
# stays valid while these files are unchanged
KERNEL_SOURCES = {
    "dkdv": ("dkdv128.cu",),
    "dq": ("dq128.cu",),
    "fwd": ("fwd2t.cu",),
    "bwd_pre": ("bwd.cu",),
    "fwd_fp8": ("fwd_fp8.cu",),
}
COMMON_SOURCES = ("attn_internal.cuh", "chunk_mask.h", "sm103_ptx.cuh", "debug_checks.h")


def source_hash(kernel):
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "bwd_tcgen05_tma_gb300", "csrc")
    for n in sorted(KERNEL_SOURCES.get(kernel, ()) + COMMON_SOURCES):
        with open(os.path.join(csrc, n), "rb") as f:
            h.update(n.encode() + f.read())
    return h.hexdigest()[:16]


# --------------------------------------------------------------------- clocks


class ClockSampler:
    """nvidia-smi samples every 200 ms while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = os.path.join("/tmp", f"bench_clocks_{os.getpid()}.csv")

    def snapshot(self):
        """One immediate sample, appended to the same record (taken right before
        and right after the timed region, so even a short region has samples
        at its edges)."""
        try:
            with open(self.path, "a") as f:
                subprocess.run(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                                "--format=csv,noheader,nounits"], stdout=f,
                               stderr=subprocess.DEVNULL, timeout=10)
        except (OSError, subprocess.SubprocessError):
            pass

    def start(self):
        self.snapshot()
        try:
            self.f = open(self.path, "a")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"], stdout=self.f,
                stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.f.close()
        self.snapshot()
        sm, smax, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    smax.append(float(parts[2]))
                except ValueError:
                    continue
                for n, v in zip(names, parts[5:9]):
                    if v.lower().startswith("active"):
                        reasons.add(n)
        os.unlink(self.path)
        out = {"sm_mhz": statistics.median(sm) if sm else None,
               "sm_max_mhz": max(smax) if smax else None, "samples": len(sm),
               "reasons": sorted(reasons)}
        if len(sm) < 5:
            # too few samples to tie the number to a clock: a longer run
            # (--steps) gives one every 200 ms
            out["few_samples"] = True
        return out


# --------------------------------------------------------------------- device setup


class Problem:
    """Device buffers of one workload plus the C-ABI parameter block."""

    def __init__(self, case, dq_mode, force_general=False, pin=True):
        import numpy as np
        import torch

        from bwd_tcgen05_tma_gb300 import attn as A
        from bwd_tcgen05_tma_gb300 import inputs as I

        self.case = c = case

        def bf(x):
            return torch.from_numpy(I.bf16_bits(x).view(np.int16)).view(torch.bfloat16)

        def i32(x):
            return None if x is None else torch.from_numpy(np.ascontiguousarray(x, np.int32))

        # host copies (pinned for the end-to-end steps) and device copies of every input
        pm = (lambda t: t.pin_memory()) if pin else (lambda t: t)
        self.host_in = {k: pm(bf(v)) for k, v in c.buffers.items()}
        self.host_in["do"] = pm(bf(c.do.reshape(c.B * c.Sq, c.Hq, c.d_v)))
        if c.bias is not None:
            self.host_in["bias"] = pm(bf(c.bias))
        for k in ("q_ids", "q_pos", "kv_ids", "kv_pos"):
            t = i32(getattr(c, k))
            if t is not None:
                self.host_in[k] = pm(t)
        self.dev = {k: v.cuda() for k, v in self.host_in.items()}
        d = self.dev
        if c.layout == "3HD":
            q, k, v = d["qkv"], None, None
        elif c.layout == "HD_2HD":
            q, k, v = d["q"], d["kv"], None
        else:
            q, k, v = d["q"], d["k"], d["v"]
        self.params = A.make_params(
            layout=c.layout, fmt=c.fmt, mask=c.mask, B=c.B, Sq=c.Sq, Skv=c.Skv, Hq=c.Hq,
            Hkv=c.Hkv, d_qk=c.d_qk, d_v=c.d_v, scale=c.scale, q=q, k=k, v=v,
            q_seg_ids=d.get("q_ids"), q_seg_pos=d.get("q_pos"), kv_seg_ids=d.get("kv_ids"),
            kv_seg_pos=d.get("kv_pos"), bias=d.get("bias"), dq_mode=dq_mode,
            force_general_path=force_general,
            metadata_from_forward=True)  # one workspace: the backward reuses the metadata
        ws = max(A.attn_fwd_workspace_size(self.params), A.attn_bwd_workspace_size(self.params))
        self.ws = torch.empty(ws, dtype=torch.uint8, device="cuda")
        self.o = torch.empty((c.B * c.Sq, c.Hq, c.d_v), dtype=torch.bfloat16, device="cuda")
        self.lse = torch.empty((c.B, c.Hq, c.Sq), dtype=torch.float32, device="cuda")
        if c.layout == "3HD":
            self.grads = {"dqkv": torch.empty_like(d["qkv"])}
            self.gptr = (self.grads["dqkv"], None, None)
        elif c.layout == "HD_2HD":
            self.grads = {"dq": torch.empty_like(d["q"]), "dkv": torch.empty_like(d["kv"])}
            self.gptr = (self.grads["dq"], self.grads["dkv"], None)
        else:
            self.grads = {n: torch.empty_like(d[n[1:]]) for n in ("dq", "dk", "dv")}
            self.gptr = (self.grads["dq"], self.grads["dk"], self.grads["dv"])
        self.dbias = torch.empty_like(d["bias"]) if c.bias is not None else None
        self.A = A
        self.launches_per_step = None

    def step(self):
        A = self.A
        A.attn_fwd(self.params, self.o, self.lse, self.ws)
        A.attn_bwd(self.params, self.o, self.dev["do"], self.lse, *self.gptr, self.dbias, self.ws)

    def fwd(self):
        self.A.attn_fwd(self.params, self.o, self.lse, self.ws)

    def bwd(self):
        self.A.attn_bwd(self.params, self.o, self.dev["do"], self.lse, *self.gptr, self.dbias,
                        self.ws)

    def host_outputs(self):
        import torch

        out = {"o": torch.empty(self.o.shape, dtype=self.o.dtype).pin_memory(),
               "lse": torch.empty(self.lse.shape, dtype=self.lse.dtype).pin_memory()}
        for k, v in self.grads.items():
            out[k] = torch.empty(v.shape, dtype=v.dtype).pin_memory()
        if self.dbias is not None:
            out["dbias"] = torch.empty(self.dbias.shape, dtype=self.dbias.dtype).pin_memory()
        return out

    def check_status(self):
        s, st = self.A.attn_read_status(self.ws)
        if s != 0:
            raise RuntimeError(f"device status {s}")
        return st


class Fp8Forward:
    """The E4M3 forward on the same workload: Q / K / V rounded to E4M3 codes
    (descale factors 1), O in bf16.  Runs only where the FP8 path applies
    (d_qk = d_v = 128, no bias)."""

    def __init__(self, case, prob):
        import torch

        from bwd_tcgen05_tma_gb300 import attn as A
        from bwd_tcgen05_tma_gb300 import inputs as I

        c = case
        self.codes = {k: torch.from_numpy(I.e4m3_codes(v)).cuda() for k, v in c.buffers.items()}
        t = self.codes
        q, k, v = {"3HD": (t.get("qkv"), None, None), "HD_2HD": (t.get("q"), t.get("kv"), None),
                   "HD_HD_HD": (t.get("q"), t.get("k"), t.get("v"))}[c.layout]
        d = prob.dev  # the metadata tensors of the 16-bit problem, kept alive there
        self.params = A.make_params(
            layout=c.layout, fmt=c.fmt, mask=c.mask, B=c.B, Sq=c.Sq, Skv=c.Skv, Hq=c.Hq,
            Hkv=c.Hkv, d_qk=c.d_qk, d_v=c.d_v, scale=c.scale, q=q, k=k, v=v,
            q_seg_ids=d.get("q_ids"), q_seg_pos=d.get("q_pos"), kv_seg_ids=d.get("kv_ids"),
            kv_seg_pos=d.get("kv_pos"), dtype="fp8_e4m3", descale=(1.0, 1.0, 1.0))
        self.ws = torch.empty(A.attn_fwd_workspace_size(self.params), dtype=torch.uint8,
                              device="cuda")
        self.o = torch.empty((c.B * c.Sq, c.Hq, c.d_v), dtype=torch.bfloat16, device="cuda")
        self.lse = torch.empty((c.B, c.Hq, c.Sq), dtype=torch.float32, device="cuda")
        self.A = A

    @staticmethod
    def applies(case):
        return case.d_qk == 128 and case.d_v == 128 and case.bias is None

    def fwd(self):
        self.A.attn_fwd(self.params, self.o, self.lse, self.ws)

    def check_status(self):
        s, _ = self.A.attn_read_status(self.ws)
        if s != 0:
            raise RuntimeError(f"device status {s} (FP8 forward)")


class E2EPipeline:
    """End-to-end steps through the C ABI with host buffers, pipelined over two
    device buffer sets: the host->device copy of step i+1 (copy stream) and the
    device->host read of step i (second copy stream) overlap the kernels of
    step i (compute stream).  Every step still moves all of its inputs in and
    all of its results out."""

    def __init__(self, probs):
        import torch

        self.p = probs
        self.host_out = [p.host_outputs() for p in probs]
        self.s_in = torch.cuda.Stream()
        self.s_out = torch.cuda.Stream()
        ev = lambda: [torch.cuda.Event(), torch.cuda.Event()]
        self.ev_in, self.ev_comp, self.ev_out = ev(), ev(), ev()
        self.i = 0

    def step(self):
        import torch

        b = self.i & 1
        p = self.p[b]
        comp = torch.cuda.current_stream()
        if self.i >= 2:  # set b was last read by the kernels of step i-2
            self.s_in.wait_event(self.ev_comp[b])
        with torch.cuda.stream(self.s_in):
            for k, hv in p.host_in.items():
                p.dev[k].copy_(hv, non_blocking=True)
            self.ev_in[b].record(self.s_in)
        comp.wait_event(self.ev_in[b])
        if self.i >= 2:  # results of step i-2 read back before they are overwritten
            comp.wait_event(self.ev_out[b])
        p.step()
        self.ev_comp[b].record(comp)
        self.s_out.wait_event(self.ev_comp[b])
        with torch.cuda.stream(self.s_out):
            for k, hv in self.host_out[b].items():
                src = p.o if k == "o" else (p.lse if k == "lse" else
                                            (p.dbias if k == "dbias" else p.grads[k]))
                hv.copy_(src, non_blocking=True)
            self.ev_out[b].record(self.s_out)
        self.i += 1

    def drain(self):
        """Make the compute stream wait for every copy still in flight."""
        import torch

        comp = torch.cuda.current_stream()
        for b in range(2):
            comp.wait_event(self.ev_out[b])


def launches_per_step(case):
    """Kernels of this library launched per step (memsets excluded): the
    metadata kernel before the forward (one cooperative launch; the backward
    reuses its results); the forward; preprocess, dK/dV pass and dQ pass or
    dQ conversion.  A broadcast dBias is finished inside the dK/dV pass."""
    meta = 1
    bwd = 3
    return meta + 1 + bwd


# --------------------------------------------------------------------- CPU oracle sample


def _oracle_inputs(case):
    import numpy as np

    from oracle import attn_ref as R

    q, k, v = R.unpack_layout(case.layout, case.buffers, case.B, case.Sq, case.Skv, case.Hq,
                              case.Hkv, case.d_qk, case.d_v)
    if case.fmt == "BSHD" and case.q_ids is None:
        qi, qp = R.dense_metadata(case.B, case.Sq)
        ki, kp = R.dense_metadata(case.B, case.Skv)
    else:
        qi, qp, ki, kp = case.q_ids, case.q_pos, case.kv_ids, case.kv_pos
    G = case.Hq // case.Hkv
    bias = None if case.bias is None else case.bias[:1, :G].astype(np.float64)
    return q, k, v, qi, qp, ki, kp, G, bias


def oracle_rows(case, rows, groups=1, cached=None):
    """Runs the float64 oracle (as it stands) forward + backward on query rows
    [0, rows) of batch row 0, for KV heads [0, groups) and their query heads,
    against all keys.  Returns (algorithmic FLOPs of the sample, seconds)."""
    import numpy as np

    from oracle import attn_ref as R

    q, k, v, qi, qp, ki, kp, G, bias = cached or _oracle_inputs(case)
    sl = slice(0, rows)
    hq = slice(0, groups * G)
    qs, dos = q[:1, sl, hq], case.do[:1, sl, hq].astype(np.float64)
    ks, vs = k[:1, :, :groups], v[:1, :, :groups]
    bs = None if bias is None else bias[:, :, sl]
    t0 = time.perf_counter()
    R.attention_forward(qs, ks, vs, qi[:1, sl], qp[:1, sl], ki[:1], kp[:1], case.causal,
                        case.scale, bs)
    R.attention_backward(qs, ks, vs, dos, qi[:1, sl], qp[:1, sl], ki[:1], kp[:1], case.causal,
                         case.scale, bs)
    dt = time.perf_counter() - t0
    pairs = R.count_valid_pairs(qi[:1, sl], qp[:1, sl], ki[:1], kp[:1], case.causal) * G * groups
    ff, fb = R.attention_flops(pairs, case.d_qk, case.d_v)
    return ff + fb, dt


def oracle_calibrate(case, budget_s):
    """Picks the sample size (query rows, then KV heads) so one sample takes
    about budget_s seconds."""
    cached = _oracle_inputs(case)
    rows, groups = min(case.Sq, 256), 1
    fl, dt = oracle_rows(case, rows, groups, cached)
    while dt < budget_s / 2.5 and (rows < case.Sq or groups < case.Hkv):
        if rows < case.Sq:
            rows = min(case.Sq, rows * 2)
        else:
            groups = min(case.Hkv, groups * 2)
        fl, dt = oracle_rows(case, rows, groups, cached)
    G = case.Hq // case.Hkv
    desc = (f"float64 NumPy oracle, forward + backward of query rows [0,{rows}) of batch row 0, "
            f"query heads 0..{groups * G - 1} (KV heads 0..{groups - 1}), against all keys")
    return (rows, groups), fl, dt, desc, cached


def cpu_cores():
    return os.cpu_count() or 1


# --------------------------------------------------------------------- main paths


def run_reference(args, case):
    """The reference arm: the float64 oracle timed on the host cores, each step a
    bounded sample of the workload sized so the whole run ends in a few minutes."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    per_step = max(0.05, 120.0 / max(1, args.steps + args.warmup))
    (rows, groups), _, _, desc, cached = oracle_calibrate(case, per_step)
    for _ in range(args.warmup):
        oracle_rows(case, rows, groups, cached)
    fl_tot, t_tot, n = 0.0, 0.0, 0
    for _ in range(args.steps):
        fl, dt = oracle_rows(case, rows, groups, cached)
        fl_tot, t_tot, n = fl_tot + fl, t_tot + dt, n + 1
        if t_tot > 150:
            break
    val = fl_tot / t_tot / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": val, "unit": "TFLOP/s",
        "n_gpus": args.gpus, "steps": n, "warmup": args.warmup, "ms_per_step": 1e3 * t_tot / n,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": {"workload": WORKLOAD_DESC.get(args.workload,
                                                                       args.workload)},
        "cpu_baseline": {"value": val, "unit": "TFLOP/s", "cores": cpu_cores(), "kind": "oracle",
                         "sample": desc},
        "e2e": {"value": val, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


class Ranks:
    """Replica bookkeeping for N > 1 (one process per GPU, launched by torchrun):
    a barrier around the timed region and the maximum of a timing over ranks.
    The workload itself needs no exchange; nothing else is communicated."""

    def __init__(self, backend=None):
        self.rank = int(os.environ.get("RANK", "0"))
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.local = int(os.environ.get("LOCAL_RANK", "0"))
        self.dist = None
        self.device = "cpu"
        if self.world > 1:
            import torch
            import torch.distributed as dist

            if backend is None:
                backend = "nccl" if torch.cuda.is_available() else "gloo"
            dist.init_process_group(backend)
            self.dist = dist
            self.device = "cuda" if backend == "nccl" else "cpu"

    def barrier(self):
        if self.dist is not None:
            self.dist.barrier()

    def max(self, x):
        if self.dist is None:
            return x
        import torch

        t = torch.tensor([x], dtype=torch.float64, device=self.device)
        self.dist.all_reduce(t, op=self.dist.ReduceOp.MAX)
        return float(t.item())

    def close(self):
        if self.dist is not None:
            self.dist.destroy_process_group()
            self.dist = None


def aggregate_tflops(world, flops_per_replica, ms_max):
    """Whole-job throughput: every rank processed flops_per_replica in at most
    ms_max milliseconds."""
    return world * flops_per_replica / (ms_max * 1e-3) / 1e12


def timed(fn, steps, stream, barrier):
    import torch

    torch.cuda.synchronize()
    barrier()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        fn()
    e1.record(stream)
    torch.cuda.synchronize()
    barrier()
    return e0.elapsed_time(e1) / steps


# the other named workloads, measured after the headline one in the same run
# (timed steps each: about half a second of work or less)
OTHER_WORKLOADS = (("bshd", 200), ("cross_bias", 20), ("long_kv", 10))


def other_workloads(args, stream, barrier, max_over_ranks, world, peaks):
    """fwd+bwd TFLOP/s of every other named workload and of the headline one
    with the general masking path forced, deterministic dQ, each against the
    measured peak for its timed region's length (burst up to 0.5 s)."""
    import gc

    import torch

    from bwd_tcgen05_tma_gb300 import flops as F
    from bwd_tcgen05_tma_gb300 import inputs as I

    out = {}
    runs = [(args.workload + "_general_path", args.workload, True, 100)]
    runs += [(n, n, False, k) for n, k in OTHER_WORKLOADS]
    for key, name, force_general, steps in runs:
        try:
            case = I.workload(name)
            f_fwd, f_bwd, _ = F.attention_flops(case)
            p = Problem(case, "deterministic", force_general, pin=False)
            for _ in range(3):
                p.step()
            t = max_over_ranks(timed(p.step, steps, stream, barrier))
            st = p.check_status()
            v = aggregate_tflops(world, f_fwd + f_bwd, t)
            pk = ("bf16_tflops_sustained" if t * steps * 1e-3 > 0.5 and
                  "bf16_tflops_sustained" in peaks else "bf16_tflops")
            out[key] = {"workload": WORKLOAD_DESC.get(name, name), "value": v, "unit": "TFLOP/s",
                        "ms_per_step": t, "steps": steps, "pct_of_peak": v / float(peaks[pk]),
                        "peak_basis": pk, "path": "fast" if st.path == 0 else "general"}
            del p, case
        except Exception as e:  # a failure here must not cost the headline line
            out[key] = {"error": f"{type(e).__name__}: {e}"[:200]}
        gc.collect()
        torch.cuda.empty_cache()
    return out


def main():
    args = parse()
    from bwd_tcgen05_tma_gb300 import inputs as I

    case = I.workload(args.workload)
    if args.impl == "reference":
        run_reference(args, case)
        return

    import torch

    rk = Ranks()
    rank, world, local = rk.rank, rk.world, rk.local
    torch.cuda.set_device(local)
    barrier, max_over_ranks = rk.barrier, rk.max

    from bwd_tcgen05_tma_gb300 import build
    from bwd_tcgen05_tma_gb300 import flops as F

    build.build()
    fwd_flops, bwd_flops, pairs = F.attention_flops(case)
    total_flops = fwd_flops + bwd_flops
    prob = Problem(case, args.dq_mode, args.force_general)
    stream = torch.cuda.current_stream()
    A = prob.A

    # warm-up (also checks the device status once)
    for _ in range(max(args.warmup, 1)):
        prob.step()
    stats = prob.check_status()

    # timed region: the steps exactly as a caller runs them (no extra events
    # between the library's launches)
    clocks = ClockSampler(local)
    clocks.start()
    ms = timed(prob.step, args.steps, stream, barrier)
    clk = clocks.stop()
    stats = prob.check_status()
    ms = max_over_ranks(ms)

    # the same number of steps again, with per-stage events recorded by the
    # library around its launches: the per-kernel times and the roofline
    slots = A.TRACE_SLOTS
    ev = [[A.Event() for _ in range(2 * len(slots))] for _ in range(args.steps)]
    it = iter(ev)

    def traced_step():
        A.attn_set_trace_events(next(it))
        prob.step()

    ms_traced = timed(traced_step, args.steps, stream, barrier)
    A.attn_set_trace_events(None)
    stats = prob.check_status()
    kern_ms = {}
    for si, name in enumerate(slots):
        vals = []
        for e in ev:
            t = A.attn_event_elapsed_ms(e[2 * si], e[2 * si + 1])
            if t is not None:  # None: slot not used this step (e.g. no dBias reduction)
                vals.append(t)
        if vals:
            kern_ms[name] = statistics.mean(vals)
    # the metadata slot is recorded twice per step (fwd and bwd); events hold the last
    if args.dq_mode == "deterministic" and max(case.d_qk, case.d_v) <= 128 and "dq" in kern_ms:
        # the 128-row dQ pass runs beside the dK/dV pass (on a second stream): its
        # events span from the end of the preprocess to the end of the dQ pass
        kern_ms["dq_span_overlapping_dkdv"] = kern_ms.pop("dq")
    value = aggregate_tflops(world, total_flops, ms)

    peaks, peak_src = load_peaks()
    # a timed region of a few tens of ms runs at burst clocks; one that lasts
    # seconds settles at the power cap like the sustained GEMM loop
    timed_s = ms * args.steps * 1e-3
    sustained = timed_s > 0.5 and "bf16_tflops_sustained" in peaks
    peak_key = "bf16_tflops_sustained" if sustained else "bf16_tflops"
    peak = float(peaks[peak_key])
    dom = max((k for k in kern_ms if k in ("fwd", "bwd_pre", "dkdv", "dq", "dbias")),
              key=lambda k: kern_ms[k])
    atomic = args.dq_mode == "atomic" and case.d_qk <= 128
    kern_flops = {"fwd": fwd_flops,
                  "dkdv": bwd_flops if atomic else 2.0 * pairs * (2 * case.d_qk + 2 * case.d_v),
                  "dq": 0.0 if atomic else 2.0 * pairs * case.d_qk}
    achieved = kern_flops.get(dom, 0.0) / (kern_ms[dom] * 1e-3) / 1e12
    traffic = None
    tpath = os.path.join(ROOT, "profiles", "traffic.json")
    if os.path.exists(tpath):
        with open(tpath) as f:
            tr = json.load(f)
        rec = tr.get(args.workload, {}).get(dom)
        if rec and rec.get("source_hash") == source_hash(dom):
            traffic = rec.get("bytes_per_launch")

    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) bf16 inputs, seeded segment metadata)",
        "config": {"workload": WORKLOAD_DESC.get(args.workload, args.workload),
                   "dq_mode": args.dq_mode, "unmasked_pairs": pairs,
                   "fwd_gflop": fwd_flops / 1e9, "bwd_gflop": bwd_flops / 1e9,
                   "l2": "inputs larger than L2 (no flush needed)",
                   "path": "fast" if stats.path == 0 else "general",
                   "force_general": bool(args.force_general)},
        "pct_of_peak": value / peak,
        "pct_of_peak_basis": f"{peak_key} = {peak} TFLOP/s ({peak_src})",
        "roofline": {"kernel": dom, "bound": "tensor", "achieved": achieved, "peak": peak,
                     "unit": "TFLOP/s", "frac": achieved / peak, "traffic": traffic,
                     "peak_source": f"{peak_key} of {peak_src} (timed region {timed_s:.3f} s)"},
        "kernels_ms": kern_ms,
        "ms_per_step_traced": max_over_ranks(ms_traced),
        "clocks": clk,
        # time x clock: comparable across runs at different SM clocks
        "ms_x_sm_mhz": (ms * clk["sm_mhz"]) if clk.get("sm_mhz") else None,
        "gpu_launches": launches_per_step(case) * args.steps,
    }

    if not args.no_extras:
        t_f = max_over_ranks(timed(prob.fwd, max(20, args.steps // 4), stream, barrier))
        t_b = max_over_ranks(timed(prob.bwd, max(20, args.steps // 4), stream, barrier))
        line["fwd_tflops"] = aggregate_tflops(world, fwd_flops, t_f)
        line["bwd_tflops"] = aggregate_tflops(world, bwd_flops, t_b)
        other = "atomic" if args.dq_mode == "deterministic" else "deterministic"
        alt = Problem(case, other, args.force_general)
        for _ in range(3):
            alt.step()
        t_d = max_over_ranks(timed(alt.step, max(20, args.steps // 4), stream, barrier))
        alt.check_status()
        line["other_dq_mode"] = {"dq_mode": other, "value": aggregate_tflops(world, total_flops, t_d),
                                 "unit": "TFLOP/s", "ms_per_step": t_d}
        del alt
        if Fp8Forward.applies(case):
            # the FP8 forward (metadata, V transpose, two-pass forward) beside
            # the bf16 one; its tensor peak is the bf16 one times the nominal
            # dense ratio 4.5 / 2.25 PFLOP/s
            f8 = Fp8Forward(case, prob)
            for _ in range(3):
                f8.fwd()
            t_8 = max_over_ranks(timed(f8.fwd, max(20, args.steps // 4), stream, barrier))
            f8.check_status()
            v8 = aggregate_tflops(world, fwd_flops, t_8)
            line["fp8_forward"] = {
                "value": v8, "unit": "TFLOP/s", "ms": t_8, "dtype": "e4m3 (O bf16)",
                "flops": "the bf16 forward's (4 d per unmasked pair and head; the row-maximum "
                         "pass recomputes S and is not credited)",
                "pct_of_fp8_peak": v8 / (2.0 * peak),
                "peak_basis": f"2 x {peak_key} = {2.0 * peak} TFLOP/s (nominal fp8/bf16 ratio)"}
            del f8

    if not args.no_e2e:
        pipe = E2EPipeline([prob, Problem(case, args.dq_mode, args.force_general)])
        for _ in range(4):
            pipe.step()
        pipe.drain()
        n_e2e = max(10, args.steps // 8)

        def e2e_steps():
            for _ in range(n_e2e):
                pipe.step()
            pipe.drain()  # the last results are on the host inside the timed region

        t_e = max_over_ranks(timed(e2e_steps, 1, stream, barrier)) / n_e2e
        for p in pipe.p:
            p.check_status()
        h2d = sum(v.numel() * v.element_size() for v in prob.host_in.values())
        d2h = sum(v.numel() * v.element_size() for v in pipe.host_out[0].values())
        line["e2e"] = {"value": aggregate_tflops(world, total_flops, t_e), "unit": "TFLOP/s",
                       "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                       "ms_per_step": t_e}

    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        _, fl, dt, desc, _ = oracle_calibrate(case, 12.0)
        line["cpu_baseline"] = {"value": fl / dt / 1e12, "unit": "TFLOP/s",
                                "cores": cpu_cores(), "kind": "oracle", "sample": desc,
                                "seconds": dt}
    if (not args.no_extras and not args.no_other_workloads and world == 1 and
            args.workload == "thd_gqa" and not args.force_general):
        del prob
        line["other_workloads"] = other_workloads(args, stream, barrier, max_over_ranks, world,
                                                  peaks)
    if rank == 0:
        print(json.dumps(line), flush=True)
    rk.close()


if __name__ == "__main__":
    main()
