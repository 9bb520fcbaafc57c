#!/usr/bin/env python
"""Benchmark of load-balanced context-parallel causal attention on GB300.

One step = the whole hot path over one batch of seeded synthetic input:
  load-balance permute of q, k, v, dout -> forward (all cp shards) ->
  backward -> unpermute of out, dq, dk, dv -> one GQA decode batch.
Default workload: the Llama3.1-70B-shaped long-context GQA layer (B=1,
Hq=64, Hkv=8, S=131072, head dim 128, cp=8 load-balanced) plus the decode
batch (B=24, Hq=32, Hkv=8, D=128, cache 2048, lengths U[1024, 2048]).  The
line also carries: the same layer with load balancing off (whole step and
per-shard forward/backward times), the zero-copy step, decode alone (bf16
and int8 caches), the end-to-end step through the Python API with host
copies, the Llama2-7B-shaped and DeepSeek-V3-shaped MLA layers' steps, and
the float64 oracle timed on a bounded sample on the host cores.

Prints ONE JSON line (rank 0).  `value` is fwd+bwd TFLOP/s (unmasked pairs
only, S(S+1)/2 per head; fwd 2(Dqk+Dv), bwd 2(3Dqk+2Dv) FLOPs per pair)
summed over all ranks; each rank runs its own replica (the cp shards are
emulated on one GPU, there is no collective on the data path).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
"""

import argparse
import hashlib
import json
import math
import os
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

WORKLOADS = {
    # name: B, S, Hq, Hkv, Dqk, Dv, cp, lb, q_scale
    "llama2_7b_s8192_cp4": dict(B=1, S=8192, Hq=32, Hkv=32, Dqk=128, Dv=128, cp=4, lb=True,
                                q_scale=1.0 / math.sqrt(128)),
    "llama3_70b_s131072_cp8": dict(B=1, S=131072, Hq=64, Hkv=8, Dqk=128, Dv=128, cp=8, lb=True,
                                   q_scale=1.0),
    "deepseek_v3_mla_s32768_cp4": dict(B=1, S=32768, Hq=128, Hkv=128, Dqk=192, Dv=128, cp=4, lb=True,
                                       q_scale=1.0),
    # the same with one 64-column rope key per token shared by the heads (k_nope per head)
    "deepseek_v3_mla_rope_s32768_cp4": dict(B=1, S=32768, Hq=128, Hkv=128, Dqk=192, Dv=128, cp=4, lb=True,
                                            q_scale=1.0, rope=True),
    "tiny_s256_cp2": dict(B=1, S=256, Hq=2, Hkv=2, Dqk=64, Dv=64, cp=2, lb=True, q_scale=1.0),
    # the Llama3.1-70B head layout at shorter sequences: cases small enough for a full ncu capture
    # (traffic scaled to the 131072-token launch by the tile pairs processed)
    "llama3_70b_gqa_s16384_cp8": dict(B=1, S=16384, Hq=64, Hkv=8, Dqk=128, Dv=128, cp=8, lb=True, q_scale=1.0),
    "llama3_70b_gqa_s32768_cp8": dict(B=1, S=32768, Hq=64, Hkv=8, Dqk=128, Dv=128, cp=8, lb=True, q_scale=1.0),
    # the DeepSeek-V3 MLA head layout at a shorter sequence, for the same purpose
    "deepseek_v3_mla_s4096_cp4": dict(B=1, S=4096, Hq=128, Hkv=128, Dqk=192, Dv=128, cp=4, lb=True, q_scale=1.0),
}
# the largest single-GPU configuration (Llama3.1-70B-shaped GQA at 131072
# tokens, load-balanced) is the headline; the others ride along in the line
HEADLINE = "llama3_70b_s131072_cp8"
EXTRA_WORKLOADS = ("llama2_7b_s8192_cp4", "deepseek_v3_mla_s32768_cp4", "deepseek_v3_mla_rope_s32768_cp4")
DECODE = dict(B=24, Hq=32, Hkv=8, D=128, Smax=2048, lo=1024, hi=2048)
METRIC = "causal CP-attention fwd+bwd TFLOP/s and % of BF16 peak; decode KV-read GB/s"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
KERNEL_SOURCES = {
    "attn_fwd": "attn_fwd.cu", "attn_fwd_shard": "attn_fwd.cu", "attn_bwd_dkdv": "attn_bwd.cu",
    "attn_bwd_dq": "attn_bwd.cu", "bwd_preprocess": "attn_bwd.cu", "gqa_decode": "decode.cu",
    "attn_bwd_fused": "attn_bwd_fused.cu", "bwd_dq_round": "attn_bwd_fused.cu",
    "lb_permute": "permute.cu", "lb_unpermute": "permute.cu", "mla_decode": "mla_decode.cu",
    "attn_bwd_mla": "attn_bwd_mla.cu",
}


# ---------------------------------------------------------------------------
# work accounting
# ---------------------------------------------------------------------------

def pairs(w):
    return w["B"] * w["Hq"] * w["S"] * (w["S"] + 1) / 2


def flops_fwd(w):
    return 2.0 * pairs(w) * (w["Dqk"] + w["Dv"])


def flops_bwd(w):
    return 2.0 * pairs(w) * (3 * w["Dqk"] + 2 * w["Dv"])


def kernel_flops(name, w):
    """Algorithmic FLOPs of one launch of each attention kernel.  The fused
    backward does all five backward products (S and dP recomputes, dV, dK,
    dQ); in the two-kernel backward the dk/dv kernel owns the S and dP
    recomputes plus dV and dK, and the dq kernel is credited only with dQ (its
    own S/dP recompute is extra work)."""
    p = pairs(w)
    return {
        "attn_fwd": 2.0 * p * (w["Dqk"] + w["Dv"]),
        "attn_bwd_fused": 2.0 * p * (3 * w["Dqk"] + 2 * w["Dv"]),
        "attn_bwd_mla": 2.0 * p * (3 * w["Dqk"] + 2 * w["Dv"]),
        "attn_bwd_dkdv": 2.0 * p * (2 * w["Dqk"] + 2 * w["Dv"]),
        "attn_bwd_dq": 2.0 * p * w["Dqk"],
    }.get(name)


def decode_bytes(lens, D=DECODE["D"], Hkv=DECODE["Hkv"]):
    return int(sum(int(x) for x in lens)) * Hkv * D * 2 * 2


def kernel_bytes(name, w, lens):
    """Algorithmic HBM bytes of one launch of the streaming kernels."""
    if name == "gqa_decode":
        return decode_bytes(lens) + 2 * DECODE["B"] * DECODE["Hq"] * DECODE["D"] * 2
    if name in ("lb_permute", "lb_unpermute"):
        return None  # four different tensors per step: reported per launch below
    return None


# ---------------------------------------------------------------------------
# distributed helpers (one replica per rank)
# ---------------------------------------------------------------------------

def dist_env():
    return int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")), \
        int(os.environ.get("LOCAL_RANK", "0"))


def max_over_ranks(x, device=None):
    """Max of a float over all ranks (identity without a process group)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate_throughput(work_per_rank, seconds_max, world):
    """Whole-job throughput: the units all ranks processed / the slowest rank's time."""
    return work_per_rank * world / seconds_max


def barrier():
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        dist.barrier()


# ---------------------------------------------------------------------------
# clocks sampled during the timed region
# ---------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.thread.join(timeout=2)
        sm, smax, power, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
                power.append(float(parts[2]))
            except ValueError:
                continue
            for nm, val in zip(names, parts[4:8]):
                if val.lower().startswith("active"):
                    reasons.add(nm)
        sm.sort()
        return {"sm_mhz": sm[len(sm) // 2] if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "samples": len(sm), "power_w_max": max(power) if power else None,
                "reasons": sorted(reasons)}


# ---------------------------------------------------------------------------
# measured peaks, stored ncu traffic
# ---------------------------------------------------------------------------

def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def source_hash(kernel):
    src = KERNEL_SOURCES.get(kernel)
    if not src:
        return None
    h = hashlib.sha256()
    for f in (src, "common.cuh"):
        with open(os.path.join(ROOT, "context_causal_attention_load_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def stored_traffic(kernel, workload):
    """dram read+write bytes per launch from a committed ncu summary, or None
    if none exists or the kernel source changed since it was captured."""
    p = os.path.join(ROOT, "profiles", "dram_traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    e = d.get("%s/%s" % (kernel, workload))
    if not e or e.get("source_sha") != source_hash(kernel):
        return None
    return e.get("bytes_per_launch")


# ---------------------------------------------------------------------------
# CPU oracle baseline (bounded sample)
# ---------------------------------------------------------------------------

def oracle_sample(w, rows=256, heads=1, seed=0):
    """Run the float64 oracle forward+backward for `heads` query heads and a
    spread sample of `rows` query rows (each against every key it sees) of
    the workload.  Returns (seconds, flops of the sample, description)."""
    import numpy as np
    from oracle import cp_attention as O
    rng = np.random.default_rng(seed)
    S, Dqk, Dv = w["S"], w["Dqk"], w["Dv"]
    q = rng.standard_normal((1, rows, heads, Dqk)) * w["q_scale"]
    k = rng.standard_normal((1, S, 1, Dqk))
    v = rng.standard_normal((1, S, 1, Dv))
    dout = rng.standard_normal((1, rows, heads, Dv))
    qpos = np.linspace(0, S - 1, rows).astype(np.int64)
    kpos = np.arange(S)
    t0 = time.perf_counter()
    out, lse = O.masked_attention_fwd(q, k, v, qpos, kpos)
    O.masked_attention_bwd(q, k, v, out, lse, dout, qpos, kpos)
    dt = time.perf_counter() - t0
    npairs = float(np.sum(qpos + 1)) * heads
    fl = 2.0 * npairs * (Dqk + Dv) + 2.0 * npairs * (3 * Dqk + 2 * Dv)
    desc = "%d query heads x %d query rows spread over S=%d (every visible key), fwd+bwd" % (heads, rows, S)
    return dt, fl, desc


def blas_threads():
    for var in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
        if os.environ.get(var):
            return int(os.environ[var])
    return os.cpu_count()


def cpu_baseline(w, budget_s=12.0):
    dt, fl, desc = oracle_sample(w, rows=64)
    rows = 64
    if dt < budget_s / 4:  # grow the sample toward the budget
        rows = int(min(w["S"], 64 * max(1.0, budget_s / max(dt, 1e-3) / 2)))
        dt, fl, desc = oracle_sample(w, rows=rows)
    return {"value": fl / dt / 1e12, "unit": "TFLOP/s", "cores": blas_threads(), "kind": "oracle",
            "sample": desc + "; float64 NumPy on the host cores, %.1f s" % dt}


def run_reference(args, w, wname):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    rows = 128
    for _ in range(max(0, args.warmup)):
        oracle_sample(w, rows=rows)
    total_t, total_f = 0.0, 0.0
    for _ in range(args.steps):
        dt, fl, desc = oracle_sample(w, rows=rows)
        total_t += dt
        total_f += fl
    val = total_f / total_t / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": val, "unit": "TFLOP/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total_t / max(1, args.steps),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": {"workload": wname, **{k: w[k] for k in ("B", "S", "Hq", "Hkv", "Dqk", "Dv", "cp")},
                                        "load_balance": w["lb"]},
        "cpu_baseline": {"value": val, "unit": "TFLOP/s", "cores": blas_threads(), "kind": "oracle",
                         "sample": desc + " per step (float64 NumPy, host cores)"},
        "e2e": {"value": val, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
# GPU path
# ---------------------------------------------------------------------------

def peak_for(peaks, timed_s):
    """Dense bf16 peak that applies to a kernel timed inside a region of
    timed_s seconds: the burst figure for a short region, the sustained one
    (the rate under the power cap) for a region of a second or more."""
    if timed_s >= 1.0:
        return peaks.get("bf16_tflops_sustained", peaks.get("bf16_tflops")), "bf16_tflops_sustained"
    return peaks.get("bf16_tflops"), "bf16_tflops"


class AttnStep:
    """One training step of the attention path for workload w: load-balance
    permute of q, k, v, dout -> forward (all cp shards) -> backward ->
    unpermute of out, dq, dk, dv (permute and unpermute only with load
    balance).  Buffers are allocated once."""

    def __init__(self, w, q, k, v, dout, cpattn, kr=None):
        import torch
        self.w, self.cpattn = w, cpattn
        self.q, self.k, self.v, self.dout, self.kr = q, k, v, dout, kr
        B, S, Hq, Dv = w["B"], w["S"], w["Hq"], w["Dv"]
        dev = q.device
        self.lb = w["lb"]
        self.qp, self.kp, self.vp, self.dop = (torch.empty_like(x) for x in (q, k, v, dout))
        self.out_p = torch.empty(B, S, Hq, Dv, dtype=torch.bfloat16, device=dev)
        self.lse = torch.empty(B, Hq, S, dtype=torch.float32, device=dev)
        self.dq_p, self.dk_p, self.dv_p = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        self.out_n, self.dq_n, self.dk_n, self.dv_n = (torch.empty_like(x) for x in (self.out_p, q, k, v))
        if kr is not None:
            self.krp, self.dkr_p, self.dkr_n = (torch.empty_like(kr) for _ in range(3))

    def __call__(self, qi=None, ki=None, vi=None, di=None):
        c = self.cpattn
        cp, lb = self.w["cp"], self.lb
        qi = self.q if qi is None else qi
        ki = self.k if ki is None else ki
        vi = self.v if vi is None else vi
        di = self.dout if di is None else di
        if lb:
            c.lb_permute(qi, cp, self.qp)
            c.lb_permute(ki, cp, self.kp)
            c.lb_permute(vi, cp, self.vp)
            c.lb_permute(di, cp, self.dop)
            a, bk, cv, d = self.qp, self.kp, self.vp, self.dop
        else:
            a, bk, cv, d = qi, ki, vi, di
        if self.kr is not None:
            kri = self.kr
            if lb:
                c.lb_permute(self.kr, cp, self.krp)
                kri = self.krp
            c.attn_fwd_mla(a, bk, kri, cv, cp, lb, self.out_p, self.lse)
            c.attn_bwd_mla(a, bk, kri, cv, self.out_p, self.lse, d, cp, lb, self.dq_p, self.dk_p, self.dkr_p,
                           self.dv_p)
        else:
            c.attn_fwd(a, bk, cv, cp, lb, self.out_p, self.lse)
            c.attn_bwd(a, bk, cv, self.out_p, self.lse, d, cp, lb, self.dq_p, self.dk_p, self.dv_p)
        if lb:
            c.lb_unpermute(self.out_p, cp, self.out_n)
            c.lb_unpermute(self.dq_p, cp, self.dq_n)
            c.lb_unpermute(self.dk_p, cp, self.dk_n)
            c.lb_unpermute(self.dv_p, cp, self.dv_n)
            if self.kr is not None:
                c.lb_unpermute(self.dkr_p, cp, self.dkr_n)

    def results(self):
        if self.lb:
            return self.out_n, self.dq_n, self.dk_n, self.dv_n
        return self.out_p, self.dq_p, self.dk_p, self.dv_p


def time_steps(fn, n):
    """Device milliseconds per call of fn over n calls (CUDA events on the
    current stream, synchronised on both sides)."""
    import torch
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(n):
        fn()
    e1.record()
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / n


def kernel_table(prof, w, peaks, timed_s, lens_host=None):
    peak, peak_name = peak_for(peaks, timed_s)
    total = sum(t for _, t in prof.values()) or 1.0
    kernels = {}
    for name, (n, tot) in sorted(prof.items(), key=lambda kv: -kv[1][1]):
        e = {"launches": n, "ms_per_launch": tot / n, "share": tot / total}
        kf = kernel_flops(name, w)
        if kf is not None:
            e["tflops"] = kf / (tot / n / 1e3) / 1e12
            e["frac_of_bf16"] = e["tflops"] / peak
            e["peak"] = peak_name
        if name == "gqa_decode" and lens_host is not None:
            e["gbs"] = kernel_bytes(name, w, lens_host) / (tot / n / 1e3) / 1e9
            e["frac_of_hbm"] = e["gbs"] / peaks["hbm_gbs"]
        kernels[name] = e
    return kernels


def run_ours(args, w, wname):
    import torch
    import torch.distributed as dist

    from context_causal_attention_load_gb300 import build as cbuild
    from context_causal_attention_load_gb300 import synth

    rank, world, local = dist_env()
    if world > 1 and not dist.is_initialized():
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if rank == 0:
        cbuild.build()
    barrier()
    from context_causal_attention_load_gb300 import cpattn
    cpattn.load()

    B, S, Hq, Hkv, Dqk, Dv, cp, lb = (w[k] for k in ("B", "S", "Hq", "Hkv", "Dqk", "Dv", "cp", "lb"))
    q, k, v, dout = synth.attention_inputs_device(B, S, Hq, Hkv, Dqk, Dv, seed=args.seed + 1000 * rank,
                                                  q_scale=w["q_scale"], device=dev)
    rope = bool(w.get("rope"))
    kr = None
    if rope:  # per-head nope keys and one rope key per token (the other extras assume one key tensor)
        k, kr = k[..., :128].contiguous(), k[:, :, 0, 128:].contiguous()
        args.no_extras = True
    D = DECODE
    dq_, dkc, dvc, dlens = synth.decode_inputs(D["B"], D["Hq"], D["Hkv"], D["D"], D["Smax"], D["lo"], D["hi"],
                                               seed=args.seed + 4)
    dq_, dkc, dvc, dlens = dq_.to(dev), dkc.to(dev), dvc.to(dev), dlens.to(dev)
    lens_host = dlens.cpu().tolist()
    dec_out = torch.empty_like(dq_)
    attn = AttnStep(w, q, k, v, dout, cpattn, kr)

    def step(qi=q, ki=k, vi=v, di=dout, dqi=dq_, dkci=dkc, dvci=dvc, dli=dlens):
        attn(qi, ki, vi, di)
        cpattn.gqa_decode(dqi, dkci, dvci, dli, dec_out)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    cpattn.check_device()

    # ---- timed region ---------------------------------------------------
    # every library launch is bracketed by two CUDA events on its own stream
    # (per-kernel times for the roofline); two event records per launch are
    # negligible against launches of milliseconds
    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.3)
    barrier()
    torch.cuda.synchronize()
    cpattn.profile_start()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record()
    for _ in range(args.steps):
        step()
    ev1.record()
    torch.cuda.synchronize()
    barrier()
    prof = cpattn.profile_stop()
    clocks = sampler.stop()
    cpattn.check_device()
    ms = ev0.elapsed_time(ev1) / args.steps
    ms_max = max_over_ranks(ms, dev)
    timed_s = ms_max * args.steps / 1e3
    f_step = flops_fwd(w) + flops_bwd(w)
    value = aggregate_throughput(f_step, ms_max / 1e3, world) / 1e12
    launches = sum(n for n, _ in prof.values())

    peaks, peak_src = load_peaks()
    peak_t, peak_name = peak_for(peaks, timed_s)
    # dominant kernel of the step
    dname, (dn, dms) = max(prof.items(), key=lambda kv: kv[1][1])
    davg = dms / dn
    fl = kernel_flops(dname, w)
    if fl is not None:
        achieved = fl / (davg / 1e3) / 1e12
        roof = {"kernel": dname, "bound": "tensor", "achieved": achieved, "peak": peak_t, "unit": "TFLOP/s",
                "frac": achieved / peak_t,
                "peak_source": "%s %s (timed region %.1f s)" % (peak_src, peak_name, timed_s),
                "traffic": stored_traffic(dname, wname), "ms_per_launch": davg,
                "algorithmic_flops_per_launch": fl}
    else:
        by = kernel_bytes(dname, w, lens_host)
        peak = peaks["hbm_gbs"]
        achieved = (by / (davg / 1e3) / 1e9) if by else None
        roof = {"kernel": dname, "bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                "frac": achieved / peak if achieved else None, "peak_source": "%s hbm_gbs" % peak_src,
                "traffic": stored_traffic(dname, wname), "ms_per_launch": davg}

    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_max, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": wname, "B": B, "S": S, "Hq": Hq, "Hkv": Hkv, "Dqk": Dqk, "Dv": Dv, "cp": cp,
                   "load_balance": lb, **({"k_rope": "one 64-column rope key per token, shared by the heads"}
                                          if rope else {}),
                   "step": "lb_permute q,k,v,dout -> fwd (all cp shards) -> bwd -> lb_unpermute out,dq,dk,dv"
                           " -> one GQA decode batch",
                   "decode": "B=24 Hq=32 Hkv=8 D=128 Smax=2048 lens~U[1024,2048]",
                   "parallelism": "replicas%d" % world,
                   "l2": "inputs larger than L2 (q,k,v,dout %.0f MB + decode KV %.0f MB per step)" % (
                       (q.numel() + k.numel() + v.numel() + dout.numel()) * 2 / 1e6, 2 * dkc.numel() * 2 / 1e6)},
        "roofline": roof,
        "gpu_launches": launches,
        "kernels": kernel_table(prof, w, peaks, timed_s, lens_host),
        "clocks": clocks,
    }

    if not args.no_extras:
        def make_step():
            a = AttnStep(w, q, k, v, dout, cpattn, kr)
            o = torch.empty_like(dq_)

            def fn(qi, ki, vi, di, dqi, dkci, dvci, dli):
                a(qi, ki, vi, di)
                cpattn.gqa_decode(dqi, dkci, dvci, dli, o)
            return fn, tuple(a.results()) + (o,)

        line["e2e"] = measure_e2e(args, make_step, (q, k, v, dout, dq_, dkc, dvc, dlens), f_step, ms_max, world, dev)
        if lb:
            line["lb_off_step"] = measure_lb_off(w, q, k, v, dout, f_step, peaks, cpattn)
        line["shards"] = measure_shards(w, attn, cpattn)
        if lb and (S // (2 * cp)) % 128 == 0:
            line["zero_copy"] = measure_zero_copy(args, w, (q, k, v, dout), (dq_, dkc, dvc, dlens), dec_out, f_step,
                                                  step, world, dev, cpattn)
        line["decode"] = measure_decode(dq_, dkc, dvc, dlens, lens_host, peaks, cpattn)
        line["decode_int8"] = measure_decode_int8(dq_, dkc, dvc, dlens, lens_host, peaks, cpattn)
        line["mla_decode"] = measure_mla_decode(lens_host, peaks, cpattn, dev, args.seed)
        del attn, q, k, v, dout
        torch.cuda.empty_cache()
        line["other_workloads"] = {
            name: measure_workload(name, peaks, cpattn, dev, args.seed)
            for name in EXTRA_WORKLOADS if name != wname}
        if rank == 0 and world == 1:
            line["cpu_baseline"] = cpu_baseline(w)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def measure_e2e(args, make_step, inputs, f_step, ms_step, world, dev):
    """Same metric through the public API with every step's inputs copied from
    pinned host memory and its results copied back, inside the timed region,
    pipelined as a serving or training loop would run it: while step i
    computes, step i+1's inputs go in on one copy stream and step i-1's
    results come out on another, into and out of a second set of device
    buffers.  make_step() returns (fn, outputs): fn(*device_inputs) runs one
    step into its own output buffers.  Host copies also run at very different
    speeds from one run to the next on this shared host (about 200 GB/s each
    way when the host is quiet, several times less at other times), which the
    overlap keeps out of the step time as long as they are shorter than it."""
    import torch
    fns, outs = zip(*(make_step() for _ in range(2)))
    host_in = [x.cpu().pin_memory() for x in inputs]
    dev_in = [[torch.empty_like(x) for x in inputs] for _ in range(2)]
    host_out = [[torch.empty(x.shape, dtype=x.dtype, pin_memory=True) for x in o] for o in outs]
    h2d = sum(x.numel() * x.element_size() for x in host_in)
    d2h = sum(x.numel() * x.element_size() for x in host_out[0])
    # (up to about 15 s of steps: the first step's input copy and the last one's result copy, which no
    # compute covers, are shared by that many steps, as in a long training or serving loop)
    n = max(3, min(args.steps, int(15000.0 / max(ms_step, 1e-3))))
    comp = torch.cuda.current_stream()
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()

    def run(nsteps):
        """nsteps pipelined steps; device ms from the start event to the last
        result on the host side of the copy."""
        ev = lambda: torch.cuda.Event(enable_timing=False)
        e_in, e_done, e_out = [ev(), ev()], [ev(), ev()], [ev(), ev()]
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0.record(comp)
        s_in.wait_event(t0)
        with torch.cuda.stream(s_in):
            for h, d in zip(host_in, dev_in[0]):
                d.copy_(h, non_blocking=True)
            e_in[0].record(s_in)
        for i in range(nsteps):
            b = i & 1
            if i + 1 < nsteps:  # next step's inputs, once step i-1 (the last user of that buffer) is done
                with torch.cuda.stream(s_in):
                    if i >= 1:
                        s_in.wait_event(e_done[b ^ 1])
                    for h, d in zip(host_in, dev_in[b ^ 1]):
                        d.copy_(h, non_blocking=True)
                    e_in[b ^ 1].record(s_in)
            comp.wait_event(e_in[b])
            if i >= 2:  # step i-2's results (the same buffers) have left
                comp.wait_event(e_out[b])
            fns[b](*dev_in[b])
            e_done[b].record(comp)
            with torch.cuda.stream(s_out):
                s_out.wait_event(e_done[b])
                for h, d in zip(host_out[b], outs[b]):
                    h.copy_(d, non_blocking=True)
                e_out[b].record(s_out)
        for e in e_out:
            comp.wait_event(e)
        t1.record(comp)
        torch.cuda.synchronize()
        return t0.elapsed_time(t1)

    run(2)
    barrier()
    ms = max_over_ranks(run(n) / n, dev)
    return {"value": aggregate_throughput(f_step, ms / 1e3, world) / 1e12, "unit": "TFLOP/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": ms, "steps": n,
            "overlap": "step i+1's inputs copied in and step i-1's results copied out on two copy streams while "
                       "step i computes (double-buffered device inputs and outputs); the timed region runs from "
                       "the first input copy to the last result copy"}


def measure_lb_off(w, q, k, v, dout, f_step, peaks, cpattn, n=3):
    """fwd + bwd of all shards with load_balance = 0 (natural order, no
    permutes).  On one GPU the persistent grid spreads every shard's units
    over all SMs, so the whole step costs about the same either way; the
    per-shard times (``shards``) show the imbalance the reorder removes."""
    import torch
    cp = w["cp"]
    out = torch.empty(w["B"], w["S"], w["Hq"], w["Dv"], dtype=torch.bfloat16, device=q.device)
    lse = torch.empty(w["B"], w["Hq"], w["S"], dtype=torch.float32, device=q.device)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)

    def s():
        cpattn.attn_fwd(q, k, v, cp, 0, out, lse)
        cpattn.attn_bwd(q, k, v, out, lse, dout, cp, 0, dq, dk, dv)

    s()
    cpattn.check_device()
    ms = time_steps(s, n)
    del out, lse, dq, dk, dv
    return {"ms_per_step": ms, "tflops": f_step / (ms / 1e3) / 1e12, "steps": n,
            "what": "fwd + bwd, load_balance = 0, natural order, no permutes, no decode"}


def measure_decode(q, kc, vc, lens, lens_host, peaks, cpattn, iters=30, layers=32):
    """Decode alone, two ways.  Cold: one call per timed region with L2
    flushed before it (a 512 MB write, then a 512 MB read of another buffer
    so that the written lines are already back in HBM); the event pair's
    ticks are about 2 us apart here, so the mean over the calls is reported
    next to the median.  Steady: the calls of one decode step over `layers`
    layers, each with its own cache of the same shape (so every call streams
    its cache from HBM), back to back in one timed region, per layer."""
    import torch
    flush = torch.empty(512 * 1024 * 1024, dtype=torch.uint8, device=q.device)
    flush_rd = torch.ones(128 * 1024 * 1024, dtype=torch.float32, device=q.device)
    sink = torch.empty((), dtype=torch.float32, device=q.device)
    out = torch.empty_like(q)
    for _ in range(3):
        cpattn.gqa_decode(q, kc, vc, lens, out)
    ts = []
    for _ in range(iters):
        flush.zero_()
        torch.sum(flush_rd, dim=0, out=sink)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        cpattn.gqa_decode(q, kc, vc, lens, out)
        e1.record()
        torch.cuda.synchronize()
        ts.append(e0.elapsed_time(e1))
    del flush, flush_rd
    ts.sort()
    med = ts[len(ts) // 2]
    mean = sum(ts) / len(ts)
    by = decode_bytes(lens_host)
    gbs = by / (mean / 1e3) / 1e9
    res = {"us": mean * 1e3, "us_median": med * 1e3, "kv_bytes": by, "gbs": gbs, "frac_of_hbm": gbs / peaks["hbm_gbs"],
           "l2": "flushed before each launch (512 MB write + 512 MB read)"}
    # steady state over the layers of one decode step
    g = torch.Generator(device=q.device).manual_seed(99)
    caches = [(torch.randn(q.shape, device=q.device, generator=g).to(q.dtype),
               torch.randn(kc.shape, device=q.device, generator=g).to(kc.dtype),
               torch.randn(vc.shape, device=q.device, generator=g).to(vc.dtype)) for _ in range(layers)]
    outs = [torch.empty_like(q) for _ in range(layers)]
    for _ in range(2):
        for (qi, ki, vi), oi in zip(caches, outs):
            cpattn.gqa_decode(qi, ki, vi, lens, oi)
    torch.cuda.synchronize()
    tl = []
    for _ in range(7):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for (qi, ki, vi), oi in zip(caches, outs):
            cpattn.gqa_decode(qi, ki, vi, lens, oi)
        e1.record()
        torch.cuda.synchronize()
        tl.append(e0.elapsed_time(e1) / layers)
    cpattn.check_device()
    tl.sort()
    per = tl[len(tl) // 2]
    sgbs = by / (per / 1e3) / 1e9
    res["steady"] = {"per_layer_us": per * 1e3, "layers": layers, "gbs": sgbs, "frac_of_hbm": sgbs / peaks["hbm_gbs"],
                     "note": "one decode step: %d calls on %d distinct caches of the decode shape, back to back "
                             "(%.1f GB of caches, far above L2)" % (layers, layers,
                                                                   layers * 2 * kc.numel() * kc.element_size() / 1e9)}
    return res


def measure_zero_copy(args, w, inputs, dec_inputs, dec_out, f_step, pstep, world, dev, cpattn):
    """The same step with load_balance=2: the kernels read natural-order
    q/k/v/dout and write natural-order out/dq/dk/dv under the balanced
    schedule, so the eight permute/unpermute launches drop out.  Timed in
    rounds of one permuted step (pstep) and one zero-copy step, so that the
    two meet the same clocks: a seconds-long run under the power cap slows
    down as it goes, and a comparison with the headline's earlier timed
    region would charge that to whichever was measured later."""
    import torch
    q, k, v, dout = inputs
    dqd, dkc, dvc, dlens = dec_inputs
    cp = w["cp"]
    out = torch.empty(w["B"], w["S"], w["Hq"], w["Dv"], dtype=torch.bfloat16, device=q.device)
    lse = torch.empty(w["B"], w["Hq"], w["S"], dtype=torch.float32, device=q.device)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)

    def zstep():
        cpattn.attn_fwd(q, k, v, cp, 2, out, lse)
        cpattn.attn_bwd(q, k, v, out, lse, dout, cp, 2, dq, dk, dv)
        cpattn.gqa_decode(dqd, dkc, dvc, dlens, dec_out)

    for _ in range(3):
        zstep()
    torch.cuda.synchronize()
    cpattn.check_device()
    pstep()
    n = max(3, min(args.steps, int(3000.0 / max(time_steps(pstep, 1), 1e-3))))
    barrier()
    zt, pt, prof = [], [], {}
    for _ in range(n):
        pt.append(time_steps(pstep, 1))
        cpattn.profile_start()
        zt.append(time_steps(zstep, 1))
        for name, (c, t) in cpattn.profile_stop().items():
            c0, t0 = prof.get(name, (0, 0.0))
            prof[name] = (c0 + c, t0 + t)
    ms = max_over_ranks(sum(zt) / n, dev)
    pms = max_over_ranks(sum(pt) / n, dev)
    barrier()
    peaks, _ = load_peaks()
    return {"ms_per_step": ms, "value": aggregate_throughput(f_step, ms / 1e3, world) / 1e12, "unit": "TFLOP/s",
            "steps": n, "permuted_ms_per_step": pms, "saved_ms_vs_permuted_step": pms - ms,
            "kernels": kernel_table(prof, w, peaks, ms * n / 1e3),
            "what": "fwd + bwd with load_balance=2 (natural-order tensors, balanced schedule) + decode, timed in "
                    "rounds alternating with the permuted step (permuted_ms_per_step)"}


def measure_decode_int8(q, kc, vc, lens, lens_host, peaks, cpattn, iters=30):
    """The decode workload against an int8 cache of the same shape (values
    drawn on the device, one fp32 scale per position and KV head), timed like
    ``measure_decode``; bytes are the int8 K/V plus their scales."""
    import torch
    g = torch.Generator(device=q.device).manual_seed(7)
    kq = torch.randint(-127, 128, kc.shape, generator=g, device=q.device, dtype=torch.int32).to(torch.int8)
    vq = torch.randint(-127, 128, vc.shape, generator=g, device=q.device, dtype=torch.int32).to(torch.int8)
    ks = 0.008 + 0.008 * torch.rand(kc.shape[:3], generator=g, device=q.device)
    vs = 0.008 + 0.008 * torch.rand(vc.shape[:3], generator=g, device=q.device)
    flush = torch.empty(512 * 1024 * 1024, dtype=torch.uint8, device=q.device)
    flush_rd = torch.ones(128 * 1024 * 1024, dtype=torch.float32, device=q.device)
    sink = torch.empty((), dtype=torch.float32, device=q.device)
    out = torch.empty_like(q)
    for _ in range(3):
        cpattn.gqa_decode_int8(q, kq, vq, ks, vs, lens, out)
    ts = []
    for _ in range(iters):
        flush.zero_()
        torch.sum(flush_rd, dim=0, out=sink)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        cpattn.gqa_decode_int8(q, kq, vq, ks, vs, lens, out)
        e1.record()
        torch.cuda.synchronize()
        ts.append(e0.elapsed_time(e1))
    ts.sort()
    med = ts[len(ts) // 2]
    mean = sum(ts) / len(ts)  # event ticks are about 2 us apart: the mean resolves finer than the median
    n = int(sum(int(x) for x in lens_host))
    by = n * DECODE["Hkv"] * DECODE["D"] * 2 + n * DECODE["Hkv"] * 4 * 2
    gbs = by / (mean / 1e3) / 1e9
    return {"us": mean * 1e3, "us_median": med * 1e3, "kv_bytes": by, "gbs": gbs, "frac_of_hbm": gbs / peaks["hbm_gbs"],
            "bf16_equivalent_gbs": decode_bytes(lens_host) / (mean / 1e3) / 1e9,
            "l2": "flushed before each launch (512 MB write + 512 MB read)"}


def measure_mla_decode(lens_host, peaks, cpattn, dev, seed, iters=30):
    """Absorbed-MLA decode (DeepSeek-V3-shaped: 128 heads, 576-column latent
    rows of which the first 512 are the value) on the decode workload's
    batch and lengths, L2 flushed before each launch like ``measure_decode``.
    Bytes: the valid latent rows, q and out; FLOPs: both products over the
    valid positions."""
    import torch
    from context_causal_attention_load_gb300 import synth
    B, H, Smax = DECODE["B"], 128, DECODE["Smax"]
    q, ckv, _ = synth.mla_decode_inputs(B, H, Smax, 1, Smax, seed=seed + 6)
    lens = torch.tensor(lens_host, dtype=torch.int32)
    q, ckv, lens = q.to(dev), ckv.to(dev), lens.to(dev)
    out = torch.empty(B, H, 512, dtype=torch.bfloat16, device=dev)
    flush = torch.empty(512 * 1024 * 1024, dtype=torch.uint8, device=dev)
    flush_rd = torch.ones(128 * 1024 * 1024, dtype=torch.float32, device=dev)
    sink = torch.empty((), dtype=torch.float32, device=dev)
    for _ in range(3):
        cpattn.mla_decode(q, ckv, lens, out=out)
    cpattn.check_device()
    ts = []
    for _ in range(iters):
        flush.zero_()
        torch.sum(flush_rd, dim=0, out=sink)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        cpattn.mla_decode(q, ckv, lens, out=out)
        e1.record()
        torch.cuda.synchronize()
        ts.append(e0.elapsed_time(e1))
    ts.sort()
    med = ts[len(ts) // 2]
    mean = sum(ts) / len(ts)  # event ticks are about 2 us apart: the mean resolves finer than the median
    n = int(sum(int(x) for x in lens_host))
    by = n * 576 * 2 + q.numel() * 2 + out.numel() * 2
    fl = 2.0 * n * H * (576 + 512)
    gbs = by / (mean / 1e3) / 1e9
    return {"us": mean * 1e3, "us_median": med * 1e3, "bytes": by, "gbs": gbs, "frac_of_hbm": gbs / peaks["hbm_gbs"],
            "tflops": fl / (mean / 1e3) / 1e12, "frac_of_bf16": fl / (mean / 1e3) / 1e12 / peaks["bf16_tflops"],
            "config": "B=%d H=%d latent 576 (value 512) Smax=%d, lengths of the decode workload" % (B, H, Smax),
            "l2": "flushed before each launch (512 MB write + 512 MB read)"}


def shard_medians(fns, rounds, inner):
    """Median device ms per call of each fn, over rounds that each time every
    fn once (inner calls back to back): interleaved, so that a clock that
    drifts under the power cap during the measurement weighs on every shard
    alike rather than on the last ones timed."""
    ts = [[] for _ in fns]
    for _ in range(rounds):
        for i, f in enumerate(fns):
            ts[i].append(time_steps(f, inner))
    return [sorted(t)[len(t) // 2] for t in ts]


def measure_shards(w, attn, cpattn, rounds=3, inner=1):
    """Per-shard forward and backward times, each shard's launch alone on the
    whole GPU, with load balancing on (slot-order tensors) and off (natural
    order), plus the tile-pair counts per head.  The backward of one shard
    writes its dq rows and its fp32 dk/dv contributions."""
    import torch
    res = {}
    cp = w["cp"]
    q, k, v, dout = attn.q, attn.k, attn.v, attn.dout
    out = torch.empty(w["B"], w["S"], w["Hq"], w["Dv"], dtype=torch.bfloat16, device=q.device)
    lse = torch.empty(w["B"], w["Hq"], w["S"], dtype=torch.float32, device=q.device)
    dq = torch.empty_like(q)
    dkp = torch.empty(k.shape, dtype=torch.float32, device=q.device)
    dvp = torch.empty(v.shape, dtype=torch.float32, device=q.device)
    for lb in (True, False):
        if lb:  # slot order, as the step leaves the permuted tensors
            qq, kk, vv, dd = attn.qp, attn.kp, attn.vp, attn.dop
        else:
            qq, kk, vv, dd = q, k, v, dout
        cpattn.attn_fwd(qq, kk, vv, cp, lb, out, lse)
        fns = [lambda s=s: cpattn.attn_fwd_shard(qq, kk, vv, cp, s, lb, out, lse) for s in range(cp)]
        for f in fns:
            f()
        fwd = shard_medians(fns, rounds, inner)
        cpattn.attn_fwd(qq, kk, vv, cp, lb, out, lse)  # full out/lse for the backward
        fns = [lambda s=s: cpattn.attn_bwd_shard(qq, kk, vv, out, lse, dd, cp, s, lb, dq, dkp, dvp) for s in range(cp)]
        for f in fns:
            f()
        bwd = shard_medians(fns, rounds, inner)
        e = {"tile_pairs_per_head": cpattn.tile_counts(w["S"], cp, lb), "fwd_ms": fwd,
             "fwd_max_over_min": max(fwd) / min(fwd)}
        if bwd:
            e["bwd_ms"] = bwd
            e["bwd_max_over_min"] = max(bwd) / min(bwd)
        res["lb_on" if lb else "lb_off"] = e
    cpattn.check_device()
    del out, lse, dq, dkp, dvp
    return res


def measure_workload(name, peaks, cpattn, dev, seed, steps=None, warmup=3):
    """The attention step (no decode) of another workload, for the same line:
    step time, fwd+bwd TFLOP/s, per-kernel rates; for the Llama2-shaped and
    the MLA layer also their per-shard times at one sequence."""
    import torch
    from context_causal_attention_load_gb300 import synth
    w = WORKLOADS[name]
    B, S, Hq, Hkv, Dqk, Dv = (w[k] for k in ("B", "S", "Hq", "Hkv", "Dqk", "Dv"))
    q, k, v, dout = synth.attention_inputs_device(B, S, Hq, Hkv, Dqk, Dv, seed=seed, q_scale=w["q_scale"],
                                                  device=dev)
    kr = None
    if w.get("rope"):
        k, kr = k[..., :128].contiguous(), k[:, :, 0, 128:].contiguous()
    attn = AttnStep(w, q, k, v, dout, cpattn, kr)
    for _ in range(warmup):
        attn()
    torch.cuda.synchronize()
    cpattn.check_device()
    est = time_steps(attn, 1)
    n = steps or max(3, min(100, int(3000.0 / max(est, 1e-3))))
    cpattn.profile_start()
    ms = time_steps(attn, n)
    prof = cpattn.profile_stop()
    timed_s = ms * n / 1e3
    f_step = flops_fwd(w) + flops_bwd(w)
    peak, peak_name = peak_for(peaks, timed_s)
    res = {"ms_per_step": ms, "tflops": f_step / (ms / 1e3) / 1e12, "steps": n,
           "frac": f_step / (ms / 1e3) / 1e12 / peak, "peak": peak_name,
           "config": {k: w[k] for k in ("B", "S", "Hq", "Hkv", "Dqk", "Dv", "cp", "lb")},
           "kernels": kernel_table(prof, w, peaks, timed_s)}
    if name in ("llama2_7b_s8192_cp4", "deepseek_v3_mla_s32768_cp4"):
        res["shards"] = measure_shards(w, attn, cpattn, rounds=5, inner=10 if name.startswith("llama2") else 1)
    if w["lb"] and (S // (2 * w["cp"])) % 128 == 0:
        # the same step with load_balance = 2: natural-order tensors, no permutes
        cp = w["cp"]
        out = torch.empty(B, S, Hq, Dv, dtype=torch.bfloat16, device=dev)
        lse = torch.empty(B, Hq, S, dtype=torch.float32, device=dev)
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        if kr is not None:
            dkr = torch.empty_like(kr)

            def zstep():
                cpattn.attn_fwd_mla(q, k, kr, v, cp, 2, out, lse)
                cpattn.attn_bwd_mla(q, k, kr, v, out, lse, dout, cp, 2, dq, dk, dkr, dv)
        else:
            def zstep():
                cpattn.attn_fwd(q, k, v, cp, 2, out, lse)
                cpattn.attn_bwd(q, k, v, out, lse, dout, cp, 2, dq, dk, dv)
        for _ in range(warmup):
            zstep()
        torch.cuda.synchronize()
        cpattn.check_device()
        # rounds alternating with the permuted step, so that both meet the same clocks
        inner = max(1, int(20.0 / max(est, 1e-3)))
        rounds = max(3, min(10, int(3000.0 / (2 * inner * max(est, 1e-3)))))
        zt, pt = [], []
        for _ in range(rounds):
            pt.append(time_steps(attn, inner))
            zt.append(time_steps(zstep, inner))
        zms, pms = sum(zt) / rounds, sum(pt) / rounds
        res["zero_copy"] = {"ms_per_step": zms, "tflops": f_step / (zms / 1e3) / 1e12,
                            "frac": f_step / (zms / 1e3) / 1e12 / peak, "steps": rounds * inner,
                            "permuted_ms_per_step": pms, "saved_ms_vs_permuted_step": pms - zms,
                            "what": "fwd + bwd with load_balance=2 (natural-order tensors, balanced schedule), "
                                    "timed in rounds alternating with the permuted step (permuted_ms_per_step)"}
        del out, lse, dq, dk, dv
    del attn, q, k, v, dout
    torch.cuda.empty_cache()
    return res


def run_only(args):
    """One decode measurement alone (for profiling it): prints its JSON."""
    import torch
    from context_causal_attention_load_gb300 import build as cbuild
    from context_causal_attention_load_gb300 import synth
    cbuild.build()
    from context_causal_attention_load_gb300 import cpattn
    cpattn.load()
    dev = torch.device("cuda", 0)
    D = DECODE
    dq_, dkc, dvc, dlens = (x.to(dev) for x in synth.decode_inputs(D["B"], D["Hq"], D["Hkv"], D["D"], D["Smax"],
                                                                   D["lo"], D["hi"], seed=args.seed + 4))
    lens_host = dlens.cpu().tolist()
    peaks, _ = load_peaks()
    if args.only == "decode":
        r = measure_decode(dq_, dkc, dvc, dlens, lens_host, peaks, cpattn, iters=args.steps)
    elif args.only == "decode_int8":
        r = measure_decode_int8(dq_, dkc, dvc, dlens, lens_host, peaks, cpattn, iters=args.steps)
    else:
        r = measure_mla_decode(lens_host, peaks, cpattn, dev, args.seed, iters=args.steps)
    print(json.dumps({args.only: r}), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default=HEADLINE)
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--no-extras", action="store_true", help="skip e2e/decode/shard/cpu measurements")
    ap.add_argument("--only", choices=["decode", "decode_int8", "mla_decode"],
                    help="time one decode measurement alone (--steps launches) and print it")
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "ours":
        args.warmup = 3
    w = WORKLOADS[args.workload]
    if args.only:
        run_only(args)
    elif args.impl == "reference":
        run_reference(args, w, args.workload)
    else:
        run_ours(args, w, args.workload)


if __name__ == "__main__":
    main()
