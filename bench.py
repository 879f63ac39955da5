"""Benchmark of the GB300 training-update megakernel.

python bench.py [--gpus N] [--steps K] [--warmup W] [--config b32] [--impl ours|reference]

One step is one complete training update (forward, cross-entropy, backward,
global-norm clip, AdamW) of the ~219M-parameter top-2-of-16 MoE on synthetic
tokens: one persistent-kernel launch per microbatch.  Prints one JSON line.
Multi-GPU runs (torchrun) are independent replicas (weak scaling): the
update has no data-parallel exchange in this single-GPU design.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import moe_inputs as mi  # noqa: E402

WORKLOADS = {
    "b32": "32 x 1024 tokens, one microbatch, 219M-param top-2-of-16 MoE (d 768, 8 layers, V 32000)",
    "b2": "2 x 1024 tokens, one microbatch, 219M-param top-2-of-16 MoE (d 768, 8 layers, V 32000)",
    "accum16": "16 microbatches of 8 x 1024 tokens, one optimizer step, 219M-param MoE",
    "top8": "1 x 4096 Zipf tokens, top-8-of-32 experts d_ff 256, 219M-param MoE",
    "tiny": "2 x 32 tokens, tiny fp32 MoE (d 64, 2 layers, 4 experts)",
    "looped": "32 x 1024 tokens, looped MoE: 4 distinct layers each visited twice (8 layer visits)",
    "selective": "selective updates: 16 microbatches of 2 x 1024 tokens, shared tensors stepped after "
                 "each microbatch, experts after the 16th",
    "b32_lowmem": "b32 with both memory rules (no attention dS^T kept, one layer of expert activations)",
}
NOMINAL_BF16_TFLOPS = 2250.0   # GB300 dense bf16 tensor peak (vendor figure, without sparsity)


def workload_config(name):
    """The model configuration and launch flags of a bench workload."""
    from adamw_persistent_sm_gb300 import binding as B
    if name == "selective":
        return mi.get_config("b2", micro_count=16), B.MT_FLAG_SELECTIVE_EXPERTS
    if name == "b32_lowmem":
        return mi.get_config("b32"), B.MT_FLAG_RECOMPUTE_ATTN_DS | B.MT_FLAG_RECOMPUTE_EXPERT_ACT
    return mi.get_config(name), 0


def param_bytes_per_update(n_params: int, micro_count: int = 1) -> float:
    """Algorithmic HBM bytes of the parameter term: gradient write 4, AdamW
    reads p, g, m, v 16 and writes p, m, v 12 plus the bf16 shadow 2, bf16
    weight reads in the forward and the dgrad products 4 (38 B/param); each
    later microbatch adds a read-modify-write of the gradient (8 B/param)."""
    return n_params * (38.0 + 8.0 * (micro_count - 1))
METRIC = "MoE train-update ms & tokens/s (B2x1024, B32x1024); % bf16 tensor peak"
ARENA_HDR_BYTES = 4512   # mt_read_outputs copies the arena's control header


def flops_per_update(cfg) -> float:
    """6 x active matmul parameters x tokens + causal attention (3 x 2 B S^2 d L)."""
    d, L, hq = cfg.d_model, cfg.n_layers, cfg.n_heads * cfg.head_dim
    per_layer = 3 * hq * d + hq * d + cfg.n_experts * d + cfg.top_k * 3 * cfg.d_ff * d
    active = L * per_layer + cfg.vocab * d
    toks = cfg.tokens_per_update
    attn = 3 * 2 * cfg.batch * cfg.seq ** 2 * hq * L * cfg.micro_count
    return 6.0 * active * toks + attn


def source_digest() -> str:
    """sha256 over the CUDA sources and the C header: the kernel a profile
    was taken from."""
    import hashlib
    h = hashlib.sha256()
    for d in (os.path.join(ROOT, "adamw_persistent_sm_gb300", "csrc"), os.path.join(ROOT, "include")):
        for f in sorted(os.listdir(d)):
            if f.endswith((".cu", ".cuh", ".h")):
                with open(os.path.join(d, f), "rb") as fh:
                    h.update(f.encode() + b"\0" + fh.read())
    return h.hexdigest()[:16]


def profiled_traffic(config: str):
    """DRAM bytes (read + write) per launch from the committed ncu summary of
    this workload, or None when there is none or the kernel's sources have
    changed since it was taken."""
    path = os.path.join(ROOT, "profiles", f"megakernel_{config}_dram.md")
    if not os.path.exists(path):
        return None
    vals = {}
    with open(path) as f:
        for line in f:
            if line.startswith("- source_digest:") or line.startswith("- dram_bytes_per_launch:"):
                k, v = line[2:].split(":", 1)
                vals[k.strip()] = v.strip().strip("`")
    if vals.get("source_digest") != source_digest() or "dram_bytes_per_launch" not in vals:
        return None
    return float(vals["dram_bytes_per_launch"])


def load_peaks() -> dict:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return dict(bf16=d.get("bf16_tflops", 1900.0), bf16_sustained=d.get("bf16_tflops_sustained", 1700.0),
                    hbm=d.get("hbm_gbs", 6800.0), source="measured")
    return dict(bf16=1900.0, bf16_sustained=1700.0, hbm=6800.0, source="fallback")


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, dev_uuid: str | None):
        self.dev = dev_uuid
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "200"]
            if self.dev:
                cmd += ["-i", self.dev]
            self.proc = subprocess.Popen(cmd, stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self) -> dict | None:
        if not self.proc:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) >= 7:
                    try:
                        rows.append((float(parts[0]), float(parts[1]), parts[3:7]))
                    except ValueError:
                        pass
        os.unlink(self.path)
        if not rows:
            return None
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for _, _, r in rows for i, v in enumerate(r) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(r[0] for r in rows), "sm_max_mhz": max(r[1] for r in rows),
                "reasons": reasons, "samples": len(rows)}


# ---------------------------------------------------------------------------
# CPU oracle baseline (bounded sample)
# ---------------------------------------------------------------------------
def oracle_sample_time(cfg, params, tokens, seq_tokens: int) -> tuple[float, str]:
    """Time the oracle, as it stands, on one sequence prefix of `seq_tokens`
    positions (forward + backward) plus the matching share of the clip+AdamW
    sweep.  Returns (seconds, description)."""
    import oracle
    D = oracle.Dims.of(cfg)
    tok = tokens[0][:1, :seq_tokens]
    share = seq_tokens / cfg.tokens_per_update
    t0 = time.perf_counter()
    P = oracle.to64(params)
    grads = {k: np.zeros_like(v) for k, v in P.items()}
    oracle.forward_backward(P, tok, D, 1.0 / oracle.n_targets(*tok.shape), grads)
    sl = {k: v.reshape(-1)[: max(1, int(v.size * share))] for k, v in P.items()}
    gs = {k: grads[k].reshape(-1)[: sl[k].size] for k in sl}
    z = {k: np.zeros_like(v) for k, v in sl.items()}
    oracle.clip_adamw(sl, gs, z, z, lr=cfg.lr, beta1=cfg.beta1, beta2=cfg.beta2, eps=cfg.eps,
                      weight_decay=cfg.weight_decay, clip_norm=cfg.clip_norm, clip_eps=cfg.clip_eps,
                      step=1)
    dt = time.perf_counter() - t0
    desc = (f"oracle (NumPy float64) forward+backward of one {seq_tokens}-token sequence of the "
            f"workload plus {share:.4%} of the clip+AdamW sweep; tokens/s = {seq_tokens}/time")
    return dt, desc


def cpu_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


# ---------------------------------------------------------------------------
def run_reference(args, cfg, rank):
    """The oracle as the reference arm: rank 0 only, host cores.  A step is a
    bounded sample of the workload (one sequence prefix of --ref-tokens
    positions plus its share of the optimizer sweep); ms_per_step is that
    measured sample time, and the time of a whole update at the same rate is
    reported apart as an extrapolation."""
    if rank != 0:
        return
    params = mi.make_params(cfg)
    toks = mi.make_update_tokens(cfg)
    seq_tokens = min(cfg.seq, args.ref_tokens)
    for _ in range(args.warmup):
        oracle_sample_time(cfg, params, toks, seq_tokens)
    times = []
    desc = ""
    for _ in range(args.steps):
        dt, desc = oracle_sample_time(cfg, params, toks, seq_tokens)
        times.append(dt)
    tot = sum(times)
    tps = seq_tokens * len(times) / tot
    ms_update = cfg.tokens_per_update / tps * 1e3
    line = {
        "impl": "reference", "metric": METRIC, "value": tps, "unit": "tokens/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": tot / len(times) * 1e3,
        "step_is": f"one bounded sample of {seq_tokens} tokens (measured)",
        "ms_per_update_extrapolated": ms_update, "extrapolated_from_tokens": seq_tokens,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": {"workload": f"{args.config}: {WORKLOADS[args.config]}"},
        "cpu_baseline": {"value": tps, "unit": "tokens/s", "cores": cpu_cores(), "kind": "oracle",
                         "sample": desc},
        "e2e": {"value": tps, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def make_update_fn(tr, cfg, flags, dtoks):
    """One step of a workload: the update's microbatch launches (under
    selective updates one period: a shared step per microbatch, the expert
    step after the last)."""
    from adamw_persistent_sm_gb300 import binding as B

    def one_update(step):
        if flags & B.MT_FLAG_SELECTIVE_EXPERTS:
            n = cfg.micro_count
            for i, t in enumerate(dtoks):
                tr.micro_step(t, i, step=(step - 1) * n + i + 1, flags=flags, expert_step=step)
        else:
            tr.update(dtoks, step=step, flags=flags)
    return one_update


def measure_workload(name, dev, steps=5, warmup=3):
    """ms per update of another workload, timed with CUDA events on the
    launching stream after warm-up (inputs resident in HBM)."""
    import torch
    from adamw_persistent_sm_gb300 import binding as B
    from adamw_persistent_sm_gb300.trainer import MoETrainer
    cfg, flags = workload_config(name)
    tr = MoETrainer(cfg, dev, flags=flags)
    tr.load_params(mi.make_params(cfg))
    dtoks = [torch.as_tensor(t).to(dev) for t in mi.make_update_tokens(cfg)]
    one = make_update_fn(tr, cfg, flags, dtoks)
    for k in range(warmup):
        one(k + 1)
    torch.cuda.synchronize(dev)
    stream = torch.cuda.current_stream(dev)
    evs = []
    for k in range(steps):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        one(warmup + k + 1)
        b.record(stream)
        evs.append((a, b))
    torch.cuda.synchronize(dev)
    out = tr.outputs()
    if out.status != B.MT_OK:
        raise RuntimeError(f"{name}: {B.status_string(out.status)}")
    ms = [a.elapsed_time(b) for a, b in evs]
    med = statistics.median(ms)
    peaks = load_peaks()
    flops = flops_per_update(cfg)
    r = {"workload": WORKLOADS[name], "ms_per_update": med, "ms_min": min(ms), "ms_max": max(ms),
         "tokens_per_s": cfg.tokens_per_update / (med / 1e3), "launches_per_update": cfg.micro_count,
         "tflops": flops / (med / 1e3) / 1e12, "frac_of_measured_bf16": flops / (med / 1e3) / 1e12 / peaks["bf16"],
         "arena_gb": tr.arena_bytes / 1e9, "timed_updates": steps}
    if flags & B.MT_FLAG_SELECTIVE_EXPERTS:
        r["ms_per_microbatch"] = med / cfg.micro_count
        r["context_h100_ms_per_microbatch"] = 10.28
    pb = param_bytes_per_update(tr.n_params, 1 if flags & B.MT_FLAG_SELECTIVE_EXPERTS else cfg.micro_count)
    r["hbm_param_term_frac"] = pb / (med / 1e3) / 1e9 / peaks["hbm"]
    r["hbm_param_term_note"] = ("38 B/param parameter term only (a lower bound on the algorithmic "
                                "bytes) over the measured copy bandwidth")
    del tr, dtoks
    torch.cuda.empty_cache()
    return r


def barrier_idle_fraction(cfg, flags, dev):
    """Mean over CTAs of the time spent waiting at grid barriers over the
    launch's duration, from one traced update (MT_FLAG_TRACE)."""
    import torch
    from adamw_persistent_sm_gb300 import binding as B
    from adamw_persistent_sm_gb300.trainer import MoETrainer
    tr = MoETrainer(cfg, dev, flags=flags | B.MT_FLAG_TRACE)
    tr.load_params(mi.make_params(cfg))
    dtoks = [torch.as_tensor(t).to(dev) for t in mi.make_update_tokens(cfg)]
    for k in range(2):
        tr.update(dtoks, step=k + 1)
    out = tr.outputs()
    tv = tr.debug_view(B.MT_VIEW_TRACE, 0, torch.int64).cpu().numpy().reshape(-1, B.MT_TRACE_WORDS)
    G = out.n_ctas
    nb = min(out.n_phases, B.MT_TRACE_PHASES)
    bars = tv[:G, :2 * B.MT_TRACE_PHASES].reshape(G, B.MT_TRACE_PHASES, 2)[:, :nb].astype(np.float64)
    jobs = tv[:G, 2 * B.MT_TRACE_PHASES:].reshape(G, B.MT_TRACE_JOBS, 2)
    nj = int((jobs[0, :, 0] > 0).sum())
    span = (jobs[:, nj - 1, 0] - jobs[:, 0, 0]).astype(np.float64)
    wait = (bars[:, :, 1] - bars[:, :, 0]).sum(axis=1)
    del tr
    torch.cuda.empty_cache()
    return {"mean": float(np.mean(wait / span)), "max": float(np.max(wait / span)), "barriers": nb,
            "source": "in-kernel trace of one traced update (MT_FLAG_TRACE), per CTA: "
                      "sum of (release - arrival) at grid barriers / launch span"}


def run_ours(args, cfg, rank, world, wflags=0):
    import torch
    from adamw_persistent_sm_gb300 import binding as B
    from adamw_persistent_sm_gb300.trainer import MoETrainer

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    B.load(build_if_missing=True)
    params = mi.make_params(cfg)
    host_toks = mi.make_update_tokens(cfg)
    flags = wflags | _sched_flags(args)
    tr = MoETrainer(cfg, dev, flags=flags)
    tr.load_params(params)
    dtoks = [torch.as_tensor(t).to(dev) for t in host_toks]
    stream = torch.cuda.current_stream(dev)

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()
        torch.cuda.synchronize(dev)

    one_update = make_update_fn(tr, cfg, flags, dtoks)

    step = 1
    for _ in range(args.warmup):
        one_update(step)
        step += 1
    out = tr.outputs()
    if out.status != B.MT_OK:
        raise RuntimeError(f"device status {B.status_string(out.status)} site {out.error_site}")

    uuid = None
    try:
        uuid = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        pass
    clocks = ClockSampler(uuid)
    barrier()
    clocks.start()
    time.sleep(0.3)
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    per_launch = []
    ev0.record(stream)
    for _ in range(args.steps):
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        one_update(step)
        b.record(stream)
        per_launch.append((a, b))
        step += 1
    ev1.record(stream)
    barrier()
    clock_info = clocks.stop()
    ms_total = ev0.elapsed_time(ev1)
    upd_ms = [a.elapsed_time(b) for a, b in per_launch]
    out = tr.outputs()
    if out.status != B.MT_OK:
        raise RuntimeError(f"device status {B.status_string(out.status)} site {out.error_site}")
    ms = ms_total / args.steps
    if world > 1:
        import torch.distributed as dist
        t = torch.tensor([ms], device=dev)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        ms = float(t.item())

    # ---- end to end through the public API: pinned host tokens in, loss out --
    e2e = None
    if not args.no_e2e:
        pinned = [torch.as_tensor(t).pin_memory() for t in host_toks]
        h2d = sum(t.numel() * 4 for t in pinned)
        barrier()
        t0 = time.perf_counter()
        n_e2e = max(1, min(args.steps, 5))
        for _ in range(n_e2e):
            for i, p in enumerate(pinned):
                dtoks[i].copy_(p, non_blocking=True)
            one_update(step)
            step += 1
            o = tr.outputs()           # synchronises and reads the loss back
            if o.status != B.MT_OK:
                raise RuntimeError(B.status_string(o.status))
        e2e_ms = (time.perf_counter() - t0) * 1e3 / n_e2e
        e2e = {"value": cfg.tokens_per_update * world / (e2e_ms / 1e3), "unit": "tokens/s",
               "ms_per_step": e2e_ms, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": ARENA_HDR_BYTES}

    if rank != 0:
        return
    n_params = tr.n_params
    arena_gb = tr.arena_bytes / 1e9
    del tr
    torch.cuda.empty_cache()
    peaks = load_peaks()
    flops = flops_per_update(cfg)
    launch_ms = statistics.mean(upd_ms) / cfg.micro_count
    achieved = flops / cfg.micro_count / (launch_ms / 1e3) / 1e12
    traffic = profiled_traffic(args.config)
    roof = {"bound": "tensor", "achieved": achieved, "peak": peaks["bf16"], "unit": "TFLOP/s",
            "frac": achieved / peaks["bf16"], "traffic": traffic,
            "peak_source": f"{peaks['source']} bf16 burst (MEASURED_PEAKS.json)",
            "frac_of_nominal_dense_bf16": achieved / NOMINAL_BF16_TFLOPS,
            "nominal_peak": NOMINAL_BF16_TFLOPS,
            "algorithmic_bytes_param_term": param_bytes_per_update(n_params, cfg.micro_count) / cfg.micro_count,
            "kernel": "mt_megakernel<__nv_bfloat16> (the only kernel of the step)"}
    extra = {}
    idle = None
    if not args.no_extra and args.config == "b32" and world == 1:
        idle = barrier_idle_fraction(cfg, flags, dev)
        for name in ("b2", "top8", "accum16", "selective", "looped", "b32_lowmem"):
            extra[name] = measure_workload(name, dev)
    cpu = None
    if not args.no_cpu_baseline:
        dt, desc = oracle_sample_time(cfg, params, host_toks, min(cfg.seq, args.cpu_tokens))
        tps = min(cfg.seq, args.cpu_tokens) / dt
        cpu = {"value": tps, "unit": "tokens/s", "cores": cpu_cores(), "kind": "oracle", "sample": desc}
    line = {
        "metric": METRIC,
        "value": cfg.tokens_per_update * world / (ms / 1e3),
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms,
        "ms_per_step_min": min(upd_ms),
        "ms_per_step_median": statistics.median(upd_ms),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16" if cfg.precision == "bf16" else "f32",
        "data": "synthetic",
        "config": {"workload": f"{args.config}: {WORKLOADS[args.config]}",
                   "tokens_per_update": cfg.tokens_per_update,
                   "flops_per_update": flops,
                   "l2": "inputs larger than L2 (arena %.1f GB, params %.2f GB)" % (
                       arena_gb, n_params * 4 / 1e9),
                   "replicas": world,
                   "context_h100_ms_per_update": {"b2": [13.63, 13.77], "b32": [68.27, 68.61]}.get(args.config)},
        "tflops": achieved,
        "gpu_launches": args.steps * cfg.micro_count,
        "launches_per_update": cfg.micro_count,
        "grid_barriers_per_launch": out.n_phases,
        "roofline": roof,
        "barrier_idle_frac": idle,
        "other_workloads": extra or None,
        "clocks": clock_info,
        "e2e": e2e,
        "cpu_baseline": cpu,
        "loss": out.loss_update,
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
# profiling helpers
# ---------------------------------------------------------------------------
JOB_NAMES = {0: "barrier wait", 1: "embed", 2: "qkv", 3: "attn_fwd", 4: "wo", 5: "router", 6: "route",
             7: "gateup", 8: "down", 9: "combine", 10: "lm_head", 11: "ce", 12: "loss", 13: "lm_dgrad",
             14: "lm_wgrad", 15: "final_norm_bwd", 16: "router_wgrad", 17: "moe_bwd1", 18: "colfinal",
             19: "down_dgrad", 20: "down_wgrad", 21: "gateup_dgrad", 22: "gateup_wgrad", 23: "moe_bwd2",
             24: "wo_dgrad", 25: "wo_wgrad", 26: "attn_bwd_dq", 27: "qkv_dgrad", 28: "qkv_wgrad",
             29: "attn_norm_bwd", 30: "embed_bwd", 31: "norm_partial", 32: "wo_ksum", 33: "qkv_ksum",
             34: "adamw", 35: "attn_bwd_dkdv", 36: "router_wait", 37: "gateup_again"}


def _sched_flags(args):
    from adamw_persistent_sm_gb300 import binding as B
    return B.MT_FLAG_BARRIERS_ONLY if args.barriers_only else 0


def run_trace(args, cfg):
    """Per-job time of one update from the in-kernel trace (MT_FLAG_TRACE):
    each CTA stamps the end of every job; a job's time is the gap to the
    previous stamp."""
    import torch
    from adamw_persistent_sm_gb300 import binding as B
    from adamw_persistent_sm_gb300.trainer import MoETrainer
    tr = MoETrainer(cfg, "cuda:0", flags=B.MT_FLAG_TRACE | _sched_flags(args))
    tr.load_params(mi.make_params(cfg))
    toks = [torch.as_tensor(t).cuda() for t in mi.make_update_tokens(cfg)]
    for it in range(max(1, args.warmup)):
        tr.update(toks, step=it + 1)
    out = tr.outputs()
    assert out.status == B.MT_OK, B.status_string(out.status)
    tv = tr.debug_view(B.MT_VIEW_TRACE, 0, torch.int64).cpu().numpy().reshape(-1, B.MT_TRACE_WORDS)
    jobs = tv[:out.n_ctas, 2 * B.MT_TRACE_PHASES:].reshape(out.n_ctas, B.MT_TRACE_JOBS, 2)
    nj = int((jobs[0, :, 0] > 0).sum())
    t = jobs[:, :nj, 0].astype(np.float64)
    ids = jobs[0, :nj, 1]
    dur = np.diff(t, axis=1)
    mean, mx = {}, {}
    for j in range(1, nj):
        k = JOB_NAMES.get(int(ids[j]), str(int(ids[j])))
        mean[k] = mean.get(k, 0.0) + dur[:, j - 1].mean() / 1e6
        mx[k] = mx.get(k, 0.0) + dur[:, j - 1].max() / 1e6
    print(f"{args.config}: {nj} job stamps over {(t[:, -1] - t[:, 0]).mean() / 1e6:.2f} ms "
          f"({out.n_phases} grid barriers, {out.n_ctas} CTAs)")
    print(f"  {'job':16s} {'mean ms':>9s} {'max-over-CTAs ms':>18s}")
    for k in sorted(mx, key=lambda k: -mx[k]):
        print(f"  {k:16s} {mean[k]:9.3f} {mx[k]:18.3f}")
    # grid-barrier waits (arrival to release, mean over CTAs), grouped by the
    # job that ran before each barrier
    bars = tv[:out.n_ctas, :2 * B.MT_TRACE_PHASES].reshape(out.n_ctas, B.MT_TRACE_PHASES, 2).astype(np.float64)
    nb = min(out.n_phases, B.MT_TRACE_PHASES)
    waits = (bars[:, :nb, 1] - bars[:, :nb, 0]).mean(axis=0) / 1e6
    before, last, k = {}, "start", 0
    for jid in ids:
        if int(jid) == 0:
            if k < nb:
                before[k] = last
            k += 1
        else:
            last = JOB_NAMES.get(int(jid), str(int(jid)))
    by = {}
    for p_, w in enumerate(waits):
        by[before.get(p_, "?")] = by.get(before.get(p_, "?"), 0.0) + w
    print(f"  barrier wait by the job before the barrier ({nb} barriers, {waits.sum():.3f} ms):")
    for k_ in sorted(by, key=lambda k_: -by[k_])[:12]:
        print(f"    {k_:16s} {by[k_]:9.3f}")


OPS = ("attn_fwd", "attn_bwd", "router", "lm_ce", "adamw")


def run_op(args, cfg):
    """One step of the update alone (mt_debug_run: the update's own device
    code in the single-op kernel) on seeded inputs, timed with CUDA events:
    --op attn_fwd|attn_bwd|router|lm_ce|adamw.  Prints ms per launch and the
    algorithmic rate (FLOP/s for the tensor-core steps, bytes/s for the
    others)."""
    import torch
    from adamw_persistent_sm_gb300 import binding as B
    from adamw_persistent_sm_gb300.trainer import MoETrainer
    if args.batch:
        cfg = cfg.replace(batch=args.batch)
    if args.layers:
        cfg = cfg.replace(n_layers=args.layers, n_unique_layers=0)
    B.load(build_if_missing=True)
    tr = MoETrainer(cfg, "cuda:0")
    T, d, hq, V = cfg.tokens_per_micro, cfg.d_model, cfg.n_heads * cfg.head_dim, cfg.vocab
    dt = torch.bfloat16 if cfg.precision == "bf16" else torch.float32
    g = torch.Generator(device="cuda").manual_seed(11)

    def fill(which, n, std=1.0, dtype=dt):
        v = tr.debug_view(which, 0, dtype)
        v.copy_((torch.randn(n, device="cuda", generator=g) * std).to(dtype))

    opid = {"attn_fwd": B.MT_OP_ATTN_FWD, "attn_bwd": B.MT_OP_ATTN_BWD, "router": B.MT_OP_ROUTER,
            "lm_ce": B.MT_OP_LM_CE, "adamw": B.MT_OP_CLIP_ADAMW}[args.op]
    toks = torch.as_tensor(mi.make_tokens(cfg, 0)).cuda()
    causal_pairs = cfg.batch * cfg.n_heads * cfg.seq * (cfg.seq + 1) / 2
    if args.op in ("attn_fwd", "attn_bwd"):
        fill(B.MT_VIEW_QKV, T * 3 * hq)
        tr.debug_run(B.MT_OP_ATTN_FWD)
        fill(B.MT_VIEW_DOUT, T * hq)
        work, unit = (2 if args.op == "attn_fwd" else 4) * 2 * causal_pairs * cfg.head_dim, "TFLOP/s"
        note = "causal score/probability products: QK^T and PV (forward); S, dP, dV, dK recomputed or " \
               "accumulated plus dQ counted as twice the forward (backward)"
    elif args.op == "router":
        fill(B.MT_VIEW_XMID, T * d, 0.05, torch.float32)
        ob = 2 if cfg.precision == "bf16" else 4
        work, unit = T * (4 * d + ob * d + 4 * cfg.n_experts + 8 * cfg.top_k + ob * d + cfg.top_k * ob * d), "GB/s"
        note = ("bytes per token: x_mid read 4d, r2 write, logits 4E, choices and weights 8K, the "
                "dispatch gather's r2 read and K expert-row writes")
    elif args.op == "lm_ce":
        fill(B.MT_VIEW_FINAL_NORM, T * d)
        tr.params.normal_(0.0, 0.02, generator=g)
        tr.sync_shadow()
        work, unit = 2.0 * T * V * d, "TFLOP/s"
        note = "LM-head product 2 T V d (the fused cross-entropy rides on its epilogue and one pass)"
    else:
        n = tr.n_params
        for buf, std in ((tr.params, 0.02), (tr.grads, 1e-4), (tr.adam_m, 1e-5), (tr.adam_v, 1e-9)):
            buf.normal_(0.0, std, generator=g)
        tr.adam_v.abs_()
        work, unit = 34.0 * n, "GB/s"
        note = "34 B/param: norm pass reads g (4); AdamW reads p, g, m, v (16), writes p, m, v (12) " \
               "and the bf16 shadow (2)"

    def once():
        tr.debug_run(opid, 0, tokens=toks, step=3 if args.op == "adamw" else None)

    for _ in range(args.warmup):
        once()
    torch.cuda.synchronize()
    st = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(st)
    for _ in range(args.steps):
        once()
    e1.record(st)
    torch.cuda.synchronize()
    out = tr.outputs()
    assert out.status == B.MT_OK, B.status_string(out.status)
    ms = e0.elapsed_time(e1) / max(1, args.steps)
    rate = work / (ms / 1e3) / (1e12 if unit == "TFLOP/s" else 1e9)
    peaks = load_peaks()
    peak = peaks["bf16"] if unit == "TFLOP/s" else peaks["hbm"]
    print(json.dumps({"op": args.op, "config": cfg.name, "batch": cfg.batch, "layers": cfg.n_layers, "ms": ms, "rate": rate,
                      "unit": unit, "frac_of_measured_peak": rate / peak, "work": work, "note": note,
                      "launches": args.steps}))


def run_product(args):
    """One matrix product C = A B^T through the megakernel's product engine
    (mt_debug_gemm): --product M N K a_mn b_mn."""
    import torch
    from adamw_persistent_sm_gb300 import binding as B
    M, N, K, amn, bmn = args.product
    out_mode = {"f32": 0, "bf16": 1, "none": 2, "f32-bulk": 4, "bf16-bulk": 5}[args.product_out]
    B.load(build_if_missing=True)
    arena = torch.zeros(1 << 16, dtype=torch.uint8, device="cuda")
    B.mt_arena_init(arena.data_ptr(), arena.numel())
    st = torch.cuda.current_stream().cuda_stream
    A = (torch.randn(K, M, device="cuda") if amn else torch.randn(M, K, device="cuda")).bfloat16()
    Bm = (torch.randn(K, N, device="cuda") if bmn else torch.randn(N, K, device="cuda")).bfloat16()
    C = torch.empty(M, N, device="cuda")

    def once():
        r = B.mt_debug_gemm(A.data_ptr(), amn, Bm.data_ptr(), bmn, C.data_ptr(), M, N, K, 0, 0, 0,
                            B.MT_PREC_BF16, 1 | (out_mode << 1) | (16 if args.product_tall else 0),
                            arena.data_ptr(), arena.numel(), st)
        assert r == B.MT_OK, B.status_string(r)

    for _ in range(args.warmup):
        once()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(args.steps):
        once()
    e1.record()
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / max(1, args.steps)
    o = B.mt_read_outputs(arena.data_ptr(), st)
    assert o.status == B.MT_OK
    print(json.dumps({"product": [M, N, K, amn, bmn], "out": args.product_out, "tall": args.product_tall, "ms": ms,
                      "tflops": 2.0 * M * N * K / ms / 1e9}))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--config", default="b32", choices=sorted(WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-tokens", type=int, default=1024)
    ap.add_argument("--ref-tokens", type=int, default=256)
    ap.add_argument("--trace", action="store_true", help="print the per-job time of one update")
    ap.add_argument("--op", choices=OPS, help="time one step of the update alone (single-op kernel)")
    ap.add_argument("--batch", type=int, default=0, help="--op: override the workload's batch")
    ap.add_argument("--layers", type=int, default=0, help="--op: override the workload's layer count")
    ap.add_argument("--no-extra", action="store_true",
                    help="b32 only: skip the other workloads and the traced barrier-idle measurement")
    ap.add_argument("--barriers-only", action="store_true",
                    help="grid barriers at every hand-off (no per-block dependency counters)")
    ap.add_argument("--product", type=int, nargs=5, metavar=("M", "N", "K", "A_MN", "B_MN"),
                    help="time one product through the tensor-core engine")
    ap.add_argument("--product-tall", action="store_true",
                    help="--product: K-major operands in 128-row (A) / 256-row (B) TMA boxes")
    ap.add_argument("--product-out", default="f32", choices=["f32", "bf16", "none", "f32-bulk", "bf16-bulk"],
                    help="output of --product: fp32, bf16, accumulators read and dropped, or fp32 / bf16 "
                         "written by bulk tensor stores")
    args = ap.parse_args()
    cfg, wflags = workload_config(args.config)
    if args.product:
        run_product(args)
        return
    if args.trace:
        run_trace(args, cfg)
        return
    if args.op:
        run_op(args, cfg)
        return
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.impl == "reference":
        run_reference(args, cfg, rank)
        return
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", 0)))
        dist.init_process_group("nccl")
    try:
        run_ours(args, cfg, rank, world, wflags)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
