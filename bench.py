"""Benchmark of one speculative-decoding verify round on GB300.

Workload (one "step" = one whole verify round over one batch):
  ragged full verify round — B = 64 sequences, gamma_b ~ U{1..10} drafts each,
  committed contexts ctx_b ~ U[128, 8192], a 36-layer Qwen3-8B-shaped stack
  (d 4096, 32 q / 8 kv heads of 128, MLP 12288) with random-init bf16 weights
  N(0, 0.02), the 151936-token LM head + softmax at T = 0.7, and the
  rejection sampler with Philox uniforms (seed 0).  All inputs are synthetic.

Metric: accepted tokens per second = sum_b (n_b + 1) / verify-round time,
measured with CUDA events over K CUDA-graph replays of the round (inputs
resident in HBM; weights + KV cache of ~93 GB are far larger than L2, so no
flush is needed).  Extra keys: verify-round microseconds and whole-round HBM
GB/s, the weight-read amortisation of the linear stack (M = 5 vs M = 1),
the dominant kernel's roofline, the oracle's CPU throughput on a bounded
sample, and the end-to-end number with host buffers.

``--impl reference`` times the CPU oracle on the same workload instead.
Under torchrun every rank runs an independent replica (weak scaling, no
collective on the data path).
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

METRIC = "verify-round accepted tokens/sec (B*(gamma+1) rows, full stack + LM head + sampler)"
UNIT = "tokens/s"
WORKLOAD = ("ragged full verify round: B=64, gamma_b~U{1..10}, ctx_b~U[128,8192], 36-layer "
            "Qwen3-8B-shaped stack + 151936-vocab LM head + rejection sampler, T=0.7, Philox seed 0")
B, G_LO, G_HI, CTX_LO, CTX_HI = 64, 1, 10, 128, 8192
TEMP, SIGMA, SEED = 0.7, 1.0, 0
TYPICAL_EPS, TYPICAL_DELTA = 0.09, 0.3   # typical acceptance: threshold floor and entropy slope
CPU_SAMPLE_SEQS = 4   # sequences of the round the oracle runs (both the cpu_baseline leg and --impl reference)


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        d = json.load(open(p))
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), float(d.get("bf16_tflops_sustained", d["bf16_tflops"])), "measured"
    except Exception:
        return 6800.0, 1900.0, 1700.0, "fallback"


# --------------------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None
        self.path = os.path.join(tempfile.gettempdir(), f"spec_verify_clocks_{os.getpid()}.csv")

    def start(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.idx}", f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
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
        self.f.close()
        rows = []
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append((float(parts[1]), float(parts[2]), parts[5:9]))
            except ValueError:
                continue
        if not rows:
            return None
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for _, _, r in rows for i, v in enumerate(r) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(r[0] for r in rows), "sm_max_mhz": max(r[1] for r in rows),
                "reasons": reasons, "samples": len(rows)}


# --------------------------------------------------------------------------- workload
def make_batch():
    import synth
    return synth.ragged_batch(SEED, B, G_LO, G_HI, CTX_LO, CTX_HI)


def algorithmic_bytes(batch, dims):
    """Bytes the round must move at minimum (weights once, KV once, activations, p)."""
    lin_w = dims.layers * 2 * (dims.qkv * dims.d + dims.d * dims.Hq * dims.D + 2 * dims.I * dims.d + dims.d * dims.I)
    kv = dims.layers * 2 * int(np.sum(batch.ctx_len.astype(np.int64) + batch.gammas + 1)) * dims.Hkv * dims.D * 2
    head = 2 * dims.V * dims.d + batch.M * dims.V * 4
    return lin_w, kv, head


# DRAM bytes per algorithmic byte of attention_tc_kernel, from an ncu capture
# (dram__bytes_read.sum + dram__bytes_write.sum) of one B = 16 launch of the kernel built from the
# sources whose SHA-256 prefix is ATTN_TRAFFIC_SOURCES.  Traffic grows with the keys streamed, so the
# bench scales the ratio to its own launch; once either source file changes the ratio no longer
# describes the kernel and the bench reports traffic as null.
ATTN_DRAM_PER_ALG_BYTE = 1.032
ATTN_TRAFFIC_SOURCES = "b8241e892ef4c034"
ATTN_SOURCE_FILES = ("speculative_decoding_verify_05_gb300/csrc/attention_tc.cu",
                     "speculative_decoding_verify_05_gb300/csrc/common.cuh")


def attention_sources_digest() -> str:
    import hashlib
    h = hashlib.sha256()
    for f in ATTN_SOURCE_FILES:
        with open(os.path.join(ROOT, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def attention_traffic(ab):
    """(DRAM bytes per launch or None, why)."""
    if attention_sources_digest() != ATTN_TRAFFIC_SOURCES:
        return None, "kernel sources changed since the DRAM counters were taken"
    return ab * ATTN_DRAM_PER_ALG_BYTE, "ncu dram__bytes_read+write on a B=16 launch, scaled by algorithmic bytes"


def attention_bytes(batch, dims):
    """Per attention launch: K/V cache read + new K/V + Q read + O write."""
    keys = int(np.sum(batch.ctx_len.astype(np.int64)))
    kv = keys * dims.Hkv * dims.D * 2 * 2
    new = batch.M * dims.Hkv * dims.D * 2 * 2 * 2          # read new k,v and write them to the cache
    qo = batch.M * dims.Hq * dims.D * 2 * 2
    return kv + new + qo


def workload_config(batch, cap):
    """The `config` of both arms' lines: the workload and the batch it draws."""
    return {"workload": WORKLOAD, "B": B, "M_rows": int(batch.M), "sum_ctx": int(batch.ctx_len.sum()), "cap": int(cap)}


def round_cap(batch):
    return int((batch.ctx_len + batch.gammas + 1).max() + 15) // 16 * 16


# --------------------------------------------------------------------------- ranks
def combine_ranks(ms: float, tokens: float, device, world: int):
    """Whole-job numbers of a replicated round: the slowest rank's time and every rank's tokens
    (each rank runs its own B-sequence batch; nothing else crosses ranks)."""
    import torch
    if world <= 1:
        return float(ms), float(tokens)
    import torch.distributed as dist
    t = torch.tensor([float(ms)], device=device)
    tok = torch.tensor([float(tokens)], device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.all_reduce(tok, op=dist.ReduceOp.SUM)
    return float(t.item()), float(tok.item())


def reference_runs_here() -> bool:
    """The reference arm (the CPU oracle) runs on rank 0 only; other ranks exit without work."""
    return int(os.environ.get("RANK", "0")) == 0


# --------------------------------------------------------------------------- GPU arm
def build_round(dev, rank, S, E, synth, fused_swiglu=True, fused_sampler=True):
    """Resident state of the benchmark round (weights, KV caches, inputs, draft distribution)
    and a function that runs one full verify round on it."""
    import torch
    dims = E.Dims()
    batch = make_batch()
    cap = round_cap(batch)
    torch.manual_seed(1234 + rank)

    # ---- resident model state: weights, KV caches (random), inputs
    sw = E.random_stack(dims, seed=1000 + rank, device=dev)
    g = torch.Generator(device=dev)
    g.manual_seed(2000 + rank)
    kcs, vcs = [], []
    for _ in range(dims.layers):
        k = torch.empty((B, dims.Hkv, cap, dims.D), dtype=torch.bfloat16, device=dev)
        v = torch.empty_like(k)
        k.normal_(0, 1, generator=g)
        v.normal_(0, 1, generator=g)
        kcs.append(k)
        vcs.append(v)
    eng = E.VerifyEngine(dims, sw, kcs, vcs, max_M=batch.M, max_rows=batch.max_rows, device=dev,
                         fused_swiglu=fused_swiglu, fused_sampler=fused_sampler)
    x0 = torch.empty((batch.M, dims.d), dtype=torch.bfloat16, device=dev).normal_(0, 1, generator=g)
    cu = torch.from_numpy(batch.cu_rows).to(dev)
    ctx = torch.from_numpy(batch.ctx_len).to(dev)
    U = torch.from_numpy(synth.uniforms_f32(SEED, batch.M)).to(dev)

    # ---- draft distribution: the target's probabilities perturbed in logit space
    # (q = softmax(log p + (sigma / T) * noise), i.e. logits + N(0, sigma^2) at temperature T)
    eng.x[:batch.M].copy_(x0)
    P0 = eng.verify_pass(eng.x[:batch.M], cu, ctx, TEMP).clone()
    qrows = np.concatenate([np.arange(batch.cu_rows[b], batch.cu_rows[b] + batch.gammas[b]) for b in range(B)])
    lp = torch.log(P0[torch.from_numpy(qrows).to(dev)].clamp_min(1e-38))
    noise = torch.empty_like(lp).normal_(0, 1, generator=g)
    q = torch.softmax(lp + (SIGMA / TEMP) * noise, dim=1).contiguous()
    drafts = torch.multinomial(q, 1, generator=g).view(-1).to(torch.int32)
    del P0, lp, noise
    out = (torch.empty(B, dtype=torch.int32, device=dev), torch.empty(batch.M, dtype=torch.int32, device=dev),
           torch.empty(B, dtype=torch.int32, device=dev))

    def step():
        eng.x[:batch.M].copy_(x0)
        eng.verify_round(eng.x[:batch.M], cu, ctx, q, drafts, U, TEMP, out=out)

    return dict(dims=dims, batch=batch, cap=cap, sw=sw, kcs=kcs, vcs=vcs, eng=eng, x0=x0, cu=cu, ctx=ctx,
                U=U, q=q, drafts=drafts, out=out, step=step)


def run_gpu(args):
    import torch
    import torch.distributed as dist

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl", init_method="env://")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    from speculative_decoding_verify_05_gb300 import binding as S
    from speculative_decoding_verify_05_gb300 import engine as E
    import synth

    hbm_peak, tc_peak, tc_sust, peak_src = peaks()
    st = build_round(dev, rank, S, E, synth, fused_swiglu=args.swiglu == "fused",
                     fused_sampler=args.sampler == "fused")
    dims, batch, cap, sw, kcs, vcs, eng = (st[k] for k in ("dims", "batch", "cap", "sw", "kcs", "vcs", "eng"))
    x0, cu, ctx, q, drafts, out, step = (st[k] for k in ("x0", "cu", "ctx", "q", "drafts", "out", "step"))
    S.reset_launch_count()

    # eager warm-up (loads every kernel), then the engine captures the round in one CUDA graph
    step()
    torch.cuda.synchronize()
    S.spec_device_status()
    S.reset_launch_count()
    replay = eng.capture_round(x0, cu, ctx, q, drafts, st["U"], TEMP, out)
    launches_per_step = S.launch_count() // 2        # the capture ran the round twice (warm-up + record)
    torch.cuda.synchronize()

    for _ in range(args.warmup):
        replay()
    torch.cuda.synchronize()
    S.spec_device_status()

    clocks = ClockSampler(local)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.3)
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    cur = torch.cuda.current_stream()
    ev0.record(cur)
    for _ in range(args.steps):
        replay()
    ev1.record(cur)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    clk = clocks.stop()
    ms = ev0.elapsed_time(ev1) / args.steps
    n_acc = out[0].cpu().numpy()
    near = int(out[2].sum().item())
    accepted = int(n_acc.sum()) + B
    S.spec_device_status()

    ms_max, tok_all = combine_ranks(ms, accepted, dev, world)
    value = tok_all / (ms_max / 1e3)

    lin_w, kv, head = algorithmic_bytes(batch, dims)
    round_gbs = (lin_w + kv + head) / (ms / 1e3) / 1e9

    # ---- per-kernel timing (eager, CUDA events on the launching stream)
    per = kernel_timings(eng, batch, dims, cu, ctx, S, hbm_peak, tc_peak, tc_sust, peak_src,
                         sampler_inputs=(q, drafts, st["U"], out))

    per["ngram_propose"] = ngram_timing(S, hbm_peak, peak_src, dev)

    # ---- weight-read amortisation of the linear stack: M = 5 verify vs M = 1 decode
    lin = linear_stack_ratio(eng, dims, S, hbm_peak, peak_src)

    # ---- the draft side (the step before the verify pass), off with --no-draft
    draft = draft_timing(S, E, batch, dev, ms) if not args.no_draft else None

    # ---- end to end through the public API with host buffers
    e2e = end_to_end(args, eng, batch, dims, q, drafts, x0, S, torch, dev)

    # ---- the other configurations, after the timed round and outside its events: batch x depth
    # points (the small-M verify batch and the largest tensor-bound one) and configuration 3
    sweep = c3 = None
    if not args.no_extra:
        sweep = {"points": sweep_points(sw, dims, dev, SWEEP_DEFAULT, hbm_peak, tc_sust),
                 "context": SWEEP_CTX, "peaks": {"hbm_gbs": hbm_peak, "bf16_tflops_sustained": tc_sust,
                                                 "source": peak_src},
                 "note": "36-layer linear stack per point (one CUDA graph) and one layer's attention over B "
                         "sequences of 2048 keys; python bench.py --sweep runs all 15 points"}
        c3 = config3(sw, dims, dev, hbm_peak, peak_src)

    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return

    cpu = cpu_baseline(eng, batch, dims, kcs, vcs, sw, q, drafts) if world >= 1 and rank == 0 and not args.no_cpu else None
    dominant = max(per.values(), key=lambda r: r["total_ms"])
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_max, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16 (fp32 accumulate; fp32 softmax, fp64 sampler sums)",
        "data": "synthetic (random-init weights, random KV cache and hidden states, seeded)",
        "config": workload_config(batch, cap),
        "l2": "inputs larger than L2 (15.1 GB weights + %.1f GB KV read per round)" % (kv / 1e9),
        "graph": "whole round captured in one CUDA graph",
        "round_us": ms * 1e3,
        "round_hbm_gbs": round_gbs,
        "round_hbm_frac": round_gbs / hbm_peak,
        "accepted_tokens_per_round": accepted,
        "mean_acceptance_length": accepted / B,
        "near_ties": near,
        "roofline": dominant["roofline"],
        "kernels": {k: {kk: vv for kk, vv in v.items() if kk != "roofline"} | {"roofline": v["roofline"]}
                    for k, v in per.items()},
        "linear_stack": lin,
        "sweep": sweep,
        "config3": c3,
        "draft_phase": draft,
        "gpu_launches": launches_per_step * args.steps,
        "launches_per_step": launches_per_step,
        "clocks": clk,
        "e2e": e2e,
        "cpu_baseline": cpu,
    }
    print(json.dumps(line))
    if world > 1:
        dist.destroy_process_group()


def kernel_timings(eng, batch, dims, cu, ctx, S, hbm_peak, tc_peak, tc_sust, peak_src, reps=3,
                   sampler_inputs=None):
    """Average launch time of each hot kernel over all 36 layers (eager, CUDA events)."""
    import torch
    M = batch.M
    res = {}
    cur = torch.cuda.current_stream()

    def timeit(fn, n):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        fn()
        torch.cuda.synchronize()
        e0.record(cur)
        for _ in range(reps):
            fn()
        e1.record(cur)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / (reps * n)

    L = dims.layers
    hq, hk = dims.Hq * dims.D, dims.Hkv * dims.D
    qkv = eng.qkv[:M]

    def attn_all():
        for li in range(L):
            S.spec_verify_attention(qkv[:, :hq], qkv[:, hq:hq + hk], qkv[:, hq + hk:], cu, ctx,
                                    eng.kc[li], eng.vc[li], eng.max_rows, O=eng.o[:M], ws=eng.ws)
    t_attn = timeit(attn_all, L)
    ab = attention_bytes(batch, dims)
    res["verify_attention"] = {"avg_launch_us": t_attn * 1e3, "launches_per_round": L,
                               "total_ms": t_attn * L,
                               "roofline": {"kernel": "verify_attention", "bound": "hbm",
                                            "achieved": ab / (t_attn / 1e3) / 1e9, "peak": hbm_peak,
                                            "unit": "GB/s", "frac": ab / (t_attn / 1e3) / 1e9 / hbm_peak,
                                            "traffic": attention_traffic(ab)[0],
                                            "traffic_source": attention_traffic(ab)[1],
                                            "algorithmic_bytes": ab,
                                            "peak_source": f"{peak_src} hbm_gbs (copy, burst)"}}
    # paged KV (128-key pages, randomly permuted) over layer 0's cache contents vs the contiguous launch
    Bc, Hkv_, cap_, D_ = eng.kc[0].shape
    max_pages = (cap_ + 127) // 128
    n_pages = Bc * max_pages
    gp = torch.Generator(device=eng.device)
    gp.manual_seed(5)
    kpool = torch.zeros((Hkv_, n_pages, 128, D_), dtype=torch.bfloat16, device=eng.device)
    vpool = torch.zeros_like(kpool)
    t_pgs = {}
    pws = S.Workspace(eng.device)     # its own scratch: the engine's stays as its captured rounds know it
    for alloc in ("in_order", "random"):
        if alloc == "random":   # pages scattered over the whole pool (worst case for locality)
            perm = torch.randperm(n_pages, generator=gp, device=eng.device).to(torch.int32)
        else:                   # each sequence's pages consecutive, as a bump allocator hands them out
            perm = torch.arange(n_pages, dtype=torch.int32, device=eng.device)
        table = perm.view(Bc, max_pages).contiguous()
        for src, pool in ((eng.kc[0], kpool), (eng.vc[0], vpool)):
            padded = torch.zeros((Bc, Hkv_, max_pages * 128, D_), dtype=torch.bfloat16, device=eng.device)
            padded[:, :, :cap_] = src
            pool[:, table.view(-1).long()] = padded.view(Bc, Hkv_, max_pages, 128, D_).permute(1, 0, 2, 3, 4).reshape(
                Hkv_, n_pages, 128, D_)
            del padded

        def attn_paged(table=table):
            S.spec_verify_attention_paged(qkv[:, :hq], qkv[:, hq:hq + hk], qkv[:, hq + hk:], cu, ctx, kpool, vpool,
                                          table, eng.max_rows, O=eng.o[:M], ws=pws)
        t_pgs[alloc] = timeit(attn_paged, 1)
    # the contiguous launch timed the same way (layer 0's cache, repeated), for a like-for-like ratio
    def attn_layer0():
        S.spec_verify_attention(qkv[:, :hq], qkv[:, hq:hq + hk], qkv[:, hq + hk:], cu, ctx,
                                eng.kc[0], eng.vc[0], eng.max_rows, O=eng.o[:M], ws=eng.ws)
    t_c0 = timeit(attn_layer0, 1)
    t_pg = t_pgs["in_order"]
    res["verify_attention_paged"] = {
        "avg_launch_us": t_pg * 1e3, "launches_per_round": 0, "total_ms": 0.0, "page_keys": 128,
        "contiguous_same_layer_us": t_c0 * 1e3,
        "vs_contiguous": t_pg / t_c0, "random_pages_us": t_pgs["random"] * 1e3,
        "random_vs_contiguous": t_pgs["random"] / t_c0,
        "roofline": {"kernel": "verify_attention (paged)", "bound": "hbm", "achieved": ab / (t_pg / 1e3) / 1e9,
                     "peak": hbm_peak, "unit": "GB/s", "frac": ab / (t_pg / 1e3) / 1e9 / hbm_peak,
                     "traffic": None, "algorithmic_bytes": ab, "peak_source": f"{peak_src} hbm_gbs"}}
    del kpool, vpool
    shapes = {"qkv": (dims.qkv, dims.d), "o": (dims.d, hq), "gate_up": (2 * dims.I, dims.d),
              "down": (dims.d, dims.I)}
    xs = {"qkv": eng.h[:M], "o": eng.o[:M], "gate_up": eng.h[:M], "down": eng.a[:M]}
    ys = {"qkv": eng.qkv[:M], "o": eng.h[:M], "gate_up": eng.a[:M] if eng.fused_swiglu else eng.gu[:M],
          "down": eng.h[:M]}
    tot_t, tot_f, tot_b = 0.0, 0.0, 0.0
    per_shape = {}
    for name, (N, K) in shapes.items():
        w_attr = {"qkv": "w_qkv", "o": "w_o", "gate_up": "w_gu", "down": "w_down"}[name]

        def lin_all(name=name, w_attr=w_attr):
            for li in range(L):
                if name == "gate_up" and eng.fused_swiglu:
                    S.spec_verify_linear_swiglu(xs[name], eng.w.layers[li].w_gu, A=ys[name], ws=eng.ws)
                else:
                    S.spec_verify_linear(xs[name], getattr(eng.w.layers[li], w_attr), Y=ys[name], ws=eng.ws)
        t = timeit(lin_all, L)
        per_shape[name] = {"us": t * 1e3, "tflops": 2.0 * M * N * K / (t / 1e3) / 1e12,
                           "weight_gbs": 2.0 * N * K / (t / 1e3) / 1e9}
        tot_t += t * L
        tot_f += 2.0 * M * N * K * L
        tot_b += 2.0 * N * K * L
    lin_tflops = tot_f / (tot_t / 1e3) / 1e12
    res["verify_linear"] = {"avg_launch_us": tot_t / (4 * L) * 1e3, "launches_per_round": 4 * L,
                            "total_ms": tot_t, "per_shape": per_shape,
                            "roofline": {"kernel": "verify_linear (tcgen05, M=%d)" % M, "bound": "tensor",
                                         "achieved": lin_tflops, "peak": tc_sust, "unit": "TFLOP/s",
                                         "frac": lin_tflops / tc_sust, "traffic": None,
                                         "algorithmic_flops": tot_f / (4 * L),
                                         "hbm_gbs": tot_b / (tot_t / 1e3) / 1e9,
                                         "peak_source": f"{peak_src} bf16_tflops_sustained (cuBLAS, in a long step)"}}
    h = eng.h[:M]

    def head():
        S.spec_lmhead_softmax(h, eng.w.w_lm, TEMP, P=eng.P[:M], ws=eng.ws)
    t_head = timeit(head, 1)
    hb = 2.0 * dims.V * dims.d + 3.0 * M * dims.V * 4
    res["lmhead_softmax"] = {"avg_launch_us": t_head * 1e3, "launches_per_round": 0 if eng.fused_sampler else 2,
                             "total_ms": 0.0 if eng.fused_sampler else t_head,
                             "roofline": {"kernel": "lmhead_softmax", "bound": "hbm",
                                          "achieved": hb / (t_head / 1e3) / 1e9, "peak": hbm_peak,
                                          "unit": "GB/s", "frac": hb / (t_head / 1e3) / 1e9 / hbm_peak,
                                          "traffic": None, "algorithmic_bytes": hb,
                                          "tflops": 2.0 * M * dims.V * dims.d / (t_head / 1e3) / 1e12,
                                          "peak_source": f"{peak_src} hbm_gbs"}}
    if sampler_inputs is not None:
        q, drafts, U, out = sampler_inputs
        B = cu.numel() - 1

        def fused():
            S.spec_lmhead_reject_sample(h, eng.w.w_lm, TEMP, q, drafts, U, cu, out=out, ws=eng.ws)
        t_f = timeit(fused, 1)
        # weights + logits written once + the final rows' logits and q read back by the sampler
        fb = 2.0 * dims.V * dims.d + 1.0 * M * dims.V * 4 + 2.0 * B * dims.V * 4
        res["lmhead_reject_sample"] = {
            "avg_launch_us": t_f * 1e3, "launches_per_round": 2 if eng.fused_sampler else 0,
            "total_ms": t_f if eng.fused_sampler else 0.0,
            "roofline": {"kernel": "lmhead_reject_sample (fused)", "bound": "hbm",
                         "achieved": fb / (t_f / 1e3) / 1e9, "peak": hbm_peak, "unit": "GB/s",
                         "frac": fb / (t_f / 1e3) / 1e9 / hbm_peak, "traffic": None, "algorithmic_bytes": fb,
                         "tflops": 2.0 * M * dims.V * dims.d / (t_f / 1e3) / 1e12,
                         "peak_source": f"{peak_src} hbm_gbs"}}
        # typical acceptance (lossy variant) on the same rows: the probabilities of this round
        S.spec_lmhead_softmax(h, eng.w.w_lm, TEMP, P=eng.P[:M], ws=eng.ws)
        t_out = (torch.empty_like(out[0]), torch.empty_like(out[1]), torch.empty_like(out[2]))

        def typical():
            S.spec_typical_sample(eng.P[:M], drafts, U, cu, TYPICAL_EPS, TYPICAL_DELTA, out=t_out)
        t_t = timeit(typical, 1)
        n_t = t_out[0].cpu().numpy().astype(np.int64)
        gam = batch.gammas.astype(np.int64)
        # rows read: one entropy pass per tested draft (n + 1 tests, gamma when all pass) + the final row
        rows = int(np.minimum(n_t + 1, gam).sum() + B)
        tb = rows * dims.V * 4.0
        res["typical_sample"] = {
            "avg_launch_us": t_t * 1e3, "launches_per_round": 0, "total_ms": 0.0,
            "epsilon": TYPICAL_EPS, "delta": TYPICAL_DELTA,
            "parity": "unpinned: the pages' threshold formula did not survive extraction; the reading "
                      "tau = max(epsilon, delta * exp(-H)) is pinned only on its closed forms",
            "accepted_tokens_per_round": int(n_t.sum()) + B,
            "roofline": {"kernel": "typical_sample", "bound": "hbm", "achieved": tb / (t_t / 1e3) / 1e9,
                         "peak": hbm_peak, "unit": "GB/s", "frac": tb / (t_t / 1e3) / 1e9 / hbm_peak,
                         "traffic": None, "algorithmic_bytes": tb, "peak_source": f"{peak_src} hbm_gbs"}}
    return res


def draft_timing(S, E, batch, dev, round_ms, gamma=4, reps=5):
    """The step before the verify pass: gamma decode steps of a Qwen3-0.6B-shaped draft stack (28
    layers, d 1024, random init) at M = B rows over the benchmark batch's contexts, captured in
    one CUDA graph.  c_hat = one draft step / one verify round (the pages' draft-cost ratio)."""
    import torch
    import synth
    dims = E.draft_dims()
    cap = int((batch.ctx_len + gamma + 1).max() + 15) // 16 * 16
    sw = E.random_stack(dims, seed=3000, device=dev)
    g = torch.Generator(device=dev)
    g.manual_seed(3001)
    kcs, vcs = [], []
    for _ in range(dims.layers):
        k = torch.empty((B, dims.Hkv, cap, dims.D), dtype=torch.bfloat16, device=dev).normal_(0, 1, generator=g)
        kcs.append(k)
        vcs.append(torch.empty_like(k).normal_(0, 1, generator=g))
    eng = E.DraftEngine(dims, sw, kcs, vcs, B, gamma, device=dev)
    tok0 = torch.randint(0, dims.V, (B,), dtype=torch.int32, device=dev, generator=g)
    ctx = torch.from_numpy(batch.ctx_len).to(dev)
    U = torch.from_numpy(synth.uniforms_f32(SEED + 11, gamma * B).reshape(gamma, B)).to(dev)
    Q = torch.empty((B * gamma, dims.V), dtype=torch.float32, device=dev)
    drafts = torch.empty(B * gamma, dtype=torch.int32, device=dev)
    stream = torch.cuda.Stream(device=dev)
    with torch.cuda.stream(stream):
        eng.draft(tok0, ctx, U, TEMP, Q, drafts)
    torch.cuda.synchronize()
    S.spec_device_status()
    graph = torch.cuda.CUDAGraph()
    S.reset_launch_count()
    with torch.cuda.graph(graph, stream=stream):
        eng.draft(tok0, ctx, U, TEMP, Q, drafts)
    launches = S.launch_count()
    for _ in range(3):
        graph.replay()
    torch.cuda.synchronize()
    cur = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(cur)
    for _ in range(reps):
        graph.replay()
    e1.record(cur)
    torch.cuda.synchronize()
    S.spec_device_status()
    t = e0.elapsed_time(e1) / reps
    wbytes = 2.0 * (dims.layers * (dims.qkv * dims.d + dims.d * dims.Hq * dims.D + 2 * dims.I * dims.d
                                   + dims.d * dims.I) + dims.V * dims.d)
    kv = float(batch.ctx_len.sum()) * dims.layers * dims.Hkv * dims.D * 2 * 2
    res = {"model": "Qwen3-0.6B-shaped (28 layers, d 1024, 16/8 heads, I 3072, tied LM head), random init",
           "B": B, "gamma": gamma, "phase_ms": t, "step_us": t / gamma * 1e3, "launches_per_phase": launches,
           "c_hat": (t / gamma) / round_ms, "step_hbm_gbs": (wbytes + kv) / (t / gamma / 1e3) / 1e9,
           "step_algorithmic_bytes": wbytes + kv}
    del eng, kcs, vcs, sw, graph
    torch.cuda.empty_cache()
    return res


def ngram_timing(S, hbm_peak, peak_src, dev, reps=5):
    """The weightless drafter on B = 64 copy-heavy histories of 128..8192 tokens (k = 4, window 3..8,
    the pages' example configuration); not part of the verify round."""
    import torch
    import synth
    tokens, cu = synth.ngram_histories(SEED + 7, B=B, len_lo=CTX_LO, len_hi=CTX_HI, vocab=151936, copy_frac=0.8)
    td, cd = torch.from_numpy(tokens).to(dev), torch.from_numpy(cu).to(dev)
    out = (torch.empty((B, 4), dtype=torch.int32, device=dev), torch.empty(B, dtype=torch.int32, device=dev))
    S.spec_ngram_propose(td, cd, 4, 3, 8, out=out)
    torch.cuda.synchronize()
    cur = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(cur)
    for _ in range(reps):
        S.spec_ngram_propose(td, cd, 4, 3, 8, out=out)
    e1.record(cur)
    torch.cuda.synchronize()
    t = e0.elapsed_time(e1) / reps
    hb = float(tokens.nbytes)   # every history read at least once
    n = out[1].cpu().numpy()
    return {"avg_launch_us": t * 1e3, "launches_per_round": 0, "total_ms": 0.0, "sequences": B,
            "history_tokens": int(len(tokens)), "with_drafts": int((n > 0).sum()), "drafts": int(n.sum()),
            "roofline": {"kernel": "ngram_propose", "bound": "hbm", "achieved": hb / (t / 1e3) / 1e9,
                         "peak": hbm_peak, "unit": "GB/s", "frac": hb / (t / 1e3) / 1e9 / hbm_peak,
                         "traffic": None, "algorithmic_bytes": hb, "peak_source": f"{peak_src} hbm_gbs"}}


def stack_chain_ops(S, eng, M, interleaved=True, bufs=None):
    """The 36-layer linear stack as one chain of products for spec_verify_linear_chain: per layer
    QKV (h -> qkv), O (o -> x, residual x), gate|up with SwiGLU (h -> a), down (a -> x, residual x).
    With `interleaved`, layer l+1's QKV projection (independent of layer l) sits between layer l's
    gate|up and its down projection, which waits for gate|up's output.  `bufs` = (layers, h, o, qkv,
    x, a) in place of the engine's."""
    layers, h, o, qkv, x, a = bufs if bufs is not None else (eng.w.layers, eng.h, eng.o, eng.qkv, eng.x, eng.a)
    per = []
    for lw in layers:
        per.append([S.linear_op(h[:M], lw.w_qkv, qkv[:M]),
                    S.linear_op(o[:M], lw.w_o, x[:M], residual=x[:M]),
                    S.linear_op(h[:M], lw.w_gu, a[:M], swiglu=True),
                    S.linear_op(a[:M], lw.w_down, x[:M], residual=x[:M])])
    if not interleaved:
        return [op for layer in per for op in layer]
    ops = [per[0][0]]
    for l, (q, o, gu, dn) in enumerate(per):
        ops += [o, gu] + ([per[l + 1][0]] if l + 1 < len(per) else []) + [dn]
    return ops


def linear_stack_ratio(eng, dims, S, hbm_peak, peak_src, reps=5):
    """36-layer linear stack (QKV, O, gate|up + SwiGLU, down) at M = 5 and M = 1 rows: the library's
    small-M path (one weight-streaming chain, spec_verify_linear_chain) and, for comparison, one
    call per product (and the optional CUDA-core path at M = 1)."""
    import torch
    cur = torch.cuda.current_stream()
    out = {"per_call": {}}
    wbytes = dims.layers * 2.0 * (dims.qkv * dims.d + dims.d * dims.Hq * dims.D + 2 * dims.I * dims.d + dims.d * dims.I)
    assert eng.fused_swiglu
    chain_ws = S.Workspace(eng.device, max(S.spec_linear_chain_workspace_bytes(stack_chain_ops(S, eng, M), M)
                                           for M in (1, 5)))
    clk = ClockSampler(torch.cuda.current_device())
    clk.start()
    for M, tag in ((1, "1"), (5, "5"), (1, "1_gemv"), (1, "1_chain"), (5, "5_chain")):
        S.spec_set_option("gemv_max_m", 4 if tag == "1_gemv" else 0)
        chain = tag.endswith("_chain")
        ops = stack_chain_ops(S, eng, M) if chain else None

        def run():
            if chain:
                S.spec_verify_linear_chain(ops, M, ws=chain_ws)
                return
            for lw in eng.w.layers:
                S.spec_verify_linear(eng.h[:M], lw.w_qkv, Y=eng.qkv[:M], ws=eng.ws)
                S.spec_verify_linear(eng.o[:M], lw.w_o, Y=eng.x[:M], residual=eng.x[:M], ws=eng.ws)
                S.spec_verify_linear_swiglu(eng.h[:M], lw.w_gu, A=eng.a[:M], ws=eng.ws)
                S.spec_verify_linear(eng.a[:M], lw.w_down, Y=eng.x[:M], residual=eng.x[:M], ws=eng.ws)
        g = torch.cuda.CUDAGraph()
        s = torch.cuda.Stream()
        with torch.cuda.stream(s):
            run()
        torch.cuda.synchronize()
        with torch.cuda.graph(g, stream=s):
            run()
        for _ in range(3):
            g.replay()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(cur)
        for _ in range(reps):
            g.replay()
        e1.record(cur)
        torch.cuda.synchronize()
        t = e0.elapsed_time(e1) / reps
        gbs = wbytes / (t / 1e3) / 1e9
        key = tag.replace("_chain", "")
        dst = out if chain else out["per_call"]
        dst[f"m{key}_us"] = t * 1e3
        dst[f"m{key}_hbm_gbs"] = gbs
        dst[f"m{key}_hbm_frac"] = gbs / hbm_peak
    S.spec_set_option("gemv_max_m", 0)
    S.spec_device_status()
    out["clocks"] = clk.stop()
    out["ratio_m5_over_m1"] = out["m5_us"] / out["m1_us"]
    out["per_call"]["ratio_m5_over_m1"] = out["per_call"]["m5_us"] / out["per_call"]["m1_us"]
    out["weights_gb"] = wbytes / 1e9
    out["note"] = ("36 layers x {QKV 6144x4096, O 4096x4096, gate|up 24576x4096 + SwiGLU, down 4096x12288}, one "
                   "CUDA graph per M; m1/m5 = the small-M path (spec_verify_linear_chain: the 144 products in "
                   "weight-streaming launches of up to 48, the next layer's QKV between gate|up and down); "
                   "per_call = one library call per product (m1_gemv: the optional CUDA-core path); peak " + peak_src)
    return out


SWEEP_B = (1, 8, 64, 256, 1024)
SWEEP_GAMMA = (1, 4, 10)
SWEEP_CTX = 2048
# points of the sweep that the default run reports under "sweep" (B, gamma): the small-M verify
# batch and the largest tensor-bound one
SWEEP_DEFAULT = ((8, 4), (1024, 4))


class SweepRig:
    """Buffers for batch x depth points on the Qwen3-8B linear shapes (one set, sized for the
    largest M asked for), over weights `sw` (gate|up interleaved for the fused SwiGLU call)."""

    def __init__(self, sw, dims, dev, m_max, points):
        import torch
        from speculative_decoding_verify_05_gb300 import binding as S
        self.S, self.sw, self.dims, self.dev = S, sw, dims, dev
        gen = torch.Generator(device=dev)
        gen.manual_seed(3000)
        self.gen = gen
        bf = dict(dtype=torch.bfloat16, device=dev)
        self.x = torch.empty((m_max, dims.d), **bf).normal_(0, 1, generator=gen)
        self.h = torch.empty_like(self.x).normal_(0, 1, generator=gen)
        self.qkv = torch.empty((m_max, dims.qkv), **bf).normal_(0, 1, generator=gen)
        self.o = torch.empty((m_max, dims.Hq * dims.D), **bf).normal_(0, 1, generator=gen)
        self.a = torch.empty((m_max, dims.I), **bf).normal_(0, 1, generator=gen)
        shapes = ((dims.qkv, dims.d), (dims.d, dims.Hq * dims.D), (dims.d, dims.I))
        need = max(max(S.spec_linear_workspace_bytes(b * (g + 1), n, k) for n, k in shapes) +
                   S.spec_swiglu_linear_workspace_bytes(b * (g + 1), dims.I, dims.d) for b, g in points)
        self.ws = S.Workspace(dev, max(need, 1 << 20))
        lw_ = dims.qkv * dims.d + dims.d * dims.Hq * dims.D + 2 * dims.I * dims.d + dims.d * dims.I
        self.wbytes = dims.layers * 2.0 * lw_
        self.flops_row = dims.layers * 2.0 * lw_

    def point(self, nb, gm, hbm_peak, tc_sust):
        import torch
        S, dims, dev = self.S, self.dims, self.dev
        import synth
        M = nb * (gm + 1)
        x, h, qkv, o, a, ws = self.x, self.h, self.qkv, self.o, self.a, self.ws
        # the small-M path (up to the chain's 64 rows): the weight-streaming chain; above it, one call
        # per product (with the weight streams marked evict-first the chain is the faster stack at every
        # M it takes: 2.94 against 3.32 ms at 40 rows, 2.97 against 3.14 ms at 64)
        chain = M <= 64
        if chain:
            ops = stack_chain_ops(S, None, M, bufs=(self.sw.layers, h, o, qkv, x, a))
            cws = S.Workspace(dev, S.spec_linear_chain_workspace_bytes(ops, M))

        def run():
            if chain:
                S.spec_verify_linear_chain(ops, M, ws=cws)
                return
            for lw in self.sw.layers:
                S.spec_verify_linear(h[:M], lw.w_qkv, Y=qkv[:M], ws=ws)
                S.spec_verify_linear(o[:M], lw.w_o, Y=x[:M], residual=x[:M], ws=ws)
                S.spec_verify_linear_swiglu(h[:M], lw.w_gu, A=a[:M], ws=ws)
                S.spec_verify_linear(a[:M], lw.w_down, Y=x[:M], residual=x[:M], ws=ws)
        cur = torch.cuda.current_stream()
        g = torch.cuda.CUDAGraph()
        st = torch.cuda.Stream()
        with torch.cuda.stream(st):
            run()
        torch.cuda.synchronize()
        with torch.cuda.graph(g, stream=st):
            run()
        reps = 3 if M > 2000 else 5
        for _ in range(2):
            g.replay()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(cur)
        for _ in range(reps):
            g.replay()
        e1.record(cur)
        torch.cuda.synchronize()
        t_lin = e0.elapsed_time(e1) / reps / 1e3
        del g
        # one layer's attention over nb sequences of SWEEP_CTX keys, gm + 1 new rows each
        batch = synth.RaggedBatch(np.full(nb, gm), np.full(nb, SWEEP_CTX))
        cap = (SWEEP_CTX + gm + 1 + 15) // 16 * 16
        kc = torch.empty((nb, dims.Hkv, cap, dims.D), dtype=torch.bfloat16, device=dev).normal_(0, 1, generator=self.gen)
        vc = torch.empty_like(kc).normal_(0, 1, generator=self.gen)
        cu = torch.from_numpy(batch.cu_rows).to(dev)
        ctx = torch.from_numpy(batch.ctx_len).to(dev)
        hq, hk = dims.Hq * dims.D, dims.Hkv * dims.D
        attn_ws = S.Workspace(dev, S.spec_attention_workspace_bytes(nb, gm + 1, dims.Hq, dims.Hkv, dims.D, cap))

        def attn():
            S.spec_verify_attention(qkv[:M, :hq], qkv[:M, hq:hq + hk], qkv[:M, hq + hk:], cu, ctx, kc, vc,
                                    gm + 1, O=o[:M], ws=attn_ws)
        for _ in range(3):
            attn()
        torch.cuda.synchronize()
        e0.record(cur)
        for _ in range(10):
            attn()
        e1.record(cur)
        torch.cuda.synchronize()
        t_att = e0.elapsed_time(e1) / 10 / 1e3
        ab = attention_bytes(batch, dims)
        S.spec_device_status()
        del kc, vc, attn_ws
        torch.cuda.empty_cache()
        return {"B": nb, "gamma": gm, "M": M, "linear_path": "chain" if chain else "one call per product",
                "linear_stack_us": t_lin * 1e6,
                "linear_hbm_frac": self.wbytes / t_lin / 1e9 / hbm_peak,
                "linear_tensor_frac": self.flops_row * M / t_lin / 1e12 / tc_sust,
                "attention_us": t_att * 1e6,
                "attention_hbm_frac": ab / t_att / 1e9 / hbm_peak}


def sweep_points(sw, dims, dev, points, hbm_peak, tc_sust):
    rig = SweepRig(sw, dims, dev, max(b * (g + 1) for b, g in points), points)
    out = [rig.point(nb, gm, hbm_peak, tc_sust) for nb, gm in points]
    del rig
    return out


def run_sweep(args):
    """Batch/depth sweep on the Qwen3-8B shapes (B x gamma, M = B (gamma + 1) from 2 to 11264 rows,
    context 2048): per point the 36-layer linear stack (one CUDA graph; % of the measured HBM copy
    peak and of the sustained bf16 tensor peak) and one layer's verify attention over a B-sequence
    cache of 2048 keys each (the cache is one layer's, reused: 36 layers at B = 1024 would not fit).
    Prints one JSON line."""
    import torch
    from speculative_decoding_verify_05_gb300 import engine as E
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    hbm_peak, tc_peak, tc_sust, peak_src = peaks()
    dims = E.Dims()
    sw = E.random_stack(dims, seed=1000, device=dev, with_head=False)
    for lw in sw.layers:
        E.set_gu_layout(lw, "interleaved")
    clk = ClockSampler(0)
    clk.start()
    pts = [(nb, gm) for nb in SWEEP_B for gm in SWEEP_GAMMA]
    points = sweep_points(sw, dims, dev, pts, hbm_peak, tc_sust)
    lw_ = dims.qkv * dims.d + dims.d * dims.Hq * dims.D + 2 * dims.I * dims.d + dims.d * dims.I
    print(json.dumps({"sweep": "batch x depth on the Qwen3-8B shapes, context %d" % SWEEP_CTX,
                      "peaks": {"hbm_gbs": hbm_peak, "bf16_tflops_sustained": tc_sust, "source": peak_src},
                      "weights_gb": dims.layers * 2.0 * lw_ / 1e9, "points": points, "clocks": clk.stop()}))


# --------------------------------------------------------------------------- configuration 3
C3_B, C3_GAMMA, C3_CTX_LO, C3_CTX_HI = 8, 4, 512, 4096
C3_SIGMAS = (0.5, 1.0, 2.0)
C3_TEMPS = (1.0, 0.0)
C3_DRAWS = 64        # draft / uniform draws per (sigma, T): 64 x 8 sequences x 4 drafts acceptance tests


def config3(sw, dims, dev, hbm_peak, peak_src, reps=10):
    """B = 8, gamma = 4, ctx ~ U[512, 4096] over the same 36-layer weights and LM head: the verify
    round (one CUDA graph) at T = 1 and T = 0, the attention and fused LM head -> sampler launches
    with their HBM fractions, and per draft-noise sigma the achieved acceptance: the expected rate
    alpha = mean over draft rows of sum_x min(p, q) and the sampler's empirical rate and mean
    accepted tokens per round over C3_DRAWS draws of drafts and uniforms.  q = softmax(z + sigma
    noise) from the target logits z of the same pass (the configuration's draft recipe)."""
    import torch
    import synth
    from speculative_decoding_verify_05_gb300 import binding as S
    from speculative_decoding_verify_05_gb300 import engine as E
    rng = np.random.default_rng(SEED + 33)
    ctx_np = rng.integers(C3_CTX_LO, C3_CTX_HI + 1, size=C3_B).astype(np.int32)
    batch = synth.RaggedBatch(np.full(C3_B, C3_GAMMA), ctx_np)
    cap = round_cap(batch)
    g = torch.Generator(device=dev)
    g.manual_seed(4000)
    kcs, vcs = [], []
    for _ in range(dims.layers):
        k = torch.empty((C3_B, dims.Hkv, cap, dims.D), dtype=torch.bfloat16, device=dev).normal_(0, 1, generator=g)
        kcs.append(k)
        vcs.append(torch.empty_like(k).normal_(0, 1, generator=g))
    eng = E.VerifyEngine(dims, sw, kcs, vcs, max_M=batch.M, max_rows=batch.max_rows, device=dev)
    M = batch.M
    x0 = torch.empty((M, dims.d), dtype=torch.bfloat16, device=dev).normal_(0, 1, generator=g)
    cu = torch.from_numpy(batch.cu_rows).to(dev)
    ctx = torch.from_numpy(batch.ctx_len).to(dev)
    qrows = torch.from_numpy(np.concatenate([np.arange(batch.cu_rows[b], batch.cu_rows[b] + C3_GAMMA)
                                             for b in range(C3_B)])).to(dev)
    # the target's probabilities at T = 1 give the logits up to a per-row constant: log p = z - logZ
    P1 = eng.verify_pass(x0, cu, ctx, 1.0).clone()
    h_final = eng.h[:M].clone()
    logp = torch.log(P1[qrows].clamp_min(1e-38))
    cur = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    out = (torch.empty(C3_B, dtype=torch.int32, device=dev), torch.empty(M, dtype=torch.int32, device=dev),
           torch.empty(C3_B, dtype=torch.int32, device=dev))
    res = {"workload": f"B={C3_B}, gamma={C3_GAMMA}, ctx~U[{C3_CTX_LO},{C3_CTX_HI}] (seeded), 36 layers + LM head "
                       f"151936 + sampler; q = softmax(z + sigma N(0,1)); {C3_DRAWS} draft/uniform draws per point",
           "M_rows": M, "sum_ctx": int(ctx_np.sum())}
    hq, hk = dims.Hq * dims.D, dims.Hkv * dims.D
    # attention: one layer's launch repeated (the round's other layers read other caches)
    qkv = eng.qkv[:M]

    def attn():
        S.spec_verify_attention(qkv[:, :hq], qkv[:, hq:hq + hk], qkv[:, hq + hk:], cu, ctx, eng.kc[0], eng.vc[0],
                                batch.max_rows, O=eng.o[:M], ws=eng.ws)
    attn()
    torch.cuda.synchronize()
    e0.record(cur)
    for _ in range(reps):
        attn()
    e1.record(cur)
    torch.cuda.synchronize()
    t_att = e0.elapsed_time(e1) / reps / 1e3
    ab = attention_bytes(batch, dims)
    res["attention_us"] = t_att * 1e6
    res["attention_hbm_frac"] = ab / t_att / 1e9 / hbm_peak
    per_T = {}
    for T in C3_TEMPS:
        noise = torch.empty_like(logp).normal_(0, 1, generator=g)
        q0 = torch.softmax(logp + noise, dim=1).contiguous()
        drafts0 = torch.multinomial(q0, 1, generator=g).view(-1).to(torch.int32)
        U0 = torch.rand(M, generator=g, device=dev)
        replay = eng.capture_round(x0, cu, ctx, q0, drafts0, U0, T, out)
        replay()
        torch.cuda.synchronize()
        e0.record(cur)
        for _ in range(reps):
            replay()
        e1.record(cur)
        torch.cuda.synchronize()
        t_round = e0.elapsed_time(e1) / reps / 1e3
        # the fused LM head -> sampler launch pair on the round's final hidden rows
        h = h_final

        def head():
            S.spec_lmhead_reject_sample(h, eng.w.w_lm, T, q0, drafts0, U0, cu, 1e-5, out=out, ws=eng.ws)
        head()
        torch.cuda.synchronize()
        e0.record(cur)
        for _ in range(reps):
            head()
        e1.record(cur)
        torch.cuda.synchronize()
        t_head = e0.elapsed_time(e1) / reps / 1e3
        hb = 2.0 * dims.V * dims.d + (M * dims.V * 4.0 if T > 0 else 0.0) + 2.0 * C3_B * dims.V * 4
        # target p at this temperature (greedy: one-hot at the argmax) for the expected rate
        if T > 0:
            p_rows = P1[qrows]
        else:
            p_rows = torch.zeros_like(P1[qrows])
            p_rows.scatter_(1, P1[qrows].argmax(dim=1, keepdim=True), 1.0)
        sig = {}
        for sigma in C3_SIGMAS:
            noise = torch.empty_like(logp).normal_(0, 1, generator=g)
            q = torch.softmax(logp + sigma * noise, dim=1).contiguous()
            alpha = float(torch.minimum(p_rows, q).sum(dim=1).mean().item())
            acc_tok, tested, accepted = 0, 0, 0
            for _ in range(C3_DRAWS):
                drafts = torch.multinomial(q, 1, generator=g).view(-1).to(torch.int32)
                U = torch.rand(M, generator=g, device=dev)
                n, _, _ = S.spec_lmhead_reject_sample(h, eng.w.w_lm, T, q, drafts, U, cu, 1e-5, out=out, ws=eng.ws)
                nn = n.cpu().numpy().astype(np.int64)
                accepted += int(nn.sum())
                tested += int(np.minimum(nn + 1, C3_GAMMA).sum())
                acc_tok += int(nn.sum()) + C3_B
            a_emp = accepted / max(tested, 1)
            e_tok = (1 - alpha ** (C3_GAMMA + 1)) / (1 - alpha) if alpha < 1 else C3_GAMMA + 1.0
            sig[str(sigma)] = {"alpha_expected": alpha, "alpha_empirical": a_emp,
                               "mean_accepted_tokens_per_seq": acc_tok / (C3_DRAWS * C3_B),
                               "closed_form_tokens_per_seq": e_tok,
                               "accepted_tokens_per_s": acc_tok / C3_DRAWS / t_round}
        S.spec_device_status()
        per_T["T=%g" % T] = {"round_us": t_round * 1e6, "lmhead_sampler_us": t_head * 1e6,
                             "lmhead_sampler_hbm_frac": hb / t_head / 1e9 / hbm_peak, "sigma": sig}
    res["per_temperature"] = per_T
    res["peak_source"] = f"{peak_src} hbm_gbs"
    del eng, kcs, vcs
    torch.cuda.empty_cache()
    return res


def end_to_end(args, eng, batch, dims, q, drafts, x0, S, torch, dev, steps=None):
    """Same round through the public API with pinned host inputs and a host read of the result.

    A serving loop's form: two input/output buffer sets, each with its own captured round
    (VerifyEngine.capture_round).  While round k runs on one set, the next round's inputs are
    copied into the other set on a copy stream; every round's H2D copies and D2H read are inside
    the timed region (wall clock)."""
    steps = steps or max(3, min(args.steps, 10))
    import synth
    host = [torch.empty(x0.shape, dtype=x0.dtype, pin_memory=True).copy_(x0.cpu()),
            torch.empty(q.shape, dtype=q.dtype, pin_memory=True).copy_(q.cpu()),
            torch.empty(drafts.shape, dtype=drafts.dtype, pin_memory=True).copy_(drafts.cpu()),
            torch.from_numpy(synth.uniforms_f32(SEED, batch.M)).pin_memory(),
            torch.from_numpy(batch.cu_rows).pin_memory(),
            torch.from_numpy(batch.ctx_len).pin_memory()]
    sets, replays, h_outs = [], [], []
    for _ in range(2):
        d_in = [torch.empty(h.shape, dtype=h.dtype, device=dev) for h in host]
        out = (torch.empty(B, dtype=torch.int32, device=dev), torch.empty(batch.M, dtype=torch.int32, device=dev),
               torch.empty(B, dtype=torch.int32, device=dev))
        for d, h in zip(d_in, host):
            d.copy_(h)
        x_d, q_d, dr_d, u_d, cu_d, ctx_d = d_in
        replays.append(eng.capture_round(x_d, cu_d, ctx_d, q_d, dr_d, u_d, TEMP, out))
        sets.append((d_in, out))
        h_outs.append([torch.empty(o.shape, dtype=o.dtype, pin_memory=True) for o in out])
    bi = sum(t.numel() * t.element_size() for t in host)
    bo = sum(t.numel() * t.element_size() for t in h_outs[0])
    main = torch.cuda.current_stream(dev)
    copy = torch.cuda.Stream(device=dev)
    ready = [torch.cuda.Event(), torch.cuda.Event()]
    done = [torch.cuda.Event(), torch.cuda.Event()]

    def h2d(k):
        with torch.cuda.stream(copy):
            copy.wait_event(done[k])          # the round that last used this set has finished
            for d, h in zip(sets[k][0], host):
                d.copy_(h, non_blocking=True)
            ready[k].record(copy)

    def run(n):
        for k in range(2):
            done[k].record(main)
        h2d(0)
        for i in range(n):
            k = i & 1
            main.wait_event(ready[k])
            replays[k]()
            done[k].record(main)
            if i + 1 < n:
                h2d(k ^ 1)
            for h, d in zip(h_outs[k], sets[k][1]):
                h.copy_(d, non_blocking=True)
        torch.cuda.synchronize()

    run(2)
    t0 = time.perf_counter()
    run(steps)
    dt = (time.perf_counter() - t0) / steps
    accepted = int(h_outs[(steps - 1) & 1][0].sum().item()) + B
    return {"value": accepted / dt, "unit": UNIT, "h2d_bytes_per_step": bi, "d2h_bytes_per_step": bo,
            "ms_per_step": dt * 1e3, "steps": steps,
            "how": "VerifyEngine.capture_round (the round's C-ABI calls recorded once in a CUDA graph), two buffer "
                   "sets: each round's pinned-host inputs copied in on a copy stream while the previous round runs, "
                   "the graph replayed, the results read back; wall clock over all steps"}


# --------------------------------------------------------------------------- oracle timing
def oracle_sample(n_seq, weights_np, kv_np, batch, x0_bits, q_sample, drafts_sample, U_sample):
    """One bounded oracle run: layer 0 + LM head + sampler on the first n_seq sequences.

    Returns (seconds for 36 layers + head + sampler, accepted tokens).
    """
    import synth
    from oracle import bf16 as obf, ops as oops, sampler as osamp, stack as ostack
    od = ostack.Dims()
    sub = synth.RaggedBatch(batch.gammas[:n_seq], batch.ctx_len[:n_seq])
    lw, final_norm, w_lm = weights_np
    kc, vc = kv_np
    x = obf.decode(x0_bits[:sub.M])
    t0 = time.perf_counter()
    x1, _, _ = ostack.layer_forward(x, lw, od, sub.cu_rows, sub.ctx_len, obf.decode(kc), obf.decode(vc))
    t_layer = time.perf_counter() - t0
    t0 = time.perf_counter()
    sw = ostack.StackWeights([], final_norm, w_lm)
    logits = ostack.head_logits(x1, sw, od)
    p = oops.target_probs(logits, TEMP)
    t_head = time.perf_counter() - t0
    t0 = time.perf_counter()
    n_acc, out, near = osamp.reject_sample(p.astype(np.float32), q_sample, drafts_sample, U_sample, sub.cu_rows)
    t_samp = time.perf_counter() - t0
    return od.layers * t_layer + t_head + t_samp, int(n_acc.sum()) + n_seq, (t_layer, t_head, t_samp)


def cpu_baseline(eng, batch, dims, kcs, vcs, sw, q, drafts, n_seq=CPU_SAMPLE_SEQS):
    """Oracle on the host cores over a bounded sample of this run's inputs (copied to the host)."""
    import torch
    from oracle import stack as ostack
    from speculative_decoding_verify_05_gb300 import binding as S
    import synth
    sub = synth.RaggedBatch(batch.gammas[:n_seq], batch.ctx_len[:n_seq])
    bits = lambda t: t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
    l0 = sw.layers[0]
    w_gu = bits(l0.w_gu)
    if l0.gu_layout == "interleaved":     # back to gate rows then up rows for the oracle
        w_gu = w_gu.reshape(-1, 2, S.GATE_UP_BLOCK, dims.d).transpose(1, 0, 2, 3).reshape(2 * dims.I, dims.d)
    lw = ostack.LayerWeights(bits(l0.w_qkv), bits(l0.w_o), w_gu, bits(l0.w_down),
                             bits(l0.attn_norm), bits(l0.mlp_norm))
    capn = int((sub.ctx_len + sub.gammas + 1).max())
    kv = (bits(kcs[0][:n_seq, :, :capn]), bits(vcs[0][:n_seq, :, :capn]))
    x0 = bits(eng.x[:sub.M])
    # the oracle's own draft inputs for the sampled sequences: same q rows / drafts
    q_s = q[:sub.n_drafts].cpu().numpy()
    d_s = drafts[:sub.n_drafts].cpu().numpy()
    U_s = synth.uniforms_f32(SEED, batch.M)[:sub.M]
    secs, acc, parts = oracle_sample(n_seq, (lw, bits(sw.final_norm), bits(sw.w_lm)), kv, batch, x0, q_s, d_s, U_s)
    cores = len(os.sched_getaffinity(0))
    return {"value": acc / secs, "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"first {n_seq} of {B} sequences ({sub.M} rows): oracle layer 0 timed and counted 36x, "
                      f"plus final norm + LM head + softmax + sampler; tokens = their accepted tokens",
            "seconds_per_round": secs, "layer_s": parts[0], "head_s": parts[1], "sampler_s": parts[2]}


# --------------------------------------------------------------------------- reference arm
def run_reference(args):
    """The oracle on the host cores, on a bounded sample of the same workload (first
    CPU_SAMPLE_SEQS sequences; layer 0 timed and counted 36x, plus the LM head and the sampler).
    `ms_per_step` is the wall time of one such step as run; `projected_ms_per_round` is the
    36-layer projection that `value` (accepted tokens per second of a full round) divides by."""
    if not reference_runs_here():
        return
    import synth
    from oracle import bf16 as obf, ops as oops, stack as ostack
    batch = make_batch()
    dims = ostack.Dims()
    n_seq = CPU_SAMPLE_SEQS
    sub = synth.RaggedBatch(batch.gammas[:n_seq], batch.ctx_len[:n_seq])
    capn = int((sub.ctx_len + sub.gammas + 1).max())
    # same distributions as the GPU arm, generated on the host (numpy Philox)
    lw = ostack.LayerWeights(
        synth.normal_bf16_bits(1001, (dims.Hq * dims.D + 2 * dims.Hkv * dims.D, dims.d), 0.02),
        synth.normal_bf16_bits(1002, (dims.d, dims.Hq * dims.D), 0.02),
        synth.normal_bf16_bits(1003, (2 * dims.I, dims.d), 0.02),
        synth.normal_bf16_bits(1004, (dims.d, dims.I), 0.02),
        synth.f32_to_bf16_bits(np.ones(dims.d, np.float32)), synth.f32_to_bf16_bits(np.ones(dims.d, np.float32)))
    w_lm = synth.normal_bf16_bits(1005, (dims.V, dims.d), 0.02)
    ones = synth.f32_to_bf16_bits(np.ones(dims.d, np.float32))
    kc = synth.normal_bf16_bits(1006, (n_seq, dims.Hkv, capn, dims.D), 1.0)
    vc = synth.normal_bf16_bits(1007, (n_seq, dims.Hkv, capn, dims.D), 1.0)
    x0 = synth.normal_bf16_bits(1008, (sub.M, dims.d), 1.0)
    # draft q from the oracle's own logits for these rows (layer 0 + head stand-in, computed once)
    x1, _, _ = ostack.layer_forward(obf.decode(x0), lw, dims, sub.cu_rows, sub.ctx_len, obf.decode(kc), obf.decode(vc))
    logits = ostack.head_logits(x1, ostack.StackWeights([], ones, w_lm), dims)
    q_s, d_s = synth.draft_distribution(logits, sub, SIGMA, TEMP, seed=SEED + 5)
    U_s = synth.uniforms_f32(SEED, batch.M)[:sub.M]
    for _ in range(args.warmup):
        oracle_sample(n_seq, (lw, ones, w_lm), (kc, vc), batch, x0, q_s, d_s, U_s)
    tot_s, tot_tok = 0.0, 0
    t_wall = time.perf_counter()
    for _ in range(args.steps):
        s, acc, _ = oracle_sample(n_seq, (lw, ones, w_lm), (kc, vc), batch, x0, q_s, d_s, U_s)
        tot_s += s
        tot_tok += acc
    wall = time.perf_counter() - t_wall
    value = tot_tok / tot_s
    cores = len(os.sched_getaffinity(0))
    sample = (f"first {n_seq} of {B} sequences ({sub.M} rows) of the same workload: oracle layer 0 timed and "
              f"counted 36x, plus final norm + LM head + softmax + sampler; {args.steps} such steps run")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * wall / args.steps,
            "projected_ms_per_round": 1e3 * tot_s / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded numpy Philox, same distributions as the GPU arm)",
            "config": workload_config(batch, round_cap(batch)),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "wall_s": wall,
            "note": "ms_per_step is the measured wall time of one sampled step; value = accepted tokens of the "
                    "sample / projected_ms_per_round (layer 0 counted 36x)"}
    print(json.dumps(line))


def run_profile_case(args):
    """Small, self-contained launches of one hot kernel for an ncu capture (no timing).

    round: one full verify round of the benchmark workload (for the launch list);
    attention: one layer of --batch (16) ragged sequences (KV ~0.6 GB at 16, above L2);
    linear: one gate|up projection (201 MB of weights) at --rows rows;
    chain: the weight-streaming chain of --layers layers' linears at --rows rows;
    swiglu: the same projection with the SwiGLU epilogue (--n interleaved gate|up rows);
    lmhead: the LM head + softmax at --rows rows.
    """
    import torch
    from speculative_decoding_verify_05_gb300 import binding as S
    from speculative_decoding_verify_05_gb300 import engine as E
    import synth
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    dims = E.Dims()
    g = torch.Generator(device=dev)
    g.manual_seed(7)
    ws = S.Workspace(dev)
    if args.profile == "round":
        # the benchmark's full verify round, run eagerly: once to warm up, then once inside
        # the NVTX range "round" (ncu --nvtx --nvtx-include "round/" lists only that one)
        st = build_round(dev, 0, S, E, synth, fused_swiglu=args.swiglu == "fused",
                         fused_sampler=args.sampler == "fused")
        st["step"]()
        torch.cuda.synchronize()
        torch.cuda.nvtx.range_push("round")
        st["step"]()
        torch.cuda.nvtx.range_pop()
    elif args.profile == "chain":
        # the small-M weight-streaming chain on --layers layers of the stack at --rows rows (4 layers:
        # 1.5 GB of weights, above L2), interleaved as the benchmark's linear stack
        dims_c = E.Dims(layers=args.layers)
        sw = E.random_stack(dims_c, seed=1000, device=dev, with_head=False)
        eng = E.VerifyEngine(dims_c, sw, [], [], max_M=args.rows, max_rows=1, device=dev)
        ops = stack_chain_ops(S, eng, args.rows)
        cws = S.Workspace(dev, S.spec_linear_chain_workspace_bytes(ops, args.rows))
        for _ in range(args.reps):
            S.spec_verify_linear_chain(ops, args.rows, ws=cws)
    elif args.profile == "attention":
        nb = args.batch
        batch = synth.ragged_batch(SEED, nb, G_LO, G_HI, CTX_LO, CTX_HI)
        cap = int((batch.ctx_len + batch.gammas + 1).max() + 15) // 16 * 16
        kc = torch.empty((nb, dims.Hkv, cap, dims.D), dtype=torch.bfloat16, device=dev).normal_(0, 1, generator=g)
        vc = torch.empty_like(kc).normal_(0, 1, generator=g)
        qkv = torch.empty((batch.M, dims.qkv), dtype=torch.bfloat16, device=dev).normal_(0, 1, generator=g)
        cu = torch.from_numpy(batch.cu_rows).to(dev)
        ctx = torch.from_numpy(batch.ctx_len).to(dev)
        hq, hk = dims.Hq * dims.D, dims.Hkv * dims.D
        for _ in range(args.reps):
            S.spec_verify_attention(qkv[:, :hq], qkv[:, hq:hq + hk], qkv[:, hq + hk:], cu, ctx, kc, vc,
                                    batch.max_rows, ws=ws)
    elif args.profile == "sampler":
        # the round's fused LM head -> sampler on synthetic inputs: the benchmark batch (368 rows), the
        # full vocabulary, draft rows q = softmax of random logits, drafts sampled from q
        batch = make_batch()
        M, K, V = batch.M, dims.d, dims.V
        W = torch.empty((V, K), dtype=torch.bfloat16, device=dev).normal_(0, 0.02, generator=g)
        X = torch.empty((M, K), dtype=torch.bfloat16, device=dev).normal_(0, 1, generator=g)
        nq = batch.n_drafts
        q = torch.softmax(torch.empty((nq, V), device=dev).normal_(0, 1, generator=g), dim=1).contiguous()
        drafts = torch.multinomial(q, 1, generator=g).view(-1).to(torch.int32)
        U = torch.from_numpy(synth.uniforms_f32(SEED, M)).to(dev)
        cu = torch.from_numpy(batch.cu_rows).to(dev)
        for _ in range(args.reps):
            S.spec_lmhead_reject_sample(X, W, TEMP, q, drafts, U, cu, ws=ws)
    else:
        M = args.rows
        if args.nsub:
            S.spec_set_option("lmhead_nsub" if args.profile == "lmhead" else "linear_nsub", args.nsub)
        if args.profile in ("linear", "swiglu"):
            N, K = args.n, args.k
        else:
            N, K = dims.V, dims.d
        W = torch.empty((N, K), dtype=torch.bfloat16, device=dev).normal_(0, 0.02, generator=g)
        X = torch.empty((M, K), dtype=torch.bfloat16, device=dev).normal_(0, 1, generator=g)
        for _ in range(args.reps):
            if args.profile == "linear":
                S.spec_verify_linear(X, W, ws=ws)
            elif args.profile == "swiglu":
                S.spec_verify_linear_swiglu(X, W, ws=ws)
            else:
                S.spec_lmhead_softmax(X, W, TEMP, ws=ws)
    torch.cuda.synchronize()
    S.spec_device_status()
    print(json.dumps({"profile": args.profile, "reps": args.reps, "ok": True}))


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu", action="store_true", help="skip the oracle CPU baseline")
    ap.add_argument("--no-draft", action="store_true", help="skip the draft-phase measurement")
    ap.add_argument("--no-extra", action="store_true", help="skip the sweep points and configuration 3")
    ap.add_argument("--profile", choices=["round", "attention", "linear", "swiglu", "lmhead", "chain", "sampler"],
                    default=None,
                    help="run a small case of one kernel for an ncu capture instead of the benchmark")
    ap.add_argument("--rows", type=int, default=368, help="rows for --profile linear/lmhead/chain")
    ap.add_argument("--layers", type=int, default=4, help="stack layers for --profile chain")
    ap.add_argument("--batch", type=int, default=16, help="sequences for --profile attention")
    ap.add_argument("--reps", type=int, default=3, help="launches for --profile")
    ap.add_argument("--n", type=int, default=24576, help="weight rows for --profile linear")
    ap.add_argument("--k", type=int, default=4096, help="reduction length for --profile linear")
    ap.add_argument("--set", action="append", default=[], metavar="NAME=VALUE",
                    help="library knob passed to spec_set_option before the run (repeatable)")
    ap.add_argument("--sampler", choices=["fused", "split"], default="fused",
                    help="LM head -> sampler in one call without materialising p (fused), or softmax + sampler")
    ap.add_argument("--swiglu", choices=["fused", "split"], default="fused",
                    help="SwiGLU in the gate|up GEMM epilogue (fused) or as its own kernel (split)")
    ap.add_argument("--sweep", action="store_true",
                    help="batch x depth sweep (B in 1..1024, gamma in 1/4/10): linear stack and attention rooflines")
    ap.add_argument("--nsub", type=int, default=0, help="linear_nsub knob for --profile linear/lmhead (0: library default)")
    args = ap.parse_args()
    if args.set and args.impl == "ours":
        from speculative_decoding_verify_05_gb300 import binding as S
        for kv in args.set:
            name, _, value = kv.partition("=")
            if S._lib.spec_set_option(name.encode(), int(value)) != 0:
                ap.error(f"--set {kv}: {S._lib.spec_last_error().decode()}")
    if args.profile:
        run_profile_case(args)
        return
    if args.sweep:
        run_sweep(args)
        return
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
