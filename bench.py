#!/usr/bin/env python
"""Benchmark of the GB300 int2 draft head: one pass of the hot path (coarse int2 pass + block
top-KCAND, then global top-RERANK + exact bf16 rerank + argmax) per step, on the vocabulary-scale
head (K=5120, N=124160, G=128, KCAND=8, RERANK=16), hidden rows M=1 by default.

Prints ONE JSON line. Timing: CUDA events on the launching stream after warm-up, synchronised
on both sides; the packed weight, scales and bf16 weight rotate over 4 device copies (716 MB of
packed head, 5 GB of bf16 head) so every step reads its weights from HBM, not from the 129 MB
L2. `--impl reference` times the CPU oracle (the plain fp64 statement of the method) on the same
workload instead. Multi-GPU (torchrun): every rank runs an independent replica (the head does
not shard here); value = job-level microseconds per call over all ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

K_DIM, N_VOCAB, GROUP, KCAND, RERANK = 5120, 124160, 128, 8, 16
COPIES = 4
METRIC = "draft-head us/call + achieved HBM GB/s vs ~8 TB/s, M=1/8/72, K=5120 N=124160"
PROFILE_TRAFFIC = os.path.join(ROOT, "profiles", "coarse_traffic.json")


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=2000)
    p.add_argument("--warmup", type=int, default=20)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--m", type=int, default=1, help="hidden rows of the headline workload")
    p.add_argument("--extra-m", default="8,72", help="supplementary row counts ('' = none)")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-variants", action="store_true",
                   help="skip the int4 / group-64 comparison lines (M=8)")
    p.add_argument("--no-soak", action="store_true",
                   help="skip the 1.5 s clock-sampling soak (profiling runs)")
    p.add_argument("--copies", type=int, default=COPIES,
                   help="rotating weight copies (4 keep every step out of L2)")
    return p.parse_args()


# ------------------------------------------------------------------------------------ helpers
def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


COARSE_SOURCES = ("coarse.cu", "coarse_kernel.cuh", "coarse_i2g128.cu", "coarse_i2g64.cu",
                  "coarse_i4g128.cu", "coarse_i4g64.cu", "dh_device.cuh")


def coarse_source_hash():
    """Fingerprint of the coarse kernel's sources: a profiled traffic figure is used only while
    it still describes the kernel being timed."""
    h = hashlib.sha256()
    for f in COARSE_SOURCES:
        with open(os.path.join(ROOT, "bit_draft_lm_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def profiled_traffic(M):
    """dram bytes per coarse launch from the committed ncu summary, if it was taken on the
    current kernel source and this row count; else None."""
    try:
        with open(PROFILE_TRAFFIC) as f:
            d = json.load(f)
        if d.get("source_hash") == coarse_source_hash() and int(d.get("M", -1)) == M:
            return float(d["dram_bytes_per_launch"])
    except Exception:
        pass
    return None


class ClockSampler:
    """nvidia-smi sampling (200 ms) of SM clock and throttle reasons while the GPU runs."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.f = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        try:
            self.p = subprocess.Popen(["nvidia-smi", "-i", str(index), f"--query-gpu={self.Q}",
                                       "--format=csv,noheader,nounits", "-lms", "200"],
                                      stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.p = None

    def stop(self):
        if self.p is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.p.terminate()
        try:
            self.p.wait(timeout=5)
        except Exception:
            self.p.kill()
        self.f.flush()
        self.f.seek(0)
        rows = [r.split(",") for r in self.f.read().strip().splitlines() if r.strip()]
        os.unlink(self.f.name)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            try:
                sm.append(float(r[1]))
                mx.append(float(r[2]))
                for name, v in zip(names, r[5:9]):
                    if v.strip() == "Active":
                        reasons.add(name)
            except (ValueError, IndexError):
                continue
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": sorted(reasons),
                "samples": len(sm)}


# ------------------------------------------------------------------------------------ workload
def workload_host(M, seed=1):
    """x [M, K] and W [N, K] bf16 bits: the vocabulary-scale recipe of synth (row 0 of x and the
    planted rows / near-tie pairs of W follow the recipe; further rows of x are fresh draws)."""
    from bit_draft_lm_gb300 import synth
    w = synth.named("head_m1_k5120_n124160")
    rng = np.random.default_rng(seed + 1000 + M)
    z = rng.standard_normal((max(M, 1) * COPIES, K_DIM))
    z /= np.sqrt(np.mean(z * z, axis=1, keepdims=True))
    xs = synth.bf16_bits(z).reshape(COPIES, max(M, 1), K_DIM)
    xs[0, 0] = w.x[0]
    return xs, w.W


# ------------------------------------------------------------------------------------ our arm
def run_ours(args, rank, world):
    import torch
    import torch.distributed as dist
    from bit_draft_lm_gb300 import build as dh_build
    from bit_draft_lm_gb300 import drafthead as dh

    dh_build.build()
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    # rows of x for every measured workload (the variant lines use 8)
    xs_h, W_h = workload_host(max([args.m] + extra_ms(args) + ([] if args.no_variants else [8])))
    W0 = torch.from_numpy(W_h.view(np.int16)).to(dev).view(torch.bfloat16)
    ncopy = max(1, args.copies)
    Ws = [W0] + [W0.clone() for _ in range(ncopy - 1)]
    packs = [dh.dh_quantize_pack_int2(Wc, GROUP) for Wc in Ws]
    torch.cuda.synchronize()
    nblk = (N_VOCAB + 63) // 64

    def measure(M, steps, warmup, record_launches, bits=2, group=GROUP, kcand=KCAND, packs=packs,
                fp8_rows=None):
        xs = [torch.from_numpy(xs_h[c, :M].copy().view(np.int16)).to(dev).view(torch.bfloat16)
              for c in range(ncopy)]
        ws = dh.new_workspace(M, N_VOCAB, K_DIM, kcand, RERANK, dev)
        cv = torch.empty(M, nblk * kcand, dtype=torch.float32, device=dev)
        ci = torch.empty(M, nblk * kcand, dtype=torch.int32, device=dev)
        rr = torch.empty(M, RERANK, dtype=torch.int32, device=dev)
        rl = torch.empty(M, RERANK, dtype=torch.float32, device=dev)
        am = torch.empty(M, dtype=torch.int32, device=dev)
        stream = torch.cuda.current_stream()

        def step(c, mode="call"):
            # call: the whole path through dh_draft_head_argmax (coarse and rerank kernels), or
            # for the FP8 head the coarse call then the FP8 rerank call; coarse: the coarse
            # kernel alone
            p, S, ZS = packs[c]
            if mode == "call" and fp8_rows is None:
                dh.dh_draft_head_argmax(xs[c], p, S, ZS, Ws[c], group, bits, kcand, RERANK,
                                        cand_val=cv, cand_id=ci, rr_id=rr, rr_logit=rl,
                                        argmax_id=am, workspace=ws)
                return
            dh.dh_draft_head_coarse_topk(xs[c], p, S, ZS, N_VOCAB, group, bits, kcand,
                                         cand_val=cv, cand_id=ci, workspace=ws)
            if mode != "coarse":
                dh.dh_draft_head_rerank_argmax_fp8(xs[c], fp8_rows[c][0], fp8_rows[c][1], cv, ci,
                                                   RERANK, rr_id=rr, rr_logit=rl, argmax_id=am,
                                                   workspace=ws)

        # eager warm-up (first launches set kernel attributes), then every timed step runs from
        # CUDA graphs: one graph per round over the weight copies, so host launch overhead is
        # not in the measurement
        for i in range(warmup):
            step(i % ncopy)
        torch.cuda.synchronize()

        def capture(n, mode="call"):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                for c in range(n):
                    step(c, mode)
            return g

        reps, rem = divmod(steps, ncopy)
        g_round = capture(ncopy)
        g_rem = capture(rem) if rem else None

        def timed(g, g_tail):
            for _ in range(max(1, warmup // ncopy)):
                g.replay()
            torch.cuda.synchronize()
            t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            if world > 1:
                dist.barrier()
            torch.cuda.synchronize()
            t0.record(stream)
            for _ in range(reps):
                g.replay()
            if g_tail is not None:
                g_tail.replay()
            t1.record(stream)
            torch.cuda.synchronize()
            if world > 1:
                dist.barrier()
            return t0.elapsed_time(t1)

        ms = timed(g_round, g_rem)
        coarse_ms = None
        if record_launches:
            # the coarse kernel alone over the same number of steps (its average launch time)
            coarse_ms = timed(capture(ncopy, "coarse"), capture(rem, "coarse") if rem else None)
        status = dh.dh_workspace_status(ws)
        if status:
            raise RuntimeError(f"kernel status word {status:#x}")
        return ms, coarse_ms

    clocks = ClockSampler(dev.index)
    time.sleep(0.3)
    ms, coarse_ms = measure(args.m, args.steps, max(args.warmup, 3), True)
    # keep the same step running ~1.5 s so the clock samples cover this workload under load
    soak_t = time.time()
    if not args.no_soak:
        soak_steps = max(1, int(1.5e3 / max(ms / args.steps, 1e-3)))
        measure(args.m, min(soak_steps, 200000), 3, False)
    soak_t = time.time() - soak_t
    clk = clocks.stop()
    if world > 1:
        t = torch.tensor([ms], device=dev)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        ms = float(t.item())

    us_step = ms * 1e3 / args.steps
    coarse_us = 1e3 * coarse_ms / args.steps
    peak, peak_kind = measured_peaks()
    alg_coarse = dh.dh_packed_bytes(N_VOCAB, K_DIM, GROUP, 2)
    alg_call = alg_coarse + args.m * RERANK * K_DIM * 2

    def launches_per_call(M):
        # coarse: passes of 8 rows up to 16 rows; beyond, a prep and a tensor-core kernel per
        # pass of up to 80 rows; then the rerank
        return ((M + 7) // 8 if M <= 16 else 2 * ((M + 79) // 80)) + 1
    launches_per_step = launches_per_call(args.m)

    extra = {}
    for M in extra_ms(args):
        steps = max(50, min(args.steps, int(3e5 / max(M, 1))))
        mm, cm = measure(M, steps, 8, True)
        u = mm * 1e3 / steps
        extra[str(M)] = {"us_per_call": round(u, 3),
                         "coarse_us": round(1e3 * cm / steps, 3),
                         "launches_per_call": launches_per_call(M),
                         "hbm_gbs_per_call": round((alg_coarse + M * RERANK * K_DIM * 2) / u / 1e3, 1),
                         "steps": steps}
    # the page's two ablations at M=8 (the comparison workload): the 4-bit head with KCAND=1, and
    # the int2 head with 64-wide groups
    # recall on the golden rows (written by the oracle alone; tests/golden/make_recall.py): the
    # timed kernels, in 8-row calls, against the brute-force exact argmax of every row
    gold = recall_golden()

    def recall(name, bits, group, kcand, pk):
        if gold is None or name not in gold["configs"]:
            return None
        from bit_draft_lm_gb300 import synth
        cfg = gold["configs"][name]
        xr = torch.from_numpy(synth.recall_rows(synth.named(gold["head"])).view(np.int16))
        xr = xr.to(dev).view(torch.bfloat16)
        am = []
        for m0 in range(0, xr.shape[0], 8):
            am.append(dh.dh_draft_head_argmax(xr[m0:m0 + 8], pk[0], pk[1], pk[2], Ws[0], group,
                                              bits, kcand, cfg["rerank"])[2])
        am = torch.cat(am).cpu().numpy()
        ex, method = np.asarray(gold["exact_argmax"]), np.asarray(cfg["method_argmax"])
        miss = np.nonzero(am != ex)[0].tolist()
        return {"rows": int(ex.size), "misses": len(miss), "miss_rows": miss,
                "oracle_method_misses": len(cfg["misses"]),
                "same_argmax_as_oracle_method": int((am == method).sum()),
                "rerank": cfg["rerank"], "kcand": kcand}

    headline_recall = recall("int2_g128_kcand8", 2, GROUP, KCAND, packs[0])
    variants = {}
    if not args.no_variants:
        for name, gname, bits, group, kc in (
                ("int4_g128_m8_kcand1", "int4_g128_kcand1", 4, 128, 1),
                ("int2_g64_m8_kcand8", "int2_g64_kcand8", 2, 64, KCAND)):
            quant = dh.dh_quantize_pack_int4 if bits == 4 else dh.dh_quantize_pack_int2
            vp = [quant(Wc, group) for Wc in Ws]
            steps = max(50, min(args.steps, 1000))
            mm, cm = measure(8, steps, 8, True, bits=bits, group=group, kcand=kc, packs=vp)
            u = mm * 1e3 / steps
            alg = dh.dh_packed_bytes(N_VOCAB, K_DIM, group, bits) + 8 * RERANK * K_DIM * 2
            variants[name] = {"us_per_call": round(u, 3), "coarse_us": round(1e3 * cm / steps, 3),
                              "algorithmic_bytes_per_call": alg,
                              "hbm_gbs_per_call": round(alg / u / 1e3, 1), "steps": steps,
                              "recall": recall(gname, bits, group, kc, vp[0])}
            del vp
            torch.cuda.synchronize()
        # the FP8 checkpoint's head at M=1: int2 codes quantised from e4m3 rows x row scale, the
        # rerank against the e4m3 rows (half the gather bytes of bf16 rows)
        from bit_draft_lm_gb300 import synth
        w8h, sch = synth.fp8_head(W_h)
        rows = [(torch.from_numpy(w8h).to(dev), torch.from_numpy(sch).to(dev))
                for _ in range(ncopy)]
        vp = [dh.dh_quantize_pack_int2_fp8(r[0], r[1], GROUP) for r in rows]
        steps = max(50, min(args.steps, 1000))
        mm, cm = measure(1, steps, 8, True, packs=vp, fp8_rows=rows)
        u = mm * 1e3 / steps
        alg = alg_coarse + RERANK * K_DIM
        variants["fp8_head_m1_kcand8"] = {"us_per_call": round(u, 3),
                                          "coarse_us": round(1e3 * cm / steps, 3),
                                          "algorithmic_bytes_per_call": alg,
                                          "hbm_gbs_per_call": round(alg / u / 1e3, 1),
                                          "steps": steps}
        del vp, rows
        torch.cuda.synchronize()

    e2e = None
    if not args.no_e2e:
        e2e = run_e2e(args, dev, Ws, xs_h, ncopy)

    line = {
        "metric": METRIC,
        "value": round(us_step / world, 3),
        "unit": "us/call",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": max(args.warmup, 3),
        "ms_per_step": round(ms / args.steps, 6),
        "higher_is_better": False,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded numpy: RMS-normed N(0,1) hidden rows; lognormal-row N(0,0.02) "
                "head with planted rows and near-tie pairs)",
        "config": {"workload": f"int2 draft head M={args.m} K={K_DIM} N={N_VOCAB} G={GROUP} "
                               f"KCAND={KCAND} RERANK={RERANK}",
                   "M": args.m, "K": K_DIM, "N": N_VOCAB, "G": GROUP, "bits": 2,
                   "kcand": KCAND, "rerank": RERANK,
                   "l2": f"inputs larger than L2: {ncopy} rotating copies of the packed head "
                         f"({ncopy * alg_coarse / 1e6:.0f} MB) and of the bf16 head",
                   "parallelism": f"replicas x{world}"},
        "hbm_gbs_per_call": round(alg_call / us_step / 1e3, 1),
        "roofline": {"bound": "hbm",
                     "kernel": "coarse_topk_kernel" if args.m <= 16 else "coarse_wide_kernel",
                     "achieved": round(alg_coarse / coarse_us / 1e3, 1), "peak": peak,
                     "unit": "GB/s", "frac": round(alg_coarse / coarse_us / 1e3 / peak, 4),
                     "peak_kind": peak_kind,
                     "traffic": profiled_traffic(args.m),
                     "algorithmic_bytes_per_launch": alg_coarse,
                     "launch_us": round(coarse_us, 3)},
        "api": "dh_draft_head_argmax (coarse + rerank kernels)",
        "launches_per_call": launches_per_step,
        "gpu_launches": args.steps * launches_per_step,
        "clocks": dict(clk, window=f"timed region + {soak_t:.1f} s of the same step"),
        "per_m": extra,
        "variants": variants,
        "recall": headline_recall,
    }
    if e2e is not None:
        line["e2e"] = e2e
    if not args.no_cpu_baseline and rank == 0:
        line["cpu_baseline"] = cpu_baseline(args.m, budget_s=15.0)
    return line


def recall_golden():
    """The recall report's stored rows and expected ids (None if the file is absent)."""
    try:
        with open(os.path.join(ROOT, "tests", "golden", "recall_k5120_n124160_m64.json")) as f:
            return json.load(f)
    except OSError:
        return None


def extra_ms(args):
    return [int(v) for v in args.extra_m.split(",") if v.strip()] if args.extra_m else []


def run_e2e(args, dev, Ws, xs_h, ncopy):
    """The C-ABI call with host buffers (DraftHead.call_host: a dh_host_plan run every step, which
    takes x from pinned host memory, runs the head, puts argmax / rr_id / rr_logit into pinned
    host memory and synchronises). dh_draft_head_host with all its arguments is timed beside
    it."""
    import torch
    from bit_draft_lm_gb300 import drafthead as dh
    M = args.m
    heads = [dh.DraftHead(Wc, GROUP, 2, KCAND, RERANK, max_tokens=M) for Wc in Ws]
    xh = [torch.from_numpy(xs_h[c, :M].copy().view(np.int16)).view(torch.bfloat16).pin_memory()
          for c in range(ncopy)]
    torch.cuda.synchronize()
    steps = min(args.steps, 2000)

    def timed(call):
        for i in range(max(args.warmup, 3)):
            call(heads[i % ncopy], xh[i % ncopy])
        t0 = time.perf_counter()
        for i in range(steps):
            call(heads[i % ncopy], xh[i % ncopy])
        return (time.perf_counter() - t0) * 1e6 / steps

    v = timed(lambda h, x: h.call_host(x))
    d = timed(lambda h, x: h.call_host(x, plan=False))
    for h in heads:
        if dh.dh_workspace_status(h.workspace):
            raise RuntimeError("kernel status word set in the end-to-end run")
    return {"value": round(v, 3), "unit": "us/call", "h2d_bytes_per_step": M * K_DIM * 2,
            "d2h_bytes_per_step": M * 4 + 2 * M * RERANK * 4, "steps": steps,
            "api": "dh_host_plan_run (C ABI, host buffers; plan prepared once per M)",
            "direct_call_value": round(d, 3)}


# ------------------------------------------------------------------------------------ oracle arm
def oracle_sample(M, rows, nthreads=None):
    """Quantise a slice of the head with the oracle (untimed) and return callables running the
    oracle's full path (coarse -> block top-K -> top-R -> rerank -> argmax) and its quantiser
    (a0) on that slice."""
    import oracle
    xs_h, W_h = workload_host(M)
    Ws = np.ascontiguousarray(W_h[:rows])
    x = np.ascontiguousarray(xs_h[0, :M])
    packed, S, ZS = oracle.quantize_pack(Ws, GROUP, 2)

    def call():
        return oracle.head(x, packed, S, ZS, Ws, G=GROUP, bits=2, kcand=KCAND, R=RERANK,
                           nthreads=nthreads)

    def quant():
        return oracle.quantize_pack(Ws, GROUP, 2, nthreads=nthreads)
    return call, quant


def _median_time(fn, budget_s, at_least=3, at_most=50):
    fn()
    times = []
    t_start = time.perf_counter()
    while (time.perf_counter() - t_start < budget_s or len(times) < at_least) and \
            len(times) < at_most:
        t0 = time.perf_counter()
        fn()
        times.append(time.perf_counter() - t0)
    return statistics.median(times), len(times)


def cpu_baseline(M, budget_s):
    """The oracle as it stands, on the host cores, on bounded slices of the same head; times per
    call scaled to the full vocabulary (each slice's rows are a fixed fraction of N). The
    all-core figure is the line's value; beside it the single-thread figure and the quantiser
    (a0, load time, not part of a call), each a median of at least 3 runs."""
    import oracle
    rows = 15520                                # 1/8 of the vocabulary, whole 64-row blocks
    call, quant = oracle_sample(M, rows)
    t_all, n_all = _median_time(call, budget_s)
    t_q, n_q = _median_time(quant, 0.2 * budget_s)
    rows1 = 1940                                # 1/64 of the vocabulary, on one thread
    call1, _ = oracle_sample(M, rows1, nthreads=1)
    t_1, n_1 = _median_time(call1, 0.2 * budget_s)
    scale, scale1 = N_VOCAB / rows, N_VOCAB / rows1
    return {"value": round(t_all * scale * 1e6, 1), "unit": "us/call",
            "cores": oracle.threads(), "kind": "oracle",
            "sample": f"median of {n_all} calls of the oracle's full path on a {rows}-row slice "
                      f"(1/{int(scale)}) of the N={N_VOCAB} head at M={M}, x {scale:g}",
            "single_thread": {"value": round(t_1 * scale1 * 1e6, 1), "unit": "us/call",
                              "cores": 1,
                              "sample": f"median of {n_1} calls on a {rows1}-row slice, "
                                        f"x {scale1:g}"},
            "quantize_a0": {"value": round(t_q * scale * 1e3, 2), "unit": "ms/head",
                            "cores": oracle.threads(),
                            "sample": f"median of {n_q} oracle quantise + pack runs of the "
                                      f"{rows}-row slice, x {scale:g} (load time: not in a call)"}}


def run_reference(args):
    """--impl reference: the CPU oracle timed per step on a bounded slice of the workload."""
    import oracle
    probe, _ = oracle_sample(args.m, 1940)
    t0 = time.perf_counter()
    probe()
    t_small = max(time.perf_counter() - t0, 1e-4)
    per_step_budget = 120.0 / max(args.steps + args.warmup, 1)
    rows = int(1940 * per_step_budget / t_small) // 64 * 64
    rows = max(128, min(rows, N_VOCAB // 4))
    call = probe if rows == 1940 else oracle_sample(args.m, rows)[0]
    for _ in range(args.warmup):
        call()
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        call()
        times.append(time.perf_counter() - t0)
    scale = N_VOCAB / rows
    v = statistics.fmean(times) * scale * 1e6
    sample = (f"each step: the oracle's full path on a {rows}-row slice of the N={N_VOCAB} head "
              f"at M={args.m}, time x {scale:.3g}")
    return {"impl": "reference", "metric": METRIC, "value": round(v, 1), "unit": "us/call",
            "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(v / 1e3, 3), "higher_is_better": False, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": f"int2 draft head M={args.m} K={K_DIM} N={N_VOCAB} G={GROUP} "
                                   f"KCAND={KCAND} RERANK={RERANK}", "M": args.m},
            "cpu_baseline": {"value": round(v, 1), "unit": "us/call", "cores": oracle.threads(),
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": round(v, 1), "unit": "us/call", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def main():
    args = parse()
    rank = int(os.environ.get("RANK", 0))
    world = int(os.environ.get("WORLD_SIZE", 1))
    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args)))
        return
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", 0)))
        dist.init_process_group("nccl")
    line = run_ours(args, rank, world)
    if rank == 0:
        print(json.dumps(line))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
