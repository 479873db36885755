#!/usr/bin/env python3
"""Throughput of the DFlash speculative round on GB300.

One step = one full round of the hot path on the end-to-end workload
(36-layer Qwen3-4B-shaped bf16 target, 5-layer drafter, block 16,
1024-token seeded prompt): drafter forward over the masked block, batched
verify forward of the 16 rows, first-mismatch acceptance with KV rollback,
and the tap commit (fc + context K/V projection) of the accepted rows.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints one JSON line.  `value` is rounds/s of device time (CUDA graph of
one round, replayed K times, inputs resident in HBM; weights stream 9.9 GB
per round, far larger than L2, so no flush is needed); `e2e` is the same
workload driven through the public Python API from a host prompt to 512
tokens on the host.  `--impl reference` times the CPU oracle on a bounded
sample of the same round.  Under torchrun each rank runs an independent
replica (the round does not shard).
"""

from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "DFlash draft+verify rounds/s and accepted tok/s at block 16; % of HBM roofline"
FALLBACK_HBM_GBS = 6800.0


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--cpu-baseline-worker", action="store_true", help=argparse.SUPPRESS)
    ap.add_argument("--ncu-tap", type=int, default=0, metavar="ROWS",
                    help="run the hc tap reduce (4 layers, hc 4, hidden 4096) at ROWS rows, "
                         "3 launches, for an ncu capture")
    ap.add_argument("--ncu-batch", type=int, default=0, metavar="S",
                    help="one many-sequence round of S sequences inside NVTX range "
                         "'dflash_batch' (with --layers: a cut target), for an ncu capture")
    ap.add_argument("--int4", action="store_true",
                    help="with --ncu-rounds: the e2e workload with every model in INT4 group-64")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-workloads", action="store_true",
                    help="skip the drafter-alone, INT4, hc-tap and verify-sweep measurements")
    ap.add_argument("--layers", type=int, default=0,
                    help="(debug) override target layers; lines printed with it are not the workload")
    ap.add_argument("--ncu-dense", type=int, nargs=3, metavar=("M", "N", "K"), default=None,
                    help="profiling mode: three dense tcgen05 GEMMs of M x N x K, no JSON line")
    ap.add_argument("--ncu-prefill", action="store_true",
                    help="profiling mode: one warm-up prefill, then one inside the NVTX range "
                         "'dflash_prefill', no JSON line")
    ap.add_argument("--ncu-rounds", type=int, default=0,
                    help="profiling mode: prefill, then N eager rounds inside the NVTX range "
                         "'dflash_rounds', no timing and no JSON line")
    return ap.parse_args()


# ----------------------------------------------------------------- helpers

def rank_info():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def workload_config(w, world, timing, l2):
    """The `config` object both arms print: the same workload, with the
    arm's own timing method and cache treatment."""
    return {
        "workload": "e2e_bf16: 36-layer Qwen3-4B-shaped bf16 target (hidden 2560, 32q/8kv "
                    "heads, SwiGLU 9728, vocab 151936) + 5-layer drafter, taps at "
                    "{0,8,17,26,35}, block 16, 1024-token prompt, natural acceptance",
        "block": w.block, "prompt_len": w.prompt_len,
        "l2": l2,
        "timing": timing,
        "parallelism": f"replicas x{world}",
    }


def reduce_over_ranks(world, device, t_ms, *counts):
    """Replicas: the whole job's time is the slowest rank's timed region and
    each count (rounds, tokens) is summed over the ranks.  Returns
    (max t_ms, [sum of each count]); with one rank, the inputs unchanged."""
    if world == 1:
        return t_ms, list(counts)
    import torch
    import torch.distributed as dist
    mx = torch.tensor([float(t_ms)], dtype=torch.float64, device=device)
    sm = torch.tensor([float(c) for c in counts], dtype=torch.float64, device=device)
    dist.all_reduce(mx, op=dist.ReduceOp.MAX)
    dist.all_reduce(sm, op=dist.ReduceOp.SUM)
    return float(mx[0]), [float(v) for v in sm.tolist()]


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled during the timed region."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.f = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        self.p = None

    def __enter__(self):
        try:
            self.p = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.idx), f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=self.f, stderr=subprocess.DEVNULL)
        except OSError:
            self.p = None
        time.sleep(0.3)
        return self

    def __exit__(self, *a):
        if self.p:
            self.p.terminate()
            try:
                self.p.wait(5)
            except subprocess.TimeoutExpired:
                self.p.kill()

    def summary(self):
        self.f.flush()
        self.f.seek(0)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.f.read().splitlines():
            parts = [x.strip() for x in line.split(",")]
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
        os.unlink(self.f.name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons)}


def measured_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        try:
            d = json.load(open(p))
            for k in ("hbm_gbs_sustained", "hbm_gbs"):
                if k in d and d[k]:
                    return float(d[k]), f"measured ({k})"
        except Exception:
            pass
    return FALLBACK_HBM_GBS, "fallback (no MEASURED_PEAKS.json)"


def gemm_source_sha() -> str:
    """Hash of the skinny GEMM's sources: a committed traffic figure counts
    only while the kernel it was captured on is unchanged."""
    import hashlib
    h = hashlib.sha256()
    for f in ("gemm.cu", "gemm_dev.cuh", "gemm.cuh", "common.cuh"):
        with open(os.path.join(ROOT, "block_diffusion_speculative_gather_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def traffic_from_profiles():
    """Per-launch DRAM bytes of the GEMM from the committed ncu summary, if it
    was captured on the current kernel sources."""
    p = os.path.join(ROOT, "profiles", "gemm_skinny_traffic.json")
    if os.path.exists(p):
        try:
            d = json.load(open(p))
        except Exception:
            return None
        if d.get("kernel_sha") == gemm_source_sha():
            return d
    return None


# ----------------------------------------------------------------- the oracle on the host

def _np32(t):
    return t.detach().float().numpy()


def oracle_weights(w, model=None):
    """The oracle's weights of workload w, from the seeded generators (the
    values the GPU arm streams): target layers and drafter, INT4 layers as
    the oracle's own quantise-dequantise of the same fp32 draws."""
    from block_diffusion_speculative_gather_gb300 import synth
    from oracle import dflash_oracle as O
    m = model if model is not None else synth.ModelTensors(w)

    def layers(ls, int4):
        out = []
        for lw in ls:
            d = {}
            for k, t in lw.items():
                a = _np32(t)
                if int4 and k in synth.LAYER_KEYS:
                    a = O.dequant_int4_g64(*O.quantize_int4_g64(a))
                d[k] = a
            out.append(d)
        return out

    embed = _np32(m.embed)
    tw = O.TargetWeights(embed, layers(m.tgt, w.tgt_int4), _np32(m.final_norm_t)) \
        if w.tgt_layers else None
    dw = O.DraftWeights(layers(m.drf, w.drf_int4), _np32(m.fc), _np32(m.ctx_norm),
                        _np32(m.final_norm_d)) if w.drf_layers else None
    cfg = O.OracleConfig(hidden=w.hidden, n_q=w.n_q, n_kv=w.n_kv, head_dim=w.head_dim, ffn=w.ffn,
                         vocab=w.vocab, tgt_layers=w.tgt_layers, drf_layers=w.drf_layers,
                         tap_layers=list(w.tap_layers), block=w.block, window=w.window,
                         max_seq=w.max_seq, eos_id=w.eos_id, rms_eps=w.rms_eps,
                         rope_theta=w.rope_theta, ctx_norm=w.ctx_norm)
    return tw, dw, cfg, embed


def synthetic_cache(n_layers, n_kv, n_pos, head_dim, name):
    """The oracle's KV cache holding N(0,1) K/V (rounded to fp16, the GPU
    caches' type) at positions [0, n_pos) of every layer."""
    import numpy as np
    from block_diffusion_speculative_gather_gb300 import synth
    from oracle import dflash_oracle as O
    cache = O.KVCache(n_layers, n_kv, head_dim)
    for l in range(n_layers):
        kv = synth.normal((2, n_kv, n_pos, head_dim), 1.0, synth.KV_SEED, f"{name}.{l}")
        kv = kv.astype(np.float16).astype(np.float32)
        cache.write(l, range(n_pos), np.moveaxis(kv[0], 0, 1), np.moveaxis(kv[1], 0, 1))
    return cache


class OracleRounds:
    """Real speculative rounds of the CPU oracle from a synthetic state: the
    target's cache holds N(0,1) K/V at positions [0, n) and the drafter's
    context N(0,1) tap rows there (a 1024-token prefill through the oracle
    would take hours), the pending token a seeded id.  One round is what the
    oracle's own loop (spec_rounds) does per round: draft_forward over the
    tap context, target_forward of [t_n, d_1..d_m], argmax, accept, KV
    rollback and the tap rows of the emitted tokens appended to the
    context."""

    def __init__(self, tw, dw, cfg, n):
        import numpy as np
        from block_diffusion_speculative_gather_gb300 import synth
        from oracle import dflash_oracle as O
        self.O, self.np = O, np
        self.tw, self.dw, self.cfg, self.n = tw, dw, cfg, n
        taps = synth.tap_rows(n, cfg.n_taps * cfg.hidden)
        self.taps = list(_np32(taps))
        self.cache = synthetic_cache(len(tw.layers), cfg.n_kv, n, cfg.head_dim, "oracle-e2e-kv")
        self.t_n = int(synth.uniform_ids(1, cfg.vocab, seed=synth.PROMPT_SEED, name="t_n")[0])
        self.emitted = 0
        self.rounds = 0

    def round(self) -> float:
        O, np = self.O, self.np
        tic = time.perf_counter()
        _, d = O.draft_forward(self.dw, self.tw.embed, self.cfg, np.stack(self.taps), self.t_n,
                               self.n, self.cfg.block, lm_head=self.tw.lm_head)
        logits, vtaps = O.target_forward(self.tw, self.cfg, [self.t_n] + d, self.n, self.cache)
        y = [O.argmax_lowest(logits[i]) for i in range(len(d) + 1)]
        a, emitted, _ = O.accept(d, y, self.cfg.eos_id)
        self.cache.truncate(self.n + len(emitted))
        self.taps.extend(vtaps[i] for i in range(len(emitted)))
        self.n += len(emitted)
        self.t_n = emitted[-1]
        self.emitted += len(emitted)
        self.rounds += 1
        return time.perf_counter() - tic


def host_cpu_model() -> str:
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.startswith("Model name:"):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    import platform
    return platform.processor() or platform.machine()


def cpu_cores() -> int:
    return len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else (os.cpu_count() or 1)


def cpu_baseline_worker():
    """The cpu_baseline leg, run as its own process with one BLAS thread:
    prepares the workloads' oracle weights and synthetic states, waits for
    a line on stdin (the GPU measurements are over), then pins itself to one
    core and times one real unit of each workload, printing one JSON line."""
    import numpy as np
    from block_diffusion_speculative_gather_gb300 import synth
    from block_diffusion_speculative_gather_gb300.configs import DRAFT_INT4, E2E_BF16, HC_SWEEP
    from oracle import dflash_oracle as O
    prep0 = time.perf_counter()
    w = E2E_BF16
    tw, dw, cfg, embed = oracle_weights(w)
    rounds = OracleRounds(tw, dw, cfg, w.prompt_len)
    ctx = np.stack(rounds.taps)
    # the INT4 drafter (long-context workload): the same draws quantised
    w4 = DRAFT_INT4
    m4 = synth.ModelTensors(w4.with_(tgt_layers=0))
    _, dw4, cfg4, _ = oracle_weights(w4, m4)
    del m4
    lo = w4.n_ctx - w4.window
    taps4 = np.zeros((w4.n_ctx, cfg4.n_taps * cfg4.hidden), np.float32)
    taps4[lo:] = _np32(synth.tap_rows(w4.window, cfg4.n_taps * cfg4.hidden, name="taps-window"))
    # the verify sweep's 16384-position synthetic cache
    n16 = HC_SWEEP.prompt_len
    cache16 = synthetic_cache(len(tw.layers), cfg.n_kv, n16, cfg.head_dim, "oracle-16k-kv")
    cfg16 = O.OracleConfig(**{**cfg.__dict__, "max_seq": HC_SWEEP.max_seq})
    drafts = synth.uniform_ids(15, cfg.vocab, seed=5).tolist()
    prep_s = time.perf_counter() - prep0
    sys.stdout.write(json.dumps({"ready": True, "prep_s": round(prep_s, 1)}) + "\n")
    sys.stdout.flush()
    sys.stdin.readline()                          # the GPU measurements are over
    core = max(os.sched_getaffinity(0))
    os.sched_setaffinity(0, {core})
    res, cpu0, wall0 = {}, os.times(), time.perf_counter()

    def timed(fn):
        t = time.perf_counter()
        fn()
        return time.perf_counter() - t

    res["e2e_bf16_round_s"] = rounds.round()
    res["draft_bf16_round_s"] = timed(lambda: O.draft_forward(dw, embed, cfg, ctx, 4242, w.prompt_len,
                                                              16))
    res["draft_int4_round_s"] = timed(lambda: O.draft_forward(dw4, embed, cfg4, taps4, 4242,
                                                              w4.n_ctx, w4.block))
    sweep = {}
    for T in (1, 16):
        sweep[str(T)] = timed(lambda: O.target_forward(tw, cfg16, [17] + drafts[:T - 1], n16, cache16))
        cache16.truncate(n16)
    res["verify_16k_s_by_T"] = sweep
    cpu1, wall = os.times(), time.perf_counter() - wall0
    res["threads_busy"] = round(((cpu1.user - cpu0.user) + (cpu1.system - cpu0.system)) / wall, 2)
    res["core"] = core
    res["prep_s"] = round(prep_s, 1)
    sys.stdout.write(json.dumps(res) + "\n")
    sys.stdout.flush()


class CpuBaseline:
    """Starts the cpu_baseline worker (one BLAS thread) so that its
    preparation overlaps the GPU measurements; finish() lets it time its
    units with the GPU work over and returns the cpu_baseline object."""

    def __init__(self):
        env = dict(os.environ)
        for k in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS", "BLIS_NUM_THREADS"):
            env[k] = "1"
        env["CUDA_VISIBLE_DEVICES"] = ""          # the worker never touches a GPU
        self.p = subprocess.Popen([sys.executable, os.path.abspath(__file__), "--cpu-baseline-worker"],
                                  stdin=subprocess.PIPE, stdout=subprocess.PIPE, text=True, env=env,
                                  cwd=ROOT)

    def finish(self, timeout_s=900.0):
        try:
            ready = json.loads(self.p.stdout.readline() or "{}")
            if not ready.get("ready"):
                raise RuntimeError("worker not ready")
            self.p.stdin.write("go\n")
            self.p.stdin.flush()
            line = self.p.stdout.readline()
            self.p.wait(timeout=timeout_s)
            r = json.loads(line)
        except Exception as e:                    # pragma: no cover
            self.p.kill()
            return {"value": None, "unit": "rounds/s", "cores": 1, "kind": "oracle",
                    "sample": f"the oracle worker failed: {e}"}
        e2e = r["e2e_bf16_round_s"]
        return {
            "value": round(1.0 / e2e, 6), "unit": "rounds/s", "cores": 1, "kind": "oracle",
            "sample": ("one real round of the e2e workload (drafter forward re-projecting the "
                       "1024-row tap context, 16-row verify of the 36-layer target over a "
                       "1024-position synthetic cache, acceptance, rollback, tap commit) from a "
                       f"synthetic state: {e2e:.2f} s; fp64 numpy, one BLAS thread, pinned to "
                       f"core {r['core']} ({r['threads_busy']} threads busy)"),
            "host_cpu": host_cpu_model(), "host_cores": os.cpu_count(),
            "per_config": {
                "draft_bf16": {"unit": "draft rounds/s", "value": round(1.0 / r["draft_bf16_round_s"], 5),
                               "s": round(r["draft_bf16_round_s"], 3),
                               "what": "one drafter forward, block 16, 1024 context tap rows"},
                "draft_int4": {"unit": "draft rounds/s", "value": round(1.0 / r["draft_int4_round_s"], 5),
                               "s": round(r["draft_int4_round_s"], 3),
                               "what": "one INT4 drafter forward, block 8, window 2048 of 16384 tap rows"},
                "verify_sweep_16k": {"unit": "ms per verify", "by_T": {
                    T: round(v * 1e3, 1) for T, v in r["verify_16k_s_by_T"].items()},
                    "what": "one 36-layer verify of T rows over a 16384-position synthetic cache"},
            },
        }


# ----------------------------------------------------------------- our arm

def run_ours(args):
    import torch
    import torch.distributed as dist
    from block_diffusion_speculative_gather_gb300 import build
    build.build()
    from block_diffusion_speculative_gather_gb300 import capi, synth
    from block_diffusion_speculative_gather_gb300.configs import E2E_BF16
    from block_diffusion_speculative_gather_gb300.runtime import DFlash

    rank, world, local = rank_info()
    # the oracle baseline (N = 1 only): its worker prepares while the GPU
    # workloads run, started after the end-to-end timing (its preparation
    # loads the host, and the host-driven end-to-end loop lost ~12 % to it)
    cpu_leg = None
    want_cpu = not (args.no_cpu_baseline or args.ncu_dense or args.ncu_prefill or args.ncu_rounds
                    or args.ncu_tap or args.ncu_batch or args.layers) and rank == 0 and world == 1
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    if args.ncu_tap:
        from block_diffusion_speculative_gather_gb300.configs import HC_TAP
        hc, rows = HC_TAP, args.ncu_tap
        gen = torch.Generator("cuda").manual_seed(2)
        streams = [torch.randn(rows, hc["hc"] * hc["hidden"], device="cuda", generator=gen)
                   .to(torch.bfloat16) for _ in range(hc["n_layers"])]
        outb = torch.empty(rows, hc["n_layers"] * hc["hidden"], device="cuda")
        for _ in range(3):
            capi.dflash_tap_reduce(streams, rows, hc["hc"], hc["hidden"], outb)
        torch.cuda.synchronize()
        print(f"ncu tap done: {rows} rows", flush=True)
        return
    if args.ncu_dense:
        m, n, k = args.ncu_dense
        gen = torch.Generator(device="cuda").manual_seed(9)
        wd = (torch.randn(n, k, device="cuda", generator=gen) * 0.02).to(torch.bfloat16)
        xd = torch.randn(m, k, device="cuda", generator=gen).to(torch.bfloat16)
        yd = torch.empty(m, n, device="cuda")
        errw = torch.zeros(2, dtype=torch.int32, device="cuda")
        for _ in range(3):
            capi.dflash_linear_dense(wd, xd, yd, errw)
        torch.cuda.synchronize()
        assert errw.tolist() == [0, 0]
        print(f"ncu dense done: {m} x {n} x {k}", flush=True)
        return
    w = E2E_BF16
    if args.int4:
        w = w.with_(name="e2e_int4", tgt_int4=True, lm_int4=True, drf_int4=True)
    if args.layers:
        from block_diffusion_speculative_gather_gb300.configs import evenly_spaced_taps
        w = w.with_(tgt_layers=args.layers,
                    tap_layers=evenly_spaced_taps(args.layers, min(5, args.layers)))
    model = synth.ModelTensors(w)
    dec = DFlash(w, model)
    model_for_sweep = model if not (args.no_workloads or args.layers) else None
    del model
    prompt = torch.from_numpy(synth.uniform_ids(w.prompt_len, w.vocab))
    B = w.block

    def barrier():
        if world > 1:
            dist.barrier()

    if args.ncu_prefill:
        dec.prefill(prompt, w.n_new)
        torch.cuda.synchronize()
        torch.cuda.nvtx.range_push("dflash_prefill")
        dec.prefill(prompt, w.n_new)
        torch.cuda.synchronize()
        torch.cuda.nvtx.range_pop()
        dec.check()
        print("ncu prefill done", flush=True)
        dec.close()
        return
    if args.ncu_batch:
        from block_diffusion_speculative_gather_gb300.runtime import DFlashBatch
        dec.close()
        S = args.ncu_batch
        bdec = DFlashBatch(w, model_for_sweep if model_for_sweep is not None else synth.ModelTensors(w), S)
        prompts = [torch.from_numpy(synth.uniform_ids(w.prompt_len, w.vocab, seed=100 + i))
                   for i in range(S)]
        bdec.prefill(prompts, w.n_new)
        bdec.verify(bdec.draft())
        torch.cuda.synchronize()
        torch.cuda.nvtx.range_push("dflash_batch")
        bdec.verify(bdec.draft())
        torch.cuda.synchronize()
        torch.cuda.nvtx.range_pop()
        bdec.check()
        print(f"ncu batch done: S={S}", flush=True)
        bdec.close()
        return
    if args.ncu_rounds:
        dec.prefill(prompt, w.n_new)
        dec.verify(dec.draft())
        torch.cuda.synchronize()
        torch.cuda.nvtx.range_push("dflash_rounds")
        for _ in range(args.ncu_rounds):
            dec.verify(dec.draft())
        torch.cuda.synchronize()
        torch.cuda.nvtx.range_pop()
        dec.check()
        print(f"ncu rounds done: {args.ncu_rounds}", flush=True)
        dec.close()
        return

    # prompt prefill (dense: every row before the last 16-row chunk on the
    # dense tcgen05 GEMM), CUDA events on the launching stream, after a warm-up
    dec.prefill(prompt, w.n_new)
    torch.cuda.synchronize()
    pe0, pe1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    pe0.record()
    dec.prefill(prompt, w.n_new)
    pe1.record()
    torch.cuda.synchronize()
    prefill_ms = pe0.elapsed_time(pe1)

    # launches per round
    dec.prefill(prompt, w.n_new)
    torch.cuda.synchronize()
    l0 = capi.dflash_launch_count()
    dec.verify(dec.draft())
    torch.cuda.synchronize()
    launches_per_round = capi.dflash_launch_count() - l0
    for _ in range(args.warmup):
        dec.verify(dec.draft())
    dec.check()

    # one round captured as a CUDA graph (state lives on the device)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        dec.verify(dec.draft())
    dec.prefill(prompt, w.n_new)
    for _ in range(args.warmup):
        g.replay()
    torch.cuda.synchronize()
    st0 = dec.stats()

    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk:
        barrier()
        torch.cuda.synchronize()
        start.record()
        for _ in range(args.steps):
            g.replay()
        end.record()
        torch.cuda.synchronize()
        barrier()
    ms = start.elapsed_time(end)
    st1 = dec.stats()
    dec.check()
    clocks = clk.summary()
    rounds_total = args.steps * world
    t_max, (emitted,) = reduce_over_ranks(world, "cuda", ms, st1.emitted - st0.emitted)
    value = rounds_total / (t_max / 1e3)

    # GEMM timing: the same round captured with event nodes around each GEMM
    # (the prefill runs first, unprofiled; only the captured round is timed)
    dec.prefill(prompt, w.n_new)
    torch.cuda.synchronize()
    capi.dflash_profile(dec.ctx, 1)
    gp = torch.cuda.CUDAGraph()
    with torch.cuda.graph(gp, stream=s):
        dec.verify(dec.draft())
    prof_ms, prof_bytes, prof_launch = 0.0, 0.0, 0
    for _ in range(args.steps):
        gp.replay()
        p = capi.dflash_profile(dec.ctx, 2)
        prof_ms += p.gemm_ms
        prof_bytes += p.gemm_bytes
        prof_launch += p.gemm_launches
    capi.dflash_profile(dec.ctx, 0)
    peak, peak_src = measured_peak()
    # The GEMM family's roofline from the graph-timed round itself (PDL
    # intact): its algorithmic bytes per launch over the round's time split
    # evenly across its launches.  The round also runs the attention and the
    # row kernels, so that duration is an upper bound of the GEMMs' own and
    # `achieved` a lower bound; it follows by hand from ms_per_step.
    gemm_per_round = prof_launch / args.steps if args.steps else 0
    bytes_per_round = prof_bytes / args.steps if args.steps else 0.0
    round_s = (ms / args.steps) / 1e3
    achieved = bytes_per_round / round_s / 1e9 if round_s > 0 else None
    event_gbs = prof_bytes / (prof_ms / 1e3) / 1e9 if prof_ms > 0 else None
    traffic = traffic_from_profiles()
    # verify cost against rows (plain greedy step = 1 row, round = 16 rows)
    t1row = None
    gg = torch.cuda.CUDAGraph()
    dec.prefill(prompt, w.n_new)
    with torch.cuda.graph(gg, stream=s):
        dec.verify(None)
    dec.prefill(prompt, w.n_new)
    for _ in range(3):
        gg.replay()
    torch.cuda.synchronize()
    start.record()
    for _ in range(args.steps):
        gg.replay()
    end.record()
    torch.cuda.synchronize()
    t1row = start.elapsed_time(end) / args.steps

    result = {
        "metric": METRIC, "value": round(value, 3), "unit": "rounds/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(t_max / args.steps, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic: seeded N(0,0.02) random-init bf16 weights, uniform-random prompt",
        "config": workload_config(
            w, world,
            timing="CUDA graph of one round replayed K times, CUDA events on the replay stream",
            l2="no flush: each round streams ~9.9 GB of weights, far larger than the 129 MB L2"),
        "accepted_tok_s": round(emitted / (t_max / 1e3), 3),
        "tokens_per_round": round(emitted / rounds_total, 4),
        "verify_ms_T1": round(t1row, 4),
        "round_ms_T16": round(t_max / args.steps, 4),
        "prefill": {"prompt_tokens": w.prompt_len, "ms": round(prefill_ms, 3),
                    "path": "dense tcgen05 forward of every prompt row; the last 16-row chunk then through the final norm into the round LM head"
                            if w.prompt_len > 16 else "16-row forwards"},
        "gpu_launches": launches_per_round * args.steps,
        "attention_form": {m: {2: "tcgen05", 1: "mma.sync split-KV", 0: "partial + combine"}[
            capi.dflash_attention_form(dec.ctx, i)] for i, m in ((0, "target"), (1, "drafter"))},
        "clocks": clocks,
        "roofline": {
            "bound": "hbm",
            "kernel": f"gemm_skinny_kernel (the {gemm_per_round:.0f} weight-streaming GEMM launches "
                      "of a round)",
            "achieved": round(achieved, 1) if achieved else None, "peak": peak,
            "peak_source": peak_src, "unit": "GB/s",
            "frac": round(achieved / peak, 4) if achieved else None,
            "traffic": traffic.get("dram_bytes_per_launch") if traffic else None,
            "traffic_source": traffic.get("summary") if traffic else
                              "null: no ncu capture of the current GEMM kernel",
            "bytes_per_launch": round(bytes_per_round / gemm_per_round) if gemm_per_round else None,
            "launch_us": round(round_s * 1e6 / gemm_per_round, 3) if gemm_per_round else None,
            "bytes_per_round": bytes_per_round,
            "event_timed_gbs": round(event_gbs, 1) if event_gbs else None,
            "note": "achieved = the GEMMs' algorithmic bytes per launch / (graph-timed round time "
                    "/ GEMM launches per round), i.e. bytes_per_round / ms_per_step: the round also "
                    "holds the attention and row kernels, so this is a lower bound of the GEMMs' "
                    "own rate.  event_timed_gbs: each GEMM bracketed by CUDA event nodes (which "
                    "break the dependent-launch overlap), another lower bound",
        },
    }
    if args.layers:
        result["config"]["workload"] += f" [DEBUG: target layers overridden to {args.layers}]"

    if not args.no_e2e:
        result["e2e"] = e2e_measure(dec, w, prompt, world, barrier)
    if want_cpu:
        cpu_leg = CpuBaseline()
    del g, gp, gg            # graphs hold event nodes of this context: drop them first
    torch.cuda.synchronize()
    if not args.no_workloads and not args.layers:
        dec.close()
        result["acceptance_injected"] = measure_injected(w, model_for_sweep)
        inj16 = result["acceptance_injected"]["by_block"].get("16")
        if inj16:
            result["accepted_tok_s_injected"] = inj16["accepted_tok_s"]
        result["workloads"] = measure_workloads(args.steps, args.warmup, model_for_sweep)
        result["workloads"]["multi_sequence"] = measure_batch(w, model_for_sweep, args.steps,
                                                              args.warmup)
    if cpu_leg is not None:                     # the oracle baseline: N = 1 only
        result["cpu_baseline"] = cpu_leg.finish()
    if rank == 0:
        print(json.dumps(result), flush=True)
    dec.close()
    if world > 1:
        dist.destroy_process_group()


def _graph_time(fn, steps, warmup, stream=None):
    """Captures fn() once as a CUDA graph; returns ms per replay (events)."""
    import torch
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        fn()
    for _ in range(warmup):
        g.replay()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(steps):
        g.replay()
    b.record()
    torch.cuda.synchronize()
    return a.elapsed_time(b) / steps, g


def _gemm_bytes_per_call(dec, fn):
    """Algorithmic GEMM bytes of one call of fn (library's own accounting)."""
    import torch
    from block_diffusion_speculative_gather_gb300 import capi
    capi.dflash_profile(dec.ctx, 1)
    fn()
    torch.cuda.synchronize()
    p = capi.dflash_profile(dec.ctx, 0)
    return p.gemm_bytes, p.gemm_ms, p.gemm_launches


def measure_workloads(steps, warmup, base_model):
    """The other workloads, each reported beside the round: drafter alone
    (bf16, 1024 tap rows, block 16), INT4 drafter (16384 tap rows, window
    2048, block 8), hc tap reduce (4 x 4096 x hc 4 streams at 4 layers), and
    the verify sweep T = 1..16 over a 16384-position synthetic KV cache."""
    import torch
    from block_diffusion_speculative_gather_gb300 import capi, synth
    from block_diffusion_speculative_gather_gb300.configs import (DRAFT_BF16, DRAFT_INT4, HC_SWEEP,
                                                                  HC_TAP)
    from block_diffusion_speculative_gather_gb300.runtime import DFlash
    peak, _ = measured_peak()
    out = {}
    # --- drafter alone, bf16 and INT4
    for w in (DRAFT_BF16, DRAFT_INT4):
        m = synth.ModelTensors(w)
        dec = DFlash(w, m)
        m_keep = m
        del m
        taps = synth.tap_rows(w.n_ctx, w.n_taps * w.hidden)
        ext = taps.view(w.n_ctx, w.n_taps, w.hidden).permute(1, 0, 2).contiguous()
        del taps
        torch.cuda.synchronize()
        ext = ext.to("cuda")   # the tap rows resident in HBM, as they are when a target made them
        dec.prefill_taps(ext, hc=1, first_token=17, max_new=64)   # warm-up (first-launch costs)
        torch.cuda.synchronize()
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0 = time.perf_counter()
        ev0.record()
        dec.prefill_taps(ext, hc=1, first_token=17, max_new=64)
        ev1.record()
        torch.cuda.synchronize()
        prefill_host_s = time.perf_counter() - t0
        prefill_s = ev0.elapsed_time(ev1) / 1e3
        # the same ingest as 16-row chunks through the round's kernels, timed the same way
        os.environ["DFLASH_DENSE_INGEST"] = "0"
        try:
            dchunk = DFlash(w, m_keep)
        finally:
            del os.environ["DFLASH_DENSE_INGEST"]
        dchunk.prefill_taps(ext, hc=1, first_token=17, max_new=64)
        torch.cuda.synchronize()
        ev0.record()
        dchunk.prefill_taps(ext, hc=1, first_token=17, max_new=64)
        ev1.record()
        torch.cuda.synchronize()
        chunked_s = ev0.elapsed_time(ev1) / 1e3
        dchunk.check()
        dchunk.close()
        del dchunk, m_keep
        del ext
        dec.draft()
        torch.cuda.synchronize()
        gb, gms, gl = _gemm_bytes_per_call(dec, dec.draft)
        ms, gdraft = _graph_time(dec.draft, steps, warmup)
        del gdraft
        ctx_rows = min(w.n_ctx, w.window) if w.window else w.n_ctx
        kv_bytes = w.drf_layers * 2 * w.n_kv * (ctx_rows + w.block) * w.head_dim * 2
        total = gb + kv_bytes
        dec.check()
        # prefill of the committed context window: fc over the window's tap
        # rows + context k/v of every draft layer (dense work, run here as
        # 16-row chunks of the round's kernels)
        win_rows = ctx_rows
        prefill_flop = 2.0 * win_rows * (w.n_taps * w.hidden * w.hidden +
                                         w.drf_layers * w.hidden * 2 * w.n_kv * w.head_dim)
        out[w.name] = {
            "window_prefill": {"rows": win_rows, "s": round(prefill_s, 5),
                               "host_s": round(prefill_host_s, 5),
                               "timing": "CUDA events on the launching stream, tap rows already in HBM",
                               "tflops": round(prefill_flop / prefill_s / 1e12, 2),
                               "chunked_16_rows_s": round(chunked_s, 5),
                               "chunked_16_rows_tflops": round(prefill_flop / chunked_s / 1e12, 2),
                               "path": "dense tcgen05 GEMM in 1024-row passes (fc bf16; context K/V " +
                                       ("f16 from the INT4 weights dequantised)" if w.drf_int4 else "bf16)")},
            "draft_rounds_s": round(1e3 / ms, 2), "ms_per_round": round(ms, 4),
            "bytes_per_round": int(total), "hbm_gbs": round(total / (ms / 1e3) / 1e9, 1),
            "frac_of_peak": round(total / (ms / 1e3) / 1e9 / peak, 4),
            "gemm_gbs_event_timed": round(gb / (gms / 1e3) / 1e9, 1) if gms else None,
            "gemm_launches": gl, "block": w.block, "context_rows": w.n_ctx, "window": w.window,
            "weights": "INT4 g64 + bf16 scales (projections), bf16 LM head" if w.drf_int4
                       else "bf16",
        }
        dec.close()
        del dec
        torch.cuda.empty_cache()
    # --- hc tap reduce
    hc = HC_TAP
    rows_res = {}
    for rows in hc["rows"]:
        streams = [torch.randn(rows, hc["hc"] * hc["hidden"], device="cuda",
                               generator=torch.Generator("cuda").manual_seed(2)).to(torch.bfloat16)
                   for _ in range(hc["n_layers"])]
        outb = torch.empty(rows, hc["n_layers"] * hc["hidden"], device="cuda")
        fn = lambda: capi.dflash_tap_reduce(streams, rows, hc["hc"], hc["hidden"], outb)
        ms, gtap = _graph_time(fn, max(steps, 20), warmup)
        del gtap
        nbytes = rows * hc["n_layers"] * hc["hidden"] * (hc["hc"] * 2 + 4)
        rows_res[str(rows)] = {"us": round(ms * 1e3, 2), "bytes": nbytes,
                               "gbs": round(nbytes / (ms / 1e3) / 1e9, 1)}
    out["hc_tap"] = {"hc": hc["hc"], "hidden": hc["hidden"], "tap_layers": hc["n_layers"],
                     "by_rows": rows_res}
    # --- the e2e round with every model 4-bit: target layers, drafter layers
    #     and the LM head in INT4 group-64 (quantised on the device from the
    #     same bf16 draws), natural acceptance
    from block_diffusion_speculative_gather_gb300.configs import E2E_BF16
    w4 = E2E_BF16.with_(name="e2e_int4", tgt_int4=True, lm_int4=True, drf_int4=True)
    dec = DFlash(w4, base_model)
    prompt = torch.from_numpy(synth.uniform_ids(w4.prompt_len, w4.vocab))
    dec.prefill(prompt, w4.n_new)
    torch.cuda.synchronize()
    pe0, pe1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    pe0.record()
    dec.prefill(prompt, w4.n_new)   # dense: INT4 matrices dequantised to f16 layer by layer
    pe1.record()
    torch.cuda.synchronize()
    prefill4_ms = pe0.elapsed_time(pe1)
    dec.verify(dec.draft())
    torch.cuda.synchronize()
    gb, _, gl = _gemm_bytes_per_call(dec, lambda: dec.verify(dec.draft()))
    dec.prefill(prompt, w4.n_new)
    ms, gr4 = _graph_time(lambda: dec.verify(dec.draft()), steps, warmup)
    del gr4
    dec.check()
    kv_bytes = (w4.tgt_layers * w4.n_kv * 2 * (w4.prompt_len + w4.block) * w4.head_dim * 2 +
                w4.drf_layers * w4.n_kv * 2 * (w4.prompt_len + w4.block) * w4.head_dim * 2)
    out["e2e_int4"] = {"rounds_s": round(1e3 / ms, 2), "ms_per_round": round(ms, 4),
                       "prefill_ms": round(prefill4_ms, 3),
                       "bytes_per_round": int(gb + kv_bytes), "gemm_launches": gl,
                       "hbm_gbs": round((gb + kv_bytes) / (ms / 1e3) / 1e9, 1),
                       "frac_of_peak": round((gb + kv_bytes) / (ms / 1e3) / 1e9 / peak, 4),
                       "weights": "INT4 g64 + bf16 scales: target and drafter projections and "
                                  "the LM head; embedding gather and fc bf16"}
    dec.close()
    # --- the e2e bf16 round with the opt-in tcgen05 attention (tensor-memory
    #     accumulators; splits of two chunks at this cache size)
    os.environ["DFLASH_ATTN_TC"] = "1"
    try:
        dec = DFlash(E2E_BF16, base_model)
    finally:
        del os.environ["DFLASH_ATTN_TC"]
    dec.prefill(prompt, E2E_BF16.n_new)
    dec.verify(dec.draft())
    dec.prefill(prompt, E2E_BF16.n_new)
    ms, gtc = _graph_time(lambda: dec.verify(dec.draft()), steps, warmup)
    del gtc
    dec.check()
    # the same prompt prefill as 16-row forwards of the round's kernels
    os.environ["DFLASH_DENSE_PREFILL"] = "0"
    try:
        dpc = DFlash(E2E_BF16, base_model)
    finally:
        del os.environ["DFLASH_DENSE_PREFILL"]
    dpc.prefill(prompt, E2E_BF16.n_new)
    torch.cuda.synchronize()
    pe0, pe1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    pe0.record()
    dpc.prefill(prompt, E2E_BF16.n_new)
    pe1.record()
    torch.cuda.synchronize()
    out["e2e_bf16_prefill_16_row_forwards"] = {"prompt_tokens": E2E_BF16.prompt_len,
                                               "ms": round(pe0.elapsed_time(pe1), 3)}
    dpc.check()
    dpc.close()
    del dpc
    out["e2e_bf16_attention_tcgen05"] = {
        "rounds_s": round(1e3 / ms, 2), "ms_per_round": round(ms, 4),
        "attention_form": {1: "mma.sync split-KV", 2: "tcgen05"}.get(capi.dflash_attention_form(dec.ctx, 0)),
        "note": "same round as the headline line with DFLASH_ATTN_TC=1"}
    dec.close()
    # --- the dense tcgen05 GEMM alone, at the window-ingest shapes
    bf16_peak, bf16_src = 1900.0, "fallback"
    try:
        pk = json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))
        if pk.get("bf16_tflops"):
            bf16_peak, bf16_src = float(pk["bf16_tflops"]), "measured (bf16_tflops, burst)"
    except Exception:
        pass
    dense = {}
    for m, n, k, split, what in [(2048, 2560, 12800, False, "fc over a 2048-row window (5 taps)"),
                                 (2048, 2048, 2560, True, "context K/V of one draft layer, hi + lo input")]:
        gen = torch.Generator(device="cuda").manual_seed(9)
        wd = (torch.randn(n, k, device="cuda", generator=gen) * 0.02).to(torch.bfloat16)
        xd = torch.randn(m, k, device="cuda", generator=gen).to(torch.bfloat16)
        xl = (torch.randn(m, k, device="cuda", generator=gen) * 2 ** -9).to(torch.bfloat16) if split else None
        yd = torch.empty(m, n, device="cuda")
        errw = torch.zeros(2, dtype=torch.int32, device="cuda")
        ms, gd = _graph_time(lambda: capi.dflash_linear_dense(wd, xd, yd, errw, x_lo=xl), max(steps, 20),
                             warmup)
        del gd
        assert errw.tolist() == [0, 0]
        flop = 2.0 * m * n * k * (2 if split else 1)
        tf = flop / (ms / 1e3) / 1e12
        dense[f"{m}x{n}x{k}" + ("_hilo" if split else "")] = {
            "what": what, "us": round(ms * 1e3, 2), "tflops": round(tf, 1),
            "frac_of_bf16_peak": round(tf / bf16_peak, 4)}
        del wd, xd, xl, yd
    out["dense_gemm_tcgen05"] = {"peak_tflops": bf16_peak, "peak_source": bf16_src,
                                 "note": "inputs stay in L2 across replays; the kernel is tensor-bound",
                                 "by_shape": dense}
    # --- verify sweep over a 16384-position synthetic KV cache
    w = HC_SWEEP
    dec = DFlash(w, base_model)
    kv = dec.kv_target.view(torch.float16)
    gen = torch.Generator("cuda").manual_seed(3)
    chunk = 1 << 26
    for i in range(0, kv.numel(), chunk):
        kv[i:i + chunk].normal_(generator=gen)
    n = w.prompt_len
    sweep = {}
    drafts = torch.randint(0, w.vocab, (w.block - 1,), dtype=torch.int32, device="cuda")
    for T in (1, 2, 4, 8, 16):
        def fn(T=T):
            dec.adopt_kv(n, 17, T + 1)
            dec.verify(drafts if T > 1 else None)
        ms, gsw = _graph_time(fn, steps, warmup)
        del gsw
        sweep[str(T)] = round(ms, 4)
    dec.check()
    kvb = 36 * 2 * w.n_kv * n * w.head_dim * 2
    out["verify_sweep_16k"] = {"ms_by_T": sweep, "T16_over_T1": round(sweep["16"] / sweep["1"], 3),
                               "kv_positions": n, "kv_bytes": kvb}
    dec.close()
    return out


def measure_batch(w, model, steps, warmup, sizes=(1, 8, 16)):
    """The many-sequence round (dflash_batch_*): S independent sequences of
    the e2e workload (1024-token prompts, one per seed), one batched draft
    and one batched verify per round on the dense tcgen05 GEMM; CUDA-graph
    timed, natural acceptance.  Aggregate rounds/s = S x batched rounds/s."""
    import torch
    from block_diffusion_speculative_gather_gb300 import synth
    from block_diffusion_speculative_gather_gb300.runtime import DFlashBatch
    out = {}
    for S in sizes:
        dec = DFlashBatch(w, model, S)
        prompts = [torch.from_numpy(synth.uniform_ids(w.prompt_len, w.vocab, seed=100 + i))
                   for i in range(S)]
        dec.prefill(prompts, w.n_new)
        dec.verify(dec.draft())
        dec.prefill(prompts, w.n_new)
        torch.cuda.synchronize()
        e0 = sum(dec.stats(i).emitted for i in range(S))
        ms, gb = _graph_time(lambda: dec.verify(dec.draft()), steps, warmup)
        del gb
        e1 = sum(dec.stats(i).emitted for i in range(S))
        dec.check()
        emitted = (e1 - e0) / (steps + warmup)     # per batched round, every sequence
        out[str(S)] = {"ms_per_batched_round": round(ms, 4),
                       "rounds_s_aggregate": round(S * 1e3 / ms, 2),
                       "tokens_s_aggregate": round(emitted * 1e3 / ms, 2),
                       "verify_rows_per_round": 16 * S}
        dec.close()
        del dec
        torch.cuda.empty_cache()
    return {"by_S": out, "acceptance": "natural (random-init drafter: ~1 token per sequence-round)",
            "path": "dense tcgen05 GEMM over 16 S rows (bf16 hi/lo planes, k-splits from N and K), "
                    "per-sequence attention, acceptance and tap commit"}


# Injected acceptance (a measurement device): per round the drafts are the
# greedy continuation with the first mismatch at a drawn position, so the
# verify accepts a realistic number of drafts while the drafter still runs.
# Position j of the block survives with probability ACCEPT_CONTINUE given
# that j - 1 did; 0.83 puts the mean accepted length at 5.59 tokens per
# round at block 16, the middle of the pages' reported range.
ACCEPT_CONTINUE = 0.83


def injected_schedule(g, n_new, B, prompt_len, max_seq, vocab, seed, adaptive=False):
    """Rounds of an injected run: (block length, draft row [B-1]) per round
    and the tokens they emit, following the device's block-length rule (with
    `adaptive`, the device's cap: 4 / 8 / 16 rows from the halving average of
    the accepted drafts, fp32)."""
    import numpy as np
    rng = np.random.default_rng(seed)
    gen, n = 1, prompt_len
    rows, emitted = [], []
    ema = np.float32(B - 1)
    while gen < n_new and n < max_seq:
        cap = B
        if adaptive:
            cap = min(B, 4 if ema < np.float32(1.5) else (8 if ema < np.float32(4.5) else 16))
        bl = min(cap, n_new - gen, max_seq - n)
        a = 0
        while a < bl - 1 and rng.random() < ACCEPT_CONTINUE:
            a += 1
        row = [int(g[min(gen + j, len(g) - 1)]) for j in range(B - 1)]   # correct drafts d_1..
        if a < bl - 1:
            row[a] = (row[a] + 1) % vocab                                # first mismatch
        rows.append(row)
        emitted.append(a + 1)
        ema = np.float32(0.5) * ema + np.float32(0.5) * np.float32(a)
        gen += a + 1
        n += a + 1
    return rows, emitted


def measure_injected(w, model, blocks=(16, 8, 4, "16a"), reps=3):
    """Rounds/s and accepted tok/s with injected acceptance at each block
    size, CUDA-graph timed; the emitted tokens must equal greedy decoding."""
    import torch
    from block_diffusion_speculative_gather_gb300 import synth
    from block_diffusion_speculative_gather_gb300.runtime import DFlash
    prompt = torch.from_numpy(synth.uniform_ids(w.prompt_len, w.vocab))
    out = {"continue_prob": ACCEPT_CONTINUE, "by_block": {}}
    g = None
    for Bk in blocks:
        adaptive = isinstance(Bk, str)                 # "16a": block 16, adaptive cap
        B = int(str(Bk).rstrip("a"))
        wb = w.with_(block=B, adaptive_block=adaptive)
        dec = DFlash(wb, model)
        if g is None:
            g = dec.greedy(prompt, w.n_new)           # the reference stream
        rows, emitted = injected_schedule(g, w.n_new, B, w.prompt_len, w.max_seq, w.vocab, seed=7,
                                          adaptive=adaptive)
        R = len(rows)
        table = torch.tensor(rows, dtype=torch.int32, device="cuda")
        inj = torch.empty((1, B - 1), dtype=torch.int32, device="cuda")
        ridx = torch.zeros(1, dtype=torch.int64, device="cuda")
        log_t = torch.zeros((R + 1, B), dtype=torch.int32, device="cuda")
        log_n = torch.zeros((R + 1, 1), dtype=torch.int32, device="cuda")

        def round_fn():
            dec.draft()                                    # runs and is timed; ids replaced
            torch.index_select(table, 0, ridx, out=inj)
            toks, n = dec.verify(inj[0])
            log_t.index_copy_(0, ridx, toks[None])
            log_n.index_copy_(0, ridx, n.view(1, 1))
            ridx.add_(1)

        # Everything runs on the current stream in order (a context's calls
        # must never overlap); the graph is captured on a side stream that
        # first waits for it, and replays on the current stream.
        dec.prefill(prompt, w.n_new)
        ridx.zero_()
        round_fn()                                         # warm (eager) round
        torch.cuda.synchronize()
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        gr = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gr, stream=s):
            round_fn()
        torch.cuda.synchronize()
        best = None
        for _ in range(reps):
            dec.prefill(prompt, w.n_new)
            ridx.zero_()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            for _ in range(R):
                gr.replay()
            b.record()
            torch.cuda.synchronize()
            ms = a.elapsed_time(b)
            best = ms if best is None else min(best, ms)
        dec.check()
        st = dec.stats()
        profile = [round(st.accept_hist[j] / max(1, st.rounds), 3) for j in range(B - 1)]
        ln = log_n[:R, 0].cpu().tolist()
        lt = log_t[:R].cpu().tolist()
        toks = [g[0]]
        for r in range(R):
            toks.extend(lt[r][:ln[r]])
        lossless = toks[:len(g)] == g[:len(toks)] and ln == emitted
        total = sum(ln)
        out["by_block"][str(Bk) if not adaptive else f"{B}_adaptive"] = {
            "rounds": R, "rounds_s": round(R / (best / 1e3), 2),
            "accepted_tok_s": round(total / (best / 1e3), 2),
            "tokens_per_round": round(total / R, 3), "ms_per_round": round(best / R, 4),
            "accept_profile": profile, "lossless_vs_greedy": bool(lossless)}
        del gr
        dec.close()
    return out


E2E_ROUNDS_PER_REPLAY = 16


def e2e_measure(dec, w, prompt, world=1, barrier=lambda: None):
    """Host prompt in pinned memory -> tokens on the host, through the public
    Python API (DFlash.generate_graphed): H2D of the prompt, prefill, then
    rounds replayed from a CUDA graph of 16 rounds until w.n_new tokens; every
    round's emitted tokens and the progress words come back to pinned host
    memory with each replay (one host wait per replay).  With several
    replicas: the rounds and tokens of all ranks over the slowest rank's time."""
    import torch
    host_prompt = prompt.to(torch.int32).pin_memory()
    dec.generate_graphed(host_prompt.to("cuda"), w.n_new, E2E_ROUNDS_PER_REPLAY)   # capture
    torch.cuda.synchronize()
    barrier()
    t0 = time.perf_counter()
    dev_prompt = host_prompt.to("cuda", non_blocking=True)
    tokens = dec.generate_graphed(dev_prompt, w.n_new, E2E_ROUNDS_PER_REPLAY)
    torch.cuda.synchronize()
    dt = time.perf_counter() - t0
    rounds_rank = int(dec.stats().rounds)
    dt_ms, (rounds, n_tok) = reduce_over_ranks(world, "cuda", dt * 1e3, rounds_rank, len(tokens))
    dt = dt_ms / 1e3
    rounds, n_tok = int(rounds), int(n_tok)
    return {"value": round(rounds / dt, 3), "unit": "rounds/s",
            "tokens_per_s": round(n_tok / dt, 3), "rounds": rounds, "tokens": n_tok,
            "includes": "prompt H2D + 1024-token prefill + rounds to 512 tokens; each round's "
                        "tokens and the progress words D2H per 16-round graph replay",
            "h2d_bytes_per_step": round(host_prompt.numel() * 4 / max(1, rounds_rank), 2),
            "d2h_bytes_per_step": (w.block + 1) * 4 + round(16 / E2E_ROUNDS_PER_REPLAY, 2)}


# ----------------------------------------------------------------- reference arm

def run_reference(args):
    """The oracle arm: every step is one real speculative round of the e2e
    workload by the CPU oracle (OracleRounds: drafter forward, 16-row
    verify, acceptance, rollback, tap commit) from a synthetic 1024-position
    state, on the host's cores (BLAS threads as the library starts them)."""
    rank, world, _ = rank_info()
    if rank != 0:
        return
    from block_diffusion_speculative_gather_gb300.configs import E2E_BF16
    w = E2E_BF16
    tw, dw, cfg, _ = oracle_weights(w)
    rounds = OracleRounds(tw, dw, cfg, w.prompt_len)
    for _ in range(args.warmup):
        rounds.round()
    e0 = rounds.emitted
    c0 = os.times()
    t = 0.0
    for _ in range(args.steps):
        t += rounds.round()
    c1 = os.times()
    busy = ((c1.user - c0.user) + (c1.system - c0.system)) / t if t > 0 else 0.0
    v = args.steps / t
    sample = (f"each step one real round of the e2e workload by the oracle (drafter forward "
              f"re-projecting the tap context, 16-row verify of the 36-layer target, acceptance, "
              f"rollback, tap commit) from a synthetic 1024-position state; fp64 numpy, "
              f"{cpu_cores()} host cores, {busy:.1f} threads busy on average; host CPU "
              f"{host_cpu_model()}")
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": round(v, 6), "unit": "rounds/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(t / args.steps * 1e3, 1), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic (same generators as ours)",
        "config": workload_config(
            w, world,
            timing="CPU oracle (fp64) on the host cores, one real round per step, wall clock",
            l2="not applicable (host run)"),
        "accepted_tok_s": round((rounds.emitted - e0) / t, 6),
        "cpu_baseline": {"value": round(v, 6), "unit": "rounds/s", "cores": cpu_cores(),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(v, 6), "unit": "rounds/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }), flush=True)


def main():
    args = parse()
    if args.cpu_baseline_worker:
        cpu_baseline_worker()
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
