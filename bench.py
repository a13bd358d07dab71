#!/usr/bin/env python
"""Benchmark of the SPD per-cycle hot path on one GB300 (replicas on N GPUs).

A step is one greedy SPD decode of the workload's generation length after its prompt: a
length-only rollback to the post-prefill state (the rollback operator of the method) followed by
cycles until gen_len tokens are committed.  Inputs (weights, prompt KV, draft overrides) are
resident in HBM before the timed region; the weights (>= 3.4 GB per cycle) are larger than L2, so
no flush is needed between steps.  Prints ONE JSON line on rank 0.

Default workload: the 9B-class model (L 32, d 4096, 32 q / 8 kv heads x 128, ffn 12288, vocab
151936, bf16) at n = 8, Ls = 4, prompt 2048, 512 tokens, alpha 0.9 (its other acceptance rate, 0.5,
and the 1.5B-class, the 4B-class and the 4B-class 32K-context workloads are reported under extra
keys).

  python bench.py [--gpus N --steps K --warmup W --workload NAME --alpha A]
  python bench.py --impl reference      # the CPU oracle timed on the host cores
  python bench.py --profile-cycles K    # K eager SPD cycles, for ncu launch lists and captures
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "committed tokens/s (1 seq, greedy SPD n=8) and cycle HBM GB/s vs peak"
DEFAULT_WORKLOAD = "gqa9b_bf16_n8"
EXTRA_WORKLOADS = ("dense1.5b_bf16_n8", "gqa4b_bf16_n8", "gqa4b_bf16_n8_ctx32k")
SPEC_HBM_GBS = 8000.0
TRAFFIC_FILE = os.path.join("profiles", "step_kernel_traffic.json")


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="spd", choices=["spd", "reference"])
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--alpha", type=float, default=None)
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--extra", default=",".join(EXTRA_WORKLOADS),
                    help="comma-separated workloads measured briefly after the headline one ('' for none)")
    ap.add_argument("--profile-cycles", type=int, default=0,
                    help="profiling case: prefill, then this many SPD cycles as plain (non-graph) "
                         "launches of the step kernel, one per cycle; prints one summary line")
    return ap.parse_args()


def sources_sha1() -> str:
    """SHA-1 over the CUDA sources (.cu, .cuh) in name order."""
    import hashlib
    src = os.path.join(ROOT, "speculative_pipeline_decoding_gb300", "csrc")
    h = hashlib.sha1()
    for f in sorted(os.listdir(src)):
        if f.endswith((".cu", ".cuh")):
            with open(os.path.join(src, f), "rb") as fh:
                h.update(fh.read())
    return h.hexdigest()


def step_kernel_traffic_ratio(workload: str):
    """DRAM bytes / algorithmic bytes of one ncu-captured step-kernel launch of `workload`, from the
    machine-readable capture record under profiles/ -- only while the CUDA sources are the ones that
    were captured (else None)."""
    try:
        with open(os.path.join(ROOT, TRAFFIC_FILE)) as fh:
            rec = json.load(fh)
        if rec.get("workload") != workload or rec.get("sources_sha1") != sources_sha1():
            return None
        return float(rec["dram_bytes"]) / float(rec["algorithmic_bytes"])
    except (OSError, ValueError, KeyError, TypeError):
        return None


def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as fh:
            d = json.load(fh)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


# ------------------------------------------------------------------------------------------------
# clocks during the timed region
# ------------------------------------------------------------------------------------------------
class Clocks:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out = ""
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for nm, val in zip(names, parts[3:7]):
                if val.lower().startswith("active"):
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None,
                "samples": len(sm), "reasons": sorted(reasons)}


# ------------------------------------------------------------------------------------------------
# distributed plumbing (replicas only: no data-path collective)
# ------------------------------------------------------------------------------------------------
def dist_setup(args):
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    return world, rank, local


def aggregate_tokens_per_s(world: int, steps: int, gen: int, ms_max: float) -> float:
    """Whole-job committed tokens/s: every rank decodes `gen` tokens per step; the job takes as long
    as its slowest rank."""
    return world * steps * gen / (ms_max / 1e3)


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64,
                     device="cuda" if dist.get_backend() == "nccl" else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ------------------------------------------------------------------------------------------------
# the CPU oracle (baseline / reference arm)
# ------------------------------------------------------------------------------------------------
def oracle_refs(w):
    """The oracle's own greedy AR stream after the workload's prompt (stored by
    tests/golden/make_oracle_ar.py): the reference tokens of the seeded drafts when the oracle is
    timed, so that nothing it computes comes from the GPU."""
    sys.path.insert(0, os.path.join(ROOT, "tests", "golden"))
    import make_oracle_ar
    return make_oracle_ar.stream_for(w)


def oracle_run(w, alpha, params_cpu, prompt, ref_tokens):
    """The oracle's SPD run (prefill included, untimed) with the seeded drafts of `alpha`; positions
    beyond the stored reference stream get no override (raw drafts)."""
    from oracle import spd as ospd
    import spd_inputs as si
    target, pdm = ospd.build(w, params_cpu)
    P, G = len(prompt), w.gen_len
    first, last = P + 2, min(P + G, P + len(ref_tokens))
    modes = dict(zip(range(first, last + 1), si.override_modes(w.coin_seed, alpha, first, last)))
    ref = {q: int(ref_tokens[q - P - 1]) for q in range(first, last + 1)}
    return ospd.SPDRun(target, pdm, w.n_stages, w.pdm_layers, w.anchors, prompt, P + G + w.n_stages + 2,
                       modes, ref)


def oracle_sample(run, seconds, min_cycles):
    """Cycles of the oracle until `seconds` passed (and >= min_cycles); committed tokens / s."""
    c0 = len(run.committed)
    k0 = run.cycles
    t0 = time.perf_counter()
    while True:
        run.cycle()
        el = time.perf_counter() - t0
        if el >= seconds and run.cycles - k0 >= min_cycles:
            break
    return (len(run.committed) - c0) / el, run.cycles - k0, len(run.committed) - c0, el


def cpu_cores():
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


def _oracle_child(conn, name, alpha, seconds):
    """Spawned process: builds the oracle of `name` (CPU weights, untimed prefill of the whole prompt),
    waits for the parent's go (its GPU measurements are done), times a sample of SPD cycles and sends
    the cpu_baseline record."""
    try:
        import spd_inputs as si
        w = si.WORKLOADS[name]
        params = si.generate_weights(w, device="cpu")
        prompt = si.prompt_tokens(w).tolist()
        refs = oracle_refs(w)
        if refs is None:
            conn.send({"error": f"no stored oracle reference stream for {name}"})
            return
        t0 = time.perf_counter()
        run = oracle_run(w, alpha, params, prompt, refs)
        del params
        prep = time.perf_counter() - t0
        conn.send({"ready": True})
        if conn.recv() != "go":
            return
        tps, c, toks, el = oracle_sample(run, seconds, w.n_stages + 2)
        conn.send({"value": tps, "unit": "tokens/s", "cores": cpu_cores(), "kind": "oracle",
                   "sample": f"{c} SPD cycles of the fp32 numpy oracle after its untimed prefill of the "
                             f"{len(prompt)}-token prompt ({prep:.0f} s, overlapped with the GPU legs): "
                             f"{toks} tokens in {el:.1f} s"})
    except Exception as e:  # reported in the JSON line instead of a baseline
        conn.send({"error": repr(e)})


def bench_config(w, alpha, world):
    """The `config` object of both arms: the same keys for the same workload."""
    return {"workload": w.name, "prompt": w.prompt_len, "gen": w.gen_len, "alpha": alpha,
            "n_stages": w.n_stages, "pdm_layers": w.pdm_layers, "anchors": list(w.anchors),
            "l2": "inputs larger than L2: every cycle streams all weights (>= 3.4 GB)",
            "parallelism": f"replicas x{world}"}


def default_alpha(w, args):
    """The headline acceptance rate: --alpha, else the workload's highest."""
    return args.alpha if args.alpha is not None else max(w.alphas)


# ------------------------------------------------------------------------------------------------
# per-cycle accounting from the verification trace
# ------------------------------------------------------------------------------------------------
def cycle_states(P, n, accepts, n_cycles):
    """(t, fill, exited) of every cycle of a run, rebuilt from the ordered accept outcomes."""
    t, a, k, out = P + 1, 1, 0, []
    for _ in range(n_cycles):
        ex = a == n
        out.append((t, a, ex))
        if ex:
            ok = accepts[k] if k < len(accepts) else True
            k += 1
            if ok:
                t += 1
            else:
                t, a = t - n + 2, 1
        else:
            t, a = t + 1, a + 1
    return out


def main_reference(args):
    import spd_inputs as si
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if world > 1 and rank != 0:
        return 0
    w = si.WORKLOADS[args.workload]
    alpha = default_alpha(w, args)
    refs = oracle_refs(w)
    if refs is None:
        print(json.dumps({"impl": "reference", "unavailable": f"no stored oracle reference stream for {w.name}"}))
        return 0
    params_cpu = si.generate_weights(w, device="cpu")
    prompt = si.prompt_tokens(w).tolist()
    cycles_per_step = max(2, w.n_stages // 2)
    run = oracle_run(w, alpha, params_cpu, prompt, refs)
    del params_cpu
    for _ in range(w.n_stages):  # untimed pipeline fill: the first token exits after n cycles
        run.cycle()
    for _ in range(args.warmup):
        for _ in range(cycles_per_step):
            run.cycle()
    c0 = len(run.committed)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        for _ in range(cycles_per_step):
            run.cycle()
    el = time.perf_counter() - t0
    tokens = len(run.committed) - c0
    value = tokens / el
    cores = cpu_cores()
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * el / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic",
        "config": bench_config(w, alpha, world),
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                         "sample": f"{args.steps} steps x {cycles_per_step} SPD cycles of the fp32 "
                                   f"numpy oracle after its prefill and an untimed pipeline fill of "
                                   f"{w.n_stages} cycles ({tokens} tokens committed)"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))
    return 0


class GpuWorkload:
    """One workload's engine on the GPU: weights, prefill, its plain AR stream, seeded drafts."""

    def __init__(self, name, alpha, stream):
        import torch
        import spd_inputs as si
        import speculative_pipeline_decoding_gb300 as spd
        self.w = w = si.WORKLOADS[name]
        self.alpha = alpha
        self.P, self.G, self.n = w.prompt_len, w.gen_len, w.n_stages
        self.params = si.generate_weights(w, device="cuda")
        self.prompt = si.prompt_tokens(w).tolist()
        torch.cuda.synchronize()  # weights are written on torch's stream; the engine uses its own
        self.stream = stream
        self.eng = spd.Engine(spd.Config.from_workload(w), self.params, stream=stream)
        self.first = self.eng.prefill(self.prompt)
        ar, _ = self.eng.generate_ar(self.G)
        self.ar = ar.tolist()
        self.set_alpha(alpha)

    def set_alpha(self, alpha):
        self.alpha = alpha
        self.eng.set_acceptance(alpha, self.w.coin_seed, self.ar)

    def spd_step(self):
        self.eng.rollback(self.P, self.first)
        return self.eng.generate(self.G)

    def ar_step(self):
        self.eng.rollback(self.P, self.first)
        return self.eng.generate_ar(self.G)

    def step_bytes(self, cycles):
        """Algorithmic bytes of the last SPD run's cycles, rebuilt from its verification trace."""
        from speculative_pipeline_decoding_gb300 import binding as B
        trace = self.eng.dump(B.DUMP_TRACE)[:, : self.eng.state()["exits"]]
        accepts = [bool(x) for x in trace[1]]
        total = 0.0
        for (t, a, ex) in cycle_states(self.P, self.n, accepts, cycles):
            total += sum(self.eng.cycle_bytes(t, a, ex, True).values())
        return total

    def close(self):
        import torch
        self.eng.close()
        del self.params
        torch.cuda.empty_cache()


def main_spd(args):
    import numpy as np
    import torch
    import spd_inputs as si
    from speculative_pipeline_decoding_gb300 import binding as B
    from speculative_pipeline_decoding_gb300 import build_ext

    world, rank, local = dist_setup(args)
    w = si.WORKLOADS[args.workload]
    alpha = default_alpha(w, args)
    # the CPU oracle's baseline: its process is spawned before the first GPU call and prepares its
    # (long, untimed) prefill while the GPU legs run; its timed sample starts after them
    child = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        import multiprocessing as mp
        ctx = mp.get_context("spawn")
        conn, child_conn = ctx.Pipe()
        child = ctx.Process(target=_oracle_child, args=(child_conn, w.name, alpha, args.cpu_seconds), daemon=True)
        child.start()
    build_ext.build()
    torch.cuda.set_device(local)
    stream = torch.cuda.Stream()
    W = GpuWorkload(w.name, alpha, stream)
    P, G, n = W.P, W.G, W.n
    eng = W.eng

    def timed(fn, K, Wm, clocks=None, tag="spd_other"):
        for _ in range(Wm):
            fn()
        barrier(world)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        if clocks:
            clocks.start()
        launches = 0
        torch.cuda.nvtx.range_push(tag)
        e0.record(stream)
        last = None
        for _ in range(K):
            last = fn()
            launches += last[1]["kernel_launches"] + 1  # + the rollback kernel
        e1.record(stream)
        torch.cuda.synchronize()
        torch.cuda.nvtx.range_pop()
        ck = clocks.stop() if clocks else None
        barrier(world)
        return e0.elapsed_time(e1), last, launches, ck

    # --- main measurement: SPD, one step-kernel launch per cycle replayed from a CUDA graph ---
    toks, _ = W.spd_step()
    lossless = toks.tolist() == W.ar
    clk = Clocks(local)
    ms, (toks, st), launches, clocks = timed(W.spd_step, args.steps, args.warmup, clk, tag="spd_timed")
    ms_max = max_over_ranks(ms, world)
    cycles = st["cycles"]
    value = aggregate_tokens_per_s(world, args.steps, G, ms_max)
    ms_step = ms_max / args.steps
    step_bytes = W.step_bytes(cycles)
    cycle_gbs = step_bytes / (ms_step / 1e3) / 1e9
    Kx = 3

    # --- the workload's other acceptance rates (same kernels, same bytes per full cycle) ---
    other_alphas = {}
    for a2 in w.alphas:
        if a2 == alpha:
            continue
        W.set_alpha(a2)
        ms2, (toks2, st2), _, _ = timed(W.spd_step, Kx, 1)
        b2 = W.step_bytes(st2["cycles"])
        other_alphas[str(a2)] = {"tokens_per_s": Kx * G / (ms2 / 1e3), "cycles_per_step": st2["cycles"],
                                 "rejects_per_step": st2["rejects"], "cycle_ms": ms2 / Kx / st2["cycles"],
                                 "cycle_hbm_frac": b2 / (ms2 / Kx / 1e3) / 1e9 / measured_peaks()[0],
                                 "lossless_vs_ar": toks2.tolist() == W.ar}
    W.set_alpha(alpha)

    # --- AR from the same kernels ---
    ms_ar, _, _, _ = timed(W.ar_step, Kx, 1)
    ar_tps = Kx * G / (ms_ar / 1e3)
    ar_bytes = sum(eng.cycle_bytes(P + G // 2, n, True, False).values())  # one token through all layers

    # --- target only (no draft module), and draft module serialised (its own phases first) ---
    step = B.OPT_STEP | B.OPT_PDL | B.OPT_GRAPHS
    eng.set_options(step | B.OPT_TARGET_ONLY)
    ms_tgt, (toks_t, st_t), _, _ = timed(W.spd_step, Kx, 1)
    tgt_bytes = 0.0
    tr_t = eng.dump(B.DUMP_TRACE)[:, : eng.state()["exits"]]
    for (t, a, ex) in cycle_states(P, n, [bool(x) for x in tr_t[1]], st_t["cycles"]):
        tgt_bytes += sum(eng.cycle_bytes(t, a, ex, False).values())
    eng.set_options(step)
    ms_ser, _, _, _ = timed(W.spd_step, Kx, 1)
    # post-step schedule (the pages' scheduling ablation): the draft module after the target step,
    # on its output state; same cycles and committed stream, drafting no longer hidden
    eng.set_options(step | B.OPT_POST_STEP)
    ms_post, (toks_p, st_p), _, _ = timed(W.spd_step, Kx, 1)
    t_cycle = ms_step / cycles
    t_tgt = ms_tgt / Kx / st_t["cycles"]
    t_ser = ms_ser / Kx / cycles
    t_post = ms_post / Kx / st_p["cycles"]
    post_tps = Kx * G / (ms_post / 1e3)
    post_lossless = toks_p.tolist() == W.ar and st_p["cycles"] == cycles
    # sampled decoding (T = 1, top-k 50, rejection-sampling verification) on seeded uniforms: the
    # acceptance is the draft module's (random weights: rarely), so this times cycles with the
    # sampling control step and mostly refills
    eng.set_options(B.OPT_DEFAULT)
    us = si.sampling_uniforms(w.coin_seed + 1, P + 1, P + G + n + 2)
    eng.set_sampling(1.0, 50, P + 1, np.array([us[k] for k in si.SAMPLING_STREAMS], dtype=np.float32))
    ms_smp, (_, st_s), _, _ = timed(W.spd_step, 2, 1)
    eng.set_sampling(0.0)
    t_smp = ms_smp / 2 / st_s["cycles"]
    smp_line = {"temperature": 1.0, "top_k": 50, "cycle_ms": t_smp, "tokens_per_s": 2 * G / (ms_smp / 1e3),
                "accept_rate": 1.0 - st_s["rejects"] / max(1, st_s["exits"])}

    # --- instrumented pass: phase timers of the step kernel (CTA 0, grid barrier to grid barrier),
    # draft module in its own phases so that its time is separate ---
    eng.set_options(B.OPT_STEP | B.OPT_PDL)
    eng.time_kernels(True)
    W.spd_step()
    kt = eng.kernel_times()
    eng.time_kernels(False)
    eng.set_options(B.OPT_DEFAULT)
    pdm_alone = sum(v[1] for k, v in kt.items() if k.startswith("draft_")) / cycles
    hidden = 1.0 - (t_cycle - t_tgt) / pdm_alone if pdm_alone > 0 else None
    # roofline of the dominant kernel: the step kernel itself (one launch per cycle); its bytes are
    # the cycle's algorithmic bytes, its duration the CUDA-event cycle time of the timed region
    peak, peak_src = measured_peaks()
    achieved = step_bytes / cycles / (t_cycle / 1e3) / 1e9
    traffic_ratio = step_kernel_traffic_ratio(w.name)

    # --- end to end through the public API with host buffers ---
    prompt_np = np.asarray(W.prompt, dtype="int32")
    ar_np = np.asarray(W.ar, dtype="int32")

    def e2e_step():
        eng.prefill(prompt_np)
        eng.set_acceptance(alpha, w.coin_seed, ar_np)
        return eng.generate(G)  # copies the committed tokens into a host array

    ms_e2e, (toks_e2e, _), _, _ = timed(e2e_step, Kx, 1)
    e2e_val = aggregate_tokens_per_s(world, Kx, G, max_over_ranks(ms_e2e, world))
    lossless = lossless and toks_e2e.tolist() == W.ar
    W.close()

    # --- the other workloads, briefly (same kernels): tokens/s, AR, cycle time, roofline fraction ---
    extra = {}
    if rank == 0:
        for name in [x for x in args.extra.split(",") if x and x != w.name]:
            if name not in si.WORKLOADS:
                continue
            X = GpuWorkload(name, max(si.WORKLOADS[name].alphas), stream)
            mx, (tx, sx), _, _ = timed(X.spd_step, Kx, 1)
            bx = X.step_bytes(sx["cycles"])
            ma, _, _, _ = timed(X.ar_step, 2, 1)
            X.eng.set_options(step | B.OPT_TARGET_ONLY)
            mt, (_, stt), _, _ = timed(X.spd_step, 2, 1)
            X.eng.set_options(B.OPT_DEFAULT)
            extra[name] = {"alpha": X.alpha, "tokens_per_s": Kx * X.G / (mx / 1e3),
                           "ar_tokens_per_s": 2 * X.G / (ma / 1e3), "cycles_per_step": sx["cycles"],
                           "cycle_ms": mx / Kx / sx["cycles"], "target_only_cycle_ms": mt / 2 / stt["cycles"],
                           "cycle_hbm_gbs": bx / (mx / Kx / 1e3) / 1e9,
                           "cycle_hbm_frac": bx / (mx / Kx / 1e3) / 1e9 / peak,
                           "lossless_vs_ar": tx.tolist() == X.ar}
            X.close()

    # --- CPU oracle baseline (rank 0, single GPU only): the child's timed sample starts now ---
    cpu = None
    if child is not None:
        try:
            msg = conn.recv() if conn.poll(1800) else {"error": "oracle prefill did not finish in 30 min"}
            if msg.get("ready"):
                conn.send("go")
                msg = conn.recv() if conn.poll(600) else {"error": "oracle sample did not finish"}
            cpu = msg if "error" not in msg else {"value": None, "unit": "tokens/s", "kind": "oracle",
                                                  "cores": cpu_cores(), "sample": msg["error"]}
        finally:
            child.join(timeout=30)
            if child.is_alive():
                child.terminate()

    if rank != 0:
        return 0
    kern = {k: round(v[1] / cycles, 4) for k, v in kt.items() if v[0]}
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": w.model.dtype, "data": "synthetic",
        "config": bench_config(w, alpha, world),
        "roofline": {"bound": "hbm", "kernel": "step_kernel (one SPD cycle per launch)",
                     "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "peak_source": peak_src,
                     "traffic": None if traffic_ratio is None else traffic_ratio * step_bytes / cycles,
                     "traffic_source": f"ncu dram bytes / algorithmic bytes of one captured launch ({TRAFFIC_FILE})"
                                       " x bytes_per_launch" if traffic_ratio is not None
                                       else "no capture of the current sources for this workload",
                     "launches": args.steps * cycles, "bytes_per_launch": step_bytes / cycles},
        "cpu_baseline": cpu,
        "e2e": {"value": e2e_val, "unit": "tokens/s", "h2d_bytes_per_step": 4 * P + 5 * (G - 1),
                "d2h_bytes_per_step": 4 * G, "includes": "prefill + decode per step"},
        "gpu_launches": launches,
        "clocks": clocks,
        "spd": {"lossless_vs_ar": lossless, "cycles_per_step": cycles, "rejects_per_step": st["rejects"],
                "cycle_ms": t_cycle, "cycle_hbm_gbs": cycle_gbs, "cycle_hbm_frac": cycle_gbs / peak,
                "cycle_hbm_frac_spec": cycle_gbs / SPEC_HBM_GBS, "alg_bytes_per_step": step_bytes,
                "ar_tokens_per_s": ar_tps, "ar_hbm_frac": ar_bytes * ar_tps / 1e9 / peak,
                "spd_over_ar": value / world / ar_tps,
                "spd_over_ar_byte_model": 1.0 / (alpha + (1 - alpha) * (n + 1) / 2),
                "target_only_cycle_ms": t_tgt,
                "target_only_hbm_frac": tgt_bytes / st_t["cycles"] / (t_tgt / 1e3) / 1e9 / peak,
                "serial_pdm_cycle_ms": t_ser,
                "post_step": {"cycle_ms": t_post, "tokens_per_s": post_tps,
                              "lossless_and_same_cycles": post_lossless},
                "sampled_t1": smp_line,
                "pdm_alone_ms_per_cycle": pdm_alone, "pdm_hidden_frac": hidden,
                "control_us": 1e3 * kt["control"][1] / max(1, kt["control"][0]),
                "phases_ms_per_cycle": kern,
                "other_alphas": other_alphas},
        "other_workloads": extra,
    }
    print(json.dumps(line))
    return 0


def main_profile(args):
    """Prefill, G - 1 plain AR steps (the reference stream for the draft overrides; the first token
    comes from the prefill), then K SPD cycles, all launched one by one without graphs.  Under a
    profiler the launch sequence is fixed: set-up and prefill kernels, G - 1 step-kernel launches
    (AR), then exactly one step-kernel launch per cycle, so `-k regex:step_kernel -s <G - 1 + c>`
    selects cycle c (c >= n: a full pipeline)."""
    import torch
    import spd_inputs as si
    import speculative_pipeline_decoding_gb300 as spd
    from speculative_pipeline_decoding_gb300 import binding as B
    from speculative_pipeline_decoding_gb300 import build_ext

    build_ext.build()
    w = si.WORKLOADS[args.workload]
    alpha = default_alpha(w, args)
    P, G = w.prompt_len, w.gen_len
    params = si.generate_weights(w, device="cuda")
    prompt = si.prompt_tokens(w).tolist()
    torch.cuda.synchronize()
    eng = spd.Engine(spd.Config.from_workload(w), params)
    eng.set_options(B.OPT_DEFAULT & ~B.OPT_GRAPHS)
    first = eng.prefill(prompt)
    ar, _ = eng.generate_ar(G)  # G - 1 step-kernel launches, one per token: the reference stream
    eng.rollback(P, first)
    eng.set_acceptance(alpha, w.coin_seed, ar)
    t0 = time.time()
    exits = 0
    st = eng.state()
    t_prev, a_prev = st["t"], st["a"]
    per_cycle = []  # (t, fill) before the cycle, exited, algorithmic bytes
    for _ in range(args.profile_cycles):
        info = eng.cycle()
        exits += info["exited"]
        nbytes = sum(eng.cycle_bytes(t_prev, a_prev, bool(info["exited"]), True).values())
        per_cycle.append([t_prev, a_prev, info["exited"], nbytes])
        t_prev, a_prev = info["t"], info["a"]
    torch.cuda.synchronize()
    print(json.dumps({"profile_cycles": args.profile_cycles, "ar_steps_before": G, "exits": exits,
                      "workload": w.name, "wall_s": time.time() - t0,
                      "cycles_t_fill_exited_bytes": per_cycle}))
    eng.close()
    return 0


def main():
    args = parse()
    if args.profile_cycles > 0:
        return main_profile(args)
    if args.impl == "reference":
        return main_reference(args)
    return main_spd(args)


if __name__ == "__main__":
    sys.exit(main())
