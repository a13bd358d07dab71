#!/usr/bin/env python
"""Benchmark of the SPD per-cycle hot path on one GB300 (replicas on N GPUs).

A step is one greedy SPD decode of the workload's generation length after its prompt: a
length-only rollback to the post-prefill state (the rollback operator of the method) followed by
cycles until gen_len tokens are committed.  Inputs (weights, prompt KV, draft overrides) are
resident in HBM before the timed region; the weights (>= 3.4 GB per cycle) are larger than L2, so
no flush is needed between steps.  Prints ONE JSON line on rank 0.

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
DEFAULT_WORKLOAD = "dense1.5b_bf16_n8"
SPEC_HBM_GBS = 8000.0


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
    ap.add_argument("--profile-cycles", type=int, default=0,
                    help="profiling case: prefill, then this many SPD cycles as plain (non-graph) "
                         "launches of the step kernel, one per cycle; prints one summary line")
    return ap.parse_args()


def step_kernel_traffic_ratio():
    """DRAM bytes / algorithmic bytes of one ncu-captured step-kernel launch, from the committed profile
    summary -- only while the CUDA sources are the ones that were profiled (else None)."""
    import hashlib
    src = os.path.join(ROOT, "speculative_pipeline_decoding_gb300", "csrc")
    prof = os.path.join(ROOT, "profiles", "step_kernel_dense1.5b_n8_sections.md")
    try:
        h = hashlib.sha1()
        for f in sorted(os.listdir(src)):
            if f.endswith((".cu", ".cuh")):
                with open(os.path.join(src, f), "rb") as fh:
                    h.update(fh.read())
        with open(prof) as fh:
            for line in fh:
                parts = line.split()
                if len(parts) == 4 and parts[0] == "traffic_ratio:" and parts[2] == "sources_sha1:":
                    return float(parts[1]) if parts[3] == h.hexdigest() else None
    except OSError:
        return None
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
def oracle_run(w, alpha, params_cpu, prompt, ar_tokens):
    from oracle import spd as ospd
    import spd_inputs as si
    target, pdm = ospd.build(w, params_cpu)
    P, G = len(prompt), w.gen_len
    first, last = P + 2, P + G
    modes = dict(zip(range(first, last + 1), si.override_modes(w.coin_seed, alpha, first, last)))
    ref = {q: int(ar_tokens[q - P - 1]) for q in range(first, last + 1)}
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
    import torch
    import spd_inputs as si
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if world > 1 and rank != 0:
        return 0
    w = si.WORKLOADS[args.workload]
    alpha = args.alpha if args.alpha is not None else w.alphas[0]
    params = si.generate_weights(w, device="cuda" if torch.cuda.is_available() else "cpu")
    params_cpu = {k: v.cpu() for k, v in params.items()}
    del params
    prompt = si.prompt_tokens(w).tolist()
    # the reference stream for the seeded drafts comes from the oracle itself (greedy AR)
    from oracle import model as om
    from oracle import spd as ospd
    cycles_per_step = max(2, w.n_stages // 2)
    need = min(w.gen_len, (args.warmup + args.steps) * cycles_per_step + 2 * w.n_stages + 2)
    target, _ = ospd.build(w, params_cpu)
    ar = om.greedy_ar(target, prompt, need)["tokens"]
    ar = ar + [0] * (w.gen_len - len(ar))  # positions the sample never reaches
    run = oracle_run(w, alpha, params_cpu, prompt, ar)
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
        "config": {"workload": w.name, "prompt": len(prompt), "gen": w.gen_len, "alpha": alpha,
                   "n_stages": w.n_stages, "pdm_layers": w.pdm_layers, "anchors": list(w.anchors)},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                         "sample": f"{args.steps} steps x {cycles_per_step} SPD cycles of the fp32 "
                                   f"numpy oracle after its prefill and an untimed pipeline fill of "
                                   f"{w.n_stages} cycles ({tokens} tokens committed)"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))
    return 0


def main_spd(args):
    import numpy as np
    import torch
    import spd_inputs as si
    import speculative_pipeline_decoding_gb300 as spd
    from speculative_pipeline_decoding_gb300 import binding as B
    from speculative_pipeline_decoding_gb300 import build_ext

    world, rank, local = dist_setup(args)
    build_ext.build()
    torch.cuda.set_device(local)
    w = si.WORKLOADS[args.workload]
    alpha = args.alpha if args.alpha is not None else w.alphas[0]
    m = w.model
    P, G, n = w.prompt_len, w.gen_len, w.n_stages
    params = si.generate_weights(w, device="cuda")
    prompt = si.prompt_tokens(w).tolist()
    stream = torch.cuda.Stream()
    torch.cuda.synchronize()  # weights are written on torch's stream; the engine uses its own
    eng = spd.Engine(spd.Config.from_workload(w), params, stream=stream)
    first = eng.prefill(prompt)
    ar, _ = eng.generate_ar(G)
    ar_list = ar.tolist()
    modes = si.override_modes(w.coin_seed, alpha, P + 2, P + G)
    eng.set_draft_override(P + 2, ar_list[1:], modes)

    def spd_step():
        eng.rollback(P, first)
        toks, st = eng.generate(G)
        return toks, st

    def ar_step():
        eng.rollback(P, first)
        toks, st = eng.generate_ar(G)
        return toks, st

    def timed(fn, K, W, clocks=None, tag="spd_other"):
        for _ in range(W):
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

    # --- main measurement: SPD, graphs, draft module on its own stream ---
    toks, _ = spd_step()
    lossless = toks.tolist() == ar_list
    clk = Clocks(local)
    ms, (toks, st), launches, clocks = timed(spd_step, args.steps, args.warmup, clk, tag="spd_timed")
    ms_max = max_over_ranks(ms, world)
    cycles = st["cycles"]
    value = aggregate_tokens_per_s(world, args.steps, G, ms_max)
    ms_step = ms_max / args.steps
    trace = eng.dump(B.DUMP_TRACE)[:, : eng.state()["exits"]]
    accepts = [bool(x) for x in trace[1]]
    states = cycle_states(P, n, accepts, cycles)
    bytes_kind = [0.0] * len(B.KIND_NAMES)
    for (t, a, ex) in states:
        cb = eng.cycle_bytes(t, a, ex, True)
        for k, name in enumerate(B.KIND_NAMES):
            bytes_kind[k] += cb[name]
    step_bytes = sum(bytes_kind)
    cycle_gbs = step_bytes / (ms_step / 1e3) / 1e9

    # --- AR from the same kernels ---
    ms_ar, _, _, _ = timed(ar_step, max(3, args.steps // 2), 2)
    ar_tps = max(3, args.steps // 2) * G / (ms_ar / 1e3)

    # --- target only (no draft module), and draft module serialised (its own phases first) ---
    step = B.OPT_STEP | B.OPT_PDL | B.OPT_GRAPHS
    eng.set_options(step | B.OPT_TARGET_ONLY)
    ms_tgt, (toks_t, st_t), _, _ = timed(spd_step, max(3, args.steps // 2), 1)
    eng.set_options(step)
    ms_ser, _, _, _ = timed(spd_step, max(3, args.steps // 2), 1)
    # post-step schedule (the pages' scheduling ablation): the draft module after the target step,
    # on its output state; same cycles and committed stream, drafting no longer hidden
    eng.set_options(step | B.OPT_POST_STEP)
    ms_post, (toks_p, st_p), _, _ = timed(spd_step, max(3, args.steps // 2), 1)
    Kx = max(3, args.steps // 2)
    t_cycle = ms_step / cycles
    t_tgt = ms_tgt / Kx / st_t["cycles"]
    t_ser = ms_ser / Kx / cycles
    t_post = ms_post / Kx / st_p["cycles"]
    post_tps = Kx * G / (ms_post / 1e3)
    post_lossless = toks_p.tolist() == ar_list and st_p["cycles"] == cycles
    # sampled decoding (T = 1, top-k 50, rejection-sampling verification) on seeded uniforms: the
    # acceptance is the draft module's (random weights: rarely), so this times cycles with the
    # sampling control step and mostly refills
    eng.set_options(B.OPT_DEFAULT)
    us = si.sampling_uniforms(w.coin_seed + 1, P + 1, P + G + n + 2)
    eng.set_sampling(1.0, 50, P + 1, np.array([us[k] for k in si.SAMPLING_STREAMS], dtype=np.float32))
    ms_smp, (_, st_s), _, _ = timed(spd_step, Kx, 1)
    eng.set_sampling(0.0)
    t_smp = ms_smp / Kx / st_s["cycles"]
    smp_line = {"temperature": 1.0, "top_k": 50, "cycle_ms": t_smp, "tokens_per_s": Kx * G / (ms_smp / 1e3),
                "accept_rate": 1.0 - st_s["rejects"] / max(1, st_s["exits"])}

    # --- instrumented pass: phase timers of the step kernel (CTA 0, grid barrier to grid barrier),
    # draft module in its own phases so that its time is separate ---
    eng.set_options(B.OPT_STEP | B.OPT_PDL)
    eng.time_kernels(True)
    spd_step()
    kt = eng.kernel_times()
    eng.time_kernels(False)
    eng.set_options(B.OPT_DEFAULT)
    pdm_alone = sum(v[1] for k, v in kt.items() if k.startswith("draft_")) / cycles
    hidden = 1.0 - (t_cycle - t_tgt) / pdm_alone if pdm_alone > 0 else None
    # roofline of the dominant kernel: the step kernel itself (one launch per cycle); its bytes are
    # the cycle's algorithmic bytes, its duration the CUDA-event cycle time of the timed region
    peak, peak_src = measured_peaks()
    achieved = step_bytes / cycles / (t_cycle / 1e3) / 1e9
    traffic_ratio = step_kernel_traffic_ratio()

    # --- end to end through the public API with host buffers ---
    prompt_np = __import__("numpy").asarray(prompt, dtype="int32")
    ref_np = ar_list[1:]

    def e2e_step():
        eng.prefill(prompt_np)
        eng.set_draft_override(P + 2, ref_np, modes)
        toks, st = eng.generate(G)  # copies the committed tokens into a host array
        return toks, st

    ms_e2e, (toks_e2e, _), _, _ = timed(e2e_step, max(3, args.steps // 2), 1)
    e2e_val = aggregate_tokens_per_s(world, max(3, args.steps // 2), G, max_over_ranks(ms_e2e, world))
    lossless = lossless and toks_e2e.tolist() == ar_list

    # --- CPU oracle baseline (rank 0, single GPU only) ---
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        params_cpu = {k: v.cpu() for k, v in params.items()}
        run = oracle_run(w, alpha, params_cpu, prompt, ar_list)
        tps, c, toks_c, el = oracle_sample(run, args.cpu_seconds, n + 2)
        cpu = {"value": tps, "unit": "tokens/s", "cores": cpu_cores(), "kind": "oracle",
               "sample": f"{c} SPD cycles of the fp32 numpy oracle after its (untimed) prefill: "
                         f"{toks_c} tokens in {el:.1f} s"}

    if rank != 0:
        return 0
    kern = {k: round(v[1] / cycles, 4) for k, v in kt.items() if v[0]}
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": m.dtype, "data": "synthetic",
        "config": {"workload": w.name, "prompt": P, "gen": G, "alpha": alpha, "n_stages": n,
                   "pdm_layers": w.pdm_layers, "anchors": list(w.anchors),
                   "l2": "inputs larger than L2: every cycle streams all weights (>=3.4 GB)",
                   "parallelism": f"replicas x{world}"},
        "roofline": {"bound": "hbm", "kernel": "step_kernel (one SPD cycle per launch)",
                     "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "peak_source": peak_src,
                     "traffic": None if traffic_ratio is None else traffic_ratio * step_bytes / cycles,
                     "traffic_source": "ncu dram bytes / algorithmic bytes of one captured launch "
                                       "(profiles/step_kernel_dense1.5b_n8_sections.md) x bytes_per_launch"
                                       if traffic_ratio is not None else "no capture of the current sources",
                     "launches": args.steps * cycles, "bytes_per_launch": step_bytes / cycles},
        "cpu_baseline": cpu,
        "e2e": {"value": e2e_val, "unit": "tokens/s", "h2d_bytes_per_step": 4 * P + 5 * (G - 1),
                "d2h_bytes_per_step": 4 * G, "includes": "prefill + decode per step"},
        "gpu_launches": launches,
        "clocks": clocks,
        "spd": {"lossless_vs_ar": lossless, "cycles_per_step": cycles, "rejects_per_step": st["rejects"],
                "cycle_ms": t_cycle, "cycle_hbm_gbs": cycle_gbs, "cycle_hbm_frac": cycle_gbs / peak,
                "cycle_hbm_frac_spec": cycle_gbs / SPEC_HBM_GBS, "alg_bytes_per_step": step_bytes,
                "ar_tokens_per_s": ar_tps, "spd_over_ar": value / world / ar_tps,
                "target_only_cycle_ms": t_tgt, "serial_pdm_cycle_ms": t_ser,
                "post_step": {"cycle_ms": t_post, "tokens_per_s": post_tps,
                              "lossless_and_same_cycles": post_lossless},
                "sampled_t1": smp_line,
                "pdm_alone_ms_per_cycle": pdm_alone, "pdm_hidden_frac": hidden,
                "control_us": 1e3 * kt["control"][1] / max(1, kt["control"][0]),
                "phases_ms_per_cycle": kern},
    }
    print(json.dumps(line))
    eng.close()
    return 0


def main_profile(args):
    """Prefill, G plain AR steps (the reference stream for the draft overrides), then K SPD cycles,
    all launched one by one without graphs.  Under a profiler the launch sequence is fixed: set-up
    and prefill kernels, G step-kernel launches (AR), then exactly one step-kernel launch per cycle,
    so `-k regex:step_kernel -s <G + warm-up cycles>` selects steady-state cycles."""
    import torch
    import spd_inputs as si
    import speculative_pipeline_decoding_gb300 as spd
    from speculative_pipeline_decoding_gb300 import binding as B
    from speculative_pipeline_decoding_gb300 import build_ext

    build_ext.build()
    w = si.WORKLOADS[args.workload]
    alpha = args.alpha if args.alpha is not None else w.alphas[0]
    P, G = w.prompt_len, w.gen_len
    params = si.generate_weights(w, device="cuda")
    prompt = si.prompt_tokens(w).tolist()
    torch.cuda.synchronize()
    eng = spd.Engine(spd.Config.from_workload(w), params)
    eng.set_options(B.OPT_DEFAULT & ~B.OPT_GRAPHS)
    first = eng.prefill(prompt)
    ar, _ = eng.generate_ar(G)  # G step-kernel launches, one per token: the reference stream
    eng.rollback(P, first)
    modes = si.override_modes(w.coin_seed, alpha, P + 2, P + G)
    eng.set_draft_override(P + 2, ar.tolist()[1:], modes)
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
