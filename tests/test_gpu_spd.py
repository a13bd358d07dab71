"""End-to-end parity of the CUDA path with the oracle, through the C ABI.

For each workload (seeded synthetic weights and prompt):
* GPU plain AR vs the oracle teacher-forced on the GPU stream: every token equals the oracle's
  argmax unless the oracle's top-2 gap is below 1e-2 (flagged near tie);
* GPU SPD == GPU AR bit for bit (batch invariance), for several acceptance rates and raw drafts;
* the verification trace is exactly the seeded coin set and the cycle count follows the refill
  arithmetic;
* cycle by cycle, state (t, a, v), residual and anchor rings, draft-module rows and the tokens at
  each exit agree with the oracle's SPD run on the same drafts (max-abs relative error 1e-4 for the
  fp32 workload, 2e-2 for bf16);
* host rollback restores a state from which decoding repeats exactly.
"""
import numpy as np
import pytest
import torch

import spd_inputs as si
from oracle import model as om
from oracle import sampling as osm
from oracle import spd as ospd

from speculative_pipeline_decoding_gb300.binding import (DUMP_ANCHORS, DUMP_KVLEN, DUMP_PDM_Z,
                                                        DUMP_RESID, DUMP_TRACE)

pytestmark = pytest.mark.gpu
NEAR_TIE = 1e-2


@pytest.fixture(scope="module")
def spd():
    from speculative_pipeline_decoding_gb300 import build_ext
    build_ext.build()
    import speculative_pipeline_decoding_gb300 as spd
    return spd


SMALL_BF16 = si.Workload(
    "small_bf16_gqa_n4",
    si.ModelConfig(n_layers=8, d_model=512, n_heads=8, n_kv_heads=2, head_dim=64, d_ffn=1024,
                   vocab=2048, dtype="bf16"),
    n_stages=4, pdm_layers=2, anchors=(0, 2, 4, 6, 7), prompt_len=300, gen_len=48, alphas=(0.7,))

# widths that are multiples of 8 but not of 64 (d_model 520, d_ffn 1000): the weight matrices stream
# through 2-D tensor maps (4 copies per 32-row band) with a zero-filled partial last chunk
ODD_BF16 = si.Workload(
    "odd_bf16_n4",
    si.ModelConfig(n_layers=4, d_model=520, n_heads=8, n_kv_heads=2, head_dim=64, d_ffn=1000,
                   vocab=1000, dtype="bf16"),
    n_stages=4, pdm_layers=1, anchors=(0, 2, 4), prompt_len=120, gen_len=32, alphas=(0.7,))


def rel(a, b):
    a, b = np.asarray(a, np.float64), np.asarray(b, np.float64)
    return float(np.max(np.abs(a - b)) / max(1e-30, np.max(np.abs(b))))


class Setup:
    def __init__(self, spd, w, max_new=None):
        self.w = w
        self.G = max_new or w.gen_len
        self.params = si.generate_weights(w, device="cuda")
        self.cpu = {k: v.cpu() for k, v in self.params.items()}
        self.prompt = si.prompt_tokens(w).tolist()
        self.P = len(self.prompt)
        self.eng = spd.Engine(spd.Config.from_workload(w, max_seq=self.P + self.G + w.n_stages + 2),
                              self.params)
        self.first = self.eng.prefill(self.prompt)
        self.ar, _ = self.eng.generate_ar(self.G)
        self.ar = self.ar.tolist()
        self.models = ospd.build(w, self.cpu)

    def modes(self, alpha):
        P, G = self.P, self.G
        first, last = P + 2, P + G
        return first, self.ar[1:], si.override_modes(self.w.coin_seed, alpha, first, last)

    def spd_run(self, alpha):
        self.eng.rollback(self.P, self.first)
        if alpha is not None:
            first, ref, md = self.modes(alpha)
            self.eng.set_draft_override(first, ref, md)
        else:
            self.eng.set_draft_override(self.P + 2, self.ar[1:], [0] * (self.G - 1))
        toks, stats = self.eng.generate(self.G)
        trace = self.eng.dump(DUMP_TRACE)
        k = self.eng.state()["exits"]
        return toks.tolist(), stats, trace[:, :k]


def teacher_forced_check(models, prompt, stream):
    target, _ = models
    ref = om.greedy_ar(target, prompt, len(stream), forced=stream)
    flagged = 0
    for i, (g, o, gap) in enumerate(zip(stream, ref["tokens"], ref["gaps"])):
        if g != o:
            assert gap < NEAR_TIE, f"token {i}: gpu {g} oracle {o} gap {gap}"
            flagged += 1
    return flagged, ref


def oracle_stream(S: Setup, count: int):
    """The oracle's own greedy AR tokens at positions P+1..P+count (cached on the setup): the
    reference stream of the seeded drafts in the per-cycle comparisons, so that no input of the
    oracle comes from the GPU."""
    have = getattr(S, "_oracle_ar", None)
    if have is None or len(have["tokens"]) < count:
        S._oracle_ar = om.greedy_ar(S.models[0], S.prompt, count)
    return S._oracle_ar


def per_cycle_parity(S: Setup, alpha, n_cycles, tol, post_step=False, min_cycles=None):
    """Run GPU and oracle SPD side by side on identical drafts; compare after every cycle (with
    ``post_step``: both in the post-step schedule, the draft module after the target step).

    The drafts follow the seeded-acceptance modes with the oracle's greedy AR stream as the
    reference tokens, on both sides.  Tokens: a decision the oracle took within NEAR_TIE of its top-2
    gap (the exiting token's verdict or argmax) may go the other way on the GPU.  The draft module's
    head is compared as logits (within ``tol`` of the largest, like every other tensor); its ranking
    must agree wherever the oracle's top-2 gap exceeds twice the largest logit difference (no
    rounding can flip it there).  A flip that is allowed ends the comparison, which must have
    covered ``min_cycles`` cycles."""
    w, eng = S.w, S.eng
    target, pdm = S.models
    from speculative_pipeline_decoding_gb300 import binding as Bd
    opts0 = eng.opts if hasattr(eng, "opts") else Bd.OPT_DEFAULT
    eng.set_options(opts0 | Bd.OPT_DEBUG_LOGITS)
    try:
        return _per_cycle_parity(S, alpha, n_cycles, tol, post_step, min_cycles)
    finally:
        eng.set_options(opts0)


def _per_cycle_parity(S, alpha, n_cycles, tol, post_step, min_cycles):
    from speculative_pipeline_decoding_gb300.binding import DUMP_LOGITS
    w, eng = S.w, S.eng
    target, pdm = S.models
    n, B = w.n_stages, list(w.anchors)
    ora = oracle_stream(S, S.G)
    if ora["tokens"][0] != S.first:  # the prompt's argmax itself is a near tie
        assert ora["gaps"][0] < NEAR_TIE
        pytest.skip("first token is a near tie between the GPU and the oracle")
    first = S.P + 2
    ref = [int(x) for x in ora["tokens"][1:S.G]]
    md = si.override_modes(w.coin_seed, alpha, first, S.P + S.G)
    eng.rollback(S.P, S.first)
    eng.set_draft_override(first, ref, md)
    modes = {q: m for q, m in zip(range(first, first + len(md)), md)}
    refd = {q: r for q, r in zip(range(first, first + len(ref)), ref)}
    run = ospd.SPDRun(target, pdm, w.n_stages, w.pdm_layers, w.anchors, S.prompt,
                      S.P + S.G + w.n_stages + 2, modes, refd, record=True, post_step=post_step)
    worst = {"resid": 0.0, "anch": 0.0, "pdm": 0.0, "pdm_logits": 0.0}
    done = 0
    history = []
    for c in range(n_cycles):
        info = run.cycle()
        g = eng.cycle()
        # the dumps first, so that a failing check reports how far the states had drifted
        cur = {"resid": 0.0, "anch": 0.0, "pdm": 0.0}
        resid = eng.dump(DUMP_RESID)
        for p, h in run.resid.items():
            cur["resid"] = max(cur["resid"], rel(resid[p % (n + 1)], h))
        anch = eng.dump(DUMP_ANCHORS)
        for p in run.resid:
            for b, vec in run.anchor[p].items():
                cur["anch"] = max(cur["anch"], rel(anch[p % (n + 1), B.index(b)], vec))
        z = eng.dump(DUMP_PDM_Z)
        R = info["pdm_z"].shape[0]
        cur["pdm"] = rel(z[:R], info["pdm_z"])
        cur["pdm_rows"] = [round(rel(z[i], info["pdm_z"][i]), 6) for i in range(R)]
        lg = eng.dump(DUMP_LOGITS)[1].astype(np.float64)
        ol = run._pdm_logits.astype(np.float64)
        dlog = float(np.max(np.abs(lg - ol)))
        cur["pdm_logits"] = dlog / float(np.max(np.abs(ol)))
        history.append((c, info["t"], info["a"], cur))
        assert cur["pdm_logits"] < tol, (c, history[-3:])
        if info["pdm_gap"] > 2 * dlog:
            assert g["pdm_top1"] == info["pdm_top"][0], (c, info["pdm_gap"], dlog, history[-3:])
        if g["draft_token"] != info["draft"]:  # the draft came from a ranking rounding may flip
            assert info["pdm_gap"] <= 2 * dlog, (c, g["draft_token"], info["draft"], history[-3:])
            break
        if info["exited"]:
            assert g["exited"] == 1 and g["exit_pos"] == info["exit_pos"]
            if info["target_gap"] >= NEAR_TIE:
                assert g["target_top1"] == info["target_top"][0], (c, history[-3:])
                assert g["accepted"] == int(info["accept"]), c
            elif g["accepted"] != int(info["accept"]) or g["target_top1"] != info["target_top"][0]:
                break
        st = eng.state()
        assert (st["t"], st["a"], st["v"]) == (run.t, run.a, run.v), (c, st, run.t, run.a, run.v)
        for k in worst:
            worst[k] = max(worst[k], cur[k])
        done += 1
    for k, v in worst.items():
        assert v < tol, (k, v)
    assert done >= (min_cycles if min_cycles is not None else min(n_cycles, 2 * n)), done
    worst["cycles"] = done
    return worst


# ------------------------------------------------------------------------------------------------
# tiny fp32 workload (full parity) and a small bf16 GQA workload
# ------------------------------------------------------------------------------------------------
@pytest.fixture(scope="module")
def tiny_setup(spd):
    return Setup(spd, si.WORKLOADS["tiny_f32_n2"])


@pytest.fixture(scope="module")
def small_setup(spd):
    return Setup(spd, SMALL_BF16)


def test_tiny_first_token_and_ar_stream_match_oracle(tiny_setup):
    S = tiny_setup
    flagged, ref = teacher_forced_check(S.models, S.prompt, S.ar)
    assert S.ar[0] == S.first
    assert flagged <= 2


@pytest.mark.parametrize("alpha", [0.0, 0.7, 1.0, None])
def test_tiny_spd_equals_ar_trace_equals_coins(tiny_setup, alpha):
    S = tiny_setup
    toks, stats, trace = S.spd_run(alpha)
    assert toks == S.ar
    assert list(trace[0]) == list(range(S.P + 2, S.P + S.G + 1))
    if alpha is not None:
        acc = [bool(x) for x in trace[1]]
        assert acc == si.accept_mask(S.w.coin_seed, alpha, S.P + 2, S.P + S.G)
        assert stats["cycles"] == ospd.expected_cycles(S.w.n_stages, acc)
        assert stats["rejects"] == acc.count(False)


@pytest.mark.parametrize("setup", ["tiny_setup", "small_setup"])
def test_library_acceptance_knob_equals_host_modes(request, setup):
    """spd_set_acceptance(alpha, seed, ref) draws its coins in the library; the committed stream,
    the trace and the cycle count equal those of the modes computed on the host."""
    S = request.getfixturevalue(setup)
    alpha = S.w.alphas[0]
    toks0, stats0, trace0 = S.spd_run(alpha)
    S.eng.rollback(S.P, S.first)
    S.eng.set_draft_override(S.P + 2, S.ar[1:], [0] * (S.G - 1))  # cleared below by the knob
    S.eng.set_acceptance(alpha, S.w.coin_seed, S.ar)
    toks, stats = S.eng.generate(S.G)
    trace = S.eng.dump(DUMP_TRACE)[:, : S.eng.state()["exits"]]
    assert toks.tolist() == toks0 == S.ar
    assert np.array_equal(trace, trace0)
    assert stats["cycles"] == stats0["cycles"] and stats["rejects"] == stats0["rejects"]
    # alpha < 0: raw draft-module drafts (no override), still lossless
    S.eng.rollback(S.P, S.first)
    S.eng.set_acceptance(-1.0, 0, S.ar)
    raw, _ = S.eng.generate(S.G)
    assert raw.tolist() == S.ar


def test_tiny_per_cycle_parity_with_oracle(tiny_setup):
    worst = per_cycle_parity(tiny_setup, 0.7, 60, 1e-4)
    print("tiny fp32 worst relative errors", worst)


def test_small_bf16_ar_stream_matches_oracle(small_setup):
    flagged, _ = teacher_forced_check(small_setup.models, small_setup.prompt, small_setup.ar)
    assert flagged <= 3


@pytest.mark.parametrize("alpha", [0.0, 0.7, None])
def test_small_bf16_spd_equals_ar(small_setup, alpha):
    S = small_setup
    toks, stats, trace = S.spd_run(alpha)
    assert toks == S.ar
    if alpha is not None:
        acc = [bool(x) for x in trace[1]]
        assert acc == si.accept_mask(S.w.coin_seed, alpha, S.P + 2, S.P + S.G)
        assert stats["cycles"] == ospd.expected_cycles(S.w.n_stages, acc)


def test_small_bf16_per_cycle_parity_with_oracle(small_setup):
    worst = per_cycle_parity(small_setup, 0.7, 40, 2e-2)
    print("small bf16 worst relative errors", worst)


@pytest.fixture(scope="module")
def odd_setup(spd):
    return Setup(spd, ODD_BF16)


@pytest.mark.parametrize("alpha", [0.0, 0.7])
def test_odd_widths_spd_equals_ar(odd_setup, alpha):
    S = odd_setup
    toks, stats, trace = S.spd_run(alpha)
    assert toks == S.ar
    acc = [bool(x) for x in trace[1]]
    assert acc == si.accept_mask(S.w.coin_seed, alpha, S.P + 2, S.P + S.G)


def test_odd_widths_per_cycle_parity_with_oracle(odd_setup):
    flagged, _ = teacher_forced_check(odd_setup.models, odd_setup.prompt, odd_setup.ar)
    assert flagged <= 3
    worst = per_cycle_parity(odd_setup, 0.7, 30, 2e-2)
    print("odd-width bf16 worst relative errors", worst)


def test_rollback_state_and_kv_lengths(tiny_setup):
    S = tiny_setup
    eng, n = S.eng, S.w.n_stages
    first, ref, md = S.modes(0.0)  # every draft wrong: a reject at every exit
    eng.rollback(S.P, S.first)
    eng.set_draft_override(first, ref, md)
    seen = 0
    for _ in range(4 * n):
        g = eng.cycle()
        if g["exited"] and not g["accepted"]:
            te = g["exit_pos"]
            assert (g["t"], g["a"], g["v"]) == (te + 1, 1, te)
            assert list(eng.dump(DUMP_KVLEN)) == [te] * S.w.model.n_layers
            assert g["pushed_token"] == g["target_top1"]
            seen += 1
    assert seen >= 3
    with pytest.raises(Exception):
        eng.rollback(10 ** 6, 0)      # beyond the verified length
    with pytest.raises(Exception):
        eng.rollback(0, 0)


@pytest.mark.parametrize("which", [0, 1, 2])
def test_bounded_waits_give_up_with_timeout_and_the_handle_stays_usable(tiny_setup, which):
    """Each kind of bounded device wait (grid-barrier counter, mbarrier phase, warp-role progress
    counter), run on a condition nothing satisfies with a 50 ms limit, gives up, flags the error
    word, and the host reports SPD_ETIMEOUT with the wait's site; decoding then proceeds normally."""
    import time
    from speculative_pipeline_decoding_gb300 import binding as B
    S = tiny_setup
    t0 = time.perf_counter()
    rc = S.eng.debug_wait_timeout(which, 50_000_000)
    el = time.perf_counter() - t0
    assert rc == -5, rc
    msg = B.lib().spd_last_error(S.eng.h).decode()
    assert "bounded device wait gave up" in msg and "site 7" in msg, msg
    assert el < 5.0
    assert S.eng.state()["err"] == 0
    toks, _, _ = S.spd_run(0.7)
    assert toks == S.ar


# ------------------------------------------------------------------------------------------------
# the 1.5B-class bf16 workload at full size (prompt 512, 256 tokens, n = 8, Ls = 4, alpha 0.8)
# ------------------------------------------------------------------------------------------------
@pytest.fixture(scope="module")
def dense_setup(spd):
    return Setup(spd, si.WORKLOADS["dense1.5b_bf16_n8"])


def test_dense_full_size_spd_equals_ar_and_trace(dense_setup):
    S = dense_setup
    toks, stats, trace = S.spd_run(0.8)
    assert toks == S.ar
    acc = [bool(x) for x in trace[1]]
    assert acc == si.accept_mask(S.w.coin_seed, 0.8, S.P + 2, S.P + S.G)
    assert stats["cycles"] == ospd.expected_cycles(8, acc)


def test_dense_full_size_sampled_tokens_match_oracle(dense_setup):
    """Oracle teacher-forced on the first 16 GPU tokens (the oracle's cost grows with every token)."""
    S = dense_setup
    flagged, _ = teacher_forced_check(S.models, S.prompt, S.ar[:16])
    assert flagged <= 1


def test_dense_full_size_first_cycles_parity(dense_setup):
    """Warm-up (8 cycles) and 16 steady-state cycles at full size, every cycle against the oracle."""
    worst = per_cycle_parity(dense_setup, 0.8, 24, 2e-2)
    print("dense1.5b bf16 worst relative errors", worst)


# ------------------------------------------------------------------------------------------------
# the 4B-class and 9B-class models at full width, with a 128-token prompt so that the oracle's
# fp32 prefill stays short: warm-up plus 2n steady-state cycles, every cycle against the oracle --
# residual and anchor rings, the draft module's rows after its layers (GQA, head size 128, up to
# 17 staircase rows at n = 16), both heads' top-1 and the verdicts
# ------------------------------------------------------------------------------------------------
@pytest.mark.parametrize("name", ["gqa4b_bf16_n8", "gqa9b_bf16_n4", "gqa9b_bf16_n8", "gqa9b_bf16_n16"])
def test_full_width_per_cycle_parity_short_prompt(spd, name):
    import dataclasses
    base = si.WORKLOADS[name]
    n = base.n_stages
    w = dataclasses.replace(base, prompt_len=128, gen_len=3 * n + 8)
    S = Setup(spd, w)
    try:
        worst = per_cycle_parity(S, max(base.alphas), 3 * n, 2e-2, min_cycles=2 * n)
    finally:
        S.eng.close()
        del S.params
        torch.cuda.empty_cache()
    print(name, "short-prompt per-cycle worst relative errors", worst)


# ------------------------------------------------------------------------------------------------
# prefill on the tensor cores: a prompt of 2100 tokens (65 full blocks and a ragged block of 20 rows;
# the causal attention splits its 17 key chunks over CTAs) -- the hidden states after all layers of
# the last block and the tokens after it, against the oracle
# ------------------------------------------------------------------------------------------------
LONG_PROMPT_BF16 = si.Workload(
    "small_bf16_gqa_long_prompt",
    si.ModelConfig(n_layers=8, d_model=512, n_heads=8, n_kv_heads=2, head_dim=64, d_ffn=1024,
                   vocab=2048, dtype="bf16"),
    n_stages=4, pdm_layers=2, anchors=(0, 2, 4, 6, 7), prompt_len=2100, gen_len=8, alphas=(0.7,))

HD128_LONG_PROMPT = si.Workload(
    "gqa_hd128_long_prompt",
    si.ModelConfig(n_layers=4, d_model=1024, n_heads=16, n_kv_heads=4, head_dim=128, d_ffn=2048,
                   vocab=4096, dtype="bf16"),
    n_stages=2, pdm_layers=2, anchors=(0, 2, 4), prompt_len=2049, gen_len=8, alphas=(0.7,))


@pytest.mark.parametrize("w", [LONG_PROMPT_BF16, HD128_LONG_PROMPT], ids=lambda w: w.name)
def test_long_prompt_prefill_hidden_states_match_oracle(spd, w):
    from speculative_pipeline_decoding_gb300.binding import DUMP_PREFILL_H
    S = Setup(spd, w)
    try:
        P = S.P
        cnt = P - 32 * ((P - 1) // 32)  # rows of the last prefill block
        got = S.eng.dump(DUMP_PREFILL_H)[:cnt]
        target, _ = S.models
        H, _ = target.prefill(S.prompt, target.new_cache(P + 1))
        err = rel(got, H[P - cnt:])
        assert err < 2e-2, err
        flagged, _ = teacher_forced_check(S.models, S.prompt, S.ar)
        assert flagged <= 1
    finally:
        S.eng.close()
    print(w.name, "prefill hidden-state relative error", err)


# ------------------------------------------------------------------------------------------------
# execution options: the persistent step kernel vs per-operator launches, draft module co-scheduled
# vs serialised, graphs vs eager launches -- every combination computes the same streams
# ------------------------------------------------------------------------------------------------
def _option_sets():
    from speculative_pipeline_decoding_gb300 import binding as B
    return {
        "step_serial_graphs": B.OPT_STEP | B.OPT_PDL | B.OPT_GRAPHS,
        "step_cosched_eager": B.OPT_STEP | B.OPT_PDL | B.OPT_COSCHED,
        "ops_cosched_graphs": B.OPT_GRAPHS | B.OPT_PDL | B.OPT_COSCHED,
        "ops_serial_eager": 0,
        "step_post_graphs": B.OPT_STEP | B.OPT_PDL | B.OPT_GRAPHS | B.OPT_POST_STEP,
        "ops_post_eager": B.OPT_POST_STEP,
    }


@pytest.mark.parametrize("name", ["step_serial_graphs", "step_cosched_eager", "ops_cosched_graphs",
                                  "ops_serial_eager", "step_post_graphs", "ops_post_eager"])
@pytest.mark.parametrize("setup", ["tiny_setup", "small_setup"])
def test_execution_options_give_identical_streams(request, setup, name):
    from speculative_pipeline_decoding_gb300 import binding as B
    S = request.getfixturevalue(setup)
    alpha = S.w.alphas[0]
    toks0, stats0, trace0 = S.spd_run(alpha)
    S.eng.set_options(_option_sets()[name])
    try:
        toks, stats, trace = S.spd_run(alpha)
        S.eng.rollback(S.P, S.first)
        ar, _ = S.eng.generate_ar(S.G)
    finally:
        S.eng.set_options(B.OPT_DEFAULT)
    assert toks == toks0 == S.ar
    assert ar.tolist() == S.ar
    assert np.array_equal(trace, trace0)
    assert stats["cycles"] == stats0["cycles"] and stats["rejects"] == stats0["rejects"]


# ------------------------------------------------------------------------------------------------
# the other configurations at full size (4B-class GQA, 9B-class at n = 4 / 8 / 16, 4B-class at 32K
# context): properties that hold at any size -- SPD == AR bit for bit, the verification trace is
# the seeded coin set, the cycle count follows the refill arithmetic -- and, for the 4B-class
# model, the first GPU tokens against the oracle (teacher-forced)
# ------------------------------------------------------------------------------------------------
FULL_SIZE = ["gqa4b_bf16_n8", "gqa9b_bf16_n4", "gqa9b_bf16_n8", "gqa9b_bf16_n16", "gqa4b_bf16_n8_ctx32k"]
# every full-size configuration runs by default (the 32K-token prefill takes about half a minute)
SLOW = set()


@pytest.mark.parametrize("name", FULL_SIZE)
def test_full_size_spd_equals_ar_and_trace(spd, name):
    import os
    if name in SLOW and os.environ.get("SPD_SLOW_TESTS") != "1":
        pytest.skip("set SPD_SLOW_TESTS=1")
    w = si.WORKLOADS[name]
    params = si.generate_weights(w, device="cuda")
    prompt = si.prompt_tokens(w).tolist()
    P, G = len(prompt), w.gen_len
    eng = spd.Engine(spd.Config.from_workload(w), params)
    try:
        first = eng.prefill(prompt)
        ar, _ = eng.generate_ar(G)
        ar = ar.tolist()
        assert ar[0] == first
        for alpha in w.alphas:
            eng.rollback(P, first)
            eng.set_draft_override(P + 2, ar[1:], si.override_modes(w.coin_seed, alpha, P + 2, P + G))
            toks, stats = eng.generate(G)
            assert toks.tolist() == ar, (name, alpha)
            trace = eng.dump(DUMP_TRACE)[:, : eng.state()["exits"]]
            acc = [bool(x) for x in trace[1]]
            assert list(trace[0]) == list(range(P + 2, P + G + 1))
            assert acc == si.accept_mask(w.coin_seed, alpha, P + 2, P + G)
            assert stats["cycles"] == ospd.expected_cycles(w.n_stages, acc)
            assert stats["rejects"] == acc.count(False)
    finally:
        eng.close()
        del params
        torch.cuda.empty_cache()


def _full_prompt_ar_vs_oracle(spd, names, count):
    """GPU AR at each workload's full prompt (the first `count` tokens), then the oracle teacher-forced
    on the first stream.  The workloads share the target model, so their AR streams must be equal."""
    w0 = si.WORKLOADS[names[0]]
    prompt = si.prompt_tokens(w0).tolist()
    streams = []
    for name in names:
        w = si.WORKLOADS[name]
        params = si.generate_weights(w, device="cuda")
        eng = spd.Engine(spd.Config.from_workload(w), params)
        try:
            first = eng.prefill(prompt)
            ar, _ = eng.generate_ar(count)
            streams.append(ar.tolist())
            assert streams[-1][0] == first
        finally:
            eng.close()
            if name == names[-1]:
                cpu = {k: v.cpu() for k, v in params.items() if not k.startswith("pdm")}
            del params
            torch.cuda.empty_cache()
    for st in streams[1:]:
        assert st == streams[0]
    target = om.Decoder(w0.model, cpu)
    del cpu
    ref = om.greedy_ar(target, prompt, count, forced=streams[0])
    flagged = 0
    for i, (g, o, gap) in enumerate(zip(streams[0], ref["tokens"], ref["gaps"])):
        if g != o:
            assert gap < NEAR_TIE, f"token {i}: gpu {g} oracle {o} gap {gap}"
            flagged += 1
    assert flagged <= 1
    return ref


def test_gqa4b_full_size_tokens_match_oracle(spd):
    """4B-class GQA at its full prompt (1024): the first 8 GPU tokens, oracle teacher-forced."""
    _full_prompt_ar_vs_oracle(spd, ["gqa4b_bf16_n8"], 8)


def test_gqa9b_full_size_tokens_match_oracle_at_every_width(spd):
    """9B-class at its full prompt (2048), engines of n = 4, 8, 16: the first 8 AR tokens are the same
    for the three engines and match the oracle teacher-forced on them."""
    _full_prompt_ar_vs_oracle(spd, ["gqa9b_bf16_n4", "gqa9b_bf16_n8", "gqa9b_bf16_n16"], 8)


# ------------------------------------------------------------------------------------------------
# post-step schedule (the scheduling ablation: draft module after the target step, on its output
# state) -- per-cycle parity with the oracle's post-step run, through the step kernel and through
# the per-operator launches
# ------------------------------------------------------------------------------------------------
@pytest.mark.parametrize("opts", ["step", "ops"])
@pytest.mark.parametrize("setup,tol", [("tiny_setup", 1e-4), ("small_setup", 2e-2)])
def test_post_step_per_cycle_parity_with_oracle(request, setup, tol, opts):
    from speculative_pipeline_decoding_gb300 import binding as B
    S = request.getfixturevalue(setup)
    S.eng.set_options(B.OPT_POST_STEP | (B.OPT_STEP | B.OPT_PDL if opts == "step" else 0))
    try:
        worst = per_cycle_parity(S, S.w.alphas[0], 40, tol, post_step=True)
    finally:
        S.eng.set_options(B.OPT_DEFAULT)
    print(setup, opts, "post-step worst relative errors", worst)


def test_post_step_cycle_count_and_pdm_cache_length(tiny_setup):
    """Same cycles and trace as the default schedule; the exiting row joins the draft-module cache."""
    from speculative_pipeline_decoding_gb300 import binding as B
    S = tiny_setup
    alpha = 0.7
    toks0, stats0, trace0 = S.spd_run(alpha)
    S.eng.set_options(B.OPT_DEFAULT | B.OPT_POST_STEP)
    try:
        toks, stats, trace = S.spd_run(alpha)
        assert toks == S.ar and stats["cycles"] == stats0["cycles"]
        assert np.array_equal(trace, trace0)
        first, ref, md = S.modes(alpha)
        S.eng.rollback(S.P, S.first)
        S.eng.set_draft_override(first, ref, md)
        for _ in range(30):
            g = S.eng.cycle()
            st = S.eng.state()
            # after an exit the draft-module cache holds every verified row (the exiting one included)
            if g["exited"]:
                assert st["pdm_len"] == g["exit_pos"], st
            else:
                assert st["pdm_len"] == st["v"], st
    finally:
        S.eng.set_options(B.OPT_DEFAULT)


# ------------------------------------------------------------------------------------------------
# sampled decoding (T > 0, top-k; rejection-sampling verification): the GPU streams and traces
# equal the oracle's on the same uniforms, up to the first decision the oracle took within `thr`
# of a boundary (a different rounding may take the other side there)
# ------------------------------------------------------------------------------------------------
def _uniforms(S, seed):
    first, last = S.P + 1, S.P + S.G + S.w.n_stages + 2
    u = si.sampling_uniforms(seed, first, last)
    arr = np.array([u[s] for s in si.SAMPLING_STREAMS], dtype=np.float32)
    by_pos = {s: {q: float(v) for q, v in zip(range(first, last + 1), u[s])} for s in si.SAMPLING_STREAMS}
    return first, arr, by_pos


def _first_mismatch(a, b):
    for j, (x, y) in enumerate(zip(a, b)):
        if x != y:
            return j
    return None if len(a) == len(b) else min(len(a), len(b))


@pytest.mark.parametrize("opts", ["step", "ops"])
# thr: the fp32 workload matches to rounding order; on the bf16 one the two sides' K/V caches
# occasionally round an element to different bf16 neighbours, which moves hidden states by ~2e-4
# (relative) and a probability by about as much, so a draw within 1e-3 of a boundary may differ
@pytest.mark.parametrize("setup,thr", [("tiny_setup", 1e-4), ("small_setup", 1e-3)])
def test_sampled_spd_and_ar_match_oracle(request, setup, thr, opts):
    from speculative_pipeline_decoding_gb300 import binding as B
    S = request.getfixturevalue(setup)
    target, pdm = S.models
    T, k, seed = 1.0, 50, 4242
    first, arr, u = _uniforms(S, seed)
    if opts == "ops":
        S.eng.set_options(B.OPT_GRAPHS | B.OPT_PDL | B.OPT_COSCHED)
    S.eng.set_sampling(T, k, first, arr)
    try:
        S.eng.rollback(S.P, S.first)
        toks, stats = S.eng.generate(S.G)
        toks = toks.tolist()
        trace = S.eng.dump(DUMP_TRACE)[:, : S.eng.state()["exits"]]
        S.eng.rollback(S.P, S.first)
        ar, _ = S.eng.generate_ar(S.G)
        ar = ar.tolist()
    finally:
        S.eng.set_sampling(0.0)
        S.eng.set_options(B.OPT_DEFAULT)
    smp = {"T": T, "k": k, "u_draft": u["draft"], "u_accept": u["accept"], "u_resample": u["resample"]}
    run = ospd.SPDRun(target, pdm, S.w.n_stages, S.w.pdm_layers, S.w.anchors, S.prompt,
                      S.P + S.G + S.w.n_stages + 2, sampling=smp)
    ref = run.generate(S.G)
    j = _first_mismatch(toks, ref)
    if j is not None:  # only after a near-boundary decision of the oracle
        q = S.P + 1 + j
        assert min([m for p, m in run.margins if p <= q] + [1.0]) < thr, (j, toks[j:j + 3], ref[j:j + 3])
    upto = S.G if j is None else j
    assert list(trace[0][:upto - 1]) == [p for p, _ in run.trace][:upto - 1]
    assert [bool(x) for x in trace[1][:upto - 1]] == [ok for _, ok in run.trace][:upto - 1]
    accepted = [bool(x) for x in trace[1]]
    assert stats["cycles"] == ospd.expected_cycles(S.w.n_stages, accepted)
    # sampled AR from the same kernels
    ora = osm.sampled_ar(target, S.prompt, S.G, T, k, u["ar"])
    ja = _first_mismatch(ar, ora["tokens"])
    if ja is not None:
        assert min(ora["margins"][:ja] + [1.0]) < thr, (ja, ar[ja:ja + 3], ora["tokens"][ja:ja + 3])
    print(setup, opts, "sampled SPD first mismatch", j, "AR", ja, "accepts", sum(accepted), "/", len(accepted))


# temperatures other than 1 (both sides divide each logit by T in fp32 before the weights) and a
# top-k that is not the pages' 50: a sharper and a flatter distribution
@pytest.mark.parametrize("T,k,seed", [(0.6, 8, 77), (1.7, 64, 31)])
@pytest.mark.parametrize("setup,thr", [("tiny_setup", 1e-4), ("small_setup", 1e-3)])
def test_sampled_other_temperatures_match_oracle(request, setup, thr, T, k, seed):
    S = request.getfixturevalue(setup)
    target, pdm = S.models
    first, arr, u = _uniforms(S, seed)
    S.eng.set_sampling(T, k, first, arr)
    try:
        S.eng.rollback(S.P, S.first)
        toks, stats = S.eng.generate(S.G)
        toks = toks.tolist()
        trace = S.eng.dump(DUMP_TRACE)[:, : S.eng.state()["exits"]]
        S.eng.rollback(S.P, S.first)
        ar, _ = S.eng.generate_ar(S.G)
        ar = ar.tolist()
    finally:
        S.eng.set_sampling(0.0)
    smp = {"T": T, "k": k, "u_draft": u["draft"], "u_accept": u["accept"], "u_resample": u["resample"]}
    run = ospd.SPDRun(target, pdm, S.w.n_stages, S.w.pdm_layers, S.w.anchors, S.prompt,
                      S.P + S.G + S.w.n_stages + 2, sampling=smp)
    ref = run.generate(S.G)
    j = _first_mismatch(toks, ref)
    if j is not None:
        q = S.P + 1 + j
        assert min([m for p, m in run.margins if p <= q] + [1.0]) < thr, (j, toks[j:j + 3], ref[j:j + 3])
    upto = S.G if j is None else j
    assert [bool(x) for x in trace[1][:upto - 1]] == [ok for _, ok in run.trace][:upto - 1]
    assert stats["cycles"] == ospd.expected_cycles(S.w.n_stages, [bool(x) for x in trace[1]])
    ora = osm.sampled_ar(target, S.prompt, S.G, T, k, u["ar"])
    ja = _first_mismatch(ar, ora["tokens"])
    if ja is not None:
        assert min(ora["margins"][:ja] + [1.0]) < thr, (ja, ar[ja:ja + 3], ora["tokens"][ja:ja + 3])
    # the output is a draw, not the greedy stream: at T = 1.7 over 64 tokens it leaves argmax early
    if T > 1.0:
        assert ar != S.ar[: len(ar)]
    print(setup, T, k, "sampled SPD first mismatch", j, "AR", ja, "accepts", int(trace[1].sum()), "/", trace.shape[1])


# ------------------------------------------------------------------------------------------------
# degenerate shapes: a one-stage pipeline (n = 1: the exiting token verifies the draft of the same
# cycle, SPD degenerates to AR with a draft per step) on a one-token prompt
# ------------------------------------------------------------------------------------------------
MICRO_N1 = si.Workload(
    "micro_f32_n1",
    si.ModelConfig(n_layers=4, d_model=128, n_heads=2, n_kv_heads=1, head_dim=64, d_ffn=256,
                   vocab=512, dtype="f32", init_std=0.1),
    n_stages=1, pdm_layers=1, anchors=(0, 2, 4), prompt_len=1, gen_len=24, alphas=(0.5,))


@pytest.fixture(scope="module")
def n1_setup(spd):
    return Setup(spd, MICRO_N1)


def test_one_stage_one_token_prompt_greedy(n1_setup):
    S = n1_setup
    assert S.P == 1
    flagged, _ = teacher_forced_check(S.models, S.prompt, S.ar)
    assert flagged <= 1
    for alpha in (0.0, 0.5, 1.0):
        toks, stats, trace = S.spd_run(alpha)
        assert toks == S.ar
        acc = [bool(x) for x in trace[1]]
        assert acc == si.accept_mask(S.w.coin_seed, alpha, S.P + 2, S.P + S.G)
        assert stats["cycles"] == ospd.expected_cycles(1, acc)
    S.eng.rollback(S.P, S.first)
    one, st1 = S.eng.generate(1)  # only the token of the prefill
    assert one.tolist() == [S.first] and st1["cycles"] == 0


def test_one_stage_sampled_matches_oracle(n1_setup):
    S = n1_setup
    target, pdm = S.models
    first, arr, u = _uniforms(S, 99)
    S.eng.set_sampling(1.0, 50, first, arr)
    try:
        S.eng.rollback(S.P, S.first)
        toks, stats = S.eng.generate(S.G)
        trace = S.eng.dump(DUMP_TRACE)[:, : S.eng.state()["exits"]]
    finally:
        S.eng.set_sampling(0.0)
    smp = {"T": 1.0, "k": 50, "u_draft": u["draft"], "u_accept": u["accept"], "u_resample": u["resample"]}
    run = ospd.SPDRun(target, pdm, 1, 1, S.w.anchors, S.prompt, S.P + S.G + 3, sampling=smp)
    ref = run.generate(S.G)
    j = _first_mismatch(toks.tolist(), ref)
    if j is not None:
        assert min([m for p, m in run.margins if p <= S.P + 1 + j] + [1.0]) < 1e-4
    upto = S.G if j is None else j
    assert [bool(x) for x in trace[1][:upto - 1]] == [ok for _, ok in run.trace][:upto - 1]
    assert stats["cycles"] == ospd.expected_cycles(1, [bool(x) for x in trace[1]])
