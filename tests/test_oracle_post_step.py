"""Pins of the oracle's post-step schedule (oracle/spd.py, reading 7).

The post-step schedule is the scheduling ablation of the SPD v3 summary (§4) and the SPD news
article (section 十): the draft module waits for the target step and reads its output state.  What
holds the oracle's version of it, independent of its own code:

* losslessness and the trace: the committed stream is plain greedy AR, the reject set is the coin
  set and the cycle count follows the same refill arithmetic as the pre-step schedule (the draft
  still enters stage 1 at the end of the cycle);
* feature reuse: cached rows + refreshed rows == the draft module recomputed from scratch;
* a relation between the two schedules: after the step of cycle c, every row has the depth and the
  anchors it has before the step of cycle c+1, so with the same accepted history the post-step
  draft module of cycle c and the pre-step one of cycle c+1 compute the same rows;
* a planted wrong depth (the pre-step staircase in the post-step schedule) is caught.
"""
import numpy as np
import pytest

import spd_inputs as si
from oracle import spd as ospd


@pytest.mark.parametrize("alpha", [0.0, 0.7, 1.0])
def test_post_step_lossless_trace_and_cycle_count(tiny, tiny_ar, alpha):
    w, params, prompt, models = tiny
    P, G = len(prompt), w.gen_len
    run = ospd.run_spd(w, params, prompt, G, alpha, ref=tiny_ar["tokens"], models=models, post_step=True)
    assert run.committed == tiny_ar["tokens"]
    accepted = [ok for _, ok in run.trace]
    assert [q for q, _ in run.trace] == list(range(P + 2, P + G + 1))
    assert accepted == si.accept_mask(w.coin_seed, alpha, P + 2, P + G)
    assert run.cycles == ospd.expected_cycles(w.n_stages, accepted)


def test_post_step_raw_drafts_are_lossless(tiny, tiny_ar):
    w, params, prompt, models = tiny
    run = ospd.run_spd(w, params, prompt, w.gen_len, None, models=models, post_step=True)
    assert run.committed == tiny_ar["tokens"]


def test_post_step_incremental_rows_equal_full_recompute(tiny, tiny_ar):
    w, params, prompt, models = tiny
    run = ospd.run_spd(w, params, prompt, 24, 0.7, ref=tiny_ar["tokens"], models=models,
                       check_full_recompute=True, post_step=True)
    assert run.cycles > 20


def test_post_step_depths_are_one_stage_deeper():
    # worked by hand: n = 4, t = 20, a = 4 -> in-flight rows 17..20 at 4 (exiting), 3, 2, 1
    assert [ospd.depth_after_step(i, 20, 4, 4) for i in range(15, 21)] == [4, 4, 4, 3, 2, 1]
    # warm-up, a = 2 of n = 4: rows 19, 20 at 2, 1; the prefix at n
    assert [ospd.depth_after_step(i, 20, 2, 4) for i in range(17, 21)] == [4, 4, 2, 1]


def test_post_step_cycle_sees_what_the_next_pre_step_cycle_sees(tiny, tiny_ar):
    """All drafts accepted: rows of the post-step draft module at cycle c == rows of the pre-step
    draft module at cycle c+1 (same positions), depths and values."""
    w, params, prompt, models = tiny
    target, pdm = models
    P, n = len(prompt), w.n_stages
    modes = {q: ospd.FORCE_REF for q in range(P + 2, P + 40)}
    ref = {q: tiny_ar["tokens"][q - P - 1] for q in modes}
    pre = ospd.SPDRun(target, pdm, n, w.pdm_layers, w.anchors, prompt, P + 50, modes, ref, record=True)
    post = ospd.SPDRun(target, pdm, n, w.pdm_layers, w.anchors, prompt, P + 50, modes, ref, record=True,
                       post_step=True)
    infos_pre = [pre.cycle() for _ in range(26)]
    infos_post = [post.cycle() for _ in range(25)]
    checked = 0
    for c in range(25):
        rows_post, z_post = infos_post[c]["rows"], infos_post[c]["pdm_z"]
        rows_pre = dict((i, (k, r)) for r, (i, k) in enumerate(infos_pre[c + 1]["rows"]))
        for r, (i, k) in enumerate(rows_post):
            k_pre, r_pre = rows_pre[i]
            assert k == k_pre, (c, i)
            z_pre = infos_pre[c + 1]["pdm_z"][r_pre]
            assert np.max(np.abs(z_post[r] - z_pre)) <= 1e-5 * max(1.0, float(np.max(np.abs(z_pre))))
            checked += 1
        # and the post-step rows are the pre-step rows of c+1 without the newest (depth 0) one
        assert [i for i, _ in rows_post] == [i for i, _ in infos_pre[c + 1]["rows"]][:len(rows_post)]
    assert checked >= 2 * 20  # about n rows per cycle (n = 2 here)


def test_planted_pre_step_depth_in_post_step_schedule_is_caught(tiny, tiny_ar, monkeypatch):
    w, params, prompt, models = tiny
    monkeypatch.setattr(ospd, "depth_after_step", ospd.depth_of)
    with pytest.raises(AssertionError):
        ospd.run_spd(w, params, prompt, 16, 0.7, ref=tiny_ar["tokens"], models=models, post_step=True)
