"""Pins of the oracle's SPD cycle (oracle/spd.py).

What holds it, independent of its own code:
* anchor tables and staircases worked by hand from the pages (tests/golden);
* the structural-mask rule of the SPD v3 summary (App. A.3) gives every key
  row one depth, whichever query looks at it;
* losslessness (SPD summary, 前置知识; SPD news §六): the committed stream is
  plain greedy AR token for token, for every acceptance pattern;
* the trace: the reject set is exactly the seeded coin set, the cycle count
  follows the refill arithmetic, and the pages' alpha = N/K;
* feature reuse (SPD v3 App. A.1): cached verified rows + refreshed trailing
  rows == the draft module recomputed from scratch;
* n = 1 degenerates to AR; Ls > L/n is refused;
* brute force over every prompt and every accept mask of a tiny model;
* planted mistakes in the oracle (wrong depth, wrong rollback length) are caught.
"""
import itertools

import numpy as np
import pytest
import torch

import spd_inputs as si
from conftest import golden_rows
from oracle import model as om
from oracle import spd as ospd


def test_anchor_tables_match_hand_worked_values():
    for L, n, B, lm, f in golden_rows("anchor_tables.txt"):
        L, n = int(L), int(n)
        B = [int(x) for x in B.split(",")]
        assert [ospd.lmax(k, L, n) for k in range(n + 1)] == [int(x) for x in lm.split(",")]
        assert ospd.f_table(L, n, B) == [int(x) for x in f.split(",")]


@pytest.mark.parametrize("n", [4, 8, 16])
def test_five_fusion_projections_suffice_for_printed_anchors(n):
    # SPD summary, 技术新颖性: with B = [0,8,16,24,31] only m = 5 projections are needed
    ft = ospd.f_table(32, n, [0, 8, 16, 24, 31])
    assert sorted(set(ft)) == [0, 1, 2, 3, 4]
    # depth 0 is an embedding projection (SPD v3 §3.2); depth n uses every anchor
    assert ft[0] == 0 and ft[n] == 4
    # deeper rows never see fewer anchors
    assert all(a <= b for a, b in zip(ft, ft[1:]))


def test_config_checks():
    ospd.check_config(32, 8, 4, [0, 8, 16, 24, 31])
    with pytest.raises(ValueError):
        ospd.check_config(32, 8, 5, [0, 8, 16, 24, 31])   # Ls > L/n breaks masking
    with pytest.raises(ValueError):
        ospd.check_config(32, 5, 1, [0, 8])               # n must divide L
    with pytest.raises(ValueError):
        ospd.check_config(32, 8, 4, [1, 8])               # b_0 must be the embedding
    with pytest.raises(ValueError):
        ospd.check_config(32, 8, 4, [0, 8, 8])            # strictly increasing
    with pytest.raises(ValueError):
        ospd.check_config(32, 8, 4, [0, 33])              # inside the model


def test_staircase_matches_hand_worked_layouts():
    for n, t, a, first, depths in golden_rows("staircase.txt"):
        n, t, a, first = int(n), int(t), int(a), int(first)
        got = [ospd.depth_of(i, t, a, n) for i in range(first, t + 1)]
        assert got == [int(x) for x in depths.split(",")]


def _mask_rule_depth(n, fill, t_q, d_q, T):
    """SPD v3 App. A.3: query at time t_q, depth d_q sees key T at depth min(n, d_q + t_q - T),
    redirected to the deepest block when t - T exceeds the fill level."""
    t = t_q + d_q  # the newest position at the time of this layout
    if t - T >= fill:
        return n
    return min(n, d_q + t_q - T)


@pytest.mark.parametrize("n", [1, 2, 4, 8])
def test_every_query_sees_each_key_at_its_staircase_depth(n):
    t = 40
    for a in range(1, n + 1):
        for t_q in range(t - n - 2, t + 1):
            d_q = ospd.depth_of(t_q, t, a, n)
            if d_q == n:
                continue  # verified rows are cached; their features never change
            for T in range(1, t_q + 1):
                assert _mask_rule_depth(n, a, t_q, d_q, T) == ospd.depth_of(T, t, a, n)


@pytest.mark.parametrize("alpha", [0.0, 0.7, 1.0])
def test_lossless_trace_and_cycle_count_tiny(tiny, tiny_ar, alpha):
    w, params, prompt, models = tiny
    P, G = len(prompt), w.gen_len
    run = ospd.run_spd(w, params, prompt, G, alpha, ref=tiny_ar["tokens"], models=models)
    assert run.committed == tiny_ar["tokens"]
    accepted = [ok for _, ok in run.trace]
    assert [q for q, _ in run.trace] == list(range(P + 2, P + G + 1))
    assert accepted == si.accept_mask(w.coin_seed, alpha, P + 2, P + G)
    assert run.cycles == ospd.expected_cycles(w.n_stages, accepted)
    assert run.rejects == accepted.count(False)
    # the pages' alpha = N/K (SPD news §八) is a cycle ratio, here from the trace
    N = G - 1
    assert run.cycles == N + (w.n_stages - 1) * (1 + accepted[:-1].count(False))


def test_raw_drafts_are_lossless_too(tiny, tiny_ar):
    w, params, prompt, models = tiny
    run = ospd.run_spd(w, params, prompt, w.gen_len, None, models=models)
    assert run.committed == tiny_ar["tokens"]


def test_rollback_state_after_every_reject(tiny, tiny_ar):
    w, params, prompt, models = tiny
    target, pdm = models
    P, n = len(prompt), w.n_stages
    modes = {q: (ospd.FORCE_OTHER if q % 3 == 0 else ospd.FORCE_REF) for q in range(P + 2, P + 40)}
    ref = {q: tiny_ar["tokens"][q - P - 1] for q in modes}
    run = ospd.SPDRun(target, pdm, n, w.pdm_layers, w.anchors, prompt, P + 50, modes, ref)
    seen = 0
    while run.v + 1 - P < 30:
        info = run.cycle()
        if info["exited"] and not info["accept"]:
            seen += 1
            te = info["exit_pos"]
            assert te == info["t"] - n + 1
            assert run.cache.length == [te] * target.L          # (i) every layer at t-n+1
            assert run.a == 1 and run.t == te + 1              # (ii) flushed, (iii) reseeded
            assert run.seq[te + 1] == info["target_top"][0]     # with the target's argmax
            assert set(run.resid) == {te + 1}
    assert seen >= 5


def test_incremental_draft_rows_equal_full_recompute(tiny, tiny_ar):
    w, params, prompt, models = tiny
    run = ospd.run_spd(w, params, prompt, 24, 0.7, ref=tiny_ar["tokens"], models=models,
                       check_full_recompute=True)
    assert run.cycles > 20


def test_draft_feature_special_cases(tiny):
    w, params, prompt, (target, pdm) = tiny
    d = w.model.d_model
    B = list(w.anchors)
    states = {b: np.random.default_rng(b).standard_normal(d).astype(np.float32) for b in B}
    saved = list(pdm.fc)
    try:
        eye = np.eye(d, dtype=np.float32)
        pdm.fc[2] = np.concatenate([eye, 0 * eye, 0 * eye], axis=1)
        np.testing.assert_array_equal(pdm.feature(states, B, 2), states[0])
        pdm.fc[2] = np.concatenate([0 * eye, 0 * eye, eye], axis=1)
        np.testing.assert_array_equal(pdm.feature(states, B, 2), states[B[2]])
        pdm.fc[1] = np.concatenate([eye, eye], axis=1)
        np.testing.assert_allclose(pdm.feature(states, B, 1), states[0] + states[B[1]], rtol=1e-6)
    finally:
        pdm.fc[:] = saved


def test_single_stage_degenerates_to_autoregressive():
    cfg = si.small_model(n_layers=2, d_model=32, n_heads=2, n_kv_heads=1, head_dim=16,
                         d_ffn=48, vocab=40, init_std=0.3)
    w = si.Workload("n1", cfg, 1, 2, (0, 1, 2), 5, 12, (0.5,))
    params = si.generate_weights(w)
    prompt = si.prompt_tokens(w).tolist()
    target, pdm = ospd.build(w, params)
    ar = om.greedy_ar(target, prompt, 12)
    for alpha in (None, 0.0, 0.5):
        run = ospd.run_spd(w, params, prompt, 12, alpha, ref=ar["tokens"], models=(target, pdm))
        assert run.committed == ar["tokens"]
        assert run.cycles == 11  # one cycle per token, like AR steps


def test_draft_depth_bounded_by_stage_depth():
    cfg = si.small_model(n_layers=4)
    w = si.Workload("bad", cfg, 2, 3, (0, 2, 4), 4, 4, (0.5,))
    params = si.generate_weights(w)
    target, pdm = ospd.build(w, params)
    with pytest.raises(ValueError):
        ospd.SPDRun(target, pdm, 2, 3, (0, 2, 4), [1, 2, 3, 4], 16)


# ---------------------------------------------------------------------------
# brute force: every prompt of length 2 x every accept mask of 5 verifications
# ---------------------------------------------------------------------------
def _brute_models():
    cfg = si.small_model(n_layers=2, d_model=8, n_heads=2, n_kv_heads=1, head_dim=4,
                         d_ffn=16, vocab=16, init_std=0.5)
    w = si.Workload("brute", cfg, 2, 1, (0, 1, 2), 2, 6, (0.5,))
    params = si.generate_weights(w)
    return w, params, ospd.build(w, params)


@pytest.mark.parametrize("first_token", list(range(16)))
def test_brute_force_all_prompts_all_masks(first_token):
    w, params, (target, pdm) = _brute_models()
    G, n = w.gen_len, w.n_stages
    for second in range(16):
        prompt = [first_token, second]
        P = len(prompt)
        ar = om.greedy_ar(target, prompt, G)["tokens"]
        ref = {q: ar[q - P - 1] for q in range(P + 2, P + G + 1)}
        for bits in itertools.product([True, False], repeat=G - 1):
            modes = {q: (ospd.FORCE_REF if b else ospd.FORCE_OTHER)
                     for q, b in zip(range(P + 2, P + G + 1), bits)}
            run = ospd.SPDRun(target, pdm, n, 1, w.anchors, prompt, P + G + 4, modes, ref)
            assert run.generate(G) == ar
            assert [ok for _, ok in run.trace] == list(bits)
            assert run.cycles == ospd.expected_cycles(n, list(bits))


# ---------------------------------------------------------------------------
# planted mistakes: the pins above catch them
# ---------------------------------------------------------------------------
def test_planted_wrong_depth_is_caught(tiny, tiny_ar, monkeypatch):
    w, params, prompt, models = tiny
    monkeypatch.setattr(ospd, "depth_of", lambda i, t, a, n: (t - i + 1) if t - i < a else n)
    with pytest.raises(AssertionError):
        ospd.run_spd(w, params, prompt, 16, 0.7, ref=tiny_ar["tokens"], models=models)


def test_planted_wrong_rollback_length_is_caught(tiny, tiny_ar, monkeypatch):
    w, params, prompt, models = tiny
    orig = om.KVCache.truncate
    monkeypatch.setattr(om.KVCache, "truncate", lambda self, L_: orig(self, L_ + 1))
    with pytest.raises(AssertionError):
        ospd.run_spd(w, params, prompt, 24, 0.3, ref=tiny_ar["tokens"], models=models)


def test_planted_wrong_reseed_breaks_losslessness(tiny, tiny_ar):
    """Reseeding stage 1 with the rejected draft instead of the target's argmax changes the stream."""
    w, params, prompt, models = tiny
    target, pdm = models
    P = len(prompt)
    modes = {q: ospd.FORCE_OTHER for q in range(P + 2, P + 30)}
    ref = {q: tiny_ar["tokens"][q - P - 1] for q in modes}

    class WrongReseed(ospd.SPDRun):
        def cycle(self):
            t_before = self.t
            old = {p: self.seq.get(p) for p in range(self.t - self.n + 2, self.t + 1)}
            info = super().cycle()
            if info["exited"] and not info["accept"] and old.get(self.t) is not None:
                self.seq[self.t] = old[self.t]          # keep the rejected token
                h = self.T.embed(old[self.t])
                self.resid[self.t] = h
                self.anchor[self.t] = {0: h.copy()}
            return info

    run = WrongReseed(target, pdm, w.n_stages, w.pdm_layers, w.anchors, prompt, P + 40, modes, ref)
    assert run.generate(20) != tiny_ar["tokens"][:20]
