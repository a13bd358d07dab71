"""Pins of the oracle's sampled decoding and verification (oracle/sampling.py).

What holds it, independent of its own code:

* the inverse-CDF draw against softmax probabilities computed in fp64 by scipy: over a fine grid of
  uniforms each token is drawn with its probability, and tokens outside the top k never are;
* the lossless property the pages claim for rejection sampling (SPD news 六; the speculative
  decoding engineering page §2.2): whatever the draft distribution q, the committed token follows
  the target distribution p -- Monte Carlo, and a planted variant that resamples from p instead of
  the residual fails the same check;
* special cases: q == p always accepts; a draft outside p's top k is always rejected;
* end to end on a micro model: the first sampled token of an SPD run follows the target's own
  distribution at that position, over many seeds; the trace keeps the refill arithmetic.
"""
import numpy as np
import pytest
from scipy.special import softmax

import spd_inputs as si
from oracle import model as om
from oracle import sampling as osm
from oracle import spd as ospd


def _tv(a, b):
    return 0.5 * float(np.abs(np.asarray(a, np.float64) - np.asarray(b, np.float64)).sum())


def _exact(logits, T, k):
    """fp64 softmax over the k largest logits, as a full-vocabulary vector."""
    logits = np.asarray(logits, np.float64)
    top = np.argsort(-logits, kind="stable")[:k]
    p = np.zeros(len(logits))
    p[top] = softmax(logits[top] / T)
    return p


@pytest.mark.parametrize("T,k", [(1.0, 20), (1.0, 6), (0.7, 20), (1.3, 9)])
def test_inverse_cdf_draws_follow_softmax(T, k):
    rng = np.random.default_rng(11)
    logits = rng.normal(0, 1.5, 20).astype(np.float32)
    d = osm.Dist(logits, T, k)
    N = 40000
    counts = np.zeros(20)
    for j in range(N):
        tok, _ = osm.sample(d, (j + 0.5) / N)
        counts[tok] += 1
    exact = _exact(logits, T, k)
    assert np.max(np.abs(counts / N - exact)) < 2.0 / N + 1e-5
    assert counts[exact == 0].sum() == 0


def test_canonical_order_and_ties():
    d = osm.Dist(np.array([0.5, 2.0, 0.5, 2.0, -1.0], np.float32), 1.0, 4)
    assert list(d.ids) == [1, 3, 0, 2]  # logit descending, lower id first among equals
    assert d.prob(4) == 0.0


def _verify_distribution(p_logits, q_logits, kp, kq, trials, seed, wrong=False):
    rng = np.random.default_rng(seed)
    p, q = osm.Dist(p_logits, 1.0, kp), osm.Dist(q_logits, 1.0, kq)
    out = np.zeros(len(p_logits))
    acc = 0
    for _ in range(trials):
        u = rng.random(3)
        x, _ = osm.sample(q, u[0])
        ok, tok, _ = osm.verify(p, x, q.prob(x), q.prob, u[1], u[2])
        if wrong and not ok:
            tok, _ = osm.sample(p, u[2])  # planted: resample from p instead of the residual
        out[tok] += 1
        acc += ok
    return out / trials, _exact(p_logits, 1.0, kp), acc / trials


@pytest.mark.parametrize("kp,kq", [(12, 12), (6, 12), (12, 5)])
def test_rejection_sampling_keeps_target_distribution(kp, kq):
    rng = np.random.default_rng(kp * 100 + kq)
    p_logits = rng.normal(0, 1.2, 12).astype(np.float32)
    q_logits = rng.normal(0, 1.2, 12).astype(np.float32)
    emp, exact, acc = _verify_distribution(p_logits, q_logits, kp, kq, 30000, 3)
    assert _tv(emp, exact) < 0.015
    # and the acceptance rate is the overlap sum_x min(p(x), q(x))
    assert abs(acc - np.minimum(exact, _exact(q_logits, 1.0, kq)).sum()) < 0.015


def test_planted_resample_from_p_is_caught():
    rng = np.random.default_rng(7)
    p_logits = rng.normal(0, 2.0, 12).astype(np.float32)
    q_logits = rng.normal(0, 2.0, 12).astype(np.float32)
    emp, exact, _ = _verify_distribution(p_logits, q_logits, 12, 12, 30000, 4, wrong=True)
    assert _tv(emp, exact) > 0.05


def test_verify_special_cases():
    rng = np.random.default_rng(5)
    logits = rng.normal(0, 1.0, 16).astype(np.float32)
    p = osm.Dist(logits, 1.0, 8)
    for u in np.linspace(0.0, 0.999, 50):
        x, _ = osm.sample(p, float(u))
        ok, tok, _ = osm.verify(p, x, p.prob(x), p.prob, float(u), 0.5)  # q == p
        assert ok and tok == x
    outside = int(np.argsort(logits)[0])  # lowest logit: outside p's top 8
    q = osm.Dist(-logits, 1.0, 8)           # a draft distribution that has it
    for u in np.linspace(0.0, 0.999, 20):
        ok, tok, _ = osm.verify(p, outside, q.prob(outside), q.prob, float(u), float(u))
        assert not ok and p.prob(tok) > 0


def _micro():
    cfg = si.small_model(n_layers=2, d_model=8, n_heads=2, n_kv_heads=1, head_dim=4,
                         d_ffn=16, vocab=16, init_std=0.5)
    w = si.Workload("micro", cfg, 2, 1, (0, 1, 2), 2, 6, (0.5,))
    params = si.generate_weights(w)
    return w, ospd.build(w, params)


def test_sampled_spd_first_token_follows_target_distribution():
    w, (target, pdm) = _micro()
    prompt = [3, 9]
    P, n, k = len(prompt), w.n_stages, 12
    first = om.greedy_ar(target, prompt, 1)["tokens"][0]
    # the target's distribution of position P+2 after the prompt and the greedy token P+1
    cache = target.new_cache(P + 4)
    H, _ = target.prefill(prompt + [first], cache)
    exact = _exact(target.logits(H[-1]), 1.0, k)
    runs = 2500
    counts = np.zeros(16)
    for s in range(runs):
        u = si.sampling_uniforms(1000 + s, P + 1, P + 8)
        smp = {"T": 1.0, "k": k}
        for name in ("draft", "accept", "resample"):
            smp["u_" + name] = {q: v for q, v in zip(range(P + 1, P + 9), u[name])}
        run = ospd.SPDRun(target, pdm, n, 1, w.anchors, prompt, P + 10, sampling=smp)
        toks = run.generate(2)
        counts[toks[1]] += 1
        accepted = [ok for _, ok in run.trace]
        assert run.cycles == ospd.expected_cycles(n, accepted)
    assert _tv(counts / runs, exact) < 0.04


def test_sampled_spd_trace_and_cycles_tiny(tiny):
    w, params, prompt, models = tiny
    P, G = len(prompt), 24
    u = si.sampling_uniforms(77, P + 1, P + G + w.n_stages + 2)
    smp = {"T": 1.0, "k": 50}
    for name in ("draft", "accept", "resample"):
        smp["u_" + name] = {q: v for q, v in zip(range(P + 1, P + G + w.n_stages + 3), u[name])}
    run = ospd.run_spd(w, params, prompt, G, None, models=models, sampling=smp)
    assert len(run.committed) >= G
    assert [q for q, _ in run.trace] == list(range(P + 2, P + 2 + len(run.trace)))
    assert run.cycles == ospd.expected_cycles(w.n_stages, [ok for _, ok in run.trace])
