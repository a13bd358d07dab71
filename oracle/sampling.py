"""Oracle, part 3: sampled decoding and sampled verification (temperature T > 0).

TEST INFRASTRUCTURE ONLY (see ``oracle/model.py``): only the tests, the smoke
check and the bench's CPU baseline use it.  Plain numpy, written from the pages:

* SPD news, section 六: under random sampling the streaming verification is the
  standard rejection sampling, and a rejected position is replaced by a token
  drawn from the target's distribution so that the output distribution equals
  plain decoding (lossless);
* the speculative-decoding engineering page (ybb.press, 打破自回归瓶颈), section
  二 2.1-2.2: accept the draft x with probability min(1, P(x)/Q(x)); on
  rejection draw from normalize(max(0, P - Q));
* SPD summary, 复现评估: decoding settings T in {0, 1}, top-k 50, top-p 1.0.

Readings taken (each also listed in the design notes):

1. A distribution is softmax(logits / T) over the k largest logits (top-p 1.0
   keeps all k).  The k are ordered by logit descending, lower token id first
   among equal logits; every draw walks them in that order.
2. Drawing with a uniform u in [0, 1): the first token whose running sum of
   weights w_i = exp(l_i - l_max) exceeds u times the total -- fp32 weights,
   fp32 running sums, in that order (the precision the CUDA path decides in).
3. The pages' "resample from the verification distribution" after a reject is
   read as the residual normalize(max(0, p - q)) of the standard rule: only
   it makes the output distribution equal p, which the pages claim.  If the
   residual mass is 0 the token is drawn from p.
4. Random numbers are inputs: per position q, u_draft[q] draws the draft for q,
   u_accept[q] and u_resample[q] verify q, u_ar[q] draws q in sampled AR.
5. The first generated token (position P+1) is the prompt's argmax in every
   mode, so sampled AR and sampled SPD share it; sampling starts at P+2.
"""
from __future__ import annotations

from typing import Dict, Optional, Sequence, Tuple

import numpy as np

F32 = np.float32


class Dist:
    """A top-k distribution: token ids in canonical order, fp32 weights, their running sums."""

    def __init__(self, logits: np.ndarray, T: float, k: int):
        logits = np.asarray(logits, dtype=np.float32)
        V = logits.shape[0]
        k = min(k, V)
        # canonical order: logit descending, then token id ascending (reading 1)
        order = np.lexsort((np.arange(V), -logits.astype(np.float64)))[:k]
        self.ids = order.astype(np.int64)
        lv = logits[order]
        if T != 1.0:
            lv = (lv / F32(T)).astype(np.float32)
        self.w = np.exp((lv - lv[0]).astype(np.float32)).astype(np.float32)
        self.cum = np.cumsum(self.w, dtype=np.float32)   # sequential running sums
        self.total = self.cum[-1]
        self.pos = {int(t): i for i, t in enumerate(self.ids)}

    def prob(self, token: int) -> np.float32:
        """p(token) = w / total in fp32; 0 outside the top k."""
        i = self.pos.get(int(token))
        return F32(0.0) if i is None else F32(self.w[i] / self.total)

    def probs(self) -> np.ndarray:
        return (self.w / self.total).astype(np.float32)


def draw(cum: np.ndarray, u: float) -> Tuple[int, float]:
    """Index of the first running sum above u x total (reading 2), and the decision's margin:
    the distance of u from the nearest boundary u_i = cum_i / total, relative to 1."""
    total = cum[-1]
    target = F32(u) * total
    i = int(np.searchsorted(cum, target, side="right"))
    i = min(i, len(cum) - 1)
    lo = F32(0.0) if i == 0 else cum[i - 1]
    margin = float(min(abs(float(target) - float(lo)), abs(float(cum[i]) - float(target))) / float(total))
    return i, margin


def sample(d: Dist, u: float) -> Tuple[int, float]:
    """A token drawn from d with uniform u; (token id, margin)."""
    i, m = draw(d.cum, u)
    return int(d.ids[i]), m


def verify(p: Dist, x: int, qx: np.float32, q_of, u_acc: float, u_res: float) -> Tuple[bool, int, float]:
    """Rejection-sampling verification of draft x (drawn with probability qx).

    Returns (accepted, committed token, margin of the decisions taken).  ``q_of(token)`` gives the
    draft distribution's probability of a token (0 outside its top k)."""
    px = p.prob(x)
    lhs = F32(u_acc) * F32(qx)
    margin = abs(float(lhs) - float(px)) / max(float(px), float(qx), 1e-30)
    if lhs < px:
        return True, int(x), margin
    # residual max(0, p - q) over the target's top k, in its canonical order (reading 3)
    pp = p.probs()
    r = np.array([max(F32(0.0), F32(pp[i] - F32(q_of(int(t))))) for i, t in enumerate(p.ids)], dtype=np.float32)
    rc = np.cumsum(r, dtype=np.float32)
    if rc[-1] <= 0:
        tok, m2 = sample(p, u_res)
        return False, tok, min(margin, m2)
    i, m2 = draw(rc, u_res)
    return False, int(p.ids[i]), min(margin, m2)


def sampled_ar(model, prompt: Sequence[int], gen: int, T: float, k: int, u_ar: Dict[int, float],
               max_len: Optional[int] = None) -> Dict:
    """Plain sampled autoregressive decoding of ``gen`` tokens (position P+1 greedy, reading 5)."""
    from oracle.model import top2
    P = len(prompt)
    cache = model.new_cache(max_len or (P + gen + 1))
    H, _ = model.prefill(prompt, cache)
    toks, margins = [top2(model.logits(H[-1]))[0]], []
    for i in range(gen - 1):
        pos = P + 1 + i
        h = model.embed(toks[-1])[None, :]
        for l in range(model.L):
            h = model.layer(l, h, [pos], cache)
        t, m = sample(Dist(model.logits(h[0]), T, k), u_ar[pos + 1])
        toks.append(t)
        margins.append(m)
    return {"tokens": toks, "margins": margins}


__all__ = ["Dist", "draw", "sample", "verify", "sampled_ar"]
