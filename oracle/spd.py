"""Oracle, part 2: the Speculative Pipeline Decoding cycle.

TEST INFRASTRUCTURE ONLY (see ``oracle/model.py``).  Plain fp32 CPU code that
walks the method's steps in the pages' order.  Page references use the page
title and section:

* "SPD summary" -- the rainbus.top page 投机式流水线解码 (Speculative Pipeline
  Decoding: Higher-Accruacy and Zero-Bubble Speculation via Pipeline
  Parallelism), sections 核心方法 and 方法步骤详情 (the six steps).
* "SPD news" -- the techwalker.com article on arXiv 2605.30852, sections 三-八.
* "SPD v3" -- the paperlayer.ai summary of arXiv 2605.30852v3, sections 3.1-3.4,
  section 4 (the scheduling ablation) and Appendix A.1-A.3.

Readings taken where the pages are silent or loose (each also listed in the
design notes):

1. Anchor state h^(b) is the residual stream after b decoder layers, before any
   norm; b = 0 is the token embedding (SPD v3 §3.2: at k = 0 the feature is an
   embedding projection).
2. Depth of row i before a step with newest position t and fill a: t - i when
   t - i < a, else n (the structural-mask rule of SPD v3 App. A.3 with the
   warm-up prefix at depth n of App. A.2; steady state gives the staircase of
   SPD summary step 2).
3. FC_j maps the concatenation of anchors b_0..b_j (in that order, no norm, no
   bias) to d; one FC per anchor count, shared by all depths with the same f
   (SPD summary step 3: m fusion projections).  The draft module's layers have
   the target layer's shape; it ends with its own final norm and LM head, and
   row t's output is the draft for position t+1 (SPD summary step 4).
4. Rows at depth n (verified) keep their draft-module KV; each cycle recomputes
   the rows from the first not-yet-cached verified row to t (SPD v3 App. A.1).
5. Rollback length "t-n+1" is the position of the exiting token (equal to
   t-n+1 when the pipeline is full); the greedy "resample" is the argmax.
6. Seeded acceptance (a harness knob, not on the pages): the draft for
   position q is replaced by the reference token when mode[q] = FORCE_REF,
   and by the draft module's best-ranked token other than the reference when
   mode[q] = FORCE_OTHER.
7. Post-step schedule (the ablation of SPD v3 §4 and SPD news 十: the draft
   module waits for the target step and reads its output state).  The pages
   give only its effect, so the plainest reading is taken: after the step, an
   in-flight row i has depth t - i + 1 (one stage more), the exiting row is
   at depth n, the verified prefix stays at n; the rows processed are the same
   ones (first not-yet-cached row to t), and the exiting row, which is
   committed whatever the verdict on its successor, joins the draft-module
   cache.  The draft still enters stage 1 at the end of the cycle and a
   rejected cycle's draft is discarded, so the cycle count is unchanged.
8. Sampled decoding (T > 0): drafts are drawn from the draft module's top-k
   distribution and verified by rejection sampling (oracle/sampling.py); the
   streaming order, the rollback and the cycle arithmetic are unchanged.
"""
from __future__ import annotations

from typing import Dict, List, Optional, Sequence, Tuple

import numpy as np

from .model import Decoder, KVCache, _f32, greedy_ar, top2
from . import sampling as osm

# draft-override modes (same values as spd_inputs.DRAFT_*)
RAW, FORCE_REF, FORCE_OTHER = 0, 1, 2


# ---------------------------------------------------------------------------
# anchor selection -- SPD summary, 核心方法 / step 3 (Eq. 6, 7)
# ---------------------------------------------------------------------------
def lmax(k: int, L: int, n: int) -> int:
    """Deepest layer reachable at pipeline depth k: min(L, k*L/n)."""
    return min(L, k * L // n)


def f_of(k: int, L: int, n: int, B: Sequence[int]) -> int:
    """f(k) = max{ i : b_i <= lmax(k) }."""
    lm = lmax(k, L, n)
    return max(i for i, b in enumerate(B) if b <= lm)


def f_table(L: int, n: int, B: Sequence[int]) -> List[int]:
    return [f_of(k, L, n, B) for k in range(n + 1)]


def check_config(L: int, n: int, Ls: int, B: Sequence[int]) -> None:
    """n | L, 1 <= Ls <= L/n (masking condition, SPD summary 核心方法), anchors valid."""
    if n < 1 or L % n != 0:
        raise ValueError(f"n={n} must divide L={L}")
    if not (1 <= Ls <= L // n):
        raise ValueError(f"draft depth Ls={Ls} must satisfy 1 <= Ls <= L/n = {L // n}")
    if len(B) < 1 or B[0] != 0 or any(b1 <= b0 for b0, b1 in zip(B, B[1:])) or B[-1] > L:
        raise ValueError(f"anchors {B} must start at 0, increase strictly and end <= L")


# ---------------------------------------------------------------------------
# depth staircase -- SPD summary step 2 / 6 (Eq. 3, 8), SPD v3 App. A.2-A.3
# ---------------------------------------------------------------------------
def depth_of(i: int, t: int, a: int, n: int) -> int:
    """Pre-step depth of row i: t-i for the a in-flight rows, n for the verified prefix."""
    return t - i if t - i < a else n


def depth_after_step(i: int, t: int, a: int, n: int) -> int:
    """Depth of row i after the step (post-step schedule, reading 7): in-flight rows one stage deeper."""
    return t - i + 1 if t - i < a else n


# ---------------------------------------------------------------------------
# draft module (PDM)
# ---------------------------------------------------------------------------
class DraftModule:
    """Anchor FCs, Ls causal decoder layers, final norm and its own LM head."""

    def __init__(self, cfg, params: Dict, Ls: int, m: int):
        self.fc = [(_f32(params[f"pdm.fc.{j}"]) if f"pdm.fc.{j}" in params else None)
                   for j in range(m)]
        self.stack = Decoder(cfg, params, n_layers=Ls, prefix="pdm.", with_embedding=False,
                             norm_name="norm", head_name="lm_head")

    def feature(self, anchor_states: Dict[int, np.ndarray], B: Sequence[int], f: int) -> np.ndarray:
        """FC_f applied to concat(h^(b_0), ..., h^(b_f)) of one position."""
        x = np.concatenate([anchor_states[B[i]] for i in range(f + 1)]).astype(np.float32)
        return (self.fc[f] @ x).astype(np.float32)

    def forward(self, Z: np.ndarray, positions: Sequence[int], cache: KVCache) -> np.ndarray:
        for l in range(self.stack.L):
            Z = self.stack.layer(l, Z, positions, cache)
        return Z


# ---------------------------------------------------------------------------
# the SPD decoding loop
# ---------------------------------------------------------------------------
class SPDRun:
    """Greedy SPD on one sequence, cycle by cycle.

    State before a cycle: newest in-flight position t, fill a (positions
    t-a+1..t in flight), verified length v = t-a, draft-module cache length
    ``pdm_len`` (rows at depth n whose draft-module KV is kept).
    """

    def __init__(self, target: Decoder, pdm: DraftModule, n: int, Ls: int, B: Sequence[int],
                 prompt: Sequence[int], max_len: int,
                 modes: Optional[Dict[int, int]] = None, ref: Optional[Dict[int, int]] = None,
                 check_full_recompute: bool = False, record: bool = False, post_step: bool = False,
                 sampling: Optional[Dict] = None):
        """``sampling``: None for greedy decoding, else {"T": temperature, "k": top-k, "u_draft",
        "u_accept", "u_resample": {position: uniform}} (oracle/sampling.py; the harness modes
        are not used then)."""
        L = target.L
        check_config(L, n, Ls, B)
        self.T, self.pdm, self.n, self.S, self.B = target, pdm, n, L // n, list(B)
        self.L, self.m = L, len(B)
        self.ftab = f_table(L, n, B)
        self.modes, self.ref = modes or {}, ref or {}
        self.check_full = check_full_recompute
        self.record = record
        self.post_step = post_step
        self.sampling = sampling
        self.qdist: Dict[int, "osm.Dist"] = {}   # draft distribution of each drafted position
        self.margins: List[Tuple[int, float]] = []  # (position, distance of a sampled decision from a boundary)
        self.P = len(prompt)
        # prefill: the prompt passes all L layers (verified prefix)
        self.cache = target.new_cache(max_len)
        H, states = target.prefill(prompt, self.cache, anchors=self.B)
        self.anchor: Dict[int, Dict[int, np.ndarray]] = states
        self.seq: Dict[int, int] = {p + 1: int(tok) for p, tok in enumerate(prompt)}
        self.done_layers: Dict[int, int] = {p: L for p in range(1, self.P + 1)}
        first = top2(target.logits(H[-1]))[0]
        # draft-module prefix: rows 1..P at depth n (feature reuse, SPD v3 App. A.1)
        self.pdm_cache = pdm.stack.new_cache(max_len)
        fn = self.ftab[n]
        Z = np.stack([pdm.feature(self.anchor[p], self.B, fn) for p in range(1, self.P + 1)])
        pdm.forward(Z, list(range(1, self.P + 1)), self.pdm_cache)
        self.pdm_len = self.P
        # pipeline holds the first generated token at depth 0
        self.t, self.a, self.v = self.P, 0, self.P
        self.resid: Dict[int, np.ndarray] = {}
        self._push(first)
        self.cycles = 0
        self.trace: List[Tuple[int, bool]] = []   # (verified position, accepted)
        self.rejects = 0
        self.log: List[Dict] = []

    # -- helpers ------------------------------------------------------------
    def _push(self, token: int) -> None:
        """A token enters stage 1 at position t+1 with only its embedding (g_0)."""
        self.t += 1
        self.a += 1
        p = self.t
        self.seq[p] = int(token)
        h = self.T.embed(token)
        self.resid[p] = h
        self.anchor[p] = {0: h.copy()} if 0 in self.B else {}
        self.done_layers[p] = 0

    @property
    def committed(self) -> List[int]:
        """Generated tokens known correct: positions P+1 .. v+1."""
        return [self.seq[p] for p in range(self.P + 1, self.v + 2)]

    def _depth(self, i: int) -> int:
        # t and a are those of the pre-step state in both schedules (the step does not change them)
        return (depth_after_step if self.post_step else depth_of)(i, self.t, self.a, self.n)

    def staircase(self) -> List[Tuple[int, int]]:
        """(position, depth) of the rows the draft module processes this cycle (at the time it runs)."""
        return [(i, self._depth(i)) for i in range(self.pdm_len + 1, self.t + 1)]

    def _draft_module(self) -> Tuple[List[Tuple[int, int]], np.ndarray, Tuple[int, int, float, float]]:
        """Steps 2-4: rows, anchor features, the Ls layers over the cached prefix, the head of row t."""
        n, S = self.n, self.S
        rows = self.staircase()
        # the closed-form staircase must agree with how far each row has actually run
        for i, k in rows:
            if self.done_layers[i] != (self.L if k == n else k * S):
                raise AssertionError(f"row {i}: depth {k} but {self.done_layers[i]} layers done")
        self.pdm_cache.truncate(self.pdm_len)
        Z = np.stack([self.pdm.feature(self.anchor[i], self.B, self.ftab[k]) for i, k in rows])
        Z = self.pdm.forward(Z, [i for i, _ in rows], self.pdm_cache)
        if self.check_full:
            self._check_full_recompute(rows, Z)
        self._pdm_logits = self.pdm.stack.logits(Z[-1])
        return rows, Z, top2(self._pdm_logits)

    def _draft(self, top1: int, top2_: int) -> int:
        q = self.t + 1
        mode = self.modes.get(q, RAW)
        if mode == FORCE_REF:
            return self.ref[q]
        if mode == FORCE_OTHER:
            return top1 if top1 != self.ref[q] else top2_
        return top1

    # -- one cycle ----------------------------------------------------------
    def cycle(self) -> Dict:
        n, S, t, a, v = self.n, self.S, self.t, self.a, self.v
        if not self.post_step:
            # (step 2-4) draft module on pre-step features, concurrently with the target step
            rows, Z, (p1, p2, pv1, pv2) = self._draft_module()
        # rows at depth n when the draft module ran keep their draft-module KV
        pdm_len_next = v + 1 if (self.post_step and a == n) else v
        # (step 1) target step: the token at depth j runs layers j*S .. j*S+S-1
        for j in range(a):
            p = t - j
            h = self.resid[p][None, :]
            for l in range(j * S, j * S + S):
                h = self.T.layer(l, h, [p], self.cache)
                if (l + 1) in self.B:
                    self.anchor[p][l + 1] = h[0].copy()
            self.resid[p] = h[0]
            self.done_layers[p] += S
        if self.post_step:
            # post-step schedule: the draft module waits for the step and reads its output state
            rows, Z, (p1, p2, pv1, pv2) = self._draft_module()
        if self.sampling is None:
            draft = self._draft(p1, p2)
        else:
            # the draft for t+1 is drawn from the draft module's top-k distribution of row t
            smp = self.sampling
            dq = osm.Dist(self._pdm_logits, smp["T"], smp["k"])
            draft, m = osm.sample(dq, smp["u_draft"][t + 1])
            self.qdist[t + 1] = dq
            self.margins.append((t + 1, m))
        info = {"t": t, "a": a, "rows": rows, "pdm_top": (p1, p2), "pdm_gap": pv1 - pv2,
                "draft": draft, "exited": a == n}
        if self.record:
            info["pdm_z"] = Z.copy()
        # (step 5) streaming verification
        if a == n:
            te = t - n + 1
            tl = self.T.logits(self.resid[te])
            i1, i2, v1, v2 = top2(tl)
            succ = self.seq[te + 1] if te + 1 <= t else draft
            if self.sampling is None:
                accept, reseed = succ == i1, i1
            else:
                # rejection sampling against the target's top-k distribution at t_e
                smp = self.sampling
                pd = osm.Dist(tl, smp["T"], smp["k"])
                dq = self.qdist[te + 1]
                accept, reseed, m = osm.verify(pd, succ, dq.prob(succ), dq.prob,
                                               smp["u_accept"][te + 1], smp["u_resample"][te + 1])
                self.margins.append((te + 1, m))
            self.trace.append((te + 1, accept))
            info.update(exit_pos=te, target_top=(i1, i2), target_gap=v1 - v2, accept=accept)
            del self.resid[te]
            self.v = te
            if accept:
                self.a -= 1
                self._push(draft)
            else:
                # three-step rollback: (i) truncate KV, (ii) flush in-flight, (iii) reseed
                self.rejects += 1
                self.cache.truncate(te)
                for p in range(te + 1, t + 1):
                    self.resid.pop(p, None)
                    self.anchor.pop(p, None)
                    self.done_layers.pop(p, None)
                    self.seq.pop(p, None)
                self.t, self.a = te, 0
                self._push(reseed)
        else:
            self._push(draft)
        self.pdm_len = pdm_len_next
        self.cycles += 1
        if self.record:
            self.log.append(info)
        return info

    def _check_full_recompute(self, rows, Z_inc: np.ndarray) -> None:
        """Draft-module rows recomputed from scratch over the whole G_t must equal the incremental ones."""
        all_rows = [(i, self._depth(i)) for i in range(1, self.t + 1)]
        cache = self.pdm.stack.new_cache(self.t + 1)
        Z = np.stack([self.pdm.feature(self.anchor[i], self.B, self.ftab[k]) for i, k in all_rows])
        Z = self.pdm.forward(Z, [i for i, _ in all_rows], cache)
        tail = Z[len(all_rows) - len(rows):]
        err = float(np.max(np.abs(tail - Z_inc)) / max(1e-30, float(np.max(np.abs(tail)))))
        if err > 1e-5:
            raise AssertionError(f"incremental draft rows differ from full recompute: rel {err:.3g}")

    def generate(self, gen: int, max_cycles: Optional[int] = None) -> List[int]:
        """Run cycles until ``gen`` tokens after the prompt are committed."""
        while self.v + 1 - self.P < gen:
            if max_cycles is not None and self.cycles >= max_cycles:
                break
            self.cycle()
        return self.committed[:gen]


def expected_cycles(n: int, accepted: Sequence[bool]) -> int:
    """Cycle count for positions P+2..P+G verified in order with the given outcomes.

    The first exit comes n cycles after prefill; after an accept the next exit is
    one cycle later, after a reject n cycles later (refill).  ``accepted`` lists
    the outcomes for positions P+2..P+G; the last outcome ends the run.
    """
    if not accepted:
        return 0
    return n + sum(1 if ok else n for ok in accepted[:-1])


def build(workload, params: Dict):
    """Target decoder and draft module of a workload from its parameter dict."""
    target = Decoder(workload.model, params)
    pdm = DraftModule(workload.model, params, workload.pdm_layers, len(workload.anchors))
    return target, pdm


def run_spd(workload, params: Dict, prompt: Sequence[int], gen: int, alpha: Optional[float],
            ref: Optional[Sequence[int]] = None, coin_seed: Optional[int] = None,
            check_full_recompute: bool = False, record: bool = False, models=None,
            post_step: bool = False, sampling: Optional[Dict] = None) -> SPDRun:
    """SPD greedy decode; with ``alpha`` set, drafts follow the seeded-acceptance modes."""
    import spd_inputs as si
    target, pdm = models if models is not None else build(workload, params)
    P = len(prompt)
    modes, refd = {}, {}
    if alpha is not None:
        seed = workload.coin_seed if coin_seed is None else coin_seed
        first, last = P + 2, P + gen
        for q, md in zip(range(first, last + 1), si.override_modes(seed, alpha, first, last)):
            modes[q] = md
            refd[q] = int(ref[q - P - 1])
    run = SPDRun(target, pdm, workload.n_stages, workload.pdm_layers, workload.anchors, prompt,
                 max_len=P + gen + workload.n_stages + 2, modes=modes, ref=refd,
                 check_full_recompute=check_full_recompute, record=record, post_step=post_step,
                 sampling=sampling)
    run.generate(gen)
    return run


__all__ = ["lmax", "f_of", "f_table", "check_config", "depth_of", "depth_after_step", "DraftModule", "SPDRun",
           "expected_cycles", "build", "run_spd", "greedy_ar", "RAW", "FORCE_REF", "FORCE_OTHER"]
