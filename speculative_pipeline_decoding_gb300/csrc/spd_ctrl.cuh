// Device-resident control of the SPD cycle: streaming verification, accept / three-step rollback,
// reseeding stage 1, and the bookkeeping the next cycle reads.  One block; it runs after the head
// launch of each cycle, so the host never synchronises between cycles.
//
// Cycle transition (SPD summary, 方法步骤详情 steps 1 and 5; SPD v3 §3.4):
//   pre-step state: newest position t, fill a, verified length v = t - a.
//   exit iff a == n: the token at t_e = t-n+1 has passed all L layers; y = argmax of its logits.
//     successor = token at t_e+1 (in flight, or this cycle's draft when n == 1).
//     accept (successor == y): v <- t_e, a <- a-1, then the draft enters stage 1.
//     reject: (i) every layer's KV length <- t_e (length-only: entries past it are never read and
//             are overwritten later), (ii) in-flight states flushed (a <- 0, t <- t_e),
//             (iii) y enters stage 1 at t_e+1; this cycle's draft is discarded.
//   no exit (warm-up / refill, a < n): the draft enters stage 1.
//   draft-module cache length <- the pre-step v (rows at depth n are cached, SPD v3 App. A.1); in
//   the post-step schedule the exiting row t_e was at depth n when the draft module ran, so <- t_e.
// "Entering stage 1" writes the token's embedding into the residual ring and anchor b_0 = 0.
//   sampled decoding (T > 0): the draft is drawn from the draft module's top-k distribution,
//   which is kept (slot q % (n+1)) until position q is verified; verification accepts with
//   probability min(1, p/q) and a reject reseeds with a draw from max(0, p - q) (spd_sample.cuh).
#pragma once
#include "spd_internal.cuh"
#include "spd_sample.cuh"

namespace spd {
namespace ctl {

template <typename WT>
static __device__ void push_embedding(const Dims& D, const Bufs& B, int tok, int slot, int nthreads) {
  const WT* e = reinterpret_cast<const WT*>(B.embed) + (size_t)tok * D.d;
  float* r = B.resid + (size_t)slot * D.d;
  float* a0 = B.anch + (size_t)slot * D.m * D.d;
  for (int c = threadIdx.x; c < D.d; c += nthreads) {
    const float x = WTraits<WT>::to_f(e[c]);
    r[c] = x;
    a0[c] = x;
  }
}

// Tree reduction of the per-CTA head partials over `nthreads` (a power of two) threads.
static __device__ void reduce_head(const Bufs& B, Top2 (*red)[2], int nthreads, int bar) {
  Top2 acc[2];
  top2_init(acc[0]);
  top2_init(acc[1]);
  for (int c = threadIdx.x; c < B.head_grid; c += nthreads) {
    const float* hp = B.head_part + (size_t)c * 8;
    for (int k = 0; k < 2; ++k) {
      Top2 t;
      t.v1 = hp[k * 4 + 0]; t.i1 = __float_as_int(hp[k * 4 + 1]);
      t.v2 = hp[k * 4 + 2]; t.i2 = __float_as_int(hp[k * 4 + 3]);
      top2_merge(acc[k], t);
    }
  }
  red[threadIdx.x][0] = acc[0];
  red[threadIdx.x][1] = acc[1];
  named_bar(bar, nthreads);
  for (int s = nthreads / 2; s > 0; s >>= 1) {
    if ((int)threadIdx.x < s) {
      top2_merge(red[threadIdx.x][0], red[threadIdx.x + s][0]);
      top2_merge(red[threadIdx.x][1], red[threadIdx.x + s][1]);
    }
    named_bar(bar, nthreads);
  }
}

// Shared memory of the sampled control step: one selection, the target's distribution (p) and
// the draft module's (q), and the residual weights max(0, p_i - q(id_i)) of p's tokens.
struct SampleSmem {
  smp::Sel sel;
  smp::Dist p, q;
  float resid[kMaxTopK];
};

// Block-wide part of a sampled control step: the distributions, then (cycle with an exit) the
// residual weights of p against the stored draft distribution of the verified position.
static __device__ void sampled_prologue(const Dims& D, const Bufs& B, SampleSmem& S, bool cycle, int nthreads,
                                        int bar) {
  const DevState* st = B.st;
  const int t = st->t, a = st->a, n = D.n;
  const int k = min(D.top_k, D.V);
  const bool target_only = (st->flags & SF_TARGET_ONLY) != 0;
  const bool q_now = cycle && !target_only;
  const bool p_now = !cycle || a == n;
  if (q_now) smp::topk_select(B.logits + D.V, D.V, k, D.temp, S.sel, S.q, nthreads, bar);
  if (p_now) smp::topk_select(B.logits, D.V, k, D.temp, S.sel, S.p, nthreads, bar);
  if (threadIdx.x == 0) {
    if (q_now) smp::dist_weights(S.q);
    if (p_now) smp::dist_weights(S.p);
  }
  named_bar(bar, nthreads);
  if (cycle && a == n && (int)threadIdx.x < k) {
    const int i = threadIdx.x, te = t - n + 1;
    const float pi = S.p.w[i] / S.p.cum[k - 1];
    float qi;
    if (te + 1 <= t) {  // the successor was drafted in an earlier cycle: its stored distribution
      const int slot = (te + 1) % (n + 1);
      qi = smp::stored_prob(B.q_id + slot * kMaxTopK, B.q_prob + slot * kMaxTopK, k, S.p.id[i]);
    } else {            // n == 1: this cycle's draft
      qi = target_only ? (S.p.id[i] == B.seq[t] ? 1.f : 0.f) : smp::prob_of(S.q, S.p.id[i]);
    }
    S.resid[i] = fmaxf(0.f, pi - qi);
  }
  named_bar(bar, nthreads);
}

// One SPD cycle's control step on `nthreads` threads (a power of two; `red` holds nthreads x 2;
// `S` is shared-memory scratch of the sampled step, untouched in greedy decoding).
template <typename WT>
static __device__ void control_cycle(const Dims& D, const Bufs& B, Top2 (*red)[2], int& s_tok, int& s_slot,
                              int nthreads, int bar, SampleSmem& S) {
  DevState* st = B.st;
  if (st->done || st->err) return;
  reduce_head(B, red, nthreads, bar);
  const bool sampled = D.top_k > 0;
  if (sampled) sampled_prologue(D, B, S, true, nthreads, bar);
  if (threadIdx.x == 0) {
    const int n = D.n, P = st->P;
    int t = st->t, a = st->a, v = st->v;
    const int v_pre = v;
    const bool target_only = (st->flags & SF_TARGET_ONLY) != 0;
    const bool post = (st->flags & SF_POST_STEP) != 0;
    int pdm_next = v_pre;
    s_tok = -1;
    if (t + 1 > D.max_seq) {
      set_err(st, ERR_BOUNDS, 500);
    } else {
      int p1 = red[0][1].i1, p2 = red[0][1].i2;
      if (target_only) p1 = p2 = B.seq[t];
      const int q = t + 1;
      const int mode = B.ovr_mode[q];
      const int ref = B.ovr_ref[q];
      int draft = p1;
      if (mode == 1) draft = ref;
      else if (mode == 2) draft = target_only ? (ref + 1) % D.V : ((p1 != ref) ? p1 : p2);
      const int topk = min(D.top_k, D.V);
      if (sampled) {
        // draw the draft for q = t+1 and keep its distribution until q is verified
        int* qid = B.q_id + (q % (n + 1)) * kMaxTopK;
        float* qp = B.q_prob + (q % (n + 1)) * kMaxTopK;
        if (target_only) {  // no draft module: the draft is a point mass on the token at t
          draft = B.seq[t];
          for (int i = 0; i < topk; ++i) { qid[i] = i ? -1 : draft; qp[i] = i ? 0.f : 1.f; }
        } else {
          draft = S.q.id[smp::draw(S.q.cum, topk, B.u_smp[(size_t)q])];
          for (int i = 0; i < topk; ++i) { qid[i] = S.q.id[i]; qp[i] = S.q.w[i] / S.q.cum[topk - 1]; }
        }
      }
      st->pdm_top1 = p1; st->pdm_top2 = p2; st->draft = draft;
      int push = draft;
      if (a == n) {
        const int te = t - n + 1;
        const int y = red[0][0].i1;  // the target's argmax at t_e
        const int succ = (te + 1 <= t) ? B.seq[te + 1] : draft;
        int accept = succ == y;
        int reseed = y;              // greedy: the argmax re-seeds stage 1 after a reject
        if (sampled) {
          // rejection sampling: accept iff u * q(succ) < p(succ); else a draw from the residual
          const size_t L = (size_t)D.max_seq + 2;
          const int slot = (te + 1) % (n + 1);
          const float qx = smp::stored_prob(B.q_id + slot * kMaxTopK, B.q_prob + slot * kMaxTopK, topk, succ);
          const float px = smp::prob_of(S.p, succ);
          accept = B.u_smp[L + te + 1] * qx < px;
          if (!accept) {
            float c = 0.f;
            for (int i = 0; i < topk; ++i) { c += S.resid[i]; S.resid[i] = c; }
            const float u = B.u_smp[2 * L + te + 1];
            reseed = (c > 0.f) ? S.p.id[smp::draw(S.resid, topk, u)] : S.p.id[smp::draw(S.p.cum, topk, u)];
          }
        }
        const int k = st->exits;
        if (k < D.max_seq) {
          B.trace[k] = te + 1;
          B.trace[D.max_seq + k] = accept;
        }
        st->exits = k + 1;
        st->last_exited = 1; st->last_exit_pos = te; st->last_accept = accept; st->target_top1 = y;
        v = te;
        if (post) pdm_next = te;
        if (accept) {
          a -= 1;
        } else {
          st->rejects += 1;
          for (int l = 0; l < D.L; ++l) B.kvlen[l] = te;
          a = 0;
          t = te;
          push = reseed;
        }
      } else {
        st->last_exited = 0; st->last_exit_pos = 0; st->last_accept = 0;
      }
      if (push < 0 || push >= D.V) {  // e.g. non-finite logits left no valid argmax
        set_err(st, ERR_BOUNDS, 501);
        push = -1;
      }
      if (!target_only) st->pdm_len = pdm_next;
      t += 1;
      a += 1;
      B.seq[t] = push;
      st->pushed = push;
      st->t = t; st->a = a; st->v = v;
      st->cycles += 1;
      if (v + 1 - P >= st->max_commit) st->done = 1;
      s_tok = push;
      s_slot = t % (n + 1);
    }
  }
  named_bar(bar, nthreads);
  if (s_tok >= 0) push_embedding<WT>(D, B, s_tok, s_slot, nthreads);
}

// One plain greedy AR step's control on `nthreads` threads.
template <typename WT>
static __device__ void control_ar(const Dims& D, const Bufs& B, Top2 (*red)[2], int& s_tok, int& s_slot,
                           int nthreads, int bar, SampleSmem& S) {
  DevState* st = B.st;
  if (st->done || st->err) return;
  reduce_head(B, red, nthreads, bar);
  const bool sampled = D.top_k > 0;
  if (sampled) sampled_prologue(D, B, S, false, nthreads, bar);
  if (threadIdx.x == 0) {
    s_tok = -1;
    const int t = st->t;
    if (t + 1 > D.max_seq) {
      set_err(st, ERR_BOUNDS, 510);
    } else {
      // greedy: the argmax; sampled: a draw from the top-k distribution with u_ar of position t+1
      const int y = sampled ? S.p.id[smp::draw(S.p.cum, min(D.top_k, D.V),
                                               B.u_smp[3 * ((size_t)D.max_seq + 2) + t + 1])]
                            : red[0][0].i1;
      if (y < 0 || y >= D.V) {
        set_err(st, ERR_BOUNDS, 511);
        s_tok = -1;
      }
      st->target_top1 = y;
      st->v = t;
      st->t = t + 1;
      st->a = 1;
      B.seq[t + 1] = y;
      st->pushed = y;
      st->cycles += 1;
      if (st->v + 1 - st->P >= st->max_commit) st->done = 1;
      if (y >= 0 && y < D.V) s_tok = y;
      s_slot = (t + 1) % (D.n + 1);
    }
  }
  named_bar(bar, nthreads);
  if (s_tok >= 0) push_embedding<WT>(D, B, s_tok, s_slot, nthreads);
}

}  // namespace ctl
}  // namespace spd
