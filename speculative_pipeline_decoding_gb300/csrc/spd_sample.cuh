// Sampled decoding (temperature T > 0, top-k) for the control step: the k largest logits of a
// head, their softmax weights, inverse-CDF draws, and the rejection-sampling verification of a
// draft (SPD news 六: standard rejection sampling under random sampling, lossless; the speculative
// decoding engineering page (ybb.press 打破自回归瓶颈) §2.1-2.2: accept x with probability
// min(1, P(x)/Q(x)), else draw from normalize(max(0, P - Q)); decoding settings T in {0, 1},
// top-k 50, top-p 1.0 from SPD summary 复现评估).
//
// Conventions (shared with the plain definition the tests hold this code to):
//   * the k tokens are ordered by logit descending, lower token id first among equal logits;
//   * weights w_i = exp(l_i/T - l_0/T) in fp32, running sums in that order, fp32;
//   * a draw with uniform u takes the first token whose running sum exceeds u x total;
//   * accept draft x iff u_accept * q(x) < p(x) (fp32); on a reject draw from the residual
//     max(0, p_i - q(id_i)) over p's tokens in p's order, or from p if that mass is 0.
// The uniforms are inputs (Bufs::u_smp, by position).  One block of `nthreads` threads; every
// wait is a named barrier of that block.
#pragma once
#include "spd_internal.cuh"

namespace spd {
namespace smp {

constexpr int kCtlThreads = 256;  // threads of the control step (both control kernels and CTA 0)

struct Sel {                       // shared memory of one selection
  unsigned hist[256];
  int cnt_gt[kCtlThreads], cnt_eq[kCtlThreads];
  float val[kMaxTopK];
  int idx[kMaxTopK];
  unsigned prefix;
  int want;
};

struct Dist {                      // one head's top-k distribution, canonical order
  float l[kMaxTopK];               // logits / T
  int id[kMaxTopK];
  float w[kMaxTopK];               // exp(l_i - l_0)
  float cum[kMaxTopK];             // running sums of w
  int k;
};

// Order-preserving key of a float: a larger float has a larger key.
__device__ __forceinline__ unsigned fkey(float f) {
  const unsigned b = __float_as_uint(f);
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

// Exclusive prefix sums of a[0..n) in place (n <= kCtlThreads), Hillis-Steele on the block.
__device__ __forceinline__ int scan_excl(int* a, int n, int nthreads, int bar) {
  const int tid = threadIdx.x;
  const int mine = tid < n ? a[tid] : 0;
  named_bar(bar, nthreads);
  for (int off = 1; off < n; off <<= 1) {
    const int v = (tid < n && tid >= off) ? a[tid - off] : 0;
    named_bar(bar, nthreads);
    if (tid < n) a[tid] += v;
    named_bar(bar, nthreads);
  }
  const int total = a[n - 1];
  named_bar(bar, nthreads);
  if (tid < n) a[tid] -= mine;  // inclusive -> exclusive
  named_bar(bar, nthreads);
  return total;
}

// The k largest of L[0..V) in canonical order into D (logits, ids), on the block: a radix select
// of the k-th largest key (four 8-bit passes), a gather in index order (all keys above it, then the
// lowest-index equal ones), and a rank sort of the k.  D's weights are filled by dist_weights.
static __device__ void topk_select(const float* L, int V, int k, float T, Sel& S, Dist& D, int nthreads, int bar) {
  const int tid = threadIdx.x;
  if (tid == 0) { S.prefix = 0u; S.want = k; }
  unsigned mask = 0u;
  for (int pass = 0; pass < 4; ++pass) {
    const int shift = 24 - 8 * pass;
    for (int b = tid; b < 256; b += nthreads) S.hist[b] = 0u;
    named_bar(bar, nthreads);
    const unsigned prefix = S.prefix;
    for (int i = tid; i < V; i += nthreads) {
      const unsigned key = fkey(__ldcg(L + i));
      if ((key & mask) == prefix) atomicAdd(&S.hist[(key >> shift) & 255u], 1u);
    }
    named_bar(bar, nthreads);
    if (tid == 0) {
      int cum = 0, want = S.want, b = 255;
      for (; b > 0; --b) {
        if (cum + (int)S.hist[b] >= want) break;
        cum += (int)S.hist[b];
      }
      S.want = want - cum;
      S.prefix = prefix | ((unsigned)b << shift);
    }
    mask |= 255u << shift;
    named_bar(bar, nthreads);
  }
  const unsigned kth = S.prefix;
  const int n_eq_take = S.want, n_gt = k - S.want;
  // gather: thread t owns indices [t*C, (t+1)*C)
  const int C = (V + nthreads - 1) / nthreads;
  const int i0 = min(V, tid * C), i1 = min(V, i0 + C);
  int g = 0, e = 0;
  for (int i = i0; i < i1; ++i) {
    const unsigned key = fkey(__ldcg(L + i));
    g += key > kth;
    e += key == kth;
  }
  S.cnt_gt[tid] = g;
  S.cnt_eq[tid] = e;
  scan_excl(S.cnt_gt, nthreads, nthreads, bar);
  scan_excl(S.cnt_eq, nthreads, nthreads, bar);
  int og = S.cnt_gt[tid], oe = S.cnt_eq[tid];
  for (int i = i0; i < i1; ++i) {
    const float v = __ldcg(L + i);
    const unsigned key = fkey(v);
    if (key > kth) {
      if (og < n_gt) { S.val[og] = v; S.idx[og] = i; }
      ++og;
    } else if (key == kth) {
      if (oe < n_eq_take) { S.val[n_gt + oe] = v; S.idx[n_gt + oe] = i; }
      ++oe;
    }
  }
  named_bar(bar, nthreads);
  // canonical order: rank by (logit descending, index ascending)
  if (tid < k) {
    const float v = S.val[tid];
    const int id = S.idx[tid];
    int r = 0;
    for (int j = 0; j < k; ++j) {
      const float u = S.val[j];
      r += (u > v) || (u == v && S.idx[j] < id);
    }
    D.l[r] = (T == 1.f) ? v : v / T;
    D.id[r] = id;
  }
  if (tid == 0) D.k = k;
  named_bar(bar, nthreads);
}

// Weights and running sums of D (one thread, fixed order).
__device__ __forceinline__ void dist_weights(Dist& D) {
  float c = 0.f;
  for (int i = 0; i < D.k; ++i) {
    D.w[i] = expf(D.l[i] - D.l[0]);
    c += D.w[i];
    D.cum[i] = c;
  }
}

// Index of the first running sum above u x total.
__device__ __forceinline__ int draw(const float* cum, int k, float u) {
  const float target = u * cum[k - 1];
  for (int i = 0; i < k; ++i)
    if (cum[i] > target) return i;
  return k - 1;
}

__device__ __forceinline__ float prob_of(const Dist& D, int tok) {
  for (int i = 0; i < D.k; ++i)
    if (D.id[i] == tok) return D.w[i] / D.cum[D.k - 1];
  return 0.f;
}

// q(tok) of a stored draft distribution (ids / probabilities of k entries).
__device__ __forceinline__ float stored_prob(const int* qid, const float* qp, int k, int tok) {
  for (int i = 0; i < k; ++i)
    if (qid[i] == tok) return qp[i];
  return 0.f;
}

}  // namespace smp
}  // namespace spd
