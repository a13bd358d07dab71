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
//   draft-module cache length <- the pre-step v (rows at depth n are cached, SPD v3 App. A.1).
// "Entering stage 1" writes the token's embedding into the residual ring and anchor b_0 = 0.
#include "spd_ctrl.cuh"

namespace spd {

namespace {

using ctl::push_embedding;

template <typename WT>
__global__ void __launch_bounds__(256) control_cycle_kernel(Dims D, Bufs B) {
  __shared__ Top2 red[256][2];
  __shared__ int s_tok, s_slot;
  __shared__ ctl::SampleSmem S;
  ctl::control_cycle<WT>(D, B, red, s_tok, s_slot, 256, 1, S);
}

template <typename WT>
__global__ void __launch_bounds__(256) control_ar_kernel(Dims D, Bufs B) {
  __shared__ Top2 red[256][2];
  __shared__ int s_tok, s_slot;
  __shared__ ctl::SampleSmem S;
  ctl::control_ar<WT>(D, B, red, s_tok, s_slot, 256, 1, S);
}

template <typename WT>
__global__ void prefill_embed_kernel(Dims D, Bufs B, float* h, float* anch, int pos0) {
  const int r = blockIdx.x;
  const int tok = B.seq[pos0 + r];
  const WT* e = reinterpret_cast<const WT*>(B.embed) + (size_t)tok * D.d;
  for (int c = threadIdx.x; c < D.d; c += blockDim.x) {
    const float x = WTraits<WT>::to_f(e[c]);
    h[(size_t)r * D.d + c] = x;
    anch[(size_t)r * D.m * D.d + c] = x;
  }
}

template <typename WT>
__global__ void __launch_bounds__(256) prefill_finish_kernel(Dims D, Bufs B, int P) {
  __shared__ Top2 red[256][2];
  __shared__ int s_tok;
  DevState* st = B.st;
  ctl::reduce_head(B, red, 256, 1);
  if (threadIdx.x == 0) {
    int x = red[0][0].i1;
    if (x < 0 || x >= D.V) {
      set_err(st, ERR_BOUNDS, 520);
      x = -1;
    }
    st->t = P + 1; st->a = 1; st->v = P; st->pdm_len = P; st->P = P;
    st->cycles = 0; st->exits = 0; st->rejects = 0;
    st->done = 0; st->max_commit = 0x7fffffff;
    st->last_exited = 0; st->last_exit_pos = 0; st->last_accept = 0;
    st->target_top1 = x; st->pushed = x; st->draft = -1;
    B.seq[P + 1] = x;
    for (int l = 0; l < D.L; ++l) B.kvlen[l] = P;
    s_tok = x;
  }
  __syncthreads();
  if (s_tok >= 0) push_embedding<WT>(D, B, s_tok, (P + 1) % (D.n + 1), blockDim.x);
}

template <typename WT>
__global__ void __launch_bounds__(256) rollback_kernel(Dims D, Bufs B, int keep, int reseed) {
  DevState* st = B.st;
  if (threadIdx.x == 0) {
    st->v = keep; st->t = keep + 1; st->a = 1;
    st->pdm_len = min(st->pdm_len, keep);
    st->done = 0; st->max_commit = 0x7fffffff;
    st->cycles = 0; st->exits = 0; st->rejects = 0;
    st->last_exited = 0; st->pushed = reseed;
    B.seq[keep + 1] = reseed;
    for (int l = 0; l < D.L; ++l) B.kvlen[l] = keep;
  }
  push_embedding<WT>(D, B, reseed, (keep + 1) % (D.n + 1), blockDim.x);
}

__global__ void begin_generate_kernel(Bufs B, int max_new) {
  DevState* st = B.st;
  st->max_commit = max_new;
  st->done = (st->v + 1 - st->P >= max_new) ? 1 : 0;
}

__global__ void rope_tables_kernel(float* cosv, float* sinv, int max_seq, int hd, double theta) {
  const int half = hd / 2;
  const long long total = (long long)max_seq * half;
  for (long long idx = blockIdx.x * (long long)blockDim.x + threadIdx.x; idx < total;
       idx += (long long)gridDim.x * blockDim.x) {
    const int pos = (int)(idx / half), i = (int)(idx % half);
    const double inv = pow(theta, -(2.0 * i) / (double)hd);
    const double ang = (double)pos * inv;  // position index pos = (1-based position) - 1
    cosv[idx] = (float)cos(ang);
    sinv[idx] = (float)sin(ang);
  }
}

}  // namespace

#define SPD_DISPATCH(D, KERNEL, GRID, BLOCK, STREAM, ...)                     \
  do {                                                                      \
    if ((D).dtype == SPD_DTYPE_BF16)                                        \
      KERNEL<__nv_bfloat16><<<GRID, BLOCK, 0, STREAM>>>(__VA_ARGS__);       \
    else                                                                    \
      KERNEL<float><<<GRID, BLOCK, 0, STREAM>>>(__VA_ARGS__);               \
  } while (0)

cudaError_t launch_control_cycle(const Dims& D, const Bufs& B, cudaStream_t s) {
  SPD_DISPATCH(D, control_cycle_kernel, 1, 256, s, D, B);
  return cudaGetLastError();
}
cudaError_t launch_control_ar(const Dims& D, const Bufs& B, cudaStream_t s) {
  SPD_DISPATCH(D, control_ar_kernel, 1, 256, s, D, B);
  return cudaGetLastError();
}
cudaError_t launch_prefill_embed(const Dims& D, const Bufs& B, float* h, float* anch, int pos0,
                                 int cnt, cudaStream_t s) {
  SPD_DISPATCH(D, prefill_embed_kernel, cnt, 256, s, D, B, h, anch, pos0);
  return cudaGetLastError();
}
cudaError_t launch_prefill_finish(const Dims& D, const Bufs& B, int P, cudaStream_t s) {
  SPD_DISPATCH(D, prefill_finish_kernel, 1, 256, s, D, B, P);
  return cudaGetLastError();
}
cudaError_t launch_rollback(const Dims& D, const Bufs& B, int keep_len, int reseed,
                            cudaStream_t s) {
  SPD_DISPATCH(D, rollback_kernel, 1, 256, s, D, B, keep_len, reseed);
  return cudaGetLastError();
}
cudaError_t launch_begin_generate(const Dims& D, const Bufs& B, int max_new, cudaStream_t s) {
  (void)D;
  begin_generate_kernel<<<1, 1, 0, s>>>(B, max_new);
  return cudaGetLastError();
}
cudaError_t launch_rope_tables(float* cosv, float* sinv, int max_seq, int hd, float theta,
                               cudaStream_t s) {
  rope_tables_kernel<<<256, 256, 0, s>>>(cosv, sinv, max_seq, hd, (double)theta);
  return cudaGetLastError();
}

}  // namespace spd
