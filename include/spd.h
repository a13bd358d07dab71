/*
 * spd.h -- C ABI of the Speculative Pipeline Decoding (SPD) per-cycle engine for one GPU.
 *
 * Method (page references are to the page title and section):
 *   "SPD summary" = the rainbus.top page 投机式流水线解码 (Speculative Pipeline Decoding:
 *                   Higher-Accruacy and Zero-Bubble Speculation via Pipeline Parallelism),
 *                   sections 核心方法 and 方法步骤详情 (six steps);
 *   "SPD v3"      = the paperlayer.ai summary of arXiv 2605.30852v3, sections 3.1-3.4 and
 *                   Appendix A.1-A.3;
 *   "SPD news"    = the techwalker.com article on arXiv 2605.30852, sections 三-八.
 *
 * An L-layer decoder is cut into n stages of S = L/n layers (SPD summary 核心方法; SPD v3 §3.1).
 * n in-flight tokens of one sequence sit at depths 0..n-1.  On one GPU a cycle is a
 * stage-diagonal step: at layer offset s = 0..S-1 the token at depth j runs layer j*S+s, so
 * one cycle streams every target weight once.  Concurrently the Pipeline Draft Module (PDM)
 * builds the depth-staircase feature rows (SPD summary step 2), aggregates anchor states
 * with f(k) = max{i : b_i <= lmax(k)}, lmax(k) = min(L, k*L/n) (step 3), runs Ls <= S causal
 * layers and its own LM head (step 4) and drafts the next token.  The token leaving stage n
 * goes through the target LM head; its greedy argmax verifies its successor (step 5).  On a
 * reject every layer's KV length drops to the exiting token's position (t-n+1 with a full
 * pipeline), in-flight states are flushed and stage 1 is re-seeded with the argmax.
 *
 * Conventions
 *   - Positions are 1-based.  Token ids are int32.  RoPE uses index position-1.
 *   - Every call returns SPD_OK (0) or a negative SPD_E* code; no C++ exception crosses the ABI.
 *     spd_last_error(h) describes the last failure on a handle; spd_create failures are
 *     described by spd_last_error(NULL).
 *   - "device pointer" = memory of the GPU the handle was created on.  Calls that take
 *     host arrays copy them; the caller keeps ownership of everything it passes in.
 *   - Work is enqueued on the stream given to spd_create; calls that return host data
 *     synchronise that stream.
 *   - A handle is not thread-safe: one host thread at a time.
 */
#ifndef SPD_H
#define SPD_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define SPD_OK        0
#define SPD_EINVAL   (-1)   /* bad argument or configuration                       */
#define SPD_ENOMEM   (-2)   /* device or host allocation failed                    */
#define SPD_ECUDA    (-3)   /* a CUDA runtime call failed                          */
#define SPD_ESTATE   (-4)   /* call not valid in the current state (e.g. no prefill) */
#define SPD_ETIMEOUT (-5)   /* a bounded device wait gave up (kernel error flag)    */

#define SPD_MAX_ANCHORS 8
#define SPD_MAX_STAGES  32

enum { SPD_DTYPE_F32 = 0, SPD_DTYPE_BF16 = 1 };

/* Model, pipeline and sequence limits.  Validated by spd_create:
 *   n_stages | n_layers; 1 <= pdm_layers <= n_layers/n_stages (the masking condition of the
 *   SPD summary 核心方法: the PDM fits inside one stage forward);
 *   anchors strictly increasing, anchors[0] == 0, anchors[n_anchors-1] <= n_layers;
 *   n_heads % n_kv_heads == 0; head_dim a multiple of 64 (<= 256: a 64-row GEMV tile holds 32
 *   rows of a head and their RoPE partners); d_model, d_ffn multiples of 8 (16-byte rows for the
 *   tensor copies), 16 for bf16 models. */
typedef struct spd_config {
    int32_t n_layers;       /* L                                                */
    int32_t d_model;        /* d                                                */
    int32_t n_heads;        /* query heads                                      */
    int32_t n_kv_heads;     /* key/value heads (grouped-query attention)        */
    int32_t head_dim;       /* hd                                               */
    int32_t d_ffn;          /* SwiGLU hidden size                               */
    int32_t vocab;          /* V                                                */
    int32_t n_stages;       /* n, pipeline width                                */
    int32_t pdm_layers;     /* Ls, draft-module depth                           */
    int32_t n_anchors;      /* m                                                */
    int32_t anchors[SPD_MAX_ANCHORS]; /* B = b_0..b_{m-1}                        */
    float   rope_theta;
    float   norm_eps;
    int32_t dtype;          /* SPD_DTYPE_*: storage of matrices, embeddings, KV  */
    int32_t max_seq;        /* largest position the handle will hold            */
} spd_config;

/* One decoder layer.  Matrices are row-major [out, in] (y = W x) in cfg.dtype; norm weights
 * are fp32 [d].  Shapes: wq [Hq*hd, d], wk/wv [Hkv*hd, d], wo [d, Hq*hd],
 * w_gate/w_up [d_ffn, d], w_down [d, d_ffn].  Every pointer 16-byte aligned. */
typedef struct spd_layer_weights {
    const void *attn_norm, *wq, *wk, *wv, *wo, *ffn_norm, *w_gate, *w_up, *w_down;
} spd_layer_weights;

/* All parameters, as BORROWED device pointers: the caller owns them and keeps them alive and
 * unchanged for the handle's lifetime.  The host arrays (layers, pdm_fc, pdm_layers) are read
 * during spd_create only.
 *   embed [V, d]; final_norm [d] fp32; lm_head [V, d];
 *   pdm_fc[j] [d, (j+1)*d] (FC_j over concat(h^(b_0)..h^(b_j))), NULL allowed when no depth
 *   k has f(k) == j; pdm_norm [d] fp32; pdm_lm_head [V, d]. */
typedef struct spd_weights {
    const void* embed;
    const spd_layer_weights* layers;      /* n_layers entries  */
    const void* final_norm;
    const void* lm_head;
    const void* const* pdm_fc;            /* n_anchors entries */
    const spd_layer_weights* pdm_layers;  /* pdm_layers entries */
    const void* pdm_norm;
    const void* pdm_lm_head;
} spd_weights;

typedef struct spd_handle spd_handle;

/* What one cycle did (filled by spd_cycle when info != NULL). */
typedef struct spd_cycle_info {
    int32_t t, a, v;            /* state AFTER the cycle: newest position, fill, verified length */
    int32_t exited;             /* a token left stage n this cycle                               */
    int32_t exit_pos;           /* its position (t_e), or 0                                      */
    int32_t accepted;           /* its successor was accepted (only when exited)                 */
    int32_t target_top1;        /* target argmax at the exit (the verified next token)           */
    int32_t pdm_top1, pdm_top2; /* draft-module ranking for the next position                    */
    int32_t draft_token;        /* the draft pushed into stage 1 (or discarded on reject)        */
    int32_t pushed_token;       /* the token that entered stage 1 at position t                  */
} spd_cycle_info;

typedef struct spd_stats {
    int64_t cycles;             /* cycles run by this call                         */
    int64_t exits, rejects;     /* verifications and rejections in this call       */
    int64_t committed;          /* tokens committed after the prompt (total)       */
    double  device_ms;          /* stream time of this call (CUDA events)          */
    int64_t kernel_launches;    /* kernels this call launched (graph nodes counted) */
} spd_stats;

/* Create a handle.  `cuda_stream` is a cudaStream_t on which all work is enqueued; with NULL the
 * library creates its own blocking stream (ordered with the legacy default stream).  The library
 * makes one more stream of its own for the draft module.
 * The library OWNS and allocates: target and PDM KV caches [layers][kv_heads][max_seq][hd]
 * in cfg.dtype, the residual / anchor rings of the n+1 trailing rows, activation scratch,
 * the device control block and the CUDA graphs.  Errors: SPD_EINVAL (invalid config or NULL
 * weight), SPD_ENOMEM, SPD_ECUDA.  *out is NULL on failure. */
int spd_create(const spd_config* cfg, const spd_weights* w, void* cuda_stream, spd_handle** out);

/* Free everything the handle owns (not the borrowed weights).  NULL is a no-op. */
void spd_destroy(spd_handle* h);

/* Text of the last error on h (or of the last failed spd_create when h == NULL). */
const char* spd_last_error(const spd_handle* h);

/* Prefill `P` prompt tokens (HOST array, 1 <= P, P + n + 1 <= max_seq): runs the target over
 * positions 1..P (KV of every layer, anchor states), fills the draft module's cache with the
 * prompt rows at depth n (SPD v3 App. A.1), takes the target argmax x_{P+1} (written to
 * *first_token if non-NULL, synchronising) and leaves the pipeline reseeded: x_{P+1} at depth 0,
 * fill a = 1.  Resets counters and the draft override. */
int spd_prefill(spd_handle* h, const int32_t* tokens, int32_t P, int32_t* first_token);

/* Enqueue one SPD cycle (SPD summary steps 1-5).  With info != NULL it synchronises and reports
 * the cycle.  SPD_ESTATE before a prefill. */
int spd_cycle(spd_handle* h, spd_cycle_info* info);

/* Run SPD cycles until `max_new` tokens after the prompt are committed (the first comes from
 * the prefill).  out_tokens: NULL, or a host or device array of >= max_new int32 receiving the
 * committed tokens at positions P+1..P+max_new.  *n_out (nullable) = number written.
 * stats (nullable) is filled.  SPD_ETIMEOUT if a kernel reported a bounded-wait failure,
 * SPD_ESTATE before a prefill or when the draft-module cache is out of step (see
 * spd_generate_ar). */
int spd_generate(spd_handle* h, int32_t max_new, int32_t* out_tokens, int32_t* n_out,
                 spd_stats* stats);

/* Plain greedy autoregressive decoding with the same kernels (one token through all L layers
 * per step): the baseline SPD must reproduce token for token.  Leaves the draft-module cache
 * behind; call spd_rollback (or spd_prefill) before the next SPD call. */
int spd_generate_ar(spd_handle* h, int32_t max_new, int32_t* out_tokens, int32_t* n_out,
                    spd_stats* stats);

/* The three-step rollback from the host (SPD summary step 5): every layer's KV length and the
 * draft-module cache length drop to `keep_len`, in-flight hidden states are flushed, and
 * `reseed_token` enters stage 1 at position keep_len+1 (fill 1).  Length-only: no KV data moves.
 * SPD_EINVAL unless 1 <= keep_len <= the verified length and 0 <= reseed_token < V. */
int spd_rollback(spd_handle* h, int32_t keep_len, int32_t reseed_token);

/* Seeded-acceptance harness (not part of the method): for positions first_pos..first_pos+count-1,
 * modes[i] = 0 keeps the draft module's top-1, 1 replaces the draft by ref_tokens[i], 2 takes the
 * draft module's best-ranked token that differs from ref_tokens[i].  HOST arrays.  Cleared by
 * spd_prefill.  SPD_EINVAL for positions outside 1..max_seq or bad modes. */
int spd_set_draft_override(spd_handle* h, int32_t first_pos, int32_t count,
                           const int32_t* ref_tokens, const uint8_t* modes);

/* Seeded acceptance from (alpha, seed) alone -- the same harness knob as spd_set_draft_override,
 * with the coins drawn inside the library so that a C caller reproduces a workload's acceptance
 * rate without computing them.  Not part of the method: random-init draft weights cannot reproduce
 * a trained draft module's acceptance, so each workload fixes alpha.
 *   coin(q) = (SplitMix64 output from state seed ^ q * 0x9E3779B97F4A7C15) >> 11, divided by 2^53
 *   (SplitMix64: Steele, Lea, Flood, OOPSLA 2014); keyed by the position q only.
 *   The draft for position q (P+2 <= q <= P+n_ref) becomes ref_tokens[q-P-1] when coin(q) < alpha
 *   (mode 1 of spd_set_draft_override), else the draft module's best-ranked token that differs from
 *   it (mode 2).  The draft module always runs in full; every such position is verified once on a
 *   correct prefix, so the reject set is exactly {q : coin(q) >= alpha}.
 *   ref_tokens: HOST array of n_ref tokens at positions P+1..P+n_ref (the plain greedy AR stream,
 *   e.g. from spd_generate_ar), copied.  alpha is compared in double precision; alpha < 0 switches
 *   the knob off (raw draft-module drafts).  Call after spd_prefill (which clears it).
 *   SPD_ESTATE before a prefill; SPD_EINVAL for alpha > 1, n_ref < 1, P + n_ref > max_seq or a token
 *   outside 0..V-1. */
int spd_set_acceptance(spd_handle* h, double alpha, uint64_t seed, const int32_t* ref_tokens, int32_t n_ref);

/* The modes spd_set_acceptance derives, on the host, without a handle or a GPU:
 * modes[i] = 1 if coin(first_pos + i) < alpha else 2, for i < count.  SPD_EINVAL (message in
 * spd_last_error(NULL)) for count < 0, first_pos < 0 or a NULL array with count > 0. */
int spd_acceptance_modes(double alpha, uint64_t seed, int32_t first_pos, int32_t count, uint8_t* modes);

/* Sampled decoding (temperature > 0, top-k; SPD news 六 and SPD summary 复现评估: T in {0, 1},
 * top-k 50, top-p 1.0).  Drafts are drawn from the draft module's top-k distribution and verified
 * by rejection sampling: accept with probability min(1, p/q), else the token is drawn from
 * normalize(max(0, p - q)) (the speculative decoding engineering page §2.1-2.2).  Plain AR
 * (spd_generate_ar) draws from the target's top-k distribution.  The k tokens are ordered by logit
 * descending (lower id first among equals); a draw with uniform u takes the first token whose fp32
 * running sum of exp(l_i/T - l_0/T) exceeds u times the total.
 *   temperature <= 0: greedy decoding (the default; top_k and the uniforms are ignored).
 *   top_k: 1..64 (capped at the vocabulary size).
 *   uniforms: HOST array of 4*count floats in [0, 1), copied: uniforms[s*count + i] is stream s
 *     (0 draft, 1 accept, 2 resample, 3 ar) at position first_pos + i; other positions keep their
 *     values.  The random numbers are inputs so that a caller can reproduce every draw.
 * The token at P+1 (returned by spd_prefill) stays the greedy one.  The seeded-acceptance harness
 * (spd_set_draft_override) does not apply while sampling.  SPD_EINVAL for a bad range or value. */
int spd_set_sampling(spd_handle* h, float temperature, int32_t top_k, int32_t first_pos, int32_t count,
                     const float* uniforms);

/* Self-check of the failure path (no GPU fault involved): runs one of the bounded device waits the
 * kernels use -- which = 0: the grid-barrier counter wait of the step kernel, 1: an mbarrier phase
 * wait (weight ring, tensor-core completion), 2: the shared-memory progress counter wait between the
 * step kernel's warp roles -- on a condition that nothing satisfies, with a limit of limit_ns
 * nanoseconds (1e3 .. 2e9; the kernels themselves use 2e9).  The wait gives up, the kernel sets the
 * control block's error word and returns, and the host turns it into SPD_ETIMEOUT, which this call
 * returns; the error word is cleared afterwards, so the handle stays usable.  Returns SPD_OK only if
 * the wait did not give up (a defect).  SPD_EINVAL for a bad `which` or limit. */
int spd_debug_wait_timeout(spd_handle* h, int32_t which, int64_t limit_ns);

/* Execution options (bit flags), default SPD_OPT_GRAPHS | SPD_OPT_COSCHED | SPD_OPT_PDL |
 * SPD_OPT_STEP. */
#define SPD_OPT_GRAPHS       1  /* replay captured CUDA graphs instead of eager launches      */
#define SPD_OPT_COSCHED      2  /* draft layer s rides in the GEMV launches of target sub-step s
                                   (SPD summary 方法步骤详情 steps 1 and 4 in one pass over HBM);
                                   without it the draft module runs as its own launches before
                                   the target step (serialised)                                */
#define SPD_OPT_TARGET_ONLY  4  /* skip the draft module (timing of the target step only);
                                   drafts come from the override (mode 2 then uses ref+1 mod V)
                                   or repeat the token at t                                    */
#define SPD_OPT_DEBUG_LOGITS 8  /* keep full fp32 logits of the last head launch for dumps     */
#define SPD_OPT_PDL         16  /* programmatic dependent launch: a kernel may start (and stream
                                   its weights) while its predecessor drains                   */
#define SPD_OPT_STEP        32  /* one persistent cooperative kernel per cycle / AR step (one CTA
                                   per SM, phases separated by grid barriers, weights streamed
                                   across phase boundaries); off: one launch per operator      */
#define SPD_OPT_POST_STEP   64  /* post-step schedule (the scheduling ablation, SPD v3 summary §4;
                                   SPD news 十): the draft module runs after the target step on
                                   its OUTPUT state -- in-flight rows one stage deeper (depth
                                   t-i+1), the exiting row at depth n and cached -- so drafting
                                   is serial with the step.  Overrides SPD_OPT_COSCHED; no
                                   effect with SPD_OPT_TARGET_ONLY.  The committed stream and
                                   the cycle count are those of the default schedule.          */
int spd_set_options(spd_handle* h, int32_t flags);

/* Copy internal state to a HOST buffer of `bytes` bytes (synchronising).  Layouts:
 *   SPD_DUMP_STATE   int32[24]: t, a, v, pdm_len, P, cycles, exits, rejects, err, done,
 *                    max_commit, flags, last_exited, last_exit_pos, last_accept, target_top1,
 *                    pdm_top1, pdm_top2, draft, pushed, err_where, 0, 0, 0
 *   SPD_DUMP_RESID   fp32[(n+1)][d]        target residual ring, row = position % (n+1)
 *   SPD_DUMP_ANCHORS fp32[(n+1)][m][d]     anchor ring, row = position % (n+1)
 *   SPD_DUMP_PDM_Z   fp32[(n+2)][d]        draft-module rows of the last cycle after Ls layers
 *   SPD_DUMP_LOGITS  fp32[2][V]            target / draft head logits of the last head launch
 *                                          (needs SPD_OPT_DEBUG_LOGITS)
 *   SPD_DUMP_SEQ     int32[max_seq+2]      token at each position (index = position)
 *   SPD_DUMP_TRACE   int32[2][max_seq]     per verification: position, accepted
 *   SPD_DUMP_KVLEN   int32[L]              per-layer KV length bookkeeping
 *   SPD_DUMP_PREFILL_H fp32[32][d]         residual after all L layers of the last prefill block's
 *                                          rows (row i = position P - cnt + 1 + i, cnt = the block's
 *                                          row count, 1..32); later rows are stale
 * SPD_EINVAL if `bytes` differs from the layout's size (query it with spd_dump_size). */
enum { SPD_DUMP_STATE = 0, SPD_DUMP_RESID = 1, SPD_DUMP_ANCHORS = 2, SPD_DUMP_PDM_Z = 3,
       SPD_DUMP_LOGITS = 4, SPD_DUMP_SEQ = 5, SPD_DUMP_TRACE = 6, SPD_DUMP_KVLEN = 7,
       SPD_DUMP_PREFILL_H = 8 };
size_t spd_dump_size(const spd_handle* h, int32_t what);
int spd_debug_dump(spd_handle* h, int32_t what, void* host_dst, size_t bytes);

/* Per-kernel-kind device time, for roofline reporting.  When enabled, graphs are bypassed; each
 * per-operator launch is bracketed by CUDA events on its own stream, and the step kernel records
 * the time of each of its phases (grid barrier to grid barrier, on CTA 0).  spd_kernel_times
 * returns, per kind, launches (or phase executions) and summed milliseconds, and resets them.
 * Kinds 0..8 are target-stack launches (stage-diagonal, AR or prefill): 0 qkv (with RoPE and
 * the KV append), 1 unused (kept for layout stability), 2 attention, 3 o-proj, 4 gate/up, 5 down,
 * 6 anchor FC, 7 vocab head, 8 control; kinds 9..17 are the same operators on the draft-module
 * stack.  A co-scheduled launch (SPD_OPT_COSCHED) is counted under its target kind. */
#define SPD_NUM_KINDS 18
int spd_time_kernels(spd_handle* h, int32_t enable);
int spd_kernel_times(spd_handle* h, int64_t* launches, double* ms, int32_t n_kinds);

/* Algorithmic HBM bytes of one cycle, per kernel kind (host arithmetic, no device work): every
 * weight byte the cycle streams plus every KV byte its attention reads, for a cycle whose pre-step
 * state is (newest position t, fill), that exits (exited != 0) or not, with or without the draft
 * module.  Weights: a = fill tokens each run S = L/n target layers; the draft module streams its
 * used FCs, Ls layers and LM head; the target LM head only when a token exits. */
int spd_cycle_bytes(const spd_handle* h, int32_t t, int32_t fill, int32_t exited, int32_t with_pdm,
                    double* bytes_per_kind, int32_t n_kinds);

/* ---------------------------------------------------------------------------------------------
 * Stand-alone operators (device pointers, enqueued on `cuda_stream`), for kernel-level tests.
 * ------------------------------------------------------------------------------------------- */

/* Decode attention over a KV cache: for each query row r (0..R-1) at 1-based position pos[r]
 * and each query head h, out[r][h][:] = softmax(q_r,h . K[kv(h)][0..pos[r]-1]^T / sqrt(hd)) V,
 * with kv(h) = h / (Hq/Hkv).  q: fp32 [R][Hq][hd] (already rotated); k_cache, v_cache:
 * [Hkv][max_seq][hd] in `dtype`; pos: device int32 [R] (1 <= pos <= max_seq); out: fp32
 * [R][Hq][hd].  A row whose pos lies outside 1..max_seq is not computed: its output row is set to
 * NaN (the device array cannot be checked on the host without a synchronisation).
 * Split over key chunks of 128 positions (the split count depends only on pos);
 * chunk partials are merged in chunk order by the last chunk to finish.  `workspace` (device,
 * >= spd_attention_workspace_bytes(...) bytes, 16-byte aligned) holds the partials and
 * counters; it must be zeroed before its first use and is left zeroed by each call.
 * SPD_EINVAL on bad sizes. */
size_t spd_attention_workspace_bytes(int32_t R, int32_t n_heads, int32_t n_kv_heads,
                                     int32_t head_dim, int32_t max_pos);
int spd_attention(const float* q, const void* k_cache, const void* v_cache, int32_t dtype,
                  const int32_t* pos, int32_t R, int32_t n_heads, int32_t n_kv_heads,
                  int32_t head_dim, int32_t max_seq, float* out, void* workspace,
                  size_t workspace_bytes, void* cuda_stream);

/* Decode attention without any allocation: the same operation, arguments and results as
 * spd_attention, but the split partials and merge tickets live in a scratch array inside the
 * library instead of a caller workspace.  The paper has no counterpart to this call; it exists for
 * callers that may not call cudaMalloc at all -- a plugin hosted by an application that owns the
 * GPU's memory budget, or code on a latency-critical path where an allocation could synchronise
 * the device.
 *   - The scratch is a fixed 16 MiB per GPU (16 KiB of tickets + 16 MiB - 16 KiB of partials),
 *     held by every GPU that loads the library until the process exits.  Calls whose partials
 *     (R * n_heads * ceil(max_seq/128) * (head_dim+2) * 4 bytes) or tickets (64 * n_kv_heads * 4
 *     bytes) do not fit return SPD_EINVAL with the sizes in spd_last_error(NULL).
 *   - The first call on a device looks up the array's device address with that device current;
 *     make that first call before any stream capture.
 *   - Every call shares the array and leaves its contents behind; the tickets are cleared at the
 *     start of each call (stream-ordered).  Calls that overlap on the GPU race on the array.
 *   - Allocates nothing: no cudaMalloc, cudaFree or allocating library routine. */
int spd_attention_static_scratch(const float* q, const void* k_cache, const void* v_cache,
                                 int32_t dtype, const int32_t* pos, int32_t R, int32_t n_heads,
                                 int32_t n_kv_heads, int32_t head_dim, int32_t max_seq, float* out,
                                 void* cuda_stream);

/* Causal attention of a prefill block on the tensor cores (tcgen05): R (1..32) query rows at the
 * consecutive positions pos0..pos0+R-1, whose keys and values are already in the cache, so row r
 * sees keys 1..pos0+r: out[r][h][:] = softmax(q_r,h . K[kv(h)][0..pos0+r-1]^T / sqrt(hd)) V.
 * q: fp32 [R][n_heads][hd] (rotated); k_cache, v_cache: bf16 [n_kv_heads][max_seq][hd]; out: fp32
 * [R][n_heads][hd]; hd 64 or 128; every pointer 16-byte aligned.  The query, and the probabilities,
 * enter the bf16 MMAs as high + low halves (fp32 accumulation in TMEM), so the result keeps about
 * 16 significant bits of the fp32 operands.  Long contexts are split over CTAs by 128-key chunks and
 * merged in split order.  `workspace` (device, >= spd_prefill_attention_workspace_bytes bytes) holds
 * the split partials and tickets; zero it before its first use, each call leaves the tickets zeroed.
 * This is the kernel the prefill uses for bf16 models with those head sizes.  SPD_EINVAL on bad sizes. */
size_t spd_prefill_attention_workspace_bytes(int32_t n_heads, int32_t n_kv_heads, int32_t head_dim,
                                             int32_t max_seq);
int spd_prefill_attention(const float* q, const void* k_cache, const void* v_cache, int32_t pos0, int32_t R,
                          int32_t n_heads, int32_t n_kv_heads, int32_t head_dim, int32_t max_seq, float* out,
                          void* workspace, size_t ws_bytes, void* cuda_stream);

/* Grouped GEMV with RMSNorm prologue: for group g (0..G-1), y_g = W_g . (x_g / rms(x_g) * nw)
 * (norm skipped when nw == NULL), W_g [rows, cols] row-major in `dtype`, x_g fp32 [cols],
 * y_g fp32 [rows].  Host arrays of G device pointers W[], x[], y[]; nw device fp32 [cols]
 * shared by all groups or NULL.  1 <= G <= 34, cols >= 8, cols % 8 == 0.  Same streaming engine
 * as the cycle (2-D tensor copies into a shared-memory ring, fp32 accumulation, fixed reduction
 * order); the G tensor maps live in stream-ordered scratch (cudaMallocAsync) for the launch. */
int spd_grouped_gemv(const void* const* W, const float* const* x, float* const* y, int32_t G,
                     int32_t rows, int32_t cols, int32_t dtype, const float* nw, float eps,
                     void* cuda_stream);

#ifdef __cplusplus
}
#endif
#endif /* SPD_H */
