/*
 * specverify.h -- C ABI of the GB300 (sm_103a) W4A16 weight-read library:
 * a group-128 dequantizing skinny GEMM and an int4 lm_head pass with fused
 * greedy speculative verification.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  * All array arguments are DEVICE pointers owned by the caller, 16-byte
 *    aligned, row-major and densely packed:
 *      x       [T][K]         bf16 bits (sv_bf16)
 *      Wq      [rows][K/8]    uint32; column k = 8w + i of a row is nibble i
 *                             (bits 4i..4i+3) of word w; level = nibble - 8
 *      scales  [rows][K/128]  bf16 bits, one per row and 128-column group
 *      y       [T][N]         bf16 bits
 *    Format source: page "qwen-warp and llamAmpere: two RTX 3090 engines
 *    for Qwen3.8, and what each one calls the same answer" (ai.satyajit.si),
 *    section "qwen-warp: keep the activations in bf16": eight nibbles per
 *    uint32 word along K, one bf16 scale per 128 columns, level = nibble - 8,
 *    the group scale applied in fp32 after each group's accumulate.
 *  * K is a multiple of 128; 1 <= T <= 32.
 *  * Every call is enqueued on `stream` (NULL = the legacy default stream)
 *    and returns before the GPU has run it.  It performs no host<->device
 *    copy and no synchronisation.  Results are valid once the stream has
 *    been synchronised.
 *  * A call returns SV_OK or a negative status.  On any error nothing is
 *    launched and no output is touched.
 *  * The library keeps one scratch area per device (split-tile fp32
 *    partial sums, the converted activations of calls with T > 8,
 *    completion counters, the argmax keys; about 32 MB on a 152-SM GPU),
 *    created with cudaMalloc by the first call on that device (so make that
 *    first call outside CUDA-graph capture) and reused afterwards.  Calls
 *    on one device must therefore be ordered with respect to each other
 *    (same stream, or synchronised streams); overlapping calls race on it.
 *  * Problems found by a kernel at run time (a vocab_map id outside [0, V),
 *    an internal wait that timed out) never trap: the kernel finishes and
 *    sets a sticky per-device error word, read with sv_last_device_error.
 */
#ifndef SPECVERIFY_H
#define SPECVERIFY_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef uint16_t sv_bf16;                  /* raw bf16 bits */
typedef struct CUstream_st *sv_stream;     /* a cudaStream_t */

enum sv_status {
    SV_OK = 0,
    SV_ERR_NULL = -1,    /* a required pointer is NULL                     */
    SV_ERR_SHAPE = -2,   /* a size is out of range or inconsistent         */
    SV_ERR_ALIGN = -3,   /* a pointer is not 16-byte aligned               */
    SV_ERR_CUDA = -4,    /* a CUDA runtime call or the launch failed       */
    SV_ERR_NOMEM = -5,   /* the per-device scratch area could not be made  */
    SV_ERR_DEVICE = -6   /* the current device is not sm_103 / sm_100      */
};

/* Bits of the sticky device error word. */
#define SV_DEVERR_BAD_MAP_ID  0x1   /* a vocab_map entry outside [0, V) was skipped */
#define SV_DEVERR_TIMEOUT     0x2   /* a pipeline wait gave up; outputs are invalid */
#define SV_DEVERR_SMEM_ALIGN  0x4   /* shared memory not 1024-byte aligned; nothing was computed */

/*
 * w4a16_gemm -- y[t][n] = bf16_rne( sum_g float(scales[n][g]) *
 *                          sum_{k in group g} (q(n,k) - 8) * float(x[t][k]) )
 * with fp32 products and sums; every packed weight byte and scale is read
 * from HBM once per call whatever T is ("read once per cycle regardless of
 * T": page "OpenJet Engine: CUDA LLM inference for Qwen3.8-27B", section "How it gets its speed").  Summation
 * order differs from a sequential loop (groups may be split across thread
 * blocks and added in a fixed order), so results agree with a sequential
 * fp32 sum to within fp32 rounding before the final bf16 rounding; they
 * are deterministic from run to run.
 *   x [T][K], Wq [N][K/8], scales [N][K/128], y [T][N] (written).
 *   Errors: SV_ERR_NULL, SV_ERR_SHAPE (T outside 1..32, K < 128 or
 *   K % 128 != 0, N < 1; with T > 8 also K > 131072), SV_ERR_ALIGN,
 *   SV_ERR_CUDA, SV_ERR_NOMEM.
 *   Launches: one kernel for T <= 8; for T > 8 a small conversion kernel
 *   (the activations into a per-device buffer) and then the main kernel,
 *   both on `stream`.
 */
int w4a16_gemm(const sv_bf16 *x, const uint32_t *Wq, const sv_bf16 *scales,
               int T, int K, int N, sv_bf16 *y, sv_stream stream);

/*
 * lmhead_verify -- one int4 lm_head pass over the T = 1 + n_draft verify
 * rows with on-device greedy verification.
 *   logit[t][v] = sum_g float(scales[v][g]) * sum_{k in g} (q(v,k)-8)*x[t][k]
 *   in fp32 (never rounded to bf16, never written to memory);
 *   a[t] = argmax over candidate v of logit[t][v], lowest token id on ties;
 *   accept_len = first i in [0, n_draft) with drafts[i] != a[i], else n_draft;
 *   next_token = a[accept_len]  (the model's own token at the first
 *   disagreement, or the bonus token when every draft was accepted).
 * Sources: page "qwen-warp and llamAmpere: two RTX 3090 engines for
 * Qwen3.8, and what each one calls the same answer" section "What each one calls the
 * same answer" (greedy acceptance is an argmax equality over the verify
 * rows); page "swift-qwen3.8-rtx3090" section "Body, heads and drafter"
 * (drafts are kept up to the first one the model disagrees with); page
 * "OpenJet Engine: CUDA LLM inference for Qwen3.8-27B" section "How it works" (lm_head and verification run on
 * the device and only the accepted tokens go back to the host).
 *   Candidates: all rows 0..V-1 when vocab_map == NULL (n_map ignored);
 *   otherwise rows vocab_map[0..n_map-1] of the V-row head, and every id
 *   compared or returned is a token id (vocab_map[j]), ties going to the
 *   lowest token id whatever the map order.  A draft outside the map can
 *   never match (page "swift-qwen3.8-rtx3090": every miss of the draft
 *   vocabulary is a rejection).
 *   x [1+n_draft][K]; Wq [V][K/8]; scales [V][K/128]; drafts [n_draft]
 *   int32 (may be NULL when n_draft == 0); vocab_map [n_map] int32 or NULL;
 *   accept_len, next_token: one int32 each (written).
 *   Errors: SV_ERR_NULL, SV_ERR_SHAPE (n_draft outside 0..31, K as above,
 *   V < 1, n_map outside 1..V with a map), SV_ERR_ALIGN, SV_ERR_CUDA,
 *   SV_ERR_NOMEM.  Launches as w4a16_gemm (T = 1 + n_draft).
 */
int lmhead_verify(const sv_bf16 *x, const uint32_t *Wq, const sv_bf16 *scales, int K,
                  const int32_t *drafts, int n_draft,
                  const int32_t *vocab_map, int n_map, int V,
                  int32_t *accept_len, int32_t *next_token, sv_stream stream);

/*
 * lmhead_verify_batched -- n_streams independent verify blocks in ONE pass
 * over the head (page "qwen-warp and llamAmpere: two RTX 3090 engines for
 * Qwen3.8, and what each one calls the same answer", section "What makes each
 * one a 3090 engine": four sequences with three drafts each share one weight
 * read).  Block s owns rows s*(1+n_draft) .. s*(1+n_draft)+n_draft of x and
 * drafts[s][0..n_draft-1]; accept_len[s], next_token[s] as in lmhead_verify.
 *   Requires n_streams >= 1 and T = n_streams*(1+n_draft) <= 32.
 */
int lmhead_verify_batched(const sv_bf16 *x, const uint32_t *Wq, const sv_bf16 *scales,
                          int K, const int32_t *drafts, int n_draft, int n_streams,
                          const int32_t *vocab_map, int n_map, int V,
                          int32_t *accept_len, int32_t *next_token, sv_stream stream);

/*
 * lmhead_verify_ex -- lmhead_verify_batched with flags.
 *   SV_MAP_STATIC: the caller promises that vocab_map is model data that no
 *   kernel enqueued before this call on `stream` writes (a draft
 *   vocabulary loaded once, as on page "Tesla P100 (sm_60) llama.cpp
 *   patches for Qwen3.5/3.6-35B-A3B: ~2x decode and prompt processing over
 *   the shinbunbun baseline", section "MTP draft vocabulary (patch 17)": a
 *   token list shipped with the model).  The kernel then reads the ids,
 *   gathers their scales and starts streaming their weight rows while the
 *   previous kernel of the stream is still finishing, instead of after it
 *   (programmatic dependent launch).  Not for a list that a preceding
 *   kernel maintains, such as the dynamic draft list of draft_list_add.
 *   Ignored without a vocab_map.  Other flag bits: SV_ERR_SHAPE.
 *   Everything else as lmhead_verify_batched.
 */
#define SV_MAP_STATIC 0x1
int lmhead_verify_ex(const sv_bf16 *x, const uint32_t *Wq, const sv_bf16 *scales, int K,
                     const int32_t *drafts, int n_draft, int n_streams,
                     const int32_t *vocab_map, int n_map, int V, int flags,
                     int32_t *accept_len, int32_t *next_token, sv_stream stream);

/*
 * sv_verify_cycle -- one verify cycle's weight reads in one call: the
 * given W4A16 GEMMs in order, then (when verify != NULL) the lm_head pass
 * with greedy verification of n_streams blocks, all enqueued on `stream`
 * with programmatic dependent launch, so each kernel streams its weights
 * while the previous one drains and the GPU does not wait for the host
 * between them.  Capturing this call in a CUDA graph gives the graph-per-
 * cycle form of the page "qwen-warp and llamAmpere: two RTX 3090 engines
 * for Qwen3.8, and what each one calls the same answer" (section "What
 * makes each one a 3090 engine": a decode cycle is one CUDA graph); the
 * page "OpenJet Engine: CUDA LLM inference for Qwen3.8-27B" (section "How
 * it works") runs the same cycle -- the main model over the T = 1 +
 * n_draft rows, then lm_head and verification on the device -- as one
 * persistent kernel.
 *   gemms [n_gemms] (host array, 0 <= n_gemms <= SV_CYCLE_MAX_GEMMS): each
 *   entry as the arguments of w4a16_gemm.  verify (host pointer or NULL):
 *   the arguments of lmhead_verify_batched.  The GEMMs' inputs are the
 *   caller's: this call does not chain one GEMM's output into the next.
 *   Every argument of every entry is checked before anything is enqueued
 *   (errors as w4a16_gemm and lmhead_verify_batched; SV_ERR_SHAPE when
 *   there is nothing to do); after that only a failed launch (SV_ERR_CUDA)
 *   can stop the call, leaving the kernels before it enqueued.
 */
#define SV_CYCLE_MAX_GEMMS 64
typedef struct sv_gemm_call {
    const sv_bf16 *x;          /* [T][K] */
    const uint32_t *Wq;        /* [N][K/8] */
    const sv_bf16 *scales;     /* [N][K/128] */
    int T, K, N;
    sv_bf16 *y;                /* [T][N], written */
} sv_gemm_call;
typedef struct sv_verify_call {
    const sv_bf16 *x;          /* [n_streams * (1 + n_draft)][K] */
    const uint32_t *Wq;        /* [V][K/8] */
    const sv_bf16 *scales;     /* [V][K/128] */
    int K;
    const int32_t *drafts;     /* [n_streams][n_draft] */
    int n_draft, n_streams;
    const int32_t *vocab_map;  /* [n_map] or NULL */
    int n_map, V;
    int32_t *accept_len;       /* [n_streams], written */
    int32_t *next_token;       /* [n_streams], written */
} sv_verify_call;
int sv_verify_cycle(const sv_gemm_call *gemms, int n_gemms, const sv_verify_call *verify, sv_stream stream);

/*
 * lmhead_argmax -- the same pass without the draft comparison: for each of
 * the T rows of x, ids[t] = the argmax token id (lowest id on ties) and
 * vals[t] = its fp32 logit.  This is the greedy step of a restricted draft
 * head (page "OpenJet Engine: CUDA LLM inference for Qwen3.8-27B", section "How it gets its speed": the draft
 * head scores a fixed id list; page "swift-qwen3.8-rtx3090": the draft head
 * is the lm_head restricted to the draft vocabulary).
 *   ids [T] int32, vals [T] float (written).  vals may be NULL.
 */
int lmhead_argmax(const sv_bf16 *x, const uint32_t *Wq, const sv_bf16 *scales, int K,
                  int T, const int32_t *vocab_map, int n_map, int V,
                  int32_t *ids, float *vals, sv_stream stream);

/*
 * lmhead_verify_noalloc -- the same greedy verify as lmhead_verify, for
 * callers that must not allocate GPU memory when they call: serving
 * runtimes that hand out every byte of device memory from their own arena
 * and forbid allocations behind their back, and latency-critical paths
 * that cannot take the implicit device synchronisation of cudaMalloc.
 * No source page has a counterpart to this entry point; it exists for this
 * library's users.
 *   Arguments, layouts and results are those of lmhead_verify.
 *   Scratch: a fixed device array inside the library (about 3.7 MB per
 *   device, held until the process exits), sized for at most 160 thread
 *   blocks, 32 verify rows and, with more than 7 drafts, K <= 16384; the
 *   call launches at most 160 blocks and rejects more than 31 drafts, or
 *   more than 7 drafts with K > 16384, with SV_ERR_SHAPE before it
 *   enqueues anything.  It calls no cudaMalloc, cudaFree or other
 *   allocating routine.
 *   The first call on a device resolves the array's device address and
 *   sets kernel attributes (no allocation); make that first call before
 *   any stream capture.  Each call clears the array's counters with an
 *   asynchronous memset on `stream` right before its kernels.
 *   All calls share the one array: calls that overlap on the GPU (two
 *   streams, or two host threads) race on it and must be ordered by the
 *   caller.  Device-side problems (a bad vocab_map id is skipped) are not
 *   reported through sv_last_device_error by this variant.
 */
int lmhead_verify_noalloc(const sv_bf16 *x, const uint32_t *Wq, const sv_bf16 *scales, int K,
                          const int32_t *drafts, int n_draft,
                          const int32_t *vocab_map, int n_map, int V,
                          int32_t *accept_len, int32_t *next_token, sv_stream stream);

/*
 * lmhead_verify_rescored / lmhead_argmax_rescored -- the greedy verify (or
 * the per-row argmax) with the ids of the bf16 head: the int4 lm_head pass
 * gives every verify row its top_k candidates by fp32 int4 logit (ties to
 * the lowest id), the bf16 head rescores just those rows, and the argmax is
 * taken among them (page "qwen-warp and llamAmpere: two RTX 3090 engines
 * for Qwen3.8, and what each one calls the same answer", section "What each
 * one calls the same answer": the rescoring head reads the quantized
 * lm_head's top candidates and rescores them with the bf16 head; table
 * "What one cycle reads from VRAM": 16 to 64 candidates).
 *   logit_bf16[t][c] = sum_k float(Wbf[c][k]) * float(x[t][k]) in fp32
 *   (products exact, summed in a fixed tree order); a[t] = argmax over the
 *   candidates, lowest id on ties; accept_len / next_token as in
 *   lmhead_verify.  ids / vals (argmax variant): a[t] and its bf16 logit.
 *   x [T][K] (T = 1 + n_draft for the verify, T <= 8); Wq [V][K/8] and
 *   scales [V][K/128] the int4 head; Wbf [V][K] bf16 the bf16 head
 *   (16-byte aligned); 1 <= top_k <= min(64, V).  No vocab_map.
 *   Launches three kernels on `stream`: the int4 head writing fp32 logits
 *   to a per-device buffer, a pass taking the largest logit of every
 *   128-row slice of V, and ceil(top_k / 16) blocks per verify row that
 *   select the row's top_k (threshold: the top_k-th largest slice maximum),
 *   rescore them and, in the last block, verify.  The first call on a
 *   device, or the first with a larger V, allocates that buffer (about
 *   32 * V bytes) after synchronising `stream`: make it outside stream
 *   capture.
 *   Errors: SV_ERR_NULL, SV_ERR_SHAPE (T outside 1..8, K as for
 *   w4a16_gemm and at most 65536, V < 1, top_k out of range),
 *   SV_ERR_ALIGN, SV_ERR_CUDA, SV_ERR_NOMEM.
 */
int lmhead_verify_rescored(const sv_bf16 *x, const uint32_t *Wq, const sv_bf16 *scales,
                           const sv_bf16 *Wbf, int K, const int32_t *drafts, int n_draft,
                           int top_k, int V, int32_t *accept_len, int32_t *next_token,
                           sv_stream stream);
int lmhead_argmax_rescored(const sv_bf16 *x, const uint32_t *Wq, const sv_bf16 *scales,
                           const sv_bf16 *Wbf, int K, int T, int top_k, int V,
                           int32_t *ids, float *vals, sv_stream stream);

/*
 * lmhead_verify_sampled -- exact speculative sampling verify over the 32
 * best int4 logits of each verify row (page "OpenJet Engine: CUDA LLM
 * inference for Qwen3.8-27B", sections "How it gets its speed": sampling
 * keeps the 32 best logits of each verified row, a draft is accepted with
 * probability p(draft) and a rejected one is resampled from the rest of the
 * distribution; "Limitations": temperature, top-k <= 32, top-p and min-p
 * in llama.cpp's order; page "qwen-warp and llamAmpere: two RTX 3090
 * engines for Qwen3.8, and what each one calls the same answer", section
 * "What each one calls the same answer": accept, else draw from the
 * residual, keeps the output distributed exactly as the target).
 *   Row i's distribution p_i: its 32 best fp32 int4 logits (ties to the
 *   lowest id), best first; then, in fp32 with m the best logit and
 *   d_j = l_j - m: top-k keeps the first min(top_k, 32) (top_k <= 0: all);
 *   top-p the shortest prefix whose running sum of exp(d_j) reaches
 *   top_p times their sum (top_p >= 1: no cut); min-p the prefix with
 *   exp(d_j) >= min_p (min_p <= 0: no cut); weights
 *   w_j = exp(d_j / temperature), W their sum in order (temperature <= 0:
 *   the point mass on the best candidate, i.e. the greedy verify).
 *   Drafts are point masses: row i < n_draft accepts drafts[i] iff it is
 *   kept and u[2i] * W < w_{drafts[i]}; the first rejected row draws
 *   next_token from p_i without drafts[i], and if all are accepted row
 *   n_draft draws it from p_{n_draft}: walk the candidates best first with
 *   running sum c and take the first with u[2i+1] * W' < c (W' the sum over
 *   the candidates it may take).
 *   u [2 (n_draft + 1)] fp32 device: uniforms in [0, 1), drawn by the
 *   caller for every call (row i uses u[2i] and u[2i+1]).  x [n_draft+1][K],
 *   n_draft 0..7; Wq / scales as for lmhead_verify; no vocab_map.
 *   Launches three kernels on `stream`: the int4 head's fp32 logits into
 *   the per-device buffer of lmhead_verify_rescored (same first-call
 *   allocation), the slice maxima, and one block per row that selects the
 *   row's 32 best, runs the chain and the accept test; the last block
 *   writes accept_len and next_token.
 *   Errors: SV_ERR_NULL, SV_ERR_SHAPE (n_draft out of range, K as for
 *   w4a16_gemm, V < 1, top_k > 32, NaN parameters, min_p > 1),
 *   SV_ERR_ALIGN, SV_ERR_CUDA, SV_ERR_NOMEM.
 *
 * lmhead_sampling_dist -- the distributions p_t themselves, for T rows
 * (1..8): ids [T][32] int32 (candidates kept, best first, then -1) and
 * probs [T][32] fp32 (w_j / W, then 0).  Same kernels, no verify.
 */
int lmhead_verify_sampled(const sv_bf16 *x, const uint32_t *Wq, const sv_bf16 *scales, int K,
                          const int32_t *drafts, int n_draft, int V,
                          float temperature, int top_k, float top_p, float min_p,
                          const float *u, int32_t *accept_len, int32_t *next_token,
                          sv_stream stream);
int lmhead_sampling_dist(const sv_bf16 *x, const uint32_t *Wq, const sv_bf16 *scales, int K,
                         int T, int V, float temperature, int top_k, float top_p, float min_p,
                         int32_t *ids, float *probs, sv_stream stream);

/*
 * Dynamic draft list -- the candidate list of the restricted draft head: a
 * static list of token ids (the most frequent tokens) plus the tokens of the
 * current sequence that are missing from it, added as the sequence grows,
 * at most `cap` of them (page "OpenJet Engine: CUDA LLM inference for
 * Qwen3.8-27B", section "How it gets its speed"; page "Tesla P100 (sm_60)
 * llama.cpp patches for Qwen3.5/3.6-35B-A3B: ~2x decode and prompt
 * processing over the shinbunbun baseline", sections "MTP draft vocabulary
 * (patch 17)" and "The draft vocabulary file": up to 4096 sequence tokens).
 * Added tokens keep their order of first appearance; once `cap` were added
 * the list stays as it is; tokens outside [0, V) are ignored.
 *   The list lives in a caller-owned device workspace of
 *   draft_list_bytes(V, n_static, cap) bytes (16-byte aligned; 0 means
 *   invalid sizes: V < 1, n_static < 1, cap < 0, or more than 2^28 entries).
 *   draft_list_ids(ws, V) is the device address of its id array, always
 *   n_static + cap entries: the static ids, the added tokens, then copies
 *   of the first static id in the unused slots (a repeated candidate ties
 *   with itself and changes no argmax).  It is a ready vocab_map for
 *   lmhead_argmax / lmhead_verify with n_map = n_static + cap; the greedy
 *   draft step is lmhead_argmax over it with T = 1.
 *   draft_list_init: static_ids [n_static] int32 device (ids outside [0, V)
 *   are copied but not marked; the head skips them and reports
 *   SV_DEVERR_BAD_MAP_ID); clears the list's membership bitmap and writes
 *   the header and ids.  draft_list_add: tokens [n_tokens] int32 device;
 *   one kernel of one warp, 32 tokens per round.  Both are asynchronous on
 *   `stream`; calls on one workspace must be stream-ordered.
 *   draft_list_count: *out (host) = number of added tokens; synchronous.
 *   Errors: SV_ERR_NULL, SV_ERR_SHAPE, SV_ERR_ALIGN, SV_ERR_CUDA.
 */
size_t draft_list_bytes(int V, int n_static, int cap);
int32_t *draft_list_ids(void *ws, int V);
int draft_list_init(void *ws, const int32_t *static_ids, int n_static, int V, int cap, sv_stream stream);
int draft_list_add(void *ws, const int32_t *tokens, int n_tokens, sv_stream stream);
int draft_list_count(const void *ws, int32_t *out);

/* A static, human-readable name for a status code. */
const char *sv_status_string(int status);

/*
 * sv_last_device_error -- *out = the sticky device error word of the
 * current device (SV_DEVERR_* bits), then clears it.  Synchronises the
 * device (it reads device memory with a blocking copy).  Returns SV_OK,
 * SV_ERR_NULL or SV_ERR_CUDA.
 */
int sv_last_device_error(int32_t *out);
/*   When the word holds SV_DEVERR_TIMEOUT, the call also puts the
 *   per-device scratch counters (split-tile arrivals, argmax keys, CTA
 *   completions) back to zero, so that a run which gave up on a wait cannot
 *   affect later calls. */

/*
 * sv_hbm_read -- a measurement aid: one launch that only reads `bytes` of
 * device memory at src (bulk copies into shared memory, one thread block
 * per SM, equal contiguous shares, programmatic dependent launch -- the
 * launch structure of the GEMM kernels) and writes one checksum word per
 * block to sink.  Timed back to back on a weight matrix's byte count, it is
 * the read rate a kernel of that size reaches with nothing else to do, the
 * ceiling the GEMMs are reported against.  No source page has a
 * counterpart.
 *   src: 16-byte aligned, bytes a multiple of 16 (>= 16); sink: one uint32
 *   per SM of the device (written).  Errors: SV_ERR_NULL, SV_ERR_SHAPE,
 *   SV_ERR_ALIGN, SV_ERR_CUDA, SV_ERR_NOMEM.
 */
int sv_hbm_read(const void *src, size_t bytes, uint32_t *sink, sv_stream stream);

/*
 * sv_debug_set_fma_consumers -- a measurement switch: with on != 0, later
 * calls whose launch keeps the activations resident (T <= 8, contiguous
 * rows, at least 80 units of 64 rows x 128 columns per SM) compute their
 * dot products on CUDA cores -- one mixed-precision fp16 x fp16 -> fp32 fma
 * per weight and token -- instead of with tensor-core mma; same weight
 * stream, same results within fp32 rounding order.  It exists to measure
 * the two formulations against each other at equal HBM traffic (the
 * tensor-core path is the default because it measured faster); 0 restores
 * the default.  Process-wide.  No source page has a counterpart.
 */
int sv_debug_set_fma_consumers(int on);

/*
 * sv_debug_set_tcgen05 -- a measurement switch.  Calls with 17 <= T <= 32
 * (four n8 token tiles), contiguous rows and K a multiple of 1024 run by
 * default on the 5th-generation tensor cores (tcgen05.mma, M = 128 weight
 * rows x N = 32 tokens x K = 16; the A operand in tensor memory holds the
 * fp16 products level x scale x 2^(137 - E), E the largest scale exponent
 * of the row's box of eight groups (exact for every scale of at least
 * 2^-27 times the box's largest); each box's fp32 sums are
 * accumulated in tensor memory and multiplied by 2^(E - 137) in
 * registers); on = 0 makes them run on mma.sync
 * instead (same results within fp32 rounding order), 1 restores the
 * default.  It exists to measure the two against each other.  Process-wide.
 * No source page has a counterpart.
 */
int sv_debug_set_tcgen05(int on);

/*
 * sv_debug_set_wait_stall -- a test hook for the bounded waits.  With
 * ns > 0, every later launch of the stream kernel makes the epilogue warp
 * of its first thread block wait up to ns nanoseconds on a shared-memory
 * barrier that nothing completes; the wait runs out, the kernel sets
 * SV_DEVERR_TIMEOUT and carries on (its outputs are still computed).  0
 * turns it off.  Process-wide, not per device.  No source page has a
 * counterpart: it exists to test the error path without a GPU fault.
 *   Errors: SV_ERR_SHAPE if ns > 10^9 (one second).
 */
int sv_debug_set_wait_stall(uint32_t ns);

#ifdef __cplusplus
}
#endif

#endif /* SPECVERIFY_H */
