// rescore.cuh -- top-k candidates of the int4 lm_head rescored by the bf16
// head, so that the greedy verify compares the bf16 head's ids (page
// "qwen-warp and llamAmpere: two RTX 3090 engines for Qwen3.8, and what each
// one calls the same answer", section "What each one calls the same answer":
// the rescoring head reads the quantized lm_head's top candidates and
// rescores them with the bf16 head; table "What one cycle reads from VRAM":
// 16 to 64 candidates).
//
// Three kernels on one stream (programmatic dependent launch between them):
//  1. the int4 head as a GEMM with fp32 outputs (w4a16_stream.cuh): logits
//     [T][V];
//  2. slicemax_kernel: the largest (logit, id) key of every 128-row slice of
//     V, per verify row;
//  3. rescore_kernel, grid (ceil(k / 16), T): with tau the k-th largest of
//     the row's slice maxima, k slices hold a key >= tau, so the row's k best
//     keys are all >= tau and lie in the k slices whose maximum is >= tau.
//     Every CTA of the row finds tau (warp sorts and merges of the maxima),
//     re-reads those k slices, keeps their keys >= tau (at most 128 k),
//     sorts them, and rescores its share of the k best: fp32 dot products of
//     their bf16 rows with x.  The last CTA of the grid takes each row's
//     argmax (lowest id on ties) and runs the greedy verify.
#pragma once

#include <cstdint>

#include "sv_ptx.cuh"

namespace sv {

constexpr int RS_KMAX = 64;                      // largest top_k
constexpr int RS_TMAX = 8;                       // verify rows (one n8 token tile)
constexpr int RS_THREADS = 512;
constexpr int RS_WARPS = RS_THREADS / 32;
constexpr int RS_SLICE = 128;                    // rows of V per slice
constexpr int RS_PER_CTA = RS_WARPS;             // candidates rescored per CTA (one per warp)
constexpr int RS_SEL_MAX = RS_KMAX * RS_SLICE;   // keys >= tau, worst case

__device__ __forceinline__ unsigned long long kmax(unsigned long long a, unsigned long long b) { return a > b ? a : b; }

// Bitonic sort, descending, of the 128 keys a warp holds as v[i] = element
// i*32 + lane.
__device__ __forceinline__ void warp_sort128_desc(unsigned long long (&v)[4], int lane)
{
#pragma unroll
    for (int ls = 1; ls <= 7; ++ls) {
        const int s = 1 << ls;
#pragma unroll
        for (int ld = ls - 1; ld >= 0; --ld) {
            const int d = 1 << ld;
            if (d >= 32) {
                const int dd = d >> 5;
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    if (i & dd) continue;
                    const int j = i | dd;
                    const bool desc = ((i * 32 + lane) & s) == 0;
                    const unsigned long long hi = kmax(v[i], v[j]), lo = v[i] > v[j] ? v[j] : v[i];
                    v[i] = desc ? hi : lo;
                    v[j] = desc ? lo : hi;
                }
            } else {
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const unsigned long long o = shfl_xor_u64(v[i], d);
                    const bool lower = (lane & d) == 0;
                    const bool desc = ((i * 32 + lane) & s) == 0;
                    v[i] = lower == desc ? kmax(v[i], o) : (v[i] < o ? v[i] : o);
                }
            }
        }
    }
}

// a (element lane = a0, element 32 + lane = a1) and b, both sorted
// descending, 64 keys each: a becomes the 64 best of the two, descending.
// max(a[e], b[63 - e]) holds those 64 as a bitonic sequence; a bitonic
// merge sorts it.
__device__ __forceinline__ void warp_merge64_desc(unsigned long long &a0, unsigned long long &a1,
                                                  unsigned long long b0, unsigned long long b1, int lane)
{
    const unsigned long long r1 = shfl_u64(b1, 31 - lane), r0 = shfl_u64(b0, 31 - lane);
    unsigned long long c0 = kmax(a0, r1), c1 = kmax(a1, r0);
    a0 = kmax(c0, c1);
    a1 = c0 > c1 ? c1 : c0;
#pragma unroll
    for (int d = 16; d > 0; d >>= 1) {
        const bool lower = (lane & d) == 0;
        const unsigned long long o0 = shfl_xor_u64(a0, d), o1 = shfl_xor_u64(a1, d);
        a0 = lower ? kmax(a0, o0) : (a0 < o0 ? a0 : o0);
        a1 = lower ? kmax(a1, o1) : (a1 < o1 ? a1 : o1);
    }
}

// Bitonic sort, descending, of keys[0..npad) (npad a power of two) by the
// whole CTA.
__device__ __forceinline__ void cta_sort_desc(unsigned long long *keys, int npad)
{
    for (int s = 2; s <= npad; s <<= 1) {
        for (int d = s >> 1; d > 0; d >>= 1) {
            for (int i = threadIdx.x; i < npad; i += blockDim.x) {
                const int j = i ^ d;
                if (j > i) {
                    const bool desc = (i & s) == 0;
                    const unsigned long long a = keys[i], c = keys[j];
                    if (desc ? (a < c) : (a > c)) {
                        keys[i] = c;
                        keys[j] = a;
                    }
                }
            }
            __syncthreads();
        }
    }
}

struct SliceMaxParams {
    const float *logits;                 // [T][V]
    int T, V, nS;
    unsigned long long *smax;            // [T][nS]
};

// One warp per slice, every verify row.
__global__ void __launch_bounds__(RS_THREADS) slicemax_kernel(const __grid_constant__ SliceMaxParams p)
{
    pdl_launch_dependents();
    pdl_wait_prior();                    // the logits come from the int4 pass
    const int lane = threadIdx.x & 31;
    const int sl = blockIdx.x * RS_WARPS + (threadIdx.x >> 5);
    if (sl >= p.nS) return;
    const int v0 = sl * RS_SLICE;
    float f[RS_TMAX][4];
#pragma unroll
    for (int t = 0; t < RS_TMAX; ++t)
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int r = v0 + i * 32 + lane;
            f[t][i] = (t < p.T && r < p.V) ? __ldcg(p.logits + static_cast<size_t>(t) * p.V + r) : 0.f;
        }
#pragma unroll
    for (int t = 0; t < RS_TMAX; ++t) {
        if (t >= p.T) break;
        unsigned long long m = 0ull;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int r = v0 + i * 32 + lane;
            if (r < p.V) m = kmax(m, make_key(f[t][i], static_cast<uint32_t>(r)));
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = kmax(m, shfl_xor_u64(m, o));
        if (lane == 0) p.smax[static_cast<size_t>(t) * p.nS + sl] = m;
    }
}

// Shared memory of select_row (static, in the calling kernel).
struct SelectSmem {
    unsigned long long wl[RS_WARPS][64];
    int slist[RS_KMAX];
    unsigned long long tau;
    unsigned n_sel, n_sl;
};

// The k best (logit, id) keys of one row, descending, into sel[0..k) (keys
// past the row's candidates are 0), by the whole CTA; sel holds RS_SEL_MAX
// keys.  mx: the row's nS slice maxima; row: its V fp32 logits.  With tau
// the k-th largest slice maximum, k slices hold a key >= tau, so the row's
// k best keys are >= tau and lie in the (at most k) slices whose maximum is
// >= tau; at most 128 k keys are gathered and sorted.
__device__ __forceinline__ void select_row(const unsigned long long *mx, const float *row, int nS, int V, int k,
                                           unsigned long long *sel, SelectSmem &sm)
{
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (tid == 0) {
        sm.n_sel = 0u;
        sm.n_sl = 0u;
    }
    // tau: each warp keeps the 64 best maxima of its chunks of 128, then
    // warp 0 merges the warps' lists
    {
        unsigned long long a0 = 0ull, a1 = 0ull;
        for (int c = warp; c * RS_SLICE < nS; c += RS_WARPS) {
            unsigned long long v[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int s = c * RS_SLICE + i * 32 + lane;
                v[i] = s < nS ? __ldcg(mx + s) : 0ull;
            }
            warp_sort128_desc(v, lane);
            warp_merge64_desc(a0, a1, v[0], v[1], lane);
        }
        sm.wl[warp][lane] = a0;
        sm.wl[warp][32 + lane] = a1;
    }
    __syncthreads();
    if (warp == 0) {
        unsigned long long a0 = sm.wl[0][lane], a1 = sm.wl[0][32 + lane];
        for (int w = 1; w < RS_WARPS; ++w) warp_merge64_desc(a0, a1, sm.wl[w][lane], sm.wl[w][32 + lane], lane);
        const int kk = k - 1;
        const unsigned long long tk = shfl_u64(kk < 32 ? a0 : a1, kk & 31);
        if (lane == 0) sm.tau = tk;
    }
    __syncthreads();
    // the (at most k) slices whose maximum is >= tau; with fewer than k
    // slices tau is 0 and every slice qualifies
    const unsigned long long tau = sm.tau;
    for (int s = tid; s < nS; s += RS_THREADS) {
        const unsigned long long m = __ldcg(mx + s);
        if (m != 0ull && m >= tau) {
            const unsigned at = atomicAdd(&sm.n_sl, 1u);
            if (at < static_cast<unsigned>(RS_KMAX)) sm.slist[at] = s;
        }
    }
    __syncthreads();
    // their keys >= tau (the order of sel is fixed below by sorting)
    const int nsl = min(static_cast<int>(sm.n_sl), RS_KMAX);
    for (int j = warp; j < nsl; j += RS_WARPS) {
        const int v0 = sm.slist[j] * RS_SLICE;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int r = v0 + i * 32 + lane;
            const unsigned long long key = r < V ? make_key(__ldcg(row + r), static_cast<uint32_t>(r)) : 0ull;
            const bool keep = key != 0ull && key >= tau;
            const unsigned bal = __ballot_sync(0xFFFFFFFFu, keep);
            unsigned base = 0u;
            if (lane == 0 && bal) base = atomicAdd(&sm.n_sel, static_cast<unsigned>(__popc(bal)));
            base = __shfl_sync(0xFFFFFFFFu, base, 0);
            const unsigned at = base + __popc(bal & ((1u << lane) - 1u));
            if (keep && at < static_cast<unsigned>(RS_SEL_MAX)) sel[at] = key;
        }
    }
    __syncthreads();
    const int ns = min(static_cast<int>(sm.n_sel), RS_SEL_MAX);
    int npad = 1;
    while (npad < ns || npad < k) npad <<= 1;
    for (int i = ns + tid; i < npad; i += RS_THREADS) sel[i] = 0ull;
    __syncthreads();
    cta_sort_desc(sel, npad);
}

struct RescoreParams {
    const uint16_t *x;                   // [T][K] bf16 bits
    const uint16_t *Wbf;                 // [V][K] bf16 bits
    const float *logits;                 // [T][V] from the int4 pass
    const unsigned long long *smax;      // [T][nS] from slicemax_kernel
    int nS, T, K, V, k;
    int mode;                            // 0: verify, 1: argmax
    const int32_t *drafts;               // [T-1]
    int32_t *accept_len, *next_token;    // [1]
    int32_t *ids;                        // [T]
    float *vals;                         // [T] or null
    float *cand_lg;                      // scratch [RS_TMAX][RS_KMAX]
    int32_t *cand_id;                    // scratch [RS_TMAX][RS_KMAX]
    unsigned *done;                      // scratch counter, left at 0
};

// CTA (r, t): verify row t, candidates [16 r, 16 r + 16) of the row's k best.
// Dynamic shared memory: RS_SEL_MAX keys, then the row of x.
__global__ void __launch_bounds__(RS_THREADS) rescore_kernel(const __grid_constant__ RescoreParams p)
{
    extern __shared__ __align__(16) unsigned long long sel[];
    __shared__ SelectSmem sm;
    __shared__ float lg[RS_TMAX];
    __shared__ int lid[RS_TMAX];
    __shared__ unsigned is_last;
    const int t = blockIdx.y, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    uint16_t *xs = reinterpret_cast<uint16_t *>(sel + RS_SEL_MAX);
    pdl_wait_prior();                    // logits and slice maxima come from the passes before
    const uint4 *xg = reinterpret_cast<const uint4 *>(p.x + static_cast<size_t>(t) * p.K);
    for (int c = tid; c < p.K / 8; c += RS_THREADS) reinterpret_cast<uint4 *>(xs)[c] = xg[c];
    select_row(p.smax + static_cast<size_t>(t) * p.nS, p.logits + static_cast<size_t>(t) * p.V, p.nS, p.V, p.k,
               sel, sm);
    // rescore candidate j = 16 r + warp: eight 16-byte weight loads per lane
    // in flight, x from shared memory
    const int j = blockIdx.x * RS_PER_CTA + warp;
    if (j < p.k) {
        const unsigned long long key = sel[j];
        const int id = key == 0ull ? -1 : key_id(key);
        float acc = 0.f;
        if (id >= 0 && id < p.V) {
            const uint4 *wrow = reinterpret_cast<const uint4 *>(p.Wbf + static_cast<size_t>(id) * p.K);
            const uint4 *xrow = reinterpret_cast<const uint4 *>(xs);
            const int nch = p.K / 8;
            for (int c0 = lane; c0 < nch; c0 += 32 * 8) {
                uint4 w[8];
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    const int c = c0 + 32 * u;
                    w[u] = c < nch ? wrow[c] : make_uint4(0u, 0u, 0u, 0u);
                }
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    const int c = c0 + 32 * u;
                    if (c < nch) {
                        const uint4 xv = xrow[c];
                        const uint32_t ww[4] = {w[u].x, w[u].y, w[u].z, w[u].w};
                        const uint32_t xx[4] = {xv.x, xv.y, xv.z, xv.w};
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            acc = fmaf(__uint_as_float(ww[q] << 16), __uint_as_float(xx[q] << 16), acc);
                            acc = fmaf(__uint_as_float(ww[q] & 0xFFFF0000u), __uint_as_float(xx[q] & 0xFFFF0000u),
                                       acc);
                        }
                    }
                }
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xFFFFFFFFu, acc, o);
        }
        if (lane == 0) {
            p.cand_lg[t * RS_KMAX + j] = acc;
            p.cand_id[t * RS_KMAX + j] = id;
        }
    }
    __syncthreads();
    if (tid == 0) {
        __threadfence();
        is_last = atomicAdd(p.done, 1u) == gridDim.x * gridDim.y - 1u;
    }
    __syncthreads();
    if (!is_last) return;
    __threadfence();
    // the last CTA: warp r takes row r's argmax (lowest id on ties)
    if (warp < p.T) {
        float bv = 0.f;
        int bi = -1;
        for (int c = lane; c < p.k; c += 32) {
            const int id = __ldcg(&p.cand_id[warp * RS_KMAX + c]);
            const float v = __ldcg(&p.cand_lg[warp * RS_KMAX + c]);
            if (id >= 0 && (bi < 0 || v > bv || (v == bv && id < bi))) {
                bv = v;
                bi = id;
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const float ov = __shfl_xor_sync(0xFFFFFFFFu, bv, o);
            const int oi = __shfl_xor_sync(0xFFFFFFFFu, bi, o);
            if (oi >= 0 && (bi < 0 || ov > bv || (ov == bv && oi < bi))) {
                bv = ov;
                bi = oi;
            }
        }
        if (lane == 0) {
            lid[warp] = bi;
            lg[warp] = bi < 0 ? __int_as_float(0x7fc00000) : bv;
        }
    }
    __syncthreads();
    if (tid != 0) return;
    if (p.mode == 1) {
        for (int r = 0; r < p.T; ++r) {
            p.ids[r] = lid[r];
            if (p.vals) p.vals[r] = lg[r];
        }
    } else {
        const int n_draft = p.T - 1;
        int acc = n_draft;
        for (int i = 0; i < n_draft; ++i)
            if (p.drafts[i] != lid[i]) {
                acc = i;
                break;
            }
        p.accept_len[0] = acc;
        p.next_token[0] = lid[acc];
    }
    *p.done = 0u;                        // ready for the next call
}

// ---------------------------------------------------------------------------
// Exact speculative sampling verify over the 32 best logits of each row
// (page "OpenJet Engine: CUDA LLM inference for Qwen3.8-27B", sections "How
// it gets its speed": sampling keeps the 32 best logits of each verified
// row, accepts a draft with probability p(draft) and resamples a rejected
// one from the rest of the distribution; "Limitations": temperature, top-k
// <= 32, top-p and min-p in llama.cpp's order).
//
// The drafter is a point mass on its draft d: the acceptance probability
// is p(d) and the residual distribution is p without d, renormalised.  Chain
// per row, fp32, fixed order (m the best logit, d_j = l_j - m, candidates
// best first):
//   top-k:  the first min(top_k, 32) candidates (top_k <= 0: all 32);
//   top-p:  the shortest prefix whose running sum of exp(d_j) reaches
//           top_p times their sum (top_p >= 1: no cut);
//   min-p:  the prefix with exp(d_j) >= min_p (min_p <= 0: no cut);
//   temperature: w_j = exp(d_j / temperature), W = sum in order;
//           temperature <= 0: the point mass on the best candidate.
// Row i < n_draft accepts iff u[2i] * W < w_d; a rejected row draws from
// the candidates other than d, and the last row from all of them: walk the
// candidates best first with running sum c and take the first with
// u[2i+1] * W' < c.

constexpr int SAMPLE_KEEP = 32;

struct SampleParams {
    const float *logits;                 // [T][V] from the int4 pass
    const unsigned long long *smax;      // [T][nS] from slicemax_kernel
    int nS, T, V;
    float temperature, top_p, min_p;
    int top_k;
    int mode;                            // 0: verify, 1: distributions only
    const float *u;                      // [2T] uniforms in [0, 1) (verify)
    const int32_t *drafts;               // [T-1] (verify)
    int32_t *accept_len, *next_token;    // [1] (verify)
    int32_t *out_ids;                    // [T][32] (distributions; -1 past the kept candidates)
    float *out_probs;                    // [T][32] (distributions; w_j / W, 0 past them)
    int32_t *row_acc, *row_tok;          // scratch [RS_TMAX]
    unsigned *done;                      // scratch counter, left at 0
};

// One CTA per verify row.  Dynamic shared memory: RS_SEL_MAX keys.
__global__ void __launch_bounds__(RS_THREADS) sample_kernel(const __grid_constant__ SampleParams p)
{
    extern __shared__ __align__(16) unsigned long long sel[];
    __shared__ SelectSmem sm;
    __shared__ float es[SAMPLE_KEEP], ds[SAMPLE_KEEP], ws[SAMPLE_KEEP];
    __shared__ int ids[SAMPLE_KEEP];
    __shared__ int n_keep;
    __shared__ float Wsum;
    __shared__ unsigned is_last;
    const int t = blockIdx.x, tid = threadIdx.x, lane = tid & 31;
    pdl_wait_prior();                    // logits and slice maxima come from the passes before
    const int keep = min(SAMPLE_KEEP, p.V);
    select_row(p.smax + static_cast<size_t>(t) * p.nS, p.logits + static_cast<size_t>(t) * p.V, p.nS, p.V, keep,
               sel, sm);
    if (tid < 32) {
        // the chain, by warp 0: lane j holds candidate j
        const unsigned long long key = lane < keep ? sel[lane] : 0ull;
        const float l = key ? key_value(key) : 0.f;
        ids[lane] = key ? key_id(key) : -1;
        const float m = __shfl_sync(0xFFFFFFFFu, l, 0);
        const float d = l - m;
        es[lane] = expf(d);
        ds[lane] = d;
        __syncwarp();
        if (lane == 0) {
            int n = keep;
            if (p.top_k > 0) n = min(n, p.top_k);
            if (p.temperature > 0.f) {
                if (p.top_p < 1.f) {
                    float S = 0.f;
                    for (int j = 0; j < n; ++j) S = S + es[j];
                    const float thr = p.top_p * S;
                    float c = 0.f;
                    for (int j = 0; j < n; ++j) {
                        c = c + es[j];
                        if (c >= thr) {
                            n = j + 1;
                            break;
                        }
                    }
                }
                if (p.min_p > 0.f) {
                    int k = 1;
                    while (k < n && es[k] >= p.min_p) ++k;
                    n = k;
                }
            } else {
                n = 1;
            }
            n_keep = n;
        }
        __syncwarp();
        const int n = n_keep;
        if (lane < n) ws[lane] = p.temperature > 0.f ? expf(ds[lane] / p.temperature) : 1.f;
        __syncwarp();
        if (lane == 0) {
            float W = 0.f;
            for (int j = 0; j < n; ++j) W = W + ws[j];
            Wsum = W;
        }
        __syncwarp();
        if (p.mode == 1) {
            p.out_ids[t * SAMPLE_KEEP + lane] = lane < n ? ids[lane] : -1;
            p.out_probs[t * SAMPLE_KEEP + lane] = lane < n ? ws[lane] / Wsum : 0.f;
        } else if (lane == 0) {
            const bool draft_row = t < p.T - 1;
            int jd = -1;
            int acc = 0;
            if (draft_row) {
                const int dr = p.drafts[t];
                for (int j = 0; j < n; ++j)
                    if (ids[j] == dr) {
                        jd = j;
                        break;
                    }
                acc = (jd >= 0 && p.u[2 * t] * Wsum < ws[jd]) ? 1 : 0;
            }
            // the draw from the candidates other than jd (all of them on the
            // last row); with none left the draft itself (then it was
            // accepted with probability 1)
            float Wx = 0.f;
            int last = -1;
            for (int j = 0; j < n; ++j)
                if (j != jd) {
                    Wx = Wx + ws[j];
                    last = j;
                }
            int tok = jd >= 0 ? ids[jd] : ids[0];
            if (last >= 0) {
                const float target = p.u[2 * t + 1] * Wx;
                float c = 0.f;
                int pick = last;
                for (int j = 0; j < n; ++j) {
                    if (j == jd) continue;
                    c = c + ws[j];
                    if (target < c) {
                        pick = j;
                        break;
                    }
                }
                tok = ids[pick];
            }
            p.row_acc[t] = acc;
            p.row_tok[t] = tok;
        }
    }
    if (p.mode == 1) return;
    __syncthreads();
    if (tid == 0) {
        __threadfence();
        is_last = atomicAdd(p.done, 1u) == gridDim.x - 1u;
    }
    __syncthreads();
    if (!is_last || tid != 0) return;
    __threadfence();
    const int n_draft = p.T - 1;
    int acc = n_draft;
    for (int i = 0; i < n_draft; ++i)
        if (!__ldcg(&p.row_acc[i])) {
            acc = i;
            break;
        }
    p.accept_len[0] = acc;
    p.next_token[0] = __ldcg(&p.row_tok[acc]);
    *p.done = 0u;                        // ready for the next call
}

}  // namespace sv
