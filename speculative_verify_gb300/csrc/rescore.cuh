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
//  3. rescore_kernel, grid (ceil(k / 16), T): with tau a threshold that at
//     least k slice maxima reach, the row's k best keys are all >= tau and
//     lie in the slices whose maximum is >= tau.  Every CTA of the row finds
//     such a tau reached by at most 64 slices (select_row), re-reads those
//     slices, keeps their keys >= tau (at most 128 per slice), sorts them,
//     and rescores its share of the k best: fp32 dot products of their bf16
//     rows with x.  The last CTA of the grid takes each row's argmax (lowest
//     id on ties) and runs the greedy verify.
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

// Largest 64-bit key across the warp: the largest high word, then the
// largest low word among the lanes holding it (two 32-bit reductions).
__device__ __forceinline__ unsigned long long warp_max_u64(unsigned long long v)
{
    const unsigned hi = static_cast<unsigned>(v >> 32);
    const unsigned mh = __reduce_max_sync(0xFFFFFFFFu, hi);
    const unsigned lo = __reduce_max_sync(0xFFFFFFFFu, hi == mh ? static_cast<unsigned>(v) : 0u);
    return (static_cast<unsigned long long>(mh) << 32) | lo;
}

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
        m = warp_max_u64(m);
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

// Exact threshold: the k-th largest of the nS slice maxima mx (k <= 64),
// by the whole CTA.  Each warp keeps the 64 best maxima of its chunks of
// 128 (register sort, then merge), the warps' lists are merged pairwise in
// a tree.  Ends with __syncthreads; the result is in sm.tau.
__device__ __forceinline__ void exact_tau(const unsigned long long *mx, int nS, int k, SelectSmem &sm)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
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
#pragma unroll
    for (int st = 1; st < RS_WARPS; st <<= 1) {
        __syncthreads();
        if ((warp & (2 * st - 1)) == 0) {
            warp_merge64_desc(a0, a1, sm.wl[warp + st][lane], sm.wl[warp + st][32 + lane], lane);
            sm.wl[warp][lane] = a0;
            sm.wl[warp][32 + lane] = a1;
        }
    }
    if (warp == 0) {
        const int kk = k - 1;
        const unsigned long long tk = shfl_u64(kk < 32 ? a0 : a1, kk & 31);
        if (lane == 0) sm.tau = tk;
    }
    __syncthreads();
}

// The slices whose maximum is >= sm.tau into sm.slist (their number, which
// may exceed RS_KMAX, in sm.n_sl).  Ends with __syncthreads.
__device__ __forceinline__ void list_slices(const unsigned long long *mx, int nS, SelectSmem &sm)
{
    const unsigned long long tau = sm.tau;
    for (int s = threadIdx.x; s < nS; s += RS_THREADS) {
        const unsigned long long m = __ldcg(mx + s);
        if (m != 0ull && m >= tau) {
            const unsigned at = atomicAdd(&sm.n_sl, 1u);
            if (at < static_cast<unsigned>(RS_KMAX)) sm.slist[at] = s;
        }
    }
    __syncthreads();
}

// The k best (logit, id) keys of one row (k <= 64), descending, into
// sel[0..k) (keys past the row's candidates are 0), by the whole CTA; sel
// holds RS_SEL_MAX keys.  mx: the row's nS slice maxima; row: its V fp32
// logits.  Any tau with at least k slice maxima >= tau is a valid
// threshold: the row's k best keys are then >= tau, and each lies in a
// slice whose maximum is >= tau.  The first try takes the k-th best of the
// warps' m best maxima (one chunk of 128 per warp; m = 4 for k <= 32, else
// 8); if more than RS_KMAX slices reach it, tau becomes the exact k-th
// largest maximum, which exactly k slices reach.  The keys >= tau of those
// slices (at most 128 per slice) are gathered and put in order.
__device__ __forceinline__ void select_row(const unsigned long long *mx, const float *row, int nS, int V, int k,
                                           unsigned long long *sel, SelectSmem &sm)
{
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (tid == 0) {
        sm.n_sel = 0u;
        sm.n_sl = 0u;
        sm.tau = 0ull;
    }
    bool exact = nS > RS_WARPS * RS_SLICE;
    if (!exact) {
        unsigned long long *top = &sm.wl[0][0];          // [RS_WARPS * 8]
        unsigned long long kv[4], v[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int s = warp * RS_SLICE + i * 32 + lane;
            kv[i] = s < nS ? __ldcg(mx + s) : 0ull;
            v[i] = kv[i];
        }
        const int rounds = k <= 32 ? 4 : 8;
#pragma unroll
        for (int r = 0; r < 8; ++r) {
            unsigned long long m = 0ull;
            if (r < rounds) {
                m = warp_max_u64(kmax(kmax(v[0], v[1]), kmax(v[2], v[3])));
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    if (v[i] == m) v[i] = 0ull;           // keys are unique (0: none left)
            }
            if (lane == 0) top[warp * 8 + r] = m;
        }
        __syncthreads();
        // tau: the one of the 128 whose rank is k - 1 (stays 0 if fewer
        // than k are nonzero)
        if (tid < RS_WARPS * 8) {
            const unsigned long long key = top[tid];
            int rank = 0;
            for (int j = 0; j < RS_WARPS * 8; ++j) rank += top[j] > key;
            if (key != 0ull && rank == k - 1) sm.tau = key;
        }
        __syncthreads();
        // the slices that reach tau, from the maxima still in registers
        const unsigned long long tau = sm.tau;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int s = warp * RS_SLICE + i * 32 + lane;
            const bool in = s < nS && kv[i] != 0ull && kv[i] >= tau;
            const unsigned bal = __ballot_sync(0xFFFFFFFFu, in);
            if (bal) {
                unsigned base = 0u;
                if (lane == 0) base = atomicAdd(&sm.n_sl, static_cast<unsigned>(__popc(bal)));
                base = __shfl_sync(0xFFFFFFFFu, base, 0);
                const unsigned at = base + __popc(bal & ((1u << lane) - 1u));
                if (in && at < static_cast<unsigned>(RS_KMAX)) sm.slist[at] = s;
            }
        }
        __syncthreads();
        if (sm.n_sl > static_cast<unsigned>(RS_KMAX)) {
            exact = true;
            __syncthreads();
            if (tid == 0) sm.n_sl = 0u;
        }
    }
    if (exact) {
        exact_tau(mx, nS, k, sm);
        list_slices(mx, nS, sm);
    }
    // the keys >= tau of the listed slices, two slices per warp in flight
    const unsigned long long tau = sm.tau;
    const int nsl = min(static_cast<int>(sm.n_sl), RS_KMAX);
    for (int j0 = warp; j0 < nsl; j0 += 2 * RS_WARPS) {
        float f[8];
        int r0[2];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int j = j0 + h * RS_WARPS;
            r0[h] = j < nsl ? sm.slist[j] * RS_SLICE : V;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int r = r0[h] + i * 32 + lane;
                f[h * 4 + i] = r < V ? __ldcg(row + r) : 0.f;
            }
        }
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            const int r = r0[q >> 2] + (q & 3) * 32 + lane;
            const unsigned long long key = r < V ? make_key(f[q], static_cast<uint32_t>(r)) : 0ull;
            const bool keep = key != 0ull && key >= tau;
            const unsigned bal = __ballot_sync(0xFFFFFFFFu, keep);
            if (bal) {
                unsigned base = 0u;
                if (lane == 0) base = atomicAdd(&sm.n_sel, static_cast<unsigned>(__popc(bal)));
                base = __shfl_sync(0xFFFFFFFFu, base, 0);
                const unsigned at = base + __popc(bal & ((1u << lane) - 1u));
                if (keep && at < static_cast<unsigned>(RS_SEL_MAX)) sel[at] = key;
            }
        }
    }
    __syncthreads();
    const int ns = min(static_cast<int>(sm.n_sel), RS_SEL_MAX);
    if (ns <= RS_THREADS) {
        // keys are unique: each goes to its rank (the number of larger ones)
        const unsigned long long key = tid < ns ? sel[tid] : 0ull;
        int rank = 0;
        if (tid < ns)
            for (int j = 0; j < ns; ++j) rank += sel[j] > key;
        __syncthreads();
        if (tid < ns) sel[rank] = key;
        for (int j = ns + tid; j < k; j += RS_THREADS) sel[j] = 0ull;
        __syncthreads();
    } else {
        int npad = 1;
        while (npad < ns || npad < k) npad <<= 1;
        for (int i = ns + tid; i < npad; i += RS_THREADS) sel[i] = 0ull;
        __syncthreads();
        cta_sort_desc(sel, npad);
    }
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

// Inclusive prefix sums across the warp (lane j: sum of lanes 0..j), in
// the order: for d = 1, 2, 4, 8, 16, lane j adds lane j - d.
__device__ __forceinline__ float warp_scan_f32(float v, int lane)
{
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const float o = __shfl_up_sync(0xFFFFFFFFu, v, d);
        if (lane >= d) v = v + o;
    }
    return v;
}

// One CTA per verify row.  Dynamic shared memory: RS_SEL_MAX keys.
__global__ void __launch_bounds__(RS_THREADS) sample_kernel(const __grid_constant__ SampleParams p)
{
    extern __shared__ __align__(16) unsigned long long sel[];
    __shared__ SelectSmem sm;
    __shared__ unsigned is_last;
    const int t = blockIdx.x, tid = threadIdx.x, lane = tid & 31;
    pdl_wait_prior();                    // logits and slice maxima come from the passes before
    const bool verify = p.mode == 0;
    const bool draft_row = verify && t < p.T - 1;
    // the row's inputs, loaded now so that they arrive during the selection
    int dr = -1;
    float u_acc = 0.f, u_smp = 0.f;
    if (tid < 32 && verify) {
        if (draft_row) dr = p.drafts[t];
        u_acc = p.u[2 * t];
        u_smp = p.u[2 * t + 1];
    }
    const int keep = min(SAMPLE_KEEP, p.V);
    select_row(p.smax + static_cast<size_t>(t) * p.nS, p.logits + static_cast<size_t>(t) * p.V, p.nS, p.V, keep,
               sel, sm);
    if (tid < 32) {
        // the chain, by warp 0: lane j holds candidate j
        const unsigned long long key = lane < keep ? sel[lane] : 0ull;
        const float l = key ? key_value(key) : 0.f;
        const int id = key ? key_id(key) : -1;
        const float m = __shfl_sync(0xFFFFFFFFu, l, 0);
        const float d = l - m;
        int n = keep;
        if (p.top_k > 0) n = min(n, p.top_k);
        float w;
        if (p.temperature > 0.f) {
            const float e = lane < n ? expf(d) : 0.f;
            if (p.top_p < 1.f) {
                const float c = warp_scan_f32(e, lane);
                const float thr = p.top_p * __shfl_sync(0xFFFFFFFFu, c, n - 1);
                const unsigned hit = __ballot_sync(0xFFFFFFFFu, lane < n && c >= thr);
                if (hit) n = __ffs(hit);
            }
            if (p.min_p > 0.f) {
                const unsigned low = __ballot_sync(0xFFFFFFFFu, lane >= 1 && lane < n && !(e >= p.min_p));
                if (low) n = __ffs(low) - 1;
            }
            w = lane < n ? expf(d / p.temperature) : 0.f;
        } else {
            n = 1;
            w = lane == 0 ? 1.f : 0.f;
        }
        const float W = __shfl_sync(0xFFFFFFFFu, warp_scan_f32(w, lane), n - 1);
        if (!verify) {
            p.out_ids[t * SAMPLE_KEEP + lane] = lane < n ? id : -1;
            p.out_probs[t * SAMPLE_KEEP + lane] = lane < n ? w / W : 0.f;
        } else {
            // the draft's position among the kept candidates, the accept
            // test, then the draw from the candidates other than it (all of
            // them on the last row); with none left the draft itself (it
            // was then accepted with probability 1)
            const unsigned at = __ballot_sync(0xFFFFFFFFu, draft_row && lane < n && id == dr);
            const int jd = at ? __ffs(at) - 1 : -1;
            const float w_d = __shfl_sync(0xFFFFFFFFu, w, jd >= 0 ? jd : 0);
            const int acc = (jd >= 0 && u_acc * W < w_d) ? 1 : 0;
            const float wx = lane == jd ? 0.f : w;
            const float cx = warp_scan_f32(wx, lane);
            const float Wx = __shfl_sync(0xFFFFFFFFu, cx, n - 1);
            const float target = u_smp * Wx;
            const unsigned may = __ballot_sync(0xFFFFFFFFu, lane < n && lane != jd);
            const unsigned below = __ballot_sync(0xFFFFFFFFu, lane < n && lane != jd && target < cx);
            int pick = below ? __ffs(below) - 1 : (may ? 31 - __clz(may) : jd);
            const int tok = __shfl_sync(0xFFFFFFFFu, id, pick);
            if (lane == 0) {
                p.row_acc[t] = acc;
                p.row_tok[t] = tok;
            }
        }
    }
    if (!verify) return;
    __syncthreads();
    if (tid == 0) {
        __threadfence();
        is_last = atomicAdd(p.done, 1u) == gridDim.x - 1u;
    }
    __syncthreads();
    if (!is_last || tid >= 32) return;
    __threadfence();
    const int n_draft = p.T - 1;
    const bool rejected = lane < n_draft && !__ldcg(&p.row_acc[lane]);
    const unsigned rej = __ballot_sync(0xFFFFFFFFu, rejected);
    const int acc = rej ? __ffs(rej) - 1 : n_draft;
    if (lane == 0) {
        p.accept_len[0] = acc;
        p.next_token[0] = __ldcg(&p.row_tok[acc]);
        *p.done = 0u;                    // ready for the next call
    }
}

}  // namespace sv
