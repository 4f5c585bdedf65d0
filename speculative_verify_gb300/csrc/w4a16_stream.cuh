// w4a16_stream.cuh -- the one kernel behind every export: a stream-K pass
// over 64-row tiles of a W4A16 (uint32 nibble words, bf16 group-128 scales)
// weight matrix, with either a GEMM epilogue (y = bf16) or an lm_head
// epilogue (fp32 logits -> per-CTA top-1 -> grid argmax -> greedy verify).
//
// Work decomposition.  A "unit" is one 64-row tile x one 128-column group
// (4 KB of packed weights).  Units are numbered tile-major and the grid's B
// CTAs (B <= SM count, one CTA per SM) take equal contiguous ranges, so every
// SM streams the same number of bytes whatever N and K are.  A tile whose
// units straddle two CTAs is finished by the last CTA to arrive (per-tile
// counter in the scratch area), which adds the fp32 partial sums of all the
// tile's CTAs in a fixed order: results do not depend on arrival order.
//
// Inside a CTA: warp 16 is the producer.  It streams each stage (up to GPS
// units of one tile) with 1-D bulk copies: one copy per weight row
// (contiguous along K) plus one per activation row, completing on the
// stage's mbarrier.  Warps 0..15 consume: warp w takes group (w % GPS) of
// the stage for R m16 tiles, dequantises its nibbles in registers and feeds
// them to the bf16 tensor cores as the A operand (mma.sync m16n8k16, tokens
// as the n8 B operand), and folds each group's fp32 sum into its accumulators
// with the group scale.  Every weight byte crosses HBM once per call; T only
// changes how many n8 token tiles each fragment is multiplied with.
#pragma once

#include <cstdint>
#include <cuda_bf16.h>

#include "sv_ptx.cuh"

namespace sv {

constexpr int ROWS = 64;                        // rows per tile
constexpr int NCW = 16;                         // consumer warps
constexpr int NTHREADS = (NCW + 1) * 32;        // + one producer warp
constexpr int CONSUMERS = NCW * 32;
constexpr int TMAX = 32;                        // largest T
constexpr int PART_FLOATS = TMAX * ROWS;        // one split-tile partial
constexpr uint64_t WAIT_LIMIT_NS = 2000000000ull;      // 2 s: only a broken run gets here
constexpr uint64_t WAIT_LIMIT_AFTER_ERR_NS = 1000000ull; // 1 ms once something failed

template <int NT>
struct Cfg {
    static constexpr int GPS = (NT == 1) ? 8 : 4;   // 128-column groups per stage
    static constexpr int MSETS = NCW / GPS;         // warps sharing one group slot
    static constexpr int R = 4 / MSETS;             // m16 tiles per warp
    static constexpr int TP = 8 * NT;               // tokens, padded to n8 tiles
    // Shared-memory row strides, chosen so that the 8 lanes of a quarter
    // warp hit distinct banks: weights stride = 64 (mod 128), activations
    // stride = 32 (mod 128).
    static constexpr int WSTR = GPS * 64 + 64;
    static constexpr int XSTR = GPS * 256 + 32;
    static constexpr int RED_FLOATS = GPS * TP * ROWS;
};

struct Params {
    const uint16_t *x;          // [T][K] bf16 bits
    const uint32_t *Wq;         // [rows][K/8]
    const uint16_t *scales;     // [rows][K/128]
    const int32_t *map;         // HEAD: candidate row -> token id, or null
    int T, K, G;                // G = K / 128
    int n_rows;                 // GEMM: N; HEAD: V or n_map
    int V;                      // HEAD: token ids must be < V
    long long U;                // units = tiles * G
    int nst;                    // pipeline stages
    int stage_bytes;
    // GEMM output
    uint16_t *y;                // [T][N]
    // HEAD outputs
    int mode;                   // 0: verify, 1: argmax
    const int32_t *drafts;      // [n_streams][n_draft]
    int n_draft, n_streams;
    int32_t *accept_len, *next_token;   // [n_streams]
    int32_t *ids;               // [T]
    float *vals;                // [T] or null
    // scratch (per device)
    float *part;                // [B][2][PART_FLOATS]
    unsigned *ctr;              // [B] split-tile arrival counters (kept at 0 between calls)
    unsigned long long *keys;   // [TMAX] grid argmax keys (kept at 0 between calls)
    unsigned *done;             // CTA completion counter (kept at 0 between calls)
    int *err;                   // sticky device error word
};

__device__ __forceinline__ long long cta_start(long long b, long long U, int B)
{
    return b * U / B;
}

// The CTA whose range holds unit u.
__device__ __forceinline__ int cta_of(long long u, long long U, int B)
{
    long long b = u * B / U;
    while (b + 1 < B && cta_start(b + 1, U, B) <= u) ++b;
    while (b > 0 && cta_start(b, U, B) > u) --b;
    return static_cast<int>(b);
}

template <int NT, bool HEAD>
__global__ void __launch_bounds__(NTHREADS, 1) w4a16_stream_kernel(const Params p)
{
    using C = Cfg<NT>;
    extern __shared__ __align__(128) uint8_t smem[];
    const int nst = p.nst;
    float *red = reinterpret_cast<float *>(smem + static_cast<size_t>(nst) * p.stage_bytes);
    float *lg = red;            // HEAD logits [TP][ROWS] reuse the reduction buffer
    unsigned long long *best = reinterpret_cast<unsigned long long *>(red + C::RED_FLOATS);
    volatile int *flags = reinterpret_cast<volatile int *>(best + TMAX);
    uint64_t *bars = reinterpret_cast<uint64_t *>(const_cast<int *>(flags) + 4);
    uint64_t *full = bars;
    uint64_t *empty = bars + nst;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int B = gridDim.x, b = blockIdx.x;
    const long long U = p.U;
    const int G = p.G, K = p.K, T = p.T;
    const long long u0 = cta_start(b, U, B), u1 = cta_start(b + 1, U, B);

    if (threadIdx.x == 0) {
        for (int s = 0; s < nst; ++s) {
            mbar_init(smem_addr(&full[s]), 1);
            mbar_init(smem_addr(&empty[s]), NCW);
        }
        fence_barrier_init();
        flags[0] = 0;   // a wait timed out in this CTA
        flags[1] = 0;   // this CTA finishes the current split tile
        flags[2] = 0;   // this CTA is the last one of the grid
    }
    if (threadIdx.x < TMAX) best[threadIdx.x] = 0ull;
    __syncthreads();

    if (warp == NCW) {
        // ============================================================ producer
        const uint64_t pol_w = policy_evict_first();
        const uint64_t pol_x = policy_evict_last();
        int s = 0;
        uint32_t ph = 0;
        int issued = 0;
        for (long long u = u0; u < u1;) {
            const long long tile = u / G;
            const int grp0 = static_cast<int>(u - tile * G);
            const long long tile_end = (tile + 1) * G;
            const int n = static_cast<int>(min(static_cast<long long>(C::GPS), min(u1 - u, tile_end - u)));
            if (issued >= nst) {
                const uint64_t lim = flags[0] ? WAIT_LIMIT_AFTER_ERR_NS : WAIT_LIMIT_NS;
                if (!mbar_wait_bounded(smem_addr(&empty[s]), ph ^ 1u, lim)) {
                    flags[0] = 1;
                    atomicOr(p.err, 2);
                }
            }
            // Source rows of this lane's two copies.
            long long src[2];
            bool ok[2];
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const long long rg = tile * ROWS + lane + 32 * h;
                ok[h] = rg < p.n_rows;
                src[h] = rg;
                if (ok[h] && p.map) {
                    const int id = p.map[rg];
                    if (id < 0 || id >= p.V) {
                        ok[h] = false;
                        atomicOr(p.err, 1);
                    }
                    src[h] = id;
                }
            }
            const int cnt = __popc(__ballot_sync(0xFFFFFFFFu, ok[0])) +
                            __popc(__ballot_sync(0xFFFFFFFFu, ok[1]));
            const uint32_t bytes = static_cast<uint32_t>(cnt * n * 64 + T * n * 256);
            const uint32_t fb = smem_addr(&full[s]);
            if (lane == 0) mbar_arrive_expect_tx(fb, bytes);
            __syncwarp();
            const uint32_t wdst = smem_addr(smem + static_cast<size_t>(s) * p.stage_bytes);
#pragma unroll
            for (int h = 0; h < 2; ++h)
                if (ok[h])
                    bulk_g2s(wdst + (lane + 32 * h) * C::WSTR,
                             p.Wq + static_cast<size_t>(src[h]) * (K / 8) + grp0 * 16,
                             static_cast<uint32_t>(n * 64), fb, pol_w);
            if (lane < T)
                bulk_g2s(wdst + ROWS * C::WSTR + lane * C::XSTR,
                         p.x + static_cast<size_t>(lane) * K + grp0 * 128,
                         static_cast<uint32_t>(n * 256), fb, pol_x);
            u += n;
            ++issued;
            if (++s == nst) { s = 0; ph ^= 1u; }
        }
        // Do not leave while a copy of ours may still be landing.
        int left = min(issued, nst);
        int ds = s;
        uint32_t dph = ph;
        while (left-- > 0) {
            if (--ds < 0) { ds = nst - 1; dph ^= 1u; }
            if (!mbar_wait_bounded(smem_addr(&full[ds]), dph, WAIT_LIMIT_AFTER_ERR_NS)) {
                flags[0] = 1;
                atomicOr(p.err, 2);
            }
        }
        return;
    }

    // ================================================================ consumers
    const int cw = warp;
    const int slot = cw % C::GPS;
    const int mset = cw / C::GPS;
    const int g = lane >> 2, c = lane & 3;
    const int tid = cw * 32 + lane;

    float acc[C::R][NT][4];
#pragma unroll
    for (int r = 0; r < C::R; ++r)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[r][nt][e] = 0.f;

    long long cur_tile = -1;
    const uint16_t *srow[C::R][2];   // scale row of each of this lane's rows (null: invalid)

    int s = 0;
    uint32_t ph = 0;
    for (long long u = u0; u < u1;) {
        const long long tile = u / G;
        const int grp0 = static_cast<int>(u - tile * G);
        const long long tile_end = (tile + 1) * G;
        const int n = static_cast<int>(min(static_cast<long long>(C::GPS), min(u1 - u, tile_end - u)));
        if (tile != cur_tile) {
            cur_tile = tile;
#pragma unroll
            for (int r = 0; r < C::R; ++r)
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const long long rg = tile * ROWS + (mset * C::R + r) * 16 + g + 8 * h;
                    const uint16_t *sp = nullptr;
                    if (rg < p.n_rows) {
                        long long id = rg;
                        if (p.map) id = p.map[rg];
                        if (id >= 0 && (!p.map || id < p.V)) sp = p.scales + static_cast<size_t>(id) * G;
                    }
                    srow[r][h] = sp;
                }
        }
        {
            const uint64_t lim = flags[0] ? WAIT_LIMIT_AFTER_ERR_NS : WAIT_LIMIT_NS;
            if (!mbar_wait_bounded(smem_addr(&full[s]), ph, lim)) {
                flags[0] = 1;
                atomicOr(p.err, 2);
            }
        }
        if (slot < n) {
            const int grp = grp0 + slot;
            float sc[C::R][2];
#pragma unroll
            for (int r = 0; r < C::R; ++r)
#pragma unroll
                for (int h = 0; h < 2; ++h)
                    sc[r][h] = srow[r][h] ? bf16_bits_to_float(ldg_u16(srow[r][h] + grp)) : 0.f;

            const uint32_t stage = smem_addr(smem + static_cast<size_t>(s) * p.stage_bytes);
            const uint32_t wbase = stage + (mset * C::R * 16 + g) * C::WSTR + slot * 64 + c * 16;
            uint4 wa[C::R], wb[C::R];
#pragma unroll
            for (int r = 0; r < C::R; ++r) {
                wa[r] = lds128(wbase + r * 16 * C::WSTR);
                wb[r] = lds128(wbase + (r * 16 + 8) * C::WSTR);
            }
            float gacc[C::R][NT][4];
#pragma unroll
            for (int r = 0; r < C::R; ++r)
#pragma unroll
                for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                    for (int e = 0; e < 4; ++e) gacc[r][nt][e] = 0.f;

            const uint32_t xbase = stage + ROWS * C::WSTR + slot * 256 + c * 64;
#pragma unroll
            for (int m = 0; m < 4; ++m) {
                // B fragments: token (nt*8 + g), the 8 activations of word
                // (4c + m) of the group, paired (j, j+4) like the nibbles.
                uint32_t bx[NT][4];
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    const int tok = nt * 8 + g;
                    if (tok < T) {
                        const uint4 v = lds128(xbase + tok * C::XSTR + m * 16);
                        bx[nt][0] = __byte_perm(v.x, v.z, 0x5410);   // (x0, x4)
                        bx[nt][1] = __byte_perm(v.x, v.z, 0x7632);   // (x1, x5)
                        bx[nt][2] = __byte_perm(v.y, v.w, 0x5410);   // (x2, x6)
                        bx[nt][3] = __byte_perm(v.y, v.w, 0x7632);   // (x3, x7)
                    } else {
                        bx[nt][0] = bx[nt][1] = bx[nt][2] = bx[nt][3] = 0u;
                    }
                }
#pragma unroll
                for (int r = 0; r < C::R; ++r) {
                    const uint32_t wA = (m == 0) ? wa[r].x : (m == 1) ? wa[r].y : (m == 2) ? wa[r].z : wa[r].w;
                    const uint32_t wB = (m == 0) ? wb[r].x : (m == 1) ? wb[r].y : (m == 2) ? wb[r].z : wb[r].w;
                    // k-step 2m: nibble pairs (0,4) and (1,5)
                    uint32_t a0 = dequant2(wA), a1 = dequant2(wB);
                    uint32_t a2 = dequant2(wA >> 4), a3 = dequant2(wB >> 4);
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt)
                        mma_bf16_16816(gacc[r][nt], a0, a1, a2, a3, bx[nt][0], bx[nt][1]);
                    // k-step 2m+1: nibble pairs (2,6) and (3,7)
                    a0 = dequant2(wA >> 8);
                    a1 = dequant2(wB >> 8);
                    a2 = dequant2(wA >> 12);
                    a3 = dequant2(wB >> 12);
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt)
                        mma_bf16_16816(gacc[r][nt], a0, a1, a2, a3, bx[nt][2], bx[nt][3]);
                }
            }
#pragma unroll
            for (int r = 0; r < C::R; ++r)
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    acc[r][nt][0] += sc[r][0] * gacc[r][nt][0];
                    acc[r][nt][1] += sc[r][0] * gacc[r][nt][1];
                    acc[r][nt][2] += sc[r][1] * gacc[r][nt][2];
                    acc[r][nt][3] += sc[r][1] * gacc[r][nt][3];
                }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_addr(&empty[s]));
        if (++s == nst) { s = 0; ph ^= 1u; }
        u += n;

        if (u == tile_end || u == u1) {
            // ================================================ tile flush
            // 1. warp partials -> red[slot][tok][row]
#pragma unroll
            for (int r = 0; r < C::R; ++r)
#pragma unroll
                for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int row = (mset * C::R + r) * 16 + g + 8 * (e >> 1);
                        const int tok = nt * 8 + 2 * c + (e & 1);
                        red[(slot * C::TP + tok) * ROWS + row] = acc[r][nt][e];
                        acc[r][nt][e] = 0.f;
                    }
            named_bar_sync(1, CONSUMERS);

            // 2. sum the group slots in a fixed order
            constexpr int PER = (C::TP * ROWS + CONSUMERS - 1) / CONSUMERS;
            float v[PER];
#pragma unroll
            for (int q = 0; q < PER; ++q) {
                const int pidx = tid + q * CONSUMERS;
                const int tok = pidx / ROWS, row = pidx % ROWS;
                float sum = 0.f;
                if (tok < T) {
                    sum = red[tok * ROWS + row];
#pragma unroll
                    for (int sl = 1; sl < C::GPS; ++sl) sum += red[(sl * C::TP + tok) * ROWS + row];
                }
                v[q] = sum;
            }

            // 3. split tile: publish the partial; the last CTA adds them all
            const long long ts = tile * G, te = ts + G;
            const bool complete = (u0 <= ts) && (u1 >= te);
            bool finish = true;
            if (!complete) {
                const int bf = cta_of(ts, U, B), bl = cta_of(te - 1, U, B);
                const int which = (tile == u0 / G) ? 0 : 1;
                float *mine = p.part + (static_cast<size_t>(b) * 2 + which) * PART_FLOATS;
#pragma unroll
                for (int q = 0; q < PER; ++q) {
                    const int pidx = tid + q * CONSUMERS;
                    if (pidx / ROWS < T) mine[pidx] = v[q];
                }
                __threadfence();
                named_bar_sync(1, CONSUMERS);
                if (tid == 0) {
                    const unsigned old = atomicAdd(&p.ctr[bf], 1u);
                    const int last = (old == static_cast<unsigned>(bl - bf));
                    if (last) atomicExch(&p.ctr[bf], 0u);
                    flags[1] = last;
                }
                named_bar_sync(1, CONSUMERS);
                finish = flags[1] != 0;
                if (finish) {
                    __threadfence();
#pragma unroll
                    for (int q = 0; q < PER; ++q) {
                        const int pidx = tid + q * CONSUMERS;
                        if (pidx / ROWS >= T) continue;
                        float sum = 0.f;
                        for (int bb = bf; bb <= bl; ++bb) {
                            float pv;
                            if (bb == b) {
                                pv = v[q];
                            } else {
                                const int wb2 = (tile == cta_start(bb, U, B) / G) ? 0 : 1;
                                pv = __ldcg(p.part + (static_cast<size_t>(bb) * 2 + wb2) * PART_FLOATS + pidx);
                            }
                            sum = (bb == bf) ? pv : sum + pv;
                        }
                        v[q] = sum;
                    }
                }
            }

            // 4. epilogue
            if (finish) {
                if constexpr (!HEAD) {
#pragma unroll
                    for (int q = 0; q < PER; ++q) {
                        const int pidx = tid + q * CONSUMERS;
                        const int tok = pidx / ROWS, row = pidx % ROWS;
                        const long long rg = tile * ROWS + row;
                        if (tok < T && rg < p.n_rows)
                            p.y[static_cast<size_t>(tok) * p.n_rows + rg] =
                                __bfloat16_as_ushort(__float2bfloat16_rn(v[q]));
                    }
                } else {
                    named_bar_sync(1, CONSUMERS);     // red is about to become lg
#pragma unroll
                    for (int q = 0; q < PER; ++q) {
                        const int pidx = tid + q * CONSUMERS;
                        if (pidx / ROWS < T) lg[pidx] = v[q];
                    }
                    named_bar_sync(1, CONSUMERS);
                    // token ids of rows lane and lane + 32 of this tile
                    uint32_t idh[2];
                    bool okh[2];
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const long long rg = tile * ROWS + lane + 32 * h;
                        okh[h] = rg < p.n_rows;
                        long long id = rg;
                        if (okh[h] && p.map) {
                            id = p.map[rg];
                            okh[h] = id >= 0 && id < p.V;
                        }
                        idh[h] = static_cast<uint32_t>(id);
                    }
                    for (int tok = cw; tok < T; tok += NCW) {
                        unsigned long long k0 = okh[0] ? make_key(lg[tok * ROWS + lane], idh[0]) : 0ull;
                        unsigned long long k1 = okh[1] ? make_key(lg[tok * ROWS + lane + 32], idh[1]) : 0ull;
                        unsigned long long k = k0 > k1 ? k0 : k1;
#pragma unroll
                        for (int o = 16; o > 0; o >>= 1) {
                            const unsigned long long ko = shfl_xor_u64(k, o);
                            k = ko > k ? ko : k;
                        }
                        if (lane == 0 && k > best[tok]) best[tok] = k;
                    }
                }
            }
            named_bar_sync(1, CONSUMERS);   // red / lg free again
        }
    }

    if constexpr (HEAD) {
        // ==================================================== grid argmax + verify
        if (tid < T && best[tid] != 0ull) atomicMax(&p.keys[tid], best[tid]);
        __threadfence();
        named_bar_sync(1, CONSUMERS);
        if (tid == 0) {
            const unsigned old = atomicAdd(p.done, 1u);
            flags[2] = (old == static_cast<unsigned>(B - 1));
        }
        named_bar_sync(1, CONSUMERS);
        if (flags[2]) {
            __threadfence();
            int32_t *a = reinterpret_cast<int32_t *>(red);    // [TMAX] argmax ids
            if (tid < T) {
                const unsigned long long k = __ldcg(&p.keys[tid]);
                a[tid] = (k == 0ull) ? -1 : key_id(k);
                if (p.mode == 1) {
                    p.ids[tid] = a[tid];
                    if (p.vals) p.vals[tid] = (k == 0ull) ? __int_as_float(0x7fc00000) : key_value(k);
                }
                p.keys[tid] = 0ull;
            }
            named_bar_sync(1, CONSUMERS);
            if (p.mode == 0 && tid < p.n_streams) {
                const int rows_per = p.n_draft + 1;
                const int32_t *as = a + tid * rows_per;
                const int32_t *ds = p.drafts + static_cast<size_t>(tid) * p.n_draft;
                int i = 0;
                while (i < p.n_draft && ds[i] == as[i]) ++i;
                p.accept_len[tid] = i;
                p.next_token[tid] = as[i];
            }
            if (tid == 0) *p.done = 0u;
        }
    }
}

}  // namespace sv
