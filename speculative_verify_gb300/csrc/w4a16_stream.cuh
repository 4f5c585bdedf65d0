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
// Inside a CTA: warp 16 is the producer.  Each pipeline stage holds up to
// GPS units of one tile; the producer fills it with tensor (TMA) copies --
// one 64-row x 64-byte box per group of packed weights and one box of the
// activations per group -- completing on the stage's mbarrier.  (When rows
// are gathered through a vocab_map, each weight row segment is a 1-D bulk
// copy instead.)  Warps 0..15 consume: warp w takes group (w % GPS) of the
// stage for R m16 tiles, dequantises its nibbles in registers and feeds them
// to the bf16 tensor cores as the A operand (mma.sync m16n8k16, tokens as the
// n8 B operand), and folds each group's fp32 sum into its accumulators with
// the group scale.  Scales of a tile are staged in shared memory two tiles
// ahead with cp.async.  Every weight byte crosses HBM once per call; T only
// changes how many n8 token tiles each dequantised fragment multiplies.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>

#include "sv_ptx.cuh"

namespace sv {

constexpr int ROWS = 64;                        // rows per tile
constexpr int NCW = 16;                         // consumer warps
constexpr int NTHREADS = (NCW + 1) * 32;        // + one producer warp
constexpr int CONSUMERS = NCW * 32;
constexpr int TMAX = 32;                        // largest T
constexpr int PART_FLOATS = TMAX * ROWS;        // one split-tile partial
constexpr int XBOX = 144;                       // activation box width (elements)
constexpr int XROW_BYTES = XBOX * 2;            // = 32 (mod 128): conflict-free B loads
constexpr uint64_t WAIT_LIMIT_NS = 2000000000ull;        // 2 s: only a broken run gets here
constexpr uint64_t WAIT_LIMIT_AFTER_ERR_NS = 1000000ull;  // 1 ms once something failed

template <int NT, bool GATHER>
struct Cfg {
    static constexpr int GPS = (NT == 1) ? 8 : 4;   // 128-column groups per stage
    static constexpr int MSETS = NCW / GPS;         // warps sharing one group slot
    static constexpr int R = 4 / MSETS;             // m16 tiles per warp
    static constexpr int TP = 8 * NT;               // tokens, padded to n8 tiles
    // Weights in a stage.  Contiguous rows: one dense [64 rows][64 B] block
    // per group (a quarter warp reads 2 rows x 64 B = 128 consecutive bytes).
    // Gathered rows: [64 rows][GPS*64 B + 64 B pad] (row stride = 64 mod 128).
    static constexpr int WSTR_G = GPS * 64 + 64;
    static constexpr int W_BYTES = GATHER ? ROWS * WSTR_G : GPS * ROWS * 64;
    static constexpr int RED_FLOATS = GPS * TP * ROWS;
    static constexpr int RED_BUFS = (NT == 4) ? 1 : 2;
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
    // shared-memory layout (bytes)
    int nst, stage_bytes, xslot_bytes, sbuf_bytes;
    int off_sbuf, off_ids, off_red, off_best, off_flags, off_bars;
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

// Token id of row rloc of tile `tile` (or -1 when the row does not exist).
__device__ __forceinline__ int row_id(const Params &p, int tile, int rloc)
{
    const long long rg = static_cast<long long>(tile) * ROWS + rloc;
    if (rg >= p.n_rows) return -1;
    if (!p.map) return static_cast<int>(rg);
    const int id = p.map[rg];
    if (id >= 0 && id < p.V) return id;
    atomicOr(p.err, 1);
    return -1;
}

// Stage the scales (and, for the head, the token ids) of one tile into
// shared memory.  Warp w owns rows w, w+16, w+32, w+48.  Uses 4-byte
// cp.async when a scale row has an even number of groups, plain loads
// otherwise; the caller commits / waits.
template <bool HEAD>
__device__ __forceinline__ void stage_tile_meta(const Params &p, int tile, const int (&id)[4],
                                                uint8_t *sb, int32_t *ib, int cw, int lane)
{
    const int G = p.G;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int rloc = cw + 16 * i;
        uint16_t *dst = reinterpret_cast<uint16_t *>(sb) + rloc * G;
        if (HEAD && lane == 0) ib[rloc] = id[i];
        if (id[i] < 0) {
            for (int j = lane; j < G; j += 32) dst[j] = 0;
            continue;
        }
        const uint16_t *src = p.scales + static_cast<size_t>(id[i]) * G;
        if ((G & 1) == 0) {
            for (int j = lane; j < G / 2; j += 32) cp_async_4(smem_addr(dst + 2 * j), src + 2 * j);
        } else {
            for (int j = lane; j < G; j += 32) dst[j] = ldg_u16(src + j);
        }
    }
    (void)tile;
}

__device__ __forceinline__ void tile_ids(const Params &p, int tile, int last_tile, int cw, int (&id)[4])
{
#pragma unroll
    for (int i = 0; i < 4; ++i) id[i] = (tile <= last_tile) ? row_id(p, tile, cw + 16 * i) : -1;
}

template <int NT, bool HEAD, bool GATHER>
__global__ void __launch_bounds__(NTHREADS, 1)
w4a16_stream_kernel(const __grid_constant__ Params p, const __grid_constant__ CUtensorMap tmW,
                    const __grid_constant__ CUtensorMap tmX)
{
    using C = Cfg<NT, GATHER>;
    extern __shared__ __align__(1024) uint8_t smem[];
    const int nst = p.nst;
    uint8_t *sbuf = smem + p.off_sbuf;                       // [2][sbuf_bytes]
    int32_t *idbuf = reinterpret_cast<int32_t *>(smem + p.off_ids);   // [3][ROWS]
    float *red = reinterpret_cast<float *>(smem + p.off_red);          // [RED_BUFS][RED_FLOATS]
    unsigned long long *best = reinterpret_cast<unsigned long long *>(smem + p.off_best);  // [TMAX]
    volatile int *flags = reinterpret_cast<volatile int *>(smem + p.off_flags);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + p.off_bars);
    uint64_t *empty = full + nst;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int B = gridDim.x, b = blockIdx.x;
    const long long U = p.U;
    const int G = p.G, T = p.T;
    const long long u0 = cta_start(b, U, B), u1 = cta_start(b + 1, U, B);
    const int tile_first = static_cast<int>(u0 / G);
    const int grp_first = static_cast<int>(u0 - static_cast<long long>(tile_first) * G);
    const int tile_last = static_cast<int>((u1 - 1) / G);

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
        if (lane == 0) {
            if (!GATHER) prefetch_tmap(&tmW);
            prefetch_tmap(&tmX);
        }
        int s = 0, issued = 0, tile = tile_first, grp = grp_first;
        uint32_t ph = 0;
        // gathered rows: ids of this lane's two rows, for this tile and the next
        int gid[2] = {-1, -1}, gid_next[2] = {-1, -1};
        if (GATHER) {
            gid[0] = row_id(p, tile, lane);
            gid[1] = row_id(p, tile, lane + 32);
            if (tile + 1 <= tile_last) {
                gid_next[0] = row_id(p, tile + 1, lane);
                gid_next[1] = row_id(p, tile + 1, lane + 32);
            }
        }
        for (long long u = u0; u < u1;) {
            const int n = static_cast<int>(min(static_cast<long long>(min(C::GPS, G - grp)), u1 - u));
            if (issued >= nst) {
                const uint64_t lim = flags[0] ? WAIT_LIMIT_AFTER_ERR_NS : WAIT_LIMIT_NS;
                if (!mbar_wait_bounded(smem_addr(&empty[s]), ph ^ 1u, lim)) {
                    flags[0] = 1;
                    atomicOr(p.err, 2);
                }
            }
            const uint32_t fb = smem_addr(&full[s]);
            const uint32_t stage = smem_addr(smem + static_cast<size_t>(s) * p.stage_bytes);
            uint32_t wbytes;
            if (GATHER) {
                const int cnt = __popc(__ballot_sync(0xFFFFFFFFu, gid[0] >= 0)) +
                                __popc(__ballot_sync(0xFFFFFFFFu, gid[1] >= 0));
                wbytes = static_cast<uint32_t>(cnt * n * 64);
            } else {
                wbytes = static_cast<uint32_t>(n * ROWS * 64);
            }
            if (lane == 0) mbar_arrive_expect_tx(fb, wbytes + static_cast<uint32_t>(n * T * XROW_BYTES));
            __syncwarp();
            if (GATHER) {
#pragma unroll
                for (int h = 0; h < 2; ++h)
                    if (gid[h] >= 0)
                        bulk_g2s(stage + (lane + 32 * h) * C::WSTR_G,
                                 p.Wq + static_cast<size_t>(gid[h]) * (p.K / 8) + grp * 16,
                                 static_cast<uint32_t>(n * 64), fb, pol_w);
            } else if (lane < n) {
                tma_load_2d(stage + lane * (ROWS * 64), &tmW, (grp + lane) * 16, tile * ROWS, fb, pol_w);
            }
            if (lane >= 16 && lane - 16 < n)
                tma_load_2d(stage + C::W_BYTES + (lane - 16) * p.xslot_bytes, &tmX,
                            (grp + lane - 16) * 128, 0, fb, pol_x);
            u += n;
            grp += n;
            if (grp == G) {
                grp = 0;
                ++tile;
                if (GATHER) {
                    gid[0] = gid_next[0];
                    gid[1] = gid_next[1];
                    if (tile + 1 <= tile_last) {
                        gid_next[0] = row_id(p, tile + 1, lane);
                        gid_next[1] = row_id(p, tile + 1, lane + 32);
                    }
                }
            }
            ++issued;
            if (++s == nst) { s = 0; ph ^= 1u; }
        }
        // Do not leave while a copy of ours may still be landing.
        int left = min(issued, nst), ds = s;
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

    // Tile metadata: scales of tile k live in sbuf[k & 1], ids in idbuf[k % 3].
    int idreg[4];
    {
        tile_ids(p, tile_first, tile_last, cw, idreg);
        stage_tile_meta<HEAD>(p, tile_first, idreg, sbuf, idbuf, cw, lane);
        if (tile_first + 1 <= tile_last) {
            tile_ids(p, tile_first + 1, tile_last, cw, idreg);
            stage_tile_meta<HEAD>(p, tile_first + 1, idreg, sbuf + p.sbuf_bytes, idbuf + ROWS, cw, lane);
        }
        cp_async_commit();
        tile_ids(p, tile_first + 2, tile_last, cw, idreg);     // for the first flush
        cp_async_wait_all();
        named_bar_sync(1, CONSUMERS);
    }

    float acc[C::R][NT][4];
#pragma unroll
    for (int r = 0; r < C::R; ++r)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[r][nt][e] = 0.f;

    int s = 0, tile = tile_first, grp = grp_first, k_rel = 0, nflush = 0;
    uint32_t ph = 0;
    const uint32_t sbuf0 = smem_addr(sbuf);
    for (long long u = u0; u < u1;) {
        const int n = static_cast<int>(min(static_cast<long long>(min(C::GPS, G - grp)), u1 - u));
        {
            const uint64_t lim = flags[0] ? WAIT_LIMIT_AFTER_ERR_NS : WAIT_LIMIT_NS;
            if (!mbar_wait_bounded(smem_addr(&full[s]), ph, lim)) {
                flags[0] = 1;
                atomicOr(p.err, 2);
            }
        }
        if (slot < n) {
            const int gs = grp + slot;     // group within the row
            const uint32_t stage = smem_addr(smem + static_cast<size_t>(s) * p.stage_bytes);
            uint32_t wbase;
            constexpr int RSTEP = GATHER ? 16 * C::WSTR_G : 16 * 64;   // next m16 tile
            constexpr int HSTEP = GATHER ? 8 * C::WSTR_G : 8 * 64;     // row g + 8
            if (GATHER)
                wbase = stage + (mset * C::R * 16 + g) * C::WSTR_G + slot * 64 + c * 16;
            else
                wbase = stage + slot * (ROWS * 64) + (mset * C::R * 16 + g) * 64 + c * 16;
            uint4 wa[C::R], wb[C::R];
#pragma unroll
            for (int r = 0; r < C::R; ++r) {
                wa[r] = lds128(wbase + r * RSTEP);
                wb[r] = lds128(wbase + r * RSTEP + HSTEP);
            }
            float gacc[C::R][NT][4];
#pragma unroll
            for (int r = 0; r < C::R; ++r)
#pragma unroll
                for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                    for (int e = 0; e < 4; ++e) gacc[r][nt][e] = 0.f;

            const uint32_t xbase = stage + C::W_BYTES + slot * p.xslot_bytes + c * 64;
#pragma unroll
            for (int m = 0; m < 4; ++m) {
                // B fragments: token (nt*8 + g), the 8 activations of word
                // (4c + m) of the group, paired (j, j+4) like the nibbles.
                uint32_t bx[NT][4];
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    const int tok = nt * 8 + g;
                    if (tok < T) {
                        const uint4 v = lds128(xbase + tok * XROW_BYTES + m * 16);
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
            // group scales of this lane's rows (staged in shared memory)
            const uint32_t sb = sbuf0 + (k_rel & 1) * p.sbuf_bytes;
#pragma unroll
            for (int r = 0; r < C::R; ++r) {
                const int row = (mset * C::R + r) * 16 + g;
                const float s0 = bf16_bits_to_float(lds_u16(sb + (row * G + gs) * 2));
                const float s1 = bf16_bits_to_float(lds_u16(sb + ((row + 8) * G + gs) * 2));
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    acc[r][nt][0] += s0 * gacc[r][nt][0];
                    acc[r][nt][1] += s0 * gacc[r][nt][1];
                    acc[r][nt][2] += s1 * gacc[r][nt][2];
                    acc[r][nt][3] += s1 * gacc[r][nt][3];
                }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_addr(&empty[s]));
        if (++s == nst) { s = 0; ph ^= 1u; }
        u += n;
        grp += n;

        if (grp == G || u == u1) {
            // ================================================ tile flush
            float *rbuf = red + ((C::RED_BUFS == 2) ? (nflush & 1) : 0) * C::RED_FLOATS;
            // 1. warp partials -> rbuf[slot][tok][row]
#pragma unroll
            for (int r = 0; r < C::R; ++r)
#pragma unroll
                for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int row = (mset * C::R + r) * 16 + g + 8 * (e >> 1);
                        const int tok = nt * 8 + 2 * c + (e & 1);
                        rbuf[(slot * C::TP + tok) * ROWS + row] = acc[r][nt][e];
                        acc[r][nt][e] = 0.f;
                    }
            cp_async_wait_all();                 // metadata of the next tile(s)
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
                    sum = rbuf[tok * ROWS + row];
#pragma unroll
                    for (int sl = 1; sl < C::GPS; ++sl) sum += rbuf[(sl * C::TP + tok) * ROWS + row];
                }
                v[q] = sum;
            }

            // 3. split tile: publish the partial; the last CTA adds them all
            const long long ts = static_cast<long long>(tile) * G, te = ts + G;
            const bool complete = (u0 <= ts) && (u1 >= te);
            bool finish = true;
            if (!complete) {
                const int bf = cta_of(ts, U, B), bl = cta_of(te - 1, U, B);
                const int which = (tile == tile_first) ? 0 : 1;
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
                                const int wb2 = (cta_start(bb, U, B) >= ts) ? 0 : 1;
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
                        const long long rg = static_cast<long long>(tile) * ROWS + row;
                        if (tok < T && rg < p.n_rows)
                            p.y[static_cast<size_t>(tok) * p.n_rows + rg] =
                                __bfloat16_as_ushort(__float2bfloat16_rn(v[q]));
                    }
                } else {
                    const int32_t *ids = idbuf + (k_rel % 3) * ROWS;
#pragma unroll
                    for (int q = 0; q < PER; ++q) {
                        const int pidx = tid + q * CONSUMERS;
                        const int tok = pidx / ROWS, row = pidx % ROWS;   // tok is warp-uniform
                        if (tok < T) {
                            const int id = ids[row];
                            unsigned long long k = id >= 0 ? make_key(v[q], static_cast<uint32_t>(id)) : 0ull;
#pragma unroll
                            for (int o = 16; o > 0; o >>= 1) {
                                const unsigned long long ko = shfl_xor_u64(k, o);
                                k = ko > k ? ko : k;
                            }
                            if (lane == 0 && k != 0ull) atomicMax(&best[tok], k);
                        }
                    }
                }
            }
            if (C::RED_BUFS == 1) named_bar_sync(1, CONSUMERS);   // rbuf free again

            // 5. metadata of tile k+2 into the buffers tile k used (free now)
            if (tile + 2 <= tile_last) {
                stage_tile_meta<HEAD>(p, tile + 2, idreg, sbuf + (k_rel & 1) * p.sbuf_bytes,
                                      idbuf + ((k_rel + 2) % 3) * ROWS, cw, lane);
                cp_async_commit();
            }
            tile_ids(p, tile + 3, tile_last, cw, idreg);
            ++nflush;
            ++k_rel;
            ++tile;
            grp = 0;
        }
    }

    if constexpr (HEAD) {
        // ==================================================== grid argmax + verify
        named_bar_sync(1, CONSUMERS);
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
