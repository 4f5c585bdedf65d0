// w4a16_wide.cuh -- the stream kernel for calls with more than one n8 token
// tile (9 <= T <= 32): tall row tiles, each consumer warp owning 64 rows of
// a tile for the CTA's whole share of it.
//
// Why a second kernel.  With T rows of activations, every 128-column group
// of every tile needs that group's activation block (TP tokens x 128
// columns, 8.7 KB at T = 32) in shared memory next to its weights; with the
// 64-row tiles of w4a16_stream_kernel that block is 2.2 times the group's
// 4 KB of packed weights, and the tokens' B fragments are read from shared
// memory once per 32 rows.  Here a tile has RT = 64 * NCW rows (512 with 8
// consumer warps), so a group's activation block is copied once per 16 KB or
// 32 KB of weights, and each warp loads the group's B fragments once into
// registers and reuses them for its four m16 tiles (64 rows).
//
// Work decomposition: a unit is one tile x one 128-column group; units are
// numbered tile-major and split evenly over the grid (stream-K), as in
// w4a16_stream_kernel.  A tile shared by several CTAs is finished by its
// first CTA, adding the partial sums of all its CTAs in CTA order.
//
// Warp roles: warps 0..NCW-1 are consumers; warp NCW is the producer.
//  * producer: per unit, the tile's packed weights of the group (TMA boxes
//    of up to 256 rows x 64 bytes), the group's activation block prepared by
//    xprep_kernel (one bulk copy) and, every eight groups, the scales of the
//    tile's rows for those eight groups (a TMA box of 8 x up to 256 bf16)
//    into a two-slot ring; completion on the stage's mbarrier.  Weights and
//    scales of the first stages are issued before griddepcontrol.wait.
//  * consumers: warp w takes rows 64w .. 64w+63 of every tile: it loads the
//    group's B fragments for all token tiles (16 x NT 16-byte loads), then
//    for each of its four m16 tiles loads the packed words, dequantises them
//    to fp16 levels in registers, runs 2 x NT mma.sync per k-step pair into
//    a group accumulator and adds it, times the group scale, to the tile
//    accumulators.  At the end of its share of a tile the warp writes y (a
//    GEMM) or folds the rows' logits into per-token argmax keys (the head)
//    itself; split tiles go through the scratch area.
#pragma once

#include "w4a16_stream.cuh"

namespace sv {

constexpr int WIDE_R = 4;                            // m16 tiles per consumer warp
constexpr int WIDE_WROWS = 16 * WIDE_R;              // rows per consumer warp
constexpr int WIDE_MAX_RT = 512;                     // largest tile (8 consumer warps)
constexpr int WIDE_PART_FLOATS = WIDE_MAX_RT * TMAX; // one split-tile partial, [row][TMAX]

__host__ __device__ constexpr int wide_rt(int ncw) { return ncw * WIDE_WROWS; }

// Which scale-ring box a unit reads: a box is issued at the CTA's first unit
// and at every group that is a multiple of 8; it holds groups
// [8 * floor(grp / 8), + 8) of the tile's rows.
__device__ __forceinline__ bool wide_new_box(bool first, int grp) { return first || (grp & 7) == 0; }

template <int NT, bool HEAD, int NCW>
__global__ void __launch_bounds__((NCW + 1) * 32, 1)
w4a16_wide_kernel(const __grid_constant__ Params p, const __grid_constant__ CUtensorMap tmW,
                  const __grid_constant__ CUtensorMap tmS)
{
    constexpr int RT = wide_rt(NCW);
    constexpr int BOX_ROWS = RT < 256 ? RT : 256;   // TMA box height
    constexpr int NBOX = RT / BOX_ROWS;
    constexpr int W_BYTES = RT * 64;                // one group of the tile's packed weights
    constexpr int RING_SLOT = RT * 16;              // 8 groups of bf16 scales per row
    constexpr uint32_t NTHR_C = NCW * 32;
    extern __shared__ __align__(1024) uint8_t smem[];

    const int nst = p.nst;
    uint8_t *ring = smem + p.off_sbuf;                                  // [2][RT][8] bf16
    unsigned long long *kt = reinterpret_cast<unsigned long long *>(smem + p.off_bk);   // [NCW][TMAX]
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + p.off_bars);
    uint64_t *full = bars;                  // [nst] producer -> consumers
    uint64_t *empty = bars + nst;           // [nst] consumers -> producer
    uint64_t *stall_bar = bars + 2 * nst;   // never completed (test hook)
    volatile int *flag = reinterpret_cast<volatile int *>(bars + 2 * nst + 1);   // a wait timed out

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int B = gridDim.x, b = blockIdx.x;
    const long long U = p.U;
    const int G = p.G, T = p.T;
    const long long u0 = cta_start(b, U, B), u1 = cta_start(b + 1, U, B);
    const int tile_first = static_cast<int>(u0 / G);
    const int grp_first = static_cast<int>(u0 - static_cast<long long>(tile_first) * G);
    const int n_units = static_cast<int>(u1 - u0);

    if (threadIdx.x == 0) {
        for (int s = 0; s < nst; ++s) {
            mbar_init(smem_addr(&full[s]), 1);
            mbar_init(smem_addr(&empty[s]), NCW);
        }
        mbar_init(smem_addr(stall_bar), 1);
        *flag = 0;
        fence_barrier_init();
    }
    if (HEAD)
        for (int i = threadIdx.x; i < NCW * TMAX; i += blockDim.x) kt[i] = 0ull;
    __syncthreads();
    pdl_launch_dependents();

    if (warp == NCW) {
        // ============================================================ producer
        if (lane != 0) return;
        const uint64_t pol_w = policy_evict_first();
        const uint64_t pol_x = policy_evict_last();
        prefetch_tmap(&tmW);
        prefetch_tmap(&tmS);
        const uint32_t stage_bytes = static_cast<uint32_t>(p.stage_bytes);
        const uint32_t xbytes = static_cast<uint32_t>(p.xslot_bytes);
        const int n_pre = min(nst, n_units);
        int tile = tile_first, grp = grp_first, box = -1;
        // Weights and scales (read-only model data) of the first stages go out
        // before griddepcontrol.wait; their activation blocks after it.
        for (int i = 0; i < n_units; ++i) {
            const int s = i % nst;
            const uint32_t ph = static_cast<uint32_t>((i / nst) & 1);
            if (i >= nst) wait_or_flag(p, flag, smem_addr(&empty[s]), ph ^ 1u);
            const uint32_t fb = smem_addr(&full[s]);
            const uint32_t stage = smem_addr(smem) + static_cast<uint32_t>(s) * stage_bytes;
            const bool nb = wide_new_box(i == 0, grp);
            if (nb) ++box;
            // boxes that start past the last row are not issued (their rows'
            // shared memory keeps stale values, and those rows are never output)
            int nbox = 0;
#pragma unroll
            for (int h = 0; h < NBOX; ++h) nbox += (tile * RT + h * BOX_ROWS < p.n_rows) ? 1 : 0;
            mbar_arrive_expect_tx(fb, static_cast<uint32_t>(nbox * BOX_ROWS * (nb ? 64 + 16 : 64)) + xbytes);
#pragma unroll
            for (int h = 0; h < NBOX; ++h)
                if (h < nbox)
                    tma_load_2d(stage + h * BOX_ROWS * 64, &tmW, grp * 16, tile * RT + h * BOX_ROWS, fb, pol_w);
            if (nb) {
                const uint32_t rs = smem_addr(ring) + static_cast<uint32_t>((box & 1) * RING_SLOT);
#pragma unroll
                for (int h = 0; h < NBOX; ++h)
                    if (h < nbox)
                        tma_load_2d(rs + h * BOX_ROWS * 16, &tmS, grp & ~7, tile * RT + h * BOX_ROWS, fb, pol_w);
            }
            if (i >= n_pre)
                bulk_g2s(stage + W_BYTES, p.x16 + static_cast<size_t>(grp) * xbytes, xbytes, fb, pol_x);
            if (i == n_pre - 1) {
                pdl_wait_prior();       // the activation blocks come from the conversion kernel
                int g2 = grp_first;
                for (int j = 0; j < n_pre; ++j) {
                    const uint32_t st2 = smem_addr(smem) + static_cast<uint32_t>(j) * stage_bytes;
                    bulk_g2s(st2 + W_BYTES, p.x16 + static_cast<size_t>(g2) * xbytes, xbytes,
                             smem_addr(&full[j]), pol_x);
                    if (++g2 == G) g2 = 0;
                }
            }
            if (++grp == G) { grp = 0; ++tile; }
        }
        // Do not leave while a copy of ours may still be landing.
        const int left = min(n_units, nst);
        for (int i = n_units - left; i < n_units; ++i) {
            const int s = i % nst;
            if (!mbar_wait_bounded(smem_addr(&full[s]), static_cast<uint32_t>((i / nst) & 1),
                                   WAIT_LIMIT_AFTER_ERR_NS)) {
                *flag = 1;
                atomicOr(p.err, 2);
            }
        }
        return;
    }

    // ================================================================ consumers
    const int g = lane >> 2, c = lane & 3;
    pdl_wait_prior();                   // xinv, scratch area, outputs and drafts from here on
    if (p.stall_ns != 0u && b == 0 && warp == 0) wait_or_flag_for(p, flag, smem_addr(stall_bar), 0u, p.stall_ns);

    // 2^-s of this lane's tokens nt*8 + 2c + e (the conversion's scale)
    float xinv[NT][2];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int e = 0; e < 2; ++e) xinv[nt][e] = __ldg(p.xinv + nt * 8 + 2 * c + e);

    // Contributors of the first and the last tile (the only ones that can be
    // shared): CTAs bf .. bf + nc - 1.
    const int tile_last = static_cast<int>((u1 - 1) / G);
    int bfA = b, ncA = 1, bfZ = b, ncZ = 1;
    {
        const long long ts = static_cast<long long>(tile_first) * G, te = ts + G;
        if (u0 > ts || u1 < te) {
            bfA = cta_of(ts, U, B);
            ncA = cta_of(te - 1, U, B) - bfA + 1;
        }
        const long long tz = static_cast<long long>(tile_last) * G;
        if (tile_last != tile_first && u1 < tz + G) ncZ = cta_of(tz + G - 1, U, B) - b + 1;
    }

    const uint32_t smem0 = smem_addr(smem);
    const uint32_t xsw = static_cast<uint32_t>((c & 2) * 16);
    // lane-constant offsets: packed words of row 64w + 16r + g (+8), chunk c;
    // B fragments of token nt*8 + g; scales of those rows
    const uint32_t w_lane = static_cast<uint32_t>((warp * WIDE_WROWS + g) * 64 + c * 16);
    const uint32_t x_lane = static_cast<uint32_t>(W_BYTES + g * XSTR + c * 64);
    const uint32_t s_lane = static_cast<uint32_t>((warp * WIDE_WROWS + g) * 16);
    const uint32_t ring0 = smem_addr(ring);

    float acc[WIDE_R][NT][4];
#pragma unroll
    for (int r = 0; r < WIDE_R; ++r)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[r][nt][e] = 0.f;

    int tile = tile_first, grp = grp_first, box = -1;
    for (int i = 0; i < n_units; ++i) {
        const int s = i % nst;
        if (wide_new_box(i == 0, grp)) ++box;
        wait_or_flag(p, flag, smem_addr(&full[s]), static_cast<uint32_t>((i / nst) & 1));
        const uint32_t stage = smem0 + static_cast<uint32_t>(s * p.stage_bytes);
        // B fragments of the whole group for every token tile
        uint4 bx[4][NT];
#pragma unroll
        for (int m = 0; m < 4; ++m)
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
                bx[m][nt] = lds128(stage + x_lane + nt * 8 * XSTR + ((16u * m) ^ xsw));
        const uint32_t sb = ring0 + static_cast<uint32_t>((box & 1) * RING_SLOT) + s_lane + (grp & 7) * 2;
#pragma unroll
        for (int r = 0; r < WIDE_R; ++r) {
            const uint4 wa = lds128(stage + w_lane + r * 16 * 64);
            const uint4 wb = lds128(stage + w_lane + (r * 16 + 8) * 64);
            float gacc[NT][4];      // first k-step writes, later ones accumulate
#pragma unroll
            for (int m = 0; m < 4; ++m) {
                const uint32_t wA = (m == 0) ? wa.x : (m == 1) ? wa.y : (m == 2) ? wa.z : wa.w;
                const uint32_t wB = (m == 0) ? wb.x : (m == 1) ? wb.y : (m == 2) ? wb.z : wb.w;
                // k-step 2m: nibble pairs (0,4) and (1,5); k-step 2m+1: pairs
                // (2,6) and (3,7) of the word >> 8
                uint32_t a0 = dequant2_f16_lo(wA), a1 = dequant2_f16_lo(wB);
                uint32_t a2 = dequant2_f16_hi(wA), a3 = dequant2_f16_hi(wB);
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    if (m == 0)
                        mma_f16_16816_zc(gacc[nt], a0, a1, a2, a3, bx[m][nt].x, bx[m][nt].y);
                    else
                        mma_f16_16816(gacc[nt], a0, a1, a2, a3, bx[m][nt].x, bx[m][nt].y);
                }
                const uint32_t wA8 = wA >> 8, wB8 = wB >> 8;
                a0 = dequant2_f16_lo(wA8);
                a1 = dequant2_f16_lo(wB8);
                a2 = dequant2_f16_hi(wA8);
                a3 = dequant2_f16_hi(wB8);
#pragma unroll
                for (int nt = 0; nt < NT; ++nt)
                    mma_f16_16816(gacc[nt], a0, a1, a2, a3, bx[m][nt].z, bx[m][nt].w);
            }
            const float s0 = bf16_bits_to_float(lds_u16(sb + r * 16 * 16));
            const float s1 = bf16_bits_to_float(lds_u16(sb + (r * 16 + 8) * 16));
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                acc[r][nt][0] += s0 * gacc[nt][0];
                acc[r][nt][1] += s0 * gacc[nt][1];
                acc[r][nt][2] += s1 * gacc[nt][2];
                acc[r][nt][3] += s1 * gacc[nt][3];
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_addr(&empty[s]));

        const bool tile_end = (grp == G - 1) || (i == n_units - 1);
        if (++grp == G) grp = 0;
        if (!tile_end) continue;

        // ------------------------------------------- end of this CTA's share of `tile`
#pragma unroll
        for (int r = 0; r < WIDE_R; ++r)
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                acc[r][nt][0] *= xinv[nt][0];
                acc[r][nt][1] *= xinv[nt][1];
                acc[r][nt][2] *= xinv[nt][0];
                acc[r][nt][3] *= xinv[nt][1];
            }
        const long long ts = static_cast<long long>(tile) * G, te = ts + G;
        const bool complete = (u0 <= ts) && (u1 >= te);
        bool finish = true;
        if (!complete) {
            // Split tile: finished by its first contributor bf, for which it
            // is the end of its range (the others' parts are the start of
            // theirs).  The others publish their partial sums and count
            // themselves in with a release add they do not wait for; bf
            // waits (bounded) until all nc - 1 are in, adds them after its
            // own in CTA order and resets the counter for the next launch.
            const bool first = tile == tile_first;
            const int bf = first ? bfA : bfZ;
            const int nc = first ? ncA : ncZ;
            finish = bf == b;
            if (!finish) {
                // the tile is this CTA's first: partial slot 0
                float *mine = p.part + static_cast<size_t>(b) * 2 * WIDE_PART_FLOATS;
#pragma unroll
                for (int r = 0; r < WIDE_R; ++r)
#pragma unroll
                    for (int hh = 0; hh < 2; ++hh)
#pragma unroll
                        for (int nt = 0; nt < NT; ++nt) {
                            const int row = warp * WIDE_WROWS + r * 16 + g + 8 * hh;
                            __stcg(reinterpret_cast<float2 *>(mine + row * TMAX + nt * 8 + 2 * c),
                                   make_float2(acc[r][nt][2 * hh], acc[r][nt][2 * hh + 1]));
                        }
                named_bar_sync(1, NTHR_C);
                if (threadIdx.x == 0) red_add_release_gpu(&p.ctr[bf], 1u);
            } else {
                if (warp == 0) {
                    const uint64_t t0 = global_timer_ns();
                    while (!__all_sync(0xFFFFFFFFu, ld_acquire_gpu_u32(&p.ctr[bf]) == static_cast<unsigned>(nc - 1))) {
                        if (global_timer_ns() - t0 > (*flag ? WAIT_LIMIT_AFTER_ERR_NS : WAIT_LIMIT_NS)) {
                            *flag = 1;
                            if (lane == 0) atomicOr(p.err, 2);
                            break;
                        }
                    }
                }
                named_bar_sync(1, NTHR_C);      // all nc - 1 are in
                if (threadIdx.x == 0) p.ctr[bf] = 0u;
#pragma unroll 1
                for (int j = 1; j < nc; ++j) {
                    const float *src = p.part + static_cast<size_t>(bf + j) * 2 * WIDE_PART_FLOATS;
                    float2 e2[WIDE_R][2][NT];     // one contributor's values, loads all in flight
#pragma unroll
                    for (int r = 0; r < WIDE_R; ++r)
#pragma unroll
                        for (int hh = 0; hh < 2; ++hh)
#pragma unroll
                            for (int nt = 0; nt < NT; ++nt) {
                                const int row = warp * WIDE_WROWS + r * 16 + g + 8 * hh;
                                e2[r][hh][nt] = __ldcg(reinterpret_cast<const float2 *>(src + row * TMAX + nt * 8 + 2 * c));
                            }
#pragma unroll
                    for (int r = 0; r < WIDE_R; ++r)
#pragma unroll
                        for (int hh = 0; hh < 2; ++hh)
#pragma unroll
                            for (int nt = 0; nt < NT; ++nt) {
                                acc[r][nt][2 * hh] += e2[r][hh][nt].x;
                                acc[r][nt][2 * hh + 1] += e2[r][hh][nt].y;
                            }
                }
            }
        }
        if (finish) {
            const long long row_base = static_cast<long long>(tile) * RT + warp * WIDE_WROWS;
            if constexpr (!HEAD) {
#pragma unroll
                for (int r = 0; r < WIDE_R; ++r)
#pragma unroll
                    for (int hh = 0; hh < 2; ++hh) {
                        const long long rg = row_base + r * 16 + g + 8 * hh;
                        if (rg >= p.n_rows) continue;
#pragma unroll
                        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                            for (int e = 0; e < 2; ++e) {
                                const int t = nt * 8 + 2 * c + e;
                                if (t >= T) continue;
                                const float v = acc[r][nt][2 * hh + e];
                                if (p.y32)
                                    p.y32[static_cast<size_t>(t) * p.n_rows + rg] = v;
                                else
                                    p.y[static_cast<size_t>(t) * p.n_rows + rg] =
                                        __bfloat16_as_ushort(__float2bfloat16_rn(v));
                            }
                    }
            } else {
                // best key of each token over this warp's 64 rows
#pragma unroll
                for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        unsigned long long best = 0ull;
#pragma unroll
                        for (int r = 0; r < WIDE_R; ++r)
#pragma unroll
                            for (int hh = 0; hh < 2; ++hh) {
                                const long long rg = row_base + r * 16 + g + 8 * hh;
                                if (rg < p.n_rows) {
                                    const unsigned long long k =
                                        make_key(acc[r][nt][2 * hh + e], static_cast<uint32_t>(rg));
                                    best = k > best ? k : best;
                                }
                            }
#pragma unroll
                        for (int o = 4; o < 32; o <<= 1) {
                            const unsigned long long k = shfl_xor_u64(best, o);
                            best = k > best ? k : best;
                        }
                        const int t = nt * 8 + 2 * c + e;
                        if (g == 0 && t < T && best > kt[warp * TMAX + t]) kt[warp * TMAX + t] = best;
                    }
            }
        }
#pragma unroll
        for (int r = 0; r < WIDE_R; ++r)
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e) acc[r][nt][e] = 0.f;
        ++tile;
    }

    if constexpr (HEAD) {
        // ==================================================== grid argmax + verify
        named_bar_sync(1, NTHR_C);
        if (warp == 0) {
            unsigned long long best = 0ull;    // lane t: best key of token t in this CTA
            if (lane < T)
                for (int w = 0; w < NCW; ++w) {
                    const unsigned long long v = kt[w * TMAX + lane];
                    best = v > best ? v : best;
                }
            head_grid_tail(p, best, lane, B);
        }
    }
}

}  // namespace sv
