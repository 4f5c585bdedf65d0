// w4a16_tc.cuh -- the stream kernel for four n8 token tiles (17 <= T <= 32)
// on the 5th-generation tensor cores (tcgen05, accumulators in tensor
// memory).
//
// Why.  At T = 32 every 16 x 16 block of weights meets four token tiles, and
// the legacy mma.sync path is bound by its tensor pipe (19.9 M m16n8k16 per
// lm_head pass; measured 52 % pipe-active at 2.4 TB/s).  Here one
// tcgen05.mma of M = 128 weight rows x N = 32 tokens x K = 16 does the work
// of 32 of them.
//
// Work: a unit is one 128-row tile x two 128-column groups (TC_GU); units
// are numbered tile-major and split evenly over the grid (stream-K), split
// tiles finished in CTA order as in the other kernels.
//
// Warp roles (15 warps):
//  * warp 0, producer (lane 0): per unit, the two groups' packed weights of
//    the tile's 128 rows (TMA boxes, 64-byte swizzle), the groups'
//    activations in the canonical K-major layout written by
//    xprep_kernel<true> (one bulk copy, 16 KB) and, every eight groups, the
//    rows' scales for those groups (a TMA box of 8 x 128 bf16) into a
//    four-slot ring; completion on the stage's mbarrier.  Weights and scales
//    of the first stages go out before griddepcontrol.wait.
//  * warp 1 allocates the CTA's tensor memory (all 512 columns: three
//    128-column A buffers and two 64-column accumulator pairs) and frees it
//    at the end.  Lane 0 of warps 1 and 14 issue the MMAs of the even and the
//    odd units: per group eight tcgen05.mma (A from tensor memory, B = the
//    stage's activation block, D = the group's own accumulator, cleared by
//    the first), then one set of commits per unit to the A buffer's, the
//    stage's and the accumulator pair's mbarriers.  (One hand-off costs about
//    as much as the eight MMAs of a group; two groups per unit and two
//    issuers that alternate hide part of it.)
//  * warps 2..9, dequant (two warpgroups taking units in turn):
//    thread = weight row; per group it reads its row's 16 words, turns the
//    128 nibbles into fp16 levels (pairs (j, j+4), the order the activation
//    chunks use) and stores them to its tensor-memory lane as the A operand.
//  * warps 10..13, epilogue: thread = row; per unit it reads the row's 32
//    fp32 sums of each group back from tensor memory, multiplies them by the
//    row's group scale and adds them to its fp32 accumulators (the scale
//    applied after each group's sum, as in the other kernels); at the end of
//    its share of a tile it writes y or folds the logits into per-token
//    argmax keys.
#pragma once

#include "w4a16_stream.cuh"
#include "w4a16_wide.cuh"

namespace sv {

constexpr int TC_RT = 128;                       // rows per tile (the MMA's M)
constexpr int TC_GU = 2;                         // 128-column groups per unit (one hand-off per TC_GU groups)
constexpr int TC_W_BYTES = TC_RT * 64;           // one group of a tile's packed weights
constexpr int TC_X_BYTES = 32 * 128 * 2;         // one group of 32 tokens, fp16
constexpr int TC_STAGE = TC_GU * (TC_W_BYTES + TC_X_BYTES);   // weights of the unit's groups, then their activations
constexpr int TC_RING = 4;                       // scale-ring slots
constexpr int TC_RING_SLOT = TC_RT * 16;         // 8 groups of bf16 scales per row
constexpr int TC_NDQ = 2;                        // dequant warpgroups, taking units in turn
constexpr int TC_NA = 3;                         // A buffers of TC_GU x 64 columns
constexpr int TC_NACC = 2;                       // accumulators of TC_GU x 32 columns
constexpr uint32_t TC_TMEM_COLS = 512;
constexpr uint32_t TC_ACC_COL = TC_NA * 64 * TC_GU;   // the accumulators after the A buffers
constexpr int TC_DQ0 = 2;                        // first dequant warp
constexpr int TC_EP0 = TC_DQ0 + 4 * TC_NDQ;      // first epilogue warp
constexpr int TC_MMA2 = TC_EP0 + 4;              // second MMA-issuing warp
constexpr int TC_WARPS = TC_MMA2 + 1;
constexpr int TC_MAX_STAGES = 12;                // the ring's reuse rule holds up to 13
static_assert(TC_ACC_COL + TC_NACC * 32 * TC_GU <= TC_TMEM_COLS, "tensor memory budget");
// Instruction descriptor of kind::f16: D fp32 (bits 4-5 = 1), A and B fp16
// (bits 7-9, 10-12 = 0), both K-major (bits 15, 16 = 0), N >> 3 at bits
// 17-22, M >> 4 at bits 24-28.
constexpr uint32_t TC_IDESC = (1u << 4) | ((32u >> 3) << 17) | ((128u >> 4) << 24);

// Shared-memory descriptor of a K-major operand without swizzle: start
// address >> 4 (bits 0-13), leading byte offset >> 4 (bits 16-29: 512, the
// next eight columns along K), stride byte offset >> 4 (bits 32-45: 128, the
// next eight tokens), descriptor version 1 (bits 46-48).
__device__ __forceinline__ uint64_t tc_bdesc(uint32_t saddr)
{
    return static_cast<uint64_t>((saddr >> 4) & 0x3FFFu) | (static_cast<uint64_t>(512 >> 4) << 16) |
           (static_cast<uint64_t>(128 >> 4) << 32) | (1ull << 46);
}

template <bool HEAD>
__global__ void __launch_bounds__(TC_WARPS * 32, 1)
w4a16_tc_kernel(const __grid_constant__ Params p, const __grid_constant__ CUtensorMap tmW,
                const __grid_constant__ CUtensorMap tmS)
{
    extern __shared__ __align__(1024) uint8_t smem[];
    const int nst = p.nst;
    uint8_t *ring = smem + p.off_sbuf;                                       // [TC_RING][128][8] bf16
    unsigned long long *kt = reinterpret_cast<unsigned long long *>(smem + p.off_bk);   // [4][TMAX]
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + p.off_bars);
    uint64_t *full = bars;                   // [nst]   producer -> dequant, MMA, epilogue
    uint64_t *empty = bars + nst;            // [nst]   dequant (4) + MMA commit (1) + epilogue (4) -> producer
    uint64_t *a_full = bars + 2 * nst;       // [NA]    dequant warpgroup (4) -> MMA
    uint64_t *a_empty = a_full + TC_NA;      // [NA]    MMA commit -> dequant
    uint64_t *d_full = a_empty + TC_NA;      // [NACC]  MMA commit -> epilogue
    uint64_t *d_empty = d_full + TC_NACC;    // [NACC]  epilogue (4) -> MMA
    uint64_t *mma_done = d_empty + TC_NACC;  //         MMA commit after the last unit
    uint64_t *stall_bar = mma_done + 1;      //         never completed (test hook)
    volatile int *flag = reinterpret_cast<volatile int *>(stall_bar + 1);   // a wait timed out
    volatile int *decision = flag + 1;       // split-tile protocol
    volatile uint32_t *tmem_slot = reinterpret_cast<volatile uint32_t *>(flag + 2);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int B = gridDim.x, b = blockIdx.x;
    const long long U = p.U;
    const int T = p.T;
    const int G = p.G / TC_GU;               // units per tile (each TC_GU groups)
    const long long u0 = cta_start(b, U, B), u1 = cta_start(b + 1, U, B);
    const int tile_first = static_cast<int>(u0 / G);
    const int grp_first = static_cast<int>(u0 - static_cast<long long>(tile_first) * G);
    const int n_units = static_cast<int>(u1 - u0);

    // The weight boxes are swizzled in 512-byte atoms: the dynamic shared
    // memory must start on a 1024-byte boundary (uniform for the whole grid).
    if (smem_addr(smem) & 1023u) {
        if (threadIdx.x == 0) atomicOr(p.err, 4);
        return;
    }
    if (threadIdx.x == 0) {
        for (int s = 0; s < nst; ++s) {
            mbar_init(smem_addr(&full[s]), 1);
            mbar_init(smem_addr(&empty[s]), 9);
        }
        for (int i = 0; i < TC_NA; ++i) {
            mbar_init(smem_addr(&a_full[i]), 4);
            mbar_init(smem_addr(&a_empty[i]), 1);
        }
        for (int i = 0; i < TC_NACC; ++i) {
            mbar_init(smem_addr(&d_full[i]), 1);
            mbar_init(smem_addr(&d_empty[i]), 4);
        }
        mbar_init(smem_addr(mma_done), 2);
        mbar_init(smem_addr(stall_bar), 1);
        *flag = 0;
        fence_barrier_init();
    }
    if (HEAD)
        for (int i = threadIdx.x; i < 4 * TMAX; i += blockDim.x) kt[i] = 0ull;
    if (warp == 1) {
        tmem_alloc(smem_addr(const_cast<uint32_t *>(tmem_slot)), TC_TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = *tmem_slot;
    pdl_launch_dependents();

    if (warp == 0) {
        // ============================================================ producer
        if (lane == 0) {
            const uint64_t pol_w = policy_evict_first();
            const uint64_t pol_x = policy_evict_last();
            prefetch_tmap(&tmW);
            prefetch_tmap(&tmS);
            const uint32_t s0 = smem_addr(smem);
            const int n_pre = min(nst, n_units);
            int tile = tile_first, grp = grp_first, box = -1;
            for (int i = 0; i < n_units; ++i) {
                const int s = i % nst;
                if (i >= nst) wait_or_flag(p, flag, smem_addr(&empty[s]), static_cast<uint32_t>(((i / nst) & 1) ^ 1));
                const uint32_t fb = smem_addr(&full[s]);
                const uint32_t stage = s0 + static_cast<uint32_t>(s * TC_STAGE);
                const int g0 = grp * TC_GU;              // the unit's first group
                const bool nb = wide_new_box(i == 0, g0);
                if (nb) ++box;
                mbar_arrive_expect_tx(fb, static_cast<uint32_t>(TC_STAGE + (nb ? TC_RING_SLOT : 0)));
#pragma unroll
                for (int g = 0; g < TC_GU; ++g)
                    tma_load_2d(stage + g * TC_W_BYTES, &tmW, (g0 + g) * 16, tile * TC_RT, fb, pol_w);
                if (nb)
                    tma_load_2d(smem_addr(ring) + static_cast<uint32_t>((box % TC_RING) * TC_RING_SLOT), &tmS, g0 & ~7,
                                tile * TC_RT, fb, pol_w);
                if (i >= n_pre)
                    bulk_g2s(stage + TC_GU * TC_W_BYTES, p.x16 + static_cast<size_t>(g0) * TC_X_BYTES,
                             TC_GU * TC_X_BYTES, fb, pol_x);
                if (i == n_pre - 1) {
                    pdl_wait_prior();       // the activation blocks come from the conversion kernel
                    int g2 = grp_first;
                    for (int j = 0; j < n_pre; ++j) {
                        bulk_g2s(s0 + static_cast<uint32_t>(j * TC_STAGE + TC_GU * TC_W_BYTES),
                                 p.x16 + static_cast<size_t>(g2 * TC_GU) * TC_X_BYTES, TC_GU * TC_X_BYTES,
                                 smem_addr(&full[j]), pol_x);
                        if (++g2 == G) g2 = 0;
                    }
                }
                if (++grp == G) { grp = 0; ++tile; }
            }
            // do not leave while a copy of ours may still be landing
            for (int i = n_units - n_pre; i < n_units; ++i)
                if (!mbar_wait_bounded(smem_addr(&full[i % nst]), static_cast<uint32_t>((i / nst) & 1),
                                       WAIT_LIMIT_AFTER_ERR_NS)) {
                    *flag = 1;
                    atomicOr(p.err, 2);
                }
        }
    } else if (warp == 1 || warp == TC_MMA2) {
        // ============================================================ MMA issue
        // two issuing warps take alternate units (and the accumulator of
        // that parity), so that one's barrier waits overlap the other's issue
        if (lane == 0) {
            const uint32_t s0 = smem_addr(smem);
            for (int i = (warp == 1 ? 0 : 1); i < n_units; i += 2) {
                const int s = i % nst, ab = i % TC_NA, db = i % TC_NACC;
                wait_or_flag(p, flag, smem_addr(&full[s]), static_cast<uint32_t>((i / nst) & 1));
                wait_or_flag(p, flag, smem_addr(&a_full[ab]), static_cast<uint32_t>((i / TC_NA) & 1));
                if (i >= TC_NACC)
                    wait_or_flag(p, flag, smem_addr(&d_empty[db]), static_cast<uint32_t>(((i / TC_NACC) & 1) ^ 1));
                tc_fence_after_sync();
#pragma unroll
                for (int g = 0; g < TC_GU; ++g) {
                    // group g of the unit: its own accumulator (each group's sum is scaled on its own)
                    const uint32_t d = tmem + TC_ACC_COL + 32u * (TC_GU * db + g);
                    const uint32_t a = tmem + 64u * (TC_GU * ab + g);
                    const uint32_t xs = s0 + static_cast<uint32_t>(s * TC_STAGE + TC_GU * TC_W_BYTES + g * TC_X_BYTES);
#pragma unroll
                    for (int k = 0; k < 8; ++k) tc_mma_f16_ts(d, a + 8u * k, tc_bdesc(xs + 1024u * k), TC_IDESC, k > 0);
                }
                tc_commit(smem_addr(&a_empty[ab]));
                tc_commit(smem_addr(&empty[s]));
                tc_commit(smem_addr(&d_full[db]));
            }
            tc_commit(smem_addr(mma_done));
        }
        __syncwarp();
    } else if (warp < TC_EP0) {
        // ============================================================ dequant
        // warpgroup wg takes units i with i % TC_NDQ == wg; thread = tile row
        const int wg = (warp - TC_DQ0) >> 2;
        const int q = warp & 3;                       // tensor-memory lane quarter
        const int row = 32 * q + lane;
        const uint32_t s0 = smem_addr(smem);
        const uint32_t sw = static_cast<uint32_t>((row >> 1) & 3);   // the box's 64-byte swizzle
        for (int i = wg; i < n_units; i += TC_NDQ) {
            const int s = i % nst, ab = i % TC_NA;
            wait_or_flag(p, flag, smem_addr(&full[s]), static_cast<uint32_t>((i / nst) & 1));
            if (i >= TC_NA) wait_or_flag(p, flag, smem_addr(&a_empty[ab]), static_cast<uint32_t>(((i / TC_NA) & 1) ^ 1));
            const uint32_t wrow0 = s0 + static_cast<uint32_t>(s * TC_STAGE + row * 64);
            const uint32_t tlane0 = tmem + (static_cast<uint32_t>(32 * q) << 16) + 64u * TC_GU * ab;
#pragma unroll
            for (int hf = 0; hf < 2 * TC_GU; ++hf) {  // per group: words 0..7, then 8..15, 32 columns each
                const uint32_t wrow = wrow0 + static_cast<uint32_t>((hf >> 1) * TC_W_BYTES);
                const uint32_t tlane = tlane0 + 64u * (hf >> 1);
                uint32_t v[32];
#pragma unroll
                for (int jj = 0; jj < 2; ++jj) {
                    const int j = 2 * (hf & 1) + jj;
                    const uint4 w4 = lds128(wrow + ((static_cast<uint32_t>(j) ^ sw) << 4));
                    const uint32_t ws[4] = {w4.x, w4.y, w4.z, w4.w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const uint32_t w = ws[e];
                        const int c0 = 4 * (4 * jj + e);
                        v[c0 + 0] = dequant2_f16_lo(w);           // nibbles (0, 4)
                        v[c0 + 1] = dequant2_f16_hi(w);           // (1, 5)
                        v[c0 + 2] = dequant2_f16_lo(w >> 8);      // (2, 6)
                        v[c0 + 3] = dequant2_f16_hi(w >> 8);      // (3, 7)
                    }
                }
                tmem_st32(tlane + 32u * (hf & 1), v);
            }
            tmem_wait_st();
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(smem_addr(&a_full[ab]));
                mbar_arrive(smem_addr(&empty[s]));
            }
        }
    } else {
        // ============================================================ epilogue
        const int q = warp & 3;
        const int ew = warp - TC_EP0;                 // epilogue warp 0..3
        const int row = 32 * q + lane;
        constexpr uint32_t NTHR_E = 128;
        pdl_wait_prior();                   // xinv, scratch area, outputs and drafts from here on
        if (p.stall_ns != 0u && b == 0 && ew == 0) wait_or_flag_for(p, flag, smem_addr(stall_bar), 0u, p.stall_ns);
        // contributors of the first and the last tile, as in the other kernels
        const int tile_last = static_cast<int>((u1 - 1) / G);
        int bfA = b, ncA = 1, ncZ = 1;
        bool bf_firstA = true;
        {
            const long long ts = static_cast<long long>(tile_first) * G, te = ts + G;
            if (u0 > ts || u1 < te) {
                bfA = cta_of(ts, U, B);
                ncA = cta_of(te - 1, U, B) - bfA + 1;
                bf_firstA = cta_start(bfA, U, B) == ts;
            }
            const long long tz = static_cast<long long>(tile_last) * G;
            if (tile_last != tile_first && u1 < tz + G) ncZ = cta_of(tz + G - 1, U, B) - b + 1;
        }
        const uint32_t taddr = tmem + (static_cast<uint32_t>(32 * q) << 16) + TC_ACC_COL;
        float acc[32];
#pragma unroll
        for (int t = 0; t < 32; ++t) acc[t] = 0.f;
        int tile = tile_first, grp = grp_first, box = -1;
        for (int i = 0; i < n_units; ++i) {
            const int s = i % nst, db = i % TC_NACC;
            if (wide_new_box(i == 0, grp * TC_GU)) ++box;
            wait_or_flag(p, flag, smem_addr(&full[s]), static_cast<uint32_t>((i / nst) & 1));
            wait_or_flag(p, flag, smem_addr(&d_full[db]), static_cast<uint32_t>((i / TC_NACC) & 1));
            tc_fence_after_sync();
#pragma unroll
            for (int g = 0; g < TC_GU; ++g) {
                uint32_t v[32];
                tmem_ld32(taddr + 32u * (TC_GU * db + g), v);
                tmem_wait_ld();
                const float sc = bf16_bits_to_float(lds_u16(
                    smem_addr(ring) +
                    static_cast<uint32_t>((box % TC_RING) * TC_RING_SLOT + row * 16 + ((grp * TC_GU + g) & 7) * 2)));
#pragma unroll
                for (int t = 0; t < 32; ++t) acc[t] += sc * __uint_as_float(v[t]);
            }
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(smem_addr(&d_empty[db]));
                mbar_arrive(smem_addr(&empty[s]));
            }

            const bool tile_end = (grp == G - 1) || (i == n_units - 1);
            if (++grp == G) grp = 0;
            if (!tile_end) continue;

            // ------------------------------------------- end of this CTA's share of `tile`
#pragma unroll
            for (int t = 0; t < 32; ++t) acc[t] *= __ldg(p.xinv + t);
            const long long ts = static_cast<long long>(tile) * G, te = ts + G;
            const bool complete = (u0 <= ts) && (u1 >= te);
            bool finish = true;
            if (!complete) {
                // every contributor publishes its row sums and counts itself in;
                // the last to arrive adds them all in CTA order
                const bool first = tile == tile_first;
                const int bf = first ? bfA : b;
                const int nc = first ? ncA : ncZ;
                const int slot_bf = (first ? bf_firstA : (u0 == ts)) ? 0 : 1;
                float *mine = p.part + (static_cast<size_t>(b) * 2 + (first ? 0 : 1)) * WIDE_PART_FLOATS + row * TMAX;
#pragma unroll
                for (int t = 0; t < 32; t += 4)
                    __stcg(reinterpret_cast<float4 *>(mine + t), make_float4(acc[t], acc[t + 1], acc[t + 2], acc[t + 3]));
                __threadfence();
                named_bar_sync(1, NTHR_E);
                if (ew == 0 && lane == 0) {
                    const unsigned old = atomic_add_acq_rel_gpu(&p.ctr[bf], 1u);
                    const bool last = old == static_cast<unsigned>(nc - 1);
                    if (last) p.ctr[bf] = 0u;          // everyone is in: ready for the next launch
                    *decision = last ? WIDE_FINISH : WIDE_DONE;
                }
                named_bar_sync(1, NTHR_E);
                finish = *decision == WIDE_FINISH;
                named_bar_sync(1, NTHR_E);         // the decision word is read before it is reused
                if (finish) {
                    __threadfence();
                    for (int j = 0; j < nc; ++j) {
                        const float *src = p.part + (static_cast<size_t>(bf + j) * 2 + (j == 0 ? slot_bf : 0)) *
                                                        WIDE_PART_FLOATS + row * TMAX;
                        float4 e4[8];
#pragma unroll
                        for (int t = 0; t < 8; ++t) e4[t] = __ldcg(reinterpret_cast<const float4 *>(src) + t);
#pragma unroll
                        for (int t = 0; t < 8; ++t) {
                            if (j == 0) {
                                acc[4 * t] = e4[t].x; acc[4 * t + 1] = e4[t].y;
                                acc[4 * t + 2] = e4[t].z; acc[4 * t + 3] = e4[t].w;
                            } else {
                                acc[4 * t] += e4[t].x; acc[4 * t + 1] += e4[t].y;
                                acc[4 * t + 2] += e4[t].z; acc[4 * t + 3] += e4[t].w;
                            }
                        }
                    }
                }
            }
            if (finish) {
                const long long rg = static_cast<long long>(tile) * TC_RT + row;
                if constexpr (!HEAD) {
                    if (rg < p.n_rows)
#pragma unroll
                        for (int t = 0; t < 32; ++t)
                            if (t < T) p.y[static_cast<size_t>(t) * p.n_rows + rg] = __bfloat16_as_ushort(__float2bfloat16_rn(acc[t]));
                } else {
#pragma unroll
                    for (int t = 0; t < 32; ++t) {
                        unsigned long long best = rg < p.n_rows ? make_key(acc[t], static_cast<uint32_t>(rg)) : 0ull;
#pragma unroll
                        for (int o = 16; o > 0; o >>= 1) {
                            const unsigned long long k = shfl_xor_u64(best, o);
                            best = k > best ? k : best;
                        }
                        if (lane == 0 && t < T && best > kt[ew * TMAX + t]) kt[ew * TMAX + t] = best;
                    }
                }
            }
#pragma unroll
            for (int t = 0; t < 32; ++t) acc[t] = 0.f;
            ++tile;
        }
        if constexpr (HEAD) {
            // ================================================ grid argmax + verify
            named_bar_sync(1, NTHR_E);
            if (ew == 0) {
                unsigned long long best = 0ull;     // lane t: best key of token t in this CTA
                if (lane < T)
                    for (int w = 0; w < 4; ++w) {
                        const unsigned long long k = kt[w * TMAX + lane];
                        best = k > best ? k : best;
                    }
                head_grid_tail(p, best, lane, B);
            }
        }
    }

    // ================================================================ teardown
    // Every warp gets here (no early exit after the allocation).  The MMAs
    // are complete once the last commit has arrived; then the tensor memory
    // is freed by the warp that allocated it.
    __syncthreads();
    if (warp == 1) {
        if (!mbar_wait_bounded(smem_addr(mma_done), 0u, WAIT_LIMIT_AFTER_ERR_NS)) atomicOr(p.err, 2);
        tc_fence_after_sync();
        tmem_dealloc(tmem, TC_TMEM_COLS);
    }
}

}  // namespace sv
