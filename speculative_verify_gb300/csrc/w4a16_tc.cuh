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
// Scales in the A operand.  Each weight row's group scales are taken eight
// groups (a "box") at a time.  With E the largest exponent among the row's
// eight scales, the dequant warps write level * s * 2^(137 - E) to the A
// operand in fp16: the box's largest scale lands in [2^10, 2^11), the level
// (an integer in -8..7) times the 8-bit significand of a bf16 scale has at
// most 11 significant bits, so the product is exact in fp16 for every scale
// of at least 2^-27 times the box's largest (a smaller one is rounded, by
// less than 2^-34 of the largest, below the fp32 rounding of the sum).  The tensor cores then add the products of
// all eight groups in fp32, and the epilogue multiplies the box's sums by
// 2^(E - 137): exactly the sum of the products level * s * x, which the
// per-group form adds in another order.  The product is formed in one fp16
// fma on the nibble placed in the top four mantissa bits of 16.0
// ((16 + n) * s' - 24 s' = (n - 8) * s', with 24 s' exact in fp16).
//
// Work: a unit is one 128-row tile x two 128-column groups (TC_GU); units
// are numbered tile-major and split evenly over the grid (stream-K); a split
// tile is finished by its first CTA, which adds the others' published
// partial sums after its own in CTA order.  A box is four units
// (fewer at the ends of a CTA's share); boxes never straddle tiles (the
// kernel needs K a multiple of 1024).  Units alternate between two
// pipelines, each a dequant warpgroup and an MMA warp with a private ring of
// two one-group A slots (64 tensor-memory columns each) and a private
// accumulator per box: no barrier is shared between the pipelines, and every
// waiter walks its barriers' phases in order, so no parity wait can alias a
// phase two ahead.
//
// Warp roles (16 warps):
//  * warp 0, producer (lane 0): per unit, the two groups' packed weights of
//    the tile's 128 rows (TMA boxes, 64-byte swizzle) and their activations
//    in the canonical K-major layout written by xprep_kernel<true> (one bulk
//    copy, 16 KB), completion on the stage's mbarrier.  Weights of the first
//    stages go out before griddepcontrol.wait.
//  * warps 1 and 14, MMA issue for pipelines 0 and 1 (warp 1 also allocates
//    the 512 tensor-memory columns and frees them at the end): per unit of
//    the pipeline, per group eight tcgen05.mma (A from the group's slot, B =
//    the stage's activation block; the pipeline's first MMA of a box clears
//    its accumulator) issued by one elected lane of the whole warp, a commit
//    that frees the slot, one that frees the stage, and at every box end one
//    to the box's accumulator set.
//  * warps 2..5 and 6..9, dequant warpgroups of pipelines 0 and 1: thread =
//    weight row; per box it loads the row's eight scales (16 bytes, read
//    ahead) and forms the fp16 factors, per group it reads its row's 16
//    words and stores the 128 scaled levels (pairs (j, j+4), the order the
//    activation chunks use) to its tensor-memory lane of the next slot.
//  * warps 10..13, epilogue: thread = row; per box it reads the row's two
//    accumulators (one per pipeline, each only if the box has a unit of that
//    pipeline), adds them, multiplies by 2^(E - 137) and adds the result to
//    its fp32 accumulators; at the end of its share of a tile it multiplies
//    by the tokens' 2^-s (staged in shared memory), finishes or publishes a
//    split tile, and writes y, or for the head hands the tile's logits to
//    the reducer.
//  * warp 15, reducer (head only): lane t keeps the largest (logit, lowest
//    id) key of token t over the CTA's finished tiles, read from a
//    double-buffered shared-memory tile, then runs the grid argmax and the
//    verify.
#pragma once

#include "w4a16_stream.cuh"
#include "w4a16_wide.cuh"

namespace sv {

constexpr int TC_RT = 128;                       // rows per tile (the MMA's M)
constexpr int TC_GU = 2;                         // 128-column groups per unit (one hand-off per TC_GU groups)
constexpr int TC_BOX_UNITS = 8 / TC_GU;          // units per box of eight groups
constexpr int TC_W_BYTES = TC_RT * 64;           // one group of a tile's packed weights
constexpr int TC_X_BYTES = 32 * 128 * 2;         // one group of 32 tokens, fp16
constexpr int TC_STAGE = TC_GU * (TC_W_BYTES + TC_X_BYTES);   // weights of the unit's groups, then their activations
constexpr int TC_NDQ = 2;                        // dequant warpgroups, taking units in turn
// A slots of one group (64 columns) per pipeline.  Measured on the T = 32
// lm_head: one slot 200 us, two 170, three 174.
constexpr int TC_NSLOT = 2;
constexpr int TC_NB = 2;                         // box accumulator sets (one 32-column accumulator per pipeline)
constexpr uint32_t TC_TMEM_COLS = 512;
constexpr uint32_t TC_ACC_COL = TC_NDQ * TC_NSLOT * 64;   // the accumulators after the A slots
constexpr int TC_DQ0 = 2;                        // first dequant warp
constexpr int TC_EP0 = TC_DQ0 + 4 * TC_NDQ;      // first epilogue warp
constexpr int TC_MMA2 = TC_EP0 + 4;              // second MMA-issuing warp
constexpr int TC_RED = TC_MMA2 + 1;              // head: the warp that reduces finished tiles to per-token maxima
constexpr int TC_WARPS = TC_RED + 1;
constexpr int TC_TB_BYTES = TC_RT * 32 * 4;      // head: one finished tile's logits, [row][32 tokens] fp32
// Four stages (128 KB).  Measured at T = 32: the same lm_head time as six,
// and GEMMs 0.4-1.3 us faster; a GEMM launch holding more than about 196 KB
// of shared memory (six stages plus 16-32 KB) ran 1.3-2.5 us slower.
constexpr int TC_MAX_STAGES = 4;
constexpr int TC_SHIFT = 137;                    // a box's largest scale x 2^(TC_SHIFT - E) is in [2^10, 2^11)
static_assert(TC_ACC_COL + TC_NB * TC_NDQ * 32 <= TC_TMEM_COLS, "tensor memory budget");
static_assert(TC_NDQ == 2, "two pipelines: dequant warpgroup w with MMA warp w");
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

// Largest biased exponent among eight bf16 scales (two per word).
__device__ __forceinline__ int tc_box_exp(const uint4 &s)
{
    const uint32_t w[4] = {s.x, s.y, s.z, s.w};
    uint32_t e = 0;
#pragma unroll
    for (int k = 0; k < 4; ++k) e = max(e, max((w[k] >> 7) & 0xFFu, (w[k] >> 23) & 0xFFu));
    return static_cast<int>(e);
}

// 2^k for -252 <= k <= 254 as a pair of normal fp32 factors.
__device__ __forceinline__ void tc_pow2_pair(int k, float &f1, float &f2)
{
    const int a = k / 2, c = k - a;
    f1 = __uint_as_float(static_cast<uint32_t>(a + 127) << 23);
    f2 = __uint_as_float(static_cast<uint32_t>(c + 127) << 23);
}

// The fp16x2 factor {s', s'} and addend {-24 s', -24 s'} of one bf16 scale,
// s' = s * f1 * f2 rounded to fp16 (exact when within the fp16 range).
__device__ __forceinline__ void tc_factor(uint32_t s_bits, float f1, float f2, uint32_t &s2, uint32_t &c2)
{
    const float sp = (__uint_as_float(s_bits << 16) * f1) * f2;
    const __half h = __float2half_rn(sp);
    const __half c = __float2half_rn(-24.0f * __half2float(h));
    const uint32_t hb = __half_as_ushort(h), cb = __half_as_ushort(c);
    s2 = hb | (hb << 16);
    c2 = cb | (cb << 16);
}

// Levels of nibbles (j, j+4) times the row's factor: `ws` is the word shifted
// so that the two nibbles sit at bits 6..9 and 22..25 (the top mantissa bits
// of fp16 16.0), then (16 + n) * s' - 24 s' = (n - 8) * s' in one fp16 fma.
__device__ __forceinline__ uint32_t tc_scaled_pair(uint32_t ws, uint32_t s2, uint32_t c2)
{
    uint32_t q, r;
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(q) : "r"(ws), "r"(0x03C003C0u), "r"(0x4C004C00u));
    asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(r) : "r"(q), "r"(s2), "r"(c2));
    return r;
}

// The row's eight scales of box `bx` (groups 8 bx .. 8 bx + 7) of tile `tile`.
__device__ __forceinline__ uint4 tc_load_scales(const Params &p, int tile, int bx, int row)
{
    const long long rg = static_cast<long long>(tile) * TC_RT + row;
    if (rg >= p.n_rows) return make_uint4(0u, 0u, 0u, 0u);
    return __ldg(reinterpret_cast<const uint4 *>(p.scales + rg * p.G + 8 * bx));
}

// A bounded wait that first polls once without reading the CTA's flag (the
// MMA warps' common case: the barrier has completed already).
__device__ __forceinline__ void tc_wait(const Params &p, volatile int *flag, uint32_t bar, uint32_t parity)
{
    if (!mbar_try_wait(bar, parity)) wait_or_flag(p, flag, bar, parity);
}

template <bool HEAD>
__global__ void __launch_bounds__(TC_WARPS * 32, 1)
w4a16_tc_kernel(const __grid_constant__ Params p, const __grid_constant__ CUtensorMap tmW)
{
    extern __shared__ __align__(1024) uint8_t smem[];
    const int nst = p.nst;
    uint8_t *tbuf = smem + p.off_bk;        // head: [2] finished tiles, TC_TB_BYTES each
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + p.off_bars);
    uint64_t *full = bars;                   // [nst]   producer -> the unit's dequant warpgroup and MMA warp
    uint64_t *empty = full + nst;            // [nst]   the unit's MMA commit -> producer
    uint64_t *a_full = empty + nst;          // [NDQ][NSLOT] dequant warpgroup w (4) -> MMA warp w
    uint64_t *a_empty = a_full + TC_NDQ * TC_NSLOT;   // [NDQ][NSLOT] MMA warp w's commit -> warpgroup w
    uint64_t *d_full = a_empty + TC_NDQ * TC_NSLOT;   // [NB]    MMA commits (2) at the end of a box -> epilogue
    uint64_t *d_empty = d_full + TC_NB;      // [NB]    epilogue (4) -> MMA
    uint64_t *tb_full = d_empty + TC_NB;     // [2]     head: epilogue (4) -> reducer
    uint64_t *tb_empty = tb_full + 2;        // [2]     head: reducer -> epilogue
    uint64_t *mma_done = tb_empty + 2;       //         MMA commits after the last unit
    uint64_t *stall_bar = mma_done + 1;      //         never completed (test hook)
    volatile int *flag = reinterpret_cast<volatile int *>(stall_bar + 1);   // a wait timed out
    volatile uint32_t *tmem_slot = reinterpret_cast<volatile uint32_t *>(flag + 2);
    volatile int *tb_tile = flag + 3;        // [2] head: the tile in each buffer, -1 = no more

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
            mbar_init(smem_addr(&empty[s]), 1);
        }
        for (int i = 0; i < TC_NDQ * TC_NSLOT; ++i) {
            mbar_init(smem_addr(&a_full[i]), 4);
            mbar_init(smem_addr(&a_empty[i]), 1);
        }
        for (int i = 0; i < TC_NB; ++i) {
            mbar_init(smem_addr(&d_full[i]), 2);
            mbar_init(smem_addr(&d_empty[i]), 4);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(smem_addr(&tb_full[i]), 4);
            mbar_init(smem_addr(&tb_empty[i]), 1);
        }
        mbar_init(smem_addr(mma_done), 2);
        mbar_init(smem_addr(stall_bar), 1);
        *flag = 0;
        fence_barrier_init();
    }
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
            const uint32_t s0 = smem_addr(smem);
            const int n_pre = min(nst, n_units);
            int tile = tile_first, grp = grp_first;
            for (int i = 0; i < n_units; ++i) {
                const int s = i % nst;
                if (i >= nst) wait_or_flag(p, flag, smem_addr(&empty[s]), static_cast<uint32_t>(((i / nst) & 1) ^ 1));
                const uint32_t fb = smem_addr(&full[s]);
                const uint32_t stage = s0 + static_cast<uint32_t>(s * TC_STAGE);
                const int g0 = grp * TC_GU;              // the unit's first group
                mbar_arrive_expect_tx(fb, static_cast<uint32_t>(TC_STAGE));
#pragma unroll
                for (int g = 0; g < TC_GU; ++g)
                    tma_load_2d(stage + g * TC_W_BYTES, &tmW, (g0 + g) * 16, tile * TC_RT, fb, pol_w);
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
        // Two pipelines: units i with i % 2 == w go to dequant warpgroup w
        // and MMA warp w, through the pipeline's own ring of TC_NSLOT group
        // slots, into the pipeline's accumulator of the box's set (its first
        // MMA of a box clears it).  Every waiter walks its barriers' phases
        // in order.  The whole warp runs the loop with warp-uniform operands
        // and one elected lane issues.
        const int w = warp == 1 ? 0 : 1;
        const uint32_t s0 = smem_addr(smem);
        const uint32_t slot_col = static_cast<uint32_t>(w * TC_NSLOT) * 64u;
        uint64_t *my_full = a_full + w * TC_NSLOT, *my_empty = a_empty + w * TC_NSLOT;
        int grp4 = grp_first % TC_BOX_UNITS, left = G - grp_first, nb = -1;
        int s = 0, slot = 0;
        uint32_t sph = 0u, slph = 0u;                 // phase parities of stage s, of the slot ring's lap
        bool first_in_box = true;
        for (int i = 0; i < n_units; ++i) {
            const bool box_start = i == 0 || grp4 == 0;
            const bool box_end = i == n_units - 1 || grp4 == TC_BOX_UNITS - 1;
            if (box_start) {
                ++nb;
                first_in_box = true;
                if (nb >= TC_NB)            // the set's previous box has been read out
                    tc_wait(p, flag, smem_addr(&d_empty[nb & 1]), static_cast<uint32_t>(((nb >> 1) - 1) & 1));
            }
            if (--left == 0) { left = G; grp4 = 0; } else grp4 = (grp4 + 1) & (TC_BOX_UNITS - 1);
            if ((i & 1) == w) {
                tc_wait(p, flag, smem_addr(&full[s]), sph);
                const uint32_t d = tmem + TC_ACC_COL + 32u * static_cast<uint32_t>(TC_NDQ * (nb & 1) + w);
                const uint32_t xs0 = s0 + static_cast<uint32_t>(s * TC_STAGE + TC_GU * TC_W_BYTES);
#pragma unroll
                for (int g = 0; g < TC_GU; ++g) {
                    tc_wait(p, flag, smem_addr(&my_full[slot]), slph);
                    __syncwarp();               // converged for elect.sync
                    tc_fence_after_sync();
                    tc_mma8_f16_ts_warp(d, tmem + slot_col + 64u * static_cast<uint32_t>(slot),
                                        tc_bdesc(xs0 + static_cast<uint32_t>(g * TC_X_BYTES)), TC_IDESC,
                                        (first_in_box && g == 0) ? 0u : 1u);
                    tc_commit_warp(smem_addr(&my_empty[slot]));
                    if (++slot == TC_NSLOT) { slot = 0; slph ^= 1u; }
                }
                tc_commit_warp(smem_addr(&empty[s]));
                first_in_box = false;
            }
            if (box_end) tc_commit_warp(smem_addr(&d_full[nb & 1]));
            if (++s == nst) { s = 0; sph ^= 1u; }
        }
        __syncwarp();
        tc_commit_warp(smem_addr(mma_done));
    } else if (warp < TC_EP0) {
        // ============================================================ dequant
        // warpgroup w takes units i with i % 2 == w; thread = tile row; each
        // group goes to the next slot of the pipeline's ring
        const int w = (warp - TC_DQ0) >> 2;
        const int q = warp & 3;                       // tensor-memory lane quarter
        const int row = 32 * q + lane;
        const uint32_t s0 = smem_addr(smem);
        const uint32_t sw = static_cast<uint32_t>((row >> 1) & 3);   // the box's 64-byte swizzle
        const uint32_t tl = tmem + (static_cast<uint32_t>(32 * q) << 16) + static_cast<uint32_t>(w * TC_NSLOT) * 64u;
        uint64_t *my_full = a_full + w * TC_NSLOT, *my_empty = a_empty + w * TC_NSLOT;
        int tile = tile_first, grp = grp_first;
        int key = -1, key_next = -1;                  // box (tile * boxes + bx) of `cur`, of `nxt`
        uint4 cur = make_uint4(0u, 0u, 0u, 0u), nxt = cur;
        float f1 = 0.f, f2 = 0.f;
        const int nbox = G / TC_BOX_UNITS;            // boxes per tile
        int s = 0, slot = 0;
        uint32_t sph = 0u, slph = 0u;
        bool lap0 = true;                             // the ring's first lap: no slot has been used
        for (int i = 0; i < n_units; ++i) {
            const int t_i = tile, j = grp;
            if (++grp == G) { grp = 0; ++tile; }
            if ((i & 1) == w) {
                const int bx = j / TC_BOX_UNITS, k = t_i * nbox + bx;
                if (k != key) {
                    // this box's scales (read ahead when possible), then the next box's
                    cur = (k == key_next) ? nxt : tc_load_scales(p, t_i, bx, row);
                    key = k;
                    const int nbx = bx + 1 < nbox ? bx + 1 : 0, ntile = bx + 1 < nbox ? t_i : t_i + 1;
                    key_next = ntile * nbox + nbx;
                    if (static_cast<long long>(ntile) * TC_RT < p.n_rows) nxt = tc_load_scales(p, ntile, nbx, row);
                    tc_pow2_pair(TC_SHIFT - tc_box_exp(cur), f1, f2);
                }
                // the unit's two groups are word j % 4 of the box's scales
                const uint32_t jw = static_cast<uint32_t>(j % TC_BOX_UNITS);
                const uint32_t sp = jw == 0 ? cur.x : jw == 1 ? cur.y : jw == 2 ? cur.z : cur.w;
                wait_or_flag(p, flag, smem_addr(&full[s]), sph);
                const uint32_t wrow0 = s0 + static_cast<uint32_t>(s * TC_STAGE + row * 64);
#pragma unroll
                for (int g = 0; g < TC_GU; ++g) {
                    uint32_t s2, c2;
                    tc_factor(g == 0 ? (sp & 0xFFFFu) : (sp >> 16), f1, f2, s2, c2);
                    if (!lap0)                          // the slot's previous group has been multiplied
                        wait_or_flag(p, flag, smem_addr(&my_empty[slot]), slph ^ 1u);
                    const uint32_t wrow = wrow0 + static_cast<uint32_t>(g * TC_W_BYTES);
                    const uint32_t tlane = tl + 64u * static_cast<uint32_t>(slot);
#pragma unroll
                    for (int h = 0; h < 2; ++h) {         // words 0..7, then 8..15: 32 columns each
                        uint32_t v[32];
#pragma unroll
                        for (int jj = 0; jj < 2; ++jj) {
                            const int jc = 2 * h + jj;
                            const uint4 w4 = lds128(wrow + ((static_cast<uint32_t>(jc) ^ sw) << 4));
                            const uint32_t ws[4] = {w4.x, w4.y, w4.z, w4.w};
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                const uint32_t wd = ws[e];
                                const int c0 = 4 * (4 * jj + e);
                                v[c0 + 0] = tc_scaled_pair(wd << 6, s2, c2);   // nibbles (0, 4)
                                v[c0 + 1] = tc_scaled_pair(wd << 2, s2, c2);   // (1, 5)
                                v[c0 + 2] = tc_scaled_pair(wd >> 2, s2, c2);   // (2, 6)
                                v[c0 + 3] = tc_scaled_pair(wd >> 6, s2, c2);   // (3, 7)
                            }
                        }
                        tmem_st32(tlane + 32u * h, v);
                    }
                    tmem_wait_st();
                    tc_fence_before_sync();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(smem_addr(&my_full[slot]));
                    if (++slot == TC_NSLOT) { slot = 0; slph ^= 1u; lap0 = false; }
                }
            }
            if (++s == nst) { s = 0; sph ^= 1u; }
        }
    } else if (warp < TC_RED) {
        // ============================================================ epilogue
        const int q = warp & 3;
        const int ew = warp - TC_EP0;                 // epilogue warp 0..3
        const int row = 32 * q + lane;
        constexpr uint32_t NTHR_E = 128;
        pdl_wait_prior();                   // xinv, scratch area, outputs and drafts from here on
        float *xinv_s = reinterpret_cast<float *>(smem + p.off_xinv);
        if (ew == 0) xinv_s[lane] = __ldg(p.xinv + lane);
        if (p.stall_ns != 0u && b == 0 && ew == 0) wait_or_flag_for(p, flag, smem_addr(stall_bar), 0u, p.stall_ns);
        // contributors of the first and the last tile, as in the other kernels
        const int tile_last = static_cast<int>((u1 - 1) / G);
        int bfA = b, ncA = 1, ncZ = 1;
        {
            const long long ts = static_cast<long long>(tile_first) * G, te = ts + G;
            if (u0 > ts || u1 < te) {
                bfA = cta_of(ts, U, B);
                ncA = cta_of(te - 1, U, B) - bfA + 1;
            }
            const long long tz = static_cast<long long>(tile_last) * G;
            if (tile_last != tile_first && u1 < tz + G) ncZ = cta_of(tz + G - 1, U, B) - b + 1;
        }
        named_bar_sync(1, NTHR_E);          // xinv staged
        const uint32_t taddr = tmem + (static_cast<uint32_t>(32 * q) << 16) + TC_ACC_COL;
        const int nbox = G / TC_BOX_UNITS;
        int ntb = 0;                                  // head: tiles handed to the reducer
        float acc[32];
#pragma unroll
        for (int t = 0; t < 32; ++t) acc[t] = 0.f;
        int tile = tile_first, grp = grp_first, nb = -1, i_start = 0;
        uint4 nxt = tc_load_scales(p, tile_first, grp_first / TC_BOX_UNITS, row);
        for (int i = 0; i < n_units; ++i) {
            const bool box_start = i == 0 || (grp % TC_BOX_UNITS) == 0;
            const bool box_end = i == n_units - 1 || (grp % TC_BOX_UNITS) == TC_BOX_UNITS - 1;
            const bool tile_end = (grp == G - 1) || (i == n_units - 1);
            const int bx = grp / TC_BOX_UNITS;
            if (box_start) { ++nb; i_start = i; }
            if (++grp == G) grp = 0;
            if (!box_end) continue;

            // ------------------------------------------- end of box nb
            const uint4 cur = nxt;
            {   // read the next box's scales ahead
                const int nbx = bx + 1 < nbox ? bx + 1 : 0, ntile = bx + 1 < nbox ? tile : tile + 1;
                if (i + 1 < n_units) nxt = tc_load_scales(p, ntile, nbx, row);
            }
            float m1, m2;
            tc_pow2_pair(tc_box_exp(cur) - TC_SHIFT, m1, m2);
            const int par = nb & 1;
            // a pipeline's accumulator holds this box only if the box has one of its units
            const bool has0 = i > i_start || (i_start & 1) == 0, has1 = i > i_start || (i_start & 1) == 1;
            wait_or_flag(p, flag, smem_addr(&d_full[par]), static_cast<uint32_t>((nb >> 1) & 1));
            tc_fence_after_sync();
            uint32_t v0[32], v1[32];        // the two pipelines' sums
            tmem_ld32(taddr + 64u * static_cast<uint32_t>(par), v0);
            tmem_ld32(taddr + 64u * static_cast<uint32_t>(par) + 32u, v1);
            tmem_wait_ld();
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_addr(&d_empty[par]));
#pragma unroll
            for (int t = 0; t < 32; ++t) {
                const float e0 = has0 ? __uint_as_float(v0[t]) : 0.f, e1 = has1 ? __uint_as_float(v1[t]) : 0.f;
                acc[t] += ((e0 + e1) * m1) * m2;
            }

            if (!tile_end) continue;
            // ------------------------------------------- end of this CTA's share of `tile`
#pragma unroll
            for (int t = 0; t < 32; ++t) acc[t] *= xinv_s[t];
            const long long ts = static_cast<long long>(tile) * G, te = ts + G;
            const bool complete = (u0 <= ts) && (u1 >= te);
            bool finish = true;
            if (!complete) {
                // The tile's first contributor bf finishes it: for bf the
                // tile is the end of its range and comes last, for the
                // others it is the start of theirs.  The others publish their
                // row sums and count themselves in with a release add they
                // do not wait for; bf waits (bounded) until all nc - 1 are
                // in, adds them after its own in CTA order and resets the
                // counter for the next launch.
                const bool first = tile == tile_first;
                const int bf = first ? bfA : b;
                const int nc = first ? ncA : ncZ;
                finish = bf == b;
                if (!finish) {
                    float *mine = p.part + static_cast<size_t>(b) * 2 * WIDE_PART_FLOATS + row * TMAX;
#pragma unroll
                    for (int t = 0; t < 32; t += 4)
                        __stcg(reinterpret_cast<float4 *>(mine + t), make_float4(acc[t], acc[t + 1], acc[t + 2], acc[t + 3]));
                    named_bar_sync(1, NTHR_E);
                    if (ew == 0 && lane == 0) red_add_release_gpu(&p.ctr[bf], 1u);
                } else {
                    if (ew == 0) {
                        const uint64_t t0 = global_timer_ns();
                        while (!__all_sync(0xFFFFFFFFu, ld_acquire_gpu_u32(&p.ctr[bf]) == static_cast<unsigned>(nc - 1))) {
                            if (global_timer_ns() - t0 > (*flag ? WAIT_LIMIT_AFTER_ERR_NS : WAIT_LIMIT_NS)) {
                                *flag = 1;
                                if (lane == 0) atomicOr(p.err, 2);
                                break;
                            }
                        }
                    }
                    named_bar_sync(1, NTHR_E);      // all nc - 1 are in
                    if (ew == 0 && lane == 0) p.ctr[bf] = 0u;
#pragma unroll 1
                    for (int jc = 1; jc < nc; ++jc) {
                        const float *src = p.part + static_cast<size_t>(bf + jc) * 2 * WIDE_PART_FLOATS + row * TMAX;
#pragma unroll
                        for (int hh = 0; hh < 2; ++hh) {
                            float4 e4[4];
#pragma unroll
                            for (int t = 0; t < 4; ++t) e4[t] = __ldcg(reinterpret_cast<const float4 *>(src) + 4 * hh + t);
#pragma unroll
                            for (int t = 0; t < 4; ++t) {
                                const int c = 16 * hh + 4 * t;
                                acc[c] += e4[t].x; acc[c + 1] += e4[t].y; acc[c + 2] += e4[t].z; acc[c + 3] += e4[t].w;
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
                    // hand the finished tile to the reducer warp (rows in
                    // 16-byte chunks, chunk j of row r at j ^ (r & 7))
                    const int tb = ntb & 1;
                    if (ntb >= 2) wait_or_flag(p, flag, smem_addr(&tb_empty[tb]), static_cast<uint32_t>(((ntb >> 1) - 1) & 1));
                    const uint32_t rb = smem_addr(tbuf + tb * TC_TB_BYTES + row * 128);
#pragma unroll
                    for (int jc = 0; jc < 8; ++jc)
                        sts128(rb + static_cast<uint32_t>((jc ^ (row & 7)) << 4),
                               make_uint4(__float_as_uint(acc[4 * jc]), __float_as_uint(acc[4 * jc + 1]),
                                          __float_as_uint(acc[4 * jc + 2]), __float_as_uint(acc[4 * jc + 3])));
                    if (ew == 0 && lane == 0) tb_tile[tb] = tile;
                    __syncwarp();
                    if (lane == 0) mbar_arrive(smem_addr(&tb_full[tb]));
                    ++ntb;
                }
            }
#pragma unroll
            for (int t = 0; t < 32; ++t) acc[t] = 0.f;
            ++tile;
        }
        if constexpr (HEAD) {
            // no more tiles: the sentinel
            const int tb = ntb & 1;
            if (ntb >= 2) wait_or_flag(p, flag, smem_addr(&tb_empty[tb]), static_cast<uint32_t>(((ntb >> 1) - 1) & 1));
            if (ew == 0 && lane == 0) tb_tile[tb] = -1;
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_addr(&tb_full[tb]));
        }
    } else if (HEAD) {
        // ============================================================ reducer (head)
        // lane t keeps the largest key (logit, lowest id) of token t over
        // every tile this CTA finishes; then the grid argmax and the verify
        unsigned long long best = 0ull;
        for (int k = 0;; ++k) {
            const int tb = k & 1;
            wait_or_flag(p, flag, smem_addr(&tb_full[tb]), static_cast<uint32_t>((k >> 1) & 1));
            const int tile = tb_tile[tb];
            if (tile < 0) break;
            const long long r0 = static_cast<long long>(tile) * TC_RT;
            const int nr = p.n_rows - r0 < TC_RT ? static_cast<int>(p.n_rows - r0) : TC_RT;
            const uint32_t base = smem_addr(tbuf + tb * TC_TB_BYTES) + static_cast<uint32_t>((lane & 3) * 4);
            const uint32_t jl = static_cast<uint32_t>(lane >> 2);
            for (int r = 0; r < nr; ++r) {
                const float v = lds_f32(base + static_cast<uint32_t>(r * 128) + ((jl ^ static_cast<uint32_t>(r & 7)) << 4));
                const unsigned long long key = make_key(v, static_cast<uint32_t>(r0 + r));
                best = key > best ? key : best;
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_addr(&tb_empty[tb]));
        }
        pdl_wait_prior();                   // scratch keys, drafts and outputs from here on
        head_grid_tail(p, lane < T ? best : 0ull, lane, B);
    }

    // ================================================================ teardown
    // Every warp gets here (no early exit after the allocation).  The MMAs
    // are complete once the last commits have arrived; then the tensor
    // memory is freed by the warp that allocated it.
    __syncthreads();
    if (warp == 1) {
        if (!mbar_wait_bounded(smem_addr(mma_done), 0u, WAIT_LIMIT_AFTER_ERR_NS)) atomicOr(p.err, 2);
        tc_fence_after_sync();
        tmem_dealloc(tmem, TC_TMEM_COLS);
    }
}

}  // namespace sv
