// w4a16_stream.cuh -- the one kernel behind every export: a stream-K pass
// over 64-row tiles of a W4A16 (uint32 nibble words, bf16 group-128 scales)
// weight matrix, with either a GEMM epilogue (y = bf16) or an lm_head
// epilogue (fp32 logits -> per-CTA top-1 -> grid argmax -> greedy verify).
//
// Work decomposition.  A "unit" is one 64-row tile x one 128-column group
// (4 KB of packed weights).  Units are numbered tile-major and the grid's B
// CTAs (B <= SM count, one CTA per SM) take equal contiguous ranges, so every
// SM streams the same number of bytes whatever N and K are.  A tile whose
// units straddle CTAs is finished by its first CTA, for which it is the end
// of its range: the others publish their fp32 partial sums and count
// themselves in (per-tile counter in the scratch area), and the finisher
// adds all of them in CTA order: results do not depend on arrival order.
//
// Warp roles inside a CTA (all hand-offs are mbarriers; no CTA-wide barrier
// after set-up):
// (NCW consumer warps, 16 or 8, see consumer_warps):
//  * warp NCW, producer: fills each pipeline stage (up to GPS units of one
//    tile) with tensor (TMA) copies -- one 64-row x 64-byte box of packed
//    weights and one box of activations per group -- completing on the
//    stage's mbarrier.  Gathered rows (a vocab_map) use one 1-D bulk copy per
//    row segment instead.
//  * warps 0..NCW-1, consumers: warp w takes group (w % GPS) of a stage for R
//    m16 tiles, dequantises its nibbles in registers and feeds them to the
//    bf16 tensor cores as the A operand (mma.sync m16n8k16; tokens are the
//    n8 B operand), and folds each group's fp32 sum into its accumulators
//    with the group scale.  At the end of a tile each warp hands its partial
//    sums to the epilogue warp through shared memory.
//  * warp NCW+1, epilogue: stages the scales (and token ids) of tile k+2 while
//    tile k+1 is being computed, adds the consumers' partials in a fixed
//    order, finishes split tiles, and runs the GEMM store or the lm_head
//    argmax; at the end it runs the grid-level argmax and the verify.
// Every weight byte crosses HBM once per call; T only changes how many n8
// token tiles each dequantised fragment multiplies.
//
// Back-to-back launches overlap (programmatic dependent launch): a CTA may
// start while the previous kernel of the stream is still finishing, and it
// streams packed weights and scales -- read-only model data -- right away.
// Everything that a preceding kernel may produce or use (activations, drafts,
// the vocab_map, the scratch area, the outputs) is touched only after
// griddepcontrol.wait.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>

#include "sv_ptx.cuh"

namespace sv {

constexpr int ROWS = 64;                        // rows per tile
// Consumer warps of a launch: 16 (two m16 tiles each) when one token tile
// of contiguous rows reads resident activations; otherwise 8 (all four m16
// tiles of a group, or two of four token tiles) -- activations copied into
// every stage, or gathered rows -- where fewer, wider warps measured faster.
// The producer and epilogue warps follow the consumers.
__host__ __device__ constexpr int consumer_warps(int NT, bool XRES, bool GATHER)
{
    return (NT == 1 && XRES && !GATHER) ? 16 : 8;
}
constexpr int TMAX = 32;                        // largest T
constexpr int PART_FLOATS = TMAX * ROWS;        // one split-tile partial
constexpr int PRE_PARTS = 2;                     // partials a finishing CTA copies ahead (one token tile)
constexpr int XBOX = 144;                       // bf16 activation box width (elements), one token tile
constexpr int XROW_BYTES = XBOX * 2;            // = 32 (mod 128): conflict-free B loads
constexpr int XSTR = 272;                       // bytes per token row of a converted group block
                                                // (256 + 16: = 16 mod 128, conflict-free B loads)
constexpr int XP_THREADS = 256;                 // threads of the activation-conversion kernel
constexpr int BK_STRIDE = TMAX + 1;             // u64 per lane in the best-key table (odd: no bank conflicts)
constexpr uint64_t WAIT_LIMIT_NS = 2000000000ull;        // 2 s: only a broken run gets here
constexpr uint64_t WAIT_LIMIT_AFTER_ERR_NS = 1000000ull;  // 1 ms once something failed

template <int NT, bool GATHER, int NCW_>
struct Cfg {
    static constexpr int NCW = NCW_;                // consumer warps
    static constexpr int GPS = (NT == 1) ? 8 : 4;   // 128-column groups per stage
    static constexpr int MSETS = NCW / GPS;         // warps sharing one group slot
    static constexpr int R = 4 / MSETS;             // m16 tiles per warp
    static constexpr int TP = 8 * NT;               // tokens, padded to n8 tiles
    // Weights in a stage.  Contiguous rows: one dense [64 rows][64 B] block
    // per group (a quarter warp reads 2 rows x 64 B = 128 consecutive bytes).
    // Gathered rows: [64 rows][GPS*64 B], filled by 16 four-row boxes
    // (tile::gather4; box b holds rows 4b..4b+3).  Box destinations stay
    // 128-byte aligned, so the two rows a quarter warp reads share banks (a
    // 2-way conflict on the weight loads, a few per 2 KB of weights).
    static constexpr int GROW = GPS * 64;           // one gathered row of a stage
    static constexpr int W_BYTES = GATHER ? ROWS * GROW : GPS * ROWS * 64;
    // hand-off buffer row stride (floats): TP, padded by 8 for wider tiles
    // (two-wavefront float2 stores by the consumers)
    static constexpr int RSTR = (NT == 1) ? 8 : TP + 8;
    static constexpr int RED_FLOATS = GPS * ROWS * RSTR;
};

struct Params {
    const uint16_t *x;          // [T][K] bf16 bits
    const uint8_t *x16;         // converted activations (NT > 1): [G][TP][XSTR] bytes, see xprep_kernel
    const float *xinv;          // converted activations: 2^-s_t of every token row (1 for rows >= T)
    const uint32_t *Wq;         // [rows][K/8]
    const uint16_t *scales;     // [rows][K/128]
    const int32_t *map;         // HEAD: candidate row -> token id, or null
    int T, K, G;                // G = K / 128
    int n_rows;                 // GEMM: N; HEAD: V or n_map
    int V;                      // HEAD: token ids must be < V
    long long U;                // units = tiles * G
    // shared-memory layout (bytes)
    int nst, stage_bytes, xslot_bytes, sbuf_bytes;
    int off_sbuf, off_ids, off_red, off_bars;
    int off_xres, xres_stride;  // resident activations (XRES kernels only)
    int off_xsc;                // XRES: per-token largest |x| (bf16 bits), [8] u32
    int off_pre;                // NT = 1: other contributors' partials of the tile this CTA finishes, [PRE_PARTS][ROWS][8] floats
    int off_xinv;               // tcgen05: xinv staged in shared memory, [32] floats
    int off_bk;                 // HEAD: running best key per lane and token, [32][BK_STRIDE] u64
    int off_xzero;              // XBF: 256 zero bytes, the activation row of absent tokens
    // GEMM output
    uint16_t *y;                // [T][N] bf16, or
    float *y32;                 // [T][N] fp32 when not null (the lm_head's logits for rescoring)
    // HEAD outputs
    int mode;                   // 0: verify, 1: argmax
    int map_static;             // the vocab_map is model data no preceding kernel writes:
                                // it may be read before griddepcontrol.wait
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
    // Test hook of the bounded waits: when nonzero, the epilogue warp of CTA
    // 0 first waits up to stall_ns on an mbarrier that nothing completes,
    // so that a test can watch a wait run out (the error word gets the
    // time-out bit; everything after it still runs).
    uint32_t stall_ns;
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

// Token id of row rloc of tile `tile` (or -1 when the row does not exist or
// its vocab_map entry is out of range; the latter sets the error word).
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

// A bounded wait: when it runs out, the CTA's flag (shorter limits from then
// on) and the time-out bit of the error word are set, and the caller goes on.
__device__ __forceinline__ void wait_or_flag_for(const Params &p, volatile int *flag, uint32_t bar,
                                                 uint32_t parity, uint64_t lim)
{
    if (!mbar_wait_bounded(bar, parity, lim)) {
        *flag = 1;
        atomicOr(p.err, 2);
    }
}

__device__ __forceinline__ void wait_or_flag(const Params &p, volatile int *flag, uint32_t bar,
                                             uint32_t parity)
{
    wait_or_flag_for(p, flag, bar, parity, *flag ? WAIT_LIMIT_AFTER_ERR_NS : WAIT_LIMIT_NS);
}

// Largest magnitude among the 8 bf16 values of a 16-byte chunk, as bf16 bits.
__device__ __forceinline__ unsigned chunk_absmax(const uint4 r)
{
    const unsigned hi = max(max(r.x & 0x7FFF0000u, r.y & 0x7FFF0000u), max(r.z & 0x7FFF0000u, r.w & 0x7FFF0000u)) >> 16;
    const unsigned lo = max(max(r.x & 0x7FFFu, r.y & 0x7FFFu), max(r.z & 0x7FFFu, r.w & 0x7FFFu));
    return max(hi, lo);
}

// A chunk of 8 bf16 activations (x0..x7) -> fp16 x * sc in B-fragment order:
// (x0,x4) (x1,x5) (x2,x6) (x3,x7), the pairing of the dequantised nibbles.
__device__ __forceinline__ uint4 chunk_to_f16(const uint4 r, float sc)
{
    uint4 v;
    v.x = pack_f16x2(__uint_as_float(r.x << 16) * sc, __uint_as_float(r.z << 16) * sc);
    v.y = pack_f16x2(__uint_as_float(r.x & 0xFFFF0000u) * sc, __uint_as_float(r.z & 0xFFFF0000u) * sc);
    v.z = pack_f16x2(__uint_as_float(r.y << 16) * sc, __uint_as_float(r.w << 16) * sc);
    v.w = pack_f16x2(__uint_as_float(r.y & 0xFFFF0000u) * sc, __uint_as_float(r.w & 0xFFFF0000u) * sc);
    return v;
}

// Position of chunk i (0..15) of a group inside its 256-byte row: chunk
// index XOR-swizzled (bit 1 ^= bit 3), so that the B loads of a quarter warp
// (chunks 4c + m, c = 0..3) hit distinct banks.
__device__ __forceinline__ int chunk_slot(int i)
{
    return i ^ ((i >> 2) & 2);
}

// Activations for the kernels that stream them per stage (T > 8, or rows too
// long to keep resident): x (bf16 [T][K]) is converted once per call into
// x16, laid out per 128-column group g as a block of TP token rows of XSTR
// bytes; row t holds the group's 16 chunks as fp16 x[t] * 2^s_t in
// B-fragment order at chunk_slot positions (the same encoding as the
// resident rows of the main kernel); rows T..TP-1 are zeros.  xinv[t] =
// 2^-s_t.  One CTA per token row.  The main kernel then copies ready-made
// group blocks into its stages (one bulk copy per group) and its B loads
// need neither byte permutes nor conversion.
//
// TC = true writes the layout of w4a16_tc_kernel instead: per group a block
// of 8 KB holding, for 16-byte chunk k (0..15, eight columns) and token t
// (0..31), the chunk at ((k * 4 + t / 8) * 8 + t % 8) * 16 -- "core
// matrices" of 8 tokens x 16 bytes, 128 bytes apart along the tokens and
// 512 bytes apart along K, the canonical K-major layout a tcgen05 B operand
// is described by; no chunk swizzle.
template <bool TC>
__device__ __forceinline__ size_t xprep_offset(int i, int t, int TP)
{
    if (TC) return static_cast<size_t>(i >> 4) * 8192 + static_cast<size_t>(((i & 15) * 4 + (t >> 3)) * 128 + (t & 7) * 16);
    return (static_cast<size_t>(i >> 4) * TP + t) * XSTR + chunk_slot(i & 15) * 16;
}

template <bool TC>
__global__ void __launch_bounds__(XP_THREADS) xprep_kernel(const uint16_t *x, int T, int K, int TP, uint8_t *x16,
                                                           float *xinv)
{
    pdl_launch_dependents();
    pdl_wait_prior();                   // x may come from the previous kernel
    const int t = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int cpr = K / 8;              // 16-byte chunks per row
    if (t >= T) {
        for (int i = tid; i < cpr; i += XP_THREADS)
            *reinterpret_cast<uint4 *>(x16 + xprep_offset<TC>(i, t, TP)) = make_uint4(0u, 0u, 0u, 0u);
        if (tid == 0) xinv[t] = 1.f;
        return;
    }
    const uint4 *row = reinterpret_cast<const uint4 *>(x) + static_cast<size_t>(t) * cpr;
    constexpr int XB = 12;
    const bool one_batch = cpr <= XB * XP_THREADS;
    uint4 r[XB];
    unsigned mx = 0u;
    for (int i0 = tid; i0 < cpr; i0 += XB * XP_THREADS) {
#pragma unroll
        for (int u = 0; u < XB; ++u) {
            const int i = i0 + u * XP_THREADS;
            r[u] = i < cpr ? row[i] : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int u = 0; u < XB; ++u) mx = max(mx, chunk_absmax(r[u]));
        if (one_batch) break;
    }
    __shared__ unsigned wmax[XP_THREADS / 32];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = max(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, o));
    if (lane == 0) wmax[warp] = mx;
    __syncthreads();
    mx = 0u;
#pragma unroll
    for (int w = 0; w < XP_THREADS / 32; ++w) mx = max(mx, wmax[w]);
    const int sh = xres_shift(mx);
    const float sc = __uint_as_float(static_cast<uint32_t>(127 + sh) << 23);
    for (int i0 = tid; i0 < cpr; i0 += XB * XP_THREADS) {
        if (!one_batch) {
#pragma unroll
            for (int u = 0; u < XB; ++u) {
                const int i = i0 + u * XP_THREADS;
                r[u] = i < cpr ? row[i] : make_uint4(0u, 0u, 0u, 0u);
            }
        }
#pragma unroll
        for (int u = 0; u < XB; ++u) {
            const int i = i0 + u * XP_THREADS;
            if (i < cpr) *reinterpret_cast<uint4 *>(x16 + xprep_offset<TC>(i, t, TP)) = chunk_to_f16(r[u], sc);
        }
    }
    if (tid == 0) xinv[t] = __uint_as_float(static_cast<uint32_t>(127 - sh) << 23);
}

// The consumers' hand-off buffer `red` holds one partial per group slot as
// [slot][ROWS][RSTR]: token t of row `row` at (slot * ROWS + row) * RSTR + t,
// so that the epilogue reads four tokens of a row with one 16-byte load.
// One token tile: RSTR = 8; wider tiles: TP + 8 (the padding keeps the
// consumers' two-token stores at two wavefronts per warp).
template <int NT, int GPS>
__device__ __forceinline__ int red_index(int slot, int tok, int row)
{
    constexpr int RSTR = (NT == 1) ? 8 : 8 * NT + 8;
    return (slot * ROWS + row) * RSTR + tok;
}

// Sums over the GPS group slots of tokens t0..t0+3 of tile row `row`
// (pairwise, in a fixed order); tokens >= T give 0.
template <int NT, int GPS>
__device__ __forceinline__ float4 slot_sums4(const float *red, int t0, int row, int T)
{
    static_assert(GPS % 4 == 0, "slots are added in groups of four");
    // slots in groups of four: ((s0 + s1) + (s2 + s3)) + ((s4 + s5) + (s6 + s7))
    auto add = [](float4 a, float4 b) { return make_float4(a.x + b.x, a.y + b.y, a.z + b.z, a.w + b.w); };
    auto ld = [&](int sl) { return *reinterpret_cast<const float4 *>(red + red_index<NT, GPS>(sl, t0, row)); };
    float4 v = add(add(ld(0), ld(1)), add(ld(2), ld(3)));
#pragma unroll
    for (int sl = 4; sl < GPS; sl += 4) v = add(v, add(add(ld(sl), ld(sl + 1)), add(ld(sl + 2), ld(sl + 3))));
    if (t0 + 1 >= T) v.y = 0.f;
    if (t0 + 2 >= T) v.z = 0.f;
    if (t0 + 3 >= T) v.w = 0.f;
    return v;
}

// Epilogue warp: stage the scales (and, for the head, the token ids) of one
// tile into shared memory with cp.async, then arrive on `bar` (expected
// arrivals: 32 cp.async completions + 1 plain arrival).  Rows that do not
// exist get scale 0 and id -1.
template <bool HEAD, bool GATHER>
__device__ __forceinline__ void stage_tile_meta(const Params &p, int tile, uint8_t *sb,
                                                int32_t *ib, uint32_t bar, int lane)
{
    const int G = p.G;
    uint16_t *dst = reinterpret_cast<uint16_t *>(sb);
    const int id0 = row_id(p, tile, lane), id1 = row_id(p, tile, lane + 32);
    if (HEAD || GATHER) {
        ib[lane] = id0;
        ib[lane + 32] = id1;
    }
    if (!GATHER) {
        // rows are contiguous: one contiguous block of nvalid * G scales
        const long long r0 = static_cast<long long>(tile) * ROWS;
        const int nvalid = static_cast<int>(min(static_cast<long long>(ROWS), p.n_rows - r0));
        const uint16_t *src = p.scales + r0 * G;
        const int nel = nvalid * G;
        const int n16 = nel / 8;                         // 16-byte chunks
        for (int i = lane; i < n16; i += 32) cp_async_16(smem_addr(dst + 8 * i), src + 8 * i);
        for (int i = 8 * n16 + lane; i < nel; i += 32) dst[i] = ldg_u16(src + i);
        for (int i = nel + lane; i < ROWS * G; i += 32) dst[i] = 0;
    } else if ((G & 7) == 0) {
        // gathered rows, 16-byte aligned (G*2 bytes a multiple of 16): the
        // ROWS x G/8 chunks are spread over the lanes, so one warp keeps
        // many independent small copies in flight
        __syncwarp();
        const int cpr = G / 8;
        for (int i = lane; i < ROWS * cpr; i += 32) {
            const int r = i / cpr, j = i - r * cpr;
            const int id = ib[r];
            uint16_t *d = dst + r * G + 8 * j;
            if (id < 0)
                *reinterpret_cast<uint4 *>(d) = make_uint4(0u, 0u, 0u, 0u);
            else
                cp_async_16(smem_addr(d), p.scales + static_cast<size_t>(id) * G + 8 * j);
        }
    } else {
        for (int r = 0; r < ROWS; ++r) {
            const int id = __shfl_sync(0xFFFFFFFFu, r < 32 ? id0 : id1, r & 31);
            uint16_t *d = dst + r * G;
            if (id < 0) {
                for (int j = lane; j < G; j += 32) d[j] = 0;
            } else if ((G & 1) == 0) {
                const uint16_t *src = p.scales + static_cast<size_t>(id) * G;
                for (int j = lane; j < G / 2; j += 32) cp_async_4(smem_addr(d + 2 * j), src + 2 * j);
            } else {
                const uint16_t *src = p.scales + static_cast<size_t>(id) * G;
                for (int j = lane; j < G; j += 32) d[j] = ldg_u16(src + j);
            }
        }
    }
    cp_async_mbar_arrive(bar);
    __syncwarp();
    if (lane == 0) mbar_arrive(bar);
}

// Grid-level end of a head launch, run by one warp of every CTA: lane t
// (< T) holds the CTA's best key of token t.  The keys go to the grid's
// per-token maxima (atomicMax), then the CTA counts itself in; the last CTA
// turns the maxima into ids and writes them (argmax mode) or runs the
// greedy verify of every stream, and leaves the keys and the counter at 0.
__device__ __forceinline__ void head_grid_tail(const Params &p, unsigned long long best, int lane, int B)
{
    const int T = p.T;
    // The warp's maxima, then one acquire-release count per CTA: the warp
    // barrier orders every lane's maximum before lane 0's release, and lane
    // 0's acquire (the count that completes the grid) before the last CTA's
    // reads of the keys.
    if (lane < T && best != 0ull) atomicMax(&p.keys[lane], best);
    __syncwarp();
    unsigned last = 0;
    if (lane == 0) last = (atomic_add_acq_rel_gpu(p.done, 1u) == static_cast<unsigned>(B - 1));
    last = __shfl_sync(0xFFFFFFFFu, last, 0);
    __syncwarp();
    if (last) {
        int32_t a = -1;
        unsigned long long kk = 0ull;
        if (lane < T) {
            kk = __ldcg(&p.keys[lane]);
            a = (kk == 0ull) ? -1 : key_id(kk);
            p.keys[lane] = 0ull;
        }
        if (p.mode == 1) {
            if (lane < T) {
                p.ids[lane] = a;
                if (p.vals) p.vals[lane] = (kk == 0ull) ? __int_as_float(0x7fc00000) : key_value(kk);
            }
        } else {
            const int rows_per = p.n_draft + 1;
            const int sidx = lane < p.n_streams ? lane : 0;
            int acc = -1, nxt = -1;
            for (int i = 0; i <= p.n_draft; ++i) {
                const int ai = __shfl_sync(0xFFFFFFFFu, a, (sidx * rows_per + i) & 31);
                if (acc < 0) {
                    if (i == p.n_draft || p.drafts[static_cast<size_t>(sidx) * p.n_draft + i] != ai) {
                        acc = i;
                        nxt = ai;
                    }
                }
            }
            if (lane < p.n_streams) {
                p.accept_len[lane] = acc;
                p.next_token[lane] = nxt;
            }
        }
        __syncwarp();
        if (lane == 0) *p.done = 0u;
    }
}

// FMA: the consumers compute on CUDA cores instead of tensor cores (one
// mixed-precision fp16 x fp16 -> fp32 fma per weight and token); only for
// one token tile of contiguous rows with resident activations.  It exists
// for the measured comparison of the two formulations at equal HBM traffic.
template <int NT, bool HEAD, bool GATHER, bool XRES, bool FMA = false>
__global__ void __launch_bounds__((consumer_warps(NT, XRES, GATHER) + 2) * 32, 1)
w4a16_stream_kernel(const __grid_constant__ Params p, const __grid_constant__ CUtensorMap tmW,
                    const __grid_constant__ CUtensorMap tmX)
{
    constexpr int NCW = consumer_warps(NT, XRES, GATHER);
    constexpr int PRODUCER_WARP = NCW;
    constexpr int EPILOGUE_WARP = NCW + 1;
    using C = Cfg<NT, GATHER, NCW>;
    static_assert(!XRES || NT == 1, "resident activations are laid out for one n8 token tile");
    static_assert(!FMA || (NT == 1 && XRES && !GATHER), "the CUDA-core consumers read resident rows");
    // How activations reach the B loads: resident fp16 rows (XRES); raw bf16
    // rows copied into every stage by tensor copies (XBF: one token tile
    // whose rows are too long to keep resident; permuted in registers, bf16
    // dequant); or fp16 group blocks prepared by xprep_kernel and copied into
    // every stage (XPREP: more than one token tile).
    constexpr bool XBF = !XRES && NT == 1;
    constexpr bool XPREP = !XRES && NT > 1;
    extern __shared__ __align__(1024) uint8_t smem[];
    const int nst = p.nst;
    uint8_t *sbuf = smem + p.off_sbuf;                                // [2][sbuf_bytes]
    int32_t *idbuf = reinterpret_cast<int32_t *>(smem + p.off_ids);   // [2][ROWS]
    float *red = reinterpret_cast<float *>(smem + p.off_red);         // [RED_FLOATS]
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + p.off_bars);
    uint64_t *full = bars;                    // [nst]  producer -> consumers
    uint64_t *empty = bars + nst;             // [nst]  consumers -> producer
    uint64_t *meta_full = bars + 2 * nst;     // [2]    epilogue -> consumers
    uint64_t *meta_empty = meta_full + 2;     // [2]    consumers -> epilogue
    uint64_t *red_full = meta_full + 4;       //        consumers -> epilogue
    uint64_t *red_empty = meta_full + 5;      //        epilogue -> consumers
    volatile int *flag = reinterpret_cast<volatile int *>(meta_full + 6);   // a wait timed out
    uint64_t *stall_bar = meta_full + 7;      //        never completed (test hook)

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int B = gridDim.x, b = blockIdx.x;
    const long long U = p.U;
    const int G = p.G, T = p.T;
    const long long u0 = cta_start(b, U, B), u1 = cta_start(b + 1, U, B);
    const int tile_first = static_cast<int>(u0 / G);
    const int grp_first = static_cast<int>(u0 - static_cast<long long>(tile_first) * G);
    const int tile_last = static_cast<int>((u1 - 1) / G);
    const int n_units = static_cast<int>(u1 - u0);

    if (threadIdx.x == 0) {
        for (int s = 0; s < nst; ++s) {
            mbar_init(smem_addr(&full[s]), 1);
            mbar_init(smem_addr(&empty[s]), NCW);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(smem_addr(&meta_full[i]), 33);
            mbar_init(smem_addr(&meta_empty[i]), NCW);
        }
        mbar_init(smem_addr(red_full), NCW);
        mbar_init(smem_addr(red_empty), 1);
        mbar_init(smem_addr(stall_bar), 1);
        *flag = 0;
        if (XRES)
            for (int t = 0; t < 8; ++t) reinterpret_cast<unsigned *>(smem + p.off_xsc)[t] = 0u;
        fence_barrier_init();
    }
    // XBF: the stages hold only the T real token rows; lanes of absent
    // tokens read this zero row instead.
    if (XBF && threadIdx.x < 16)
        reinterpret_cast<uint4 *>(smem + p.off_xzero)[threadIdx.x] = make_uint4(0u, 0u, 0u, 0u);
    __syncthreads();
    pdl_launch_dependents();

    if (warp == PRODUCER_WARP) {
        // ============================================================ producer
        const uint64_t pol_w = policy_evict_first();
        const uint64_t pol_x = policy_evict_last();
        if (lane == 0) {
            prefetch_tmap(&tmW);
            if (XBF) prefetch_tmap(&tmX);
        }
        int s = 0, issued = 0, tile = tile_first, grp = grp_first, rem = n_units;
        uint32_t ph = 0;
        bool waited = false;
        if (GATHER && !p.map_static) {
            pdl_wait_prior();       // the id list may come from the previous kernel
            waited = true;
        }
        // gathered rows: ids of this lane's two rows, for this tile and the next
        int gid[2] = {-1, -1}, gid_next[2] = {-1, -1};
        int grows[4] = {0, 0, 0, 0};    // lanes 0..15: rows 4*lane .. 4*lane+3 (gather box `lane`)
        int grows_tile = -1;
        if (GATHER) {
            gid[0] = row_id(p, tile, lane);
            gid[1] = row_id(p, tile, lane + 32);
            if (tile + 1 <= tile_last) {
                gid_next[0] = row_id(p, tile + 1, lane);
                gid_next[1] = row_id(p, tile + 1, lane + 32);
            }
        }
        while (rem > 0) {
            const int n = min(min(C::GPS, G - grp), rem);
            if (issued >= nst) wait_or_flag(p, flag, smem_addr(&empty[s]), ph ^ 1u);
            const uint32_t fb = smem_addr(&full[s]);
            const uint32_t stage = smem_addr(smem) + static_cast<uint32_t>(s * p.stage_bytes);
            // gathered rows: 16 boxes of 4 full rows (GPS groups, zeros for
            // absent rows and past the end of K)
            const uint32_t wbytes = GATHER ? static_cast<uint32_t>(ROWS * C::GROW) : static_cast<uint32_t>(n * ROWS * 64);
            const uint32_t xbytes = XRES  ? 0u
                                    : XBF ? static_cast<uint32_t>(n * T * XROW_BYTES)
                                          : static_cast<uint32_t>(n * p.xslot_bytes);
            if (lane == 0) mbar_arrive_expect_tx(fb, wbytes + xbytes);
            __syncwarp();
            if (GATHER) {
                // Rows at scattered addresses: lane b (< 16) loads rows
                // 4b .. 4b+3 with one four-row gather.  Absent rows get an
                // out-of-range row index and read zeros (their scale is 0
                // as well).
                if (grows_tile != tile) {
#pragma unroll
                    for (int t = 0; t < 4; ++t) {
                        const int src = (4 * lane + t) & 31;
                        const int v0 = __shfl_sync(0xFFFFFFFFu, gid[0], src);
                        const int v1 = __shfl_sync(0xFFFFFFFFu, gid[1], src);
                        const int id = (lane & 8) ? v1 : v0;       // rows >= 32 for lanes 8..15
                        grows[t] = id >= 0 ? id : p.V;
                    }
                    grows_tile = tile;
                }
                if (lane < 16)
                    tma_gather4(stage + lane * 4 * C::GROW, &tmW, grp * 16, grows[0], grows[1], grows[2], grows[3], fb,
                                pol_w);
            } else if (lane < n) {
                tma_load_2d(stage + lane * (ROWS * 64), &tmW, (grp + lane) * 16, tile * ROWS, fb, pol_w);
            }
            if (!XRES && !waited) {
                pdl_wait_prior();   // activations may come from the previous kernel
                waited = true;
            }
            if (XBF && lane >= 16 && lane - 16 < n)
                tma_load_2d(stage + C::W_BYTES + (lane - 16) * p.xslot_bytes, &tmX, (grp + lane - 16) * 128, 0, fb,
                            pol_x);
            if (XPREP && lane >= 16 && lane - 16 < n)
                bulk_g2s(stage + C::W_BYTES + (lane - 16) * p.xslot_bytes,
                         p.x16 + static_cast<size_t>(grp + lane - 16) * p.xslot_bytes,
                         static_cast<uint32_t>(p.xslot_bytes), fb, pol_x);
            rem -= n;
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
                *flag = 1;
                atomicOr(p.err, 2);
            }
        }
        return;
    }

    if (warp == EPILOGUE_WARP) {
        // ============================================================ epilogue
        if (GATHER && !p.map_static) pdl_wait_prior();   // the id list may come from the previous kernel
        stage_tile_meta<HEAD, GATHER>(p, tile_first, sbuf, idbuf, smem_addr(&meta_full[0]), lane);
        if (tile_first + 1 <= tile_last)
            stage_tile_meta<HEAD, GATHER>(p, tile_first + 1, sbuf + p.sbuf_bytes, idbuf + ROWS,
                                          smem_addr(&meta_full[1]), lane);
        // HEAD: bk[lane][t] = best key of token t over the rows this lane has
        // seen; reduced across lanes once, at the end.
        unsigned long long *bk = reinterpret_cast<unsigned long long *>(smem + p.off_bk) + lane * BK_STRIDE;
        if (HEAD)
            for (int t = 0; t < T; ++t) bk[t] = 0ull;

        // Contributors of the only tiles that can be split, the first and
        // the last: CTAs bf .. bf+nc-1, and whether the tile is bf's first
        // tile (its partial then sits in slot 0).  Worked out once here
        // (64-bit divisions) instead of at the end of the run.
        int bfA = b, ncA = 1, bfZ = b, ncZ = 1;
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
        pdl_wait_prior();                  // scratch area, outputs and drafts from here on
        if (p.stall_ns != 0u && b == 0) wait_or_flag_for(p, flag, smem_addr(stall_bar), 0u, p.stall_ns);
        for (int k = 0, tile = tile_first; tile <= tile_last; ++k, ++tile) {
            const int kb = k & 1;
            const bool first = tile == tile_first;
            const int tbf = first ? bfA : bfZ, tnc = first ? ncA : ncZ;
            // The tile this CTA finishes (its own part is the end of its
            // range): while the consumers are still on it, poll the tile's
            // counter and, once the other contributors are all in, copy their
            // partials to shared memory, so that the end of the kernel only
            // adds and stores.  Polling stops when this CTA's own sums are
            // ready; the finish below then waits and loads the rest itself.
            int npre = 0;
            const long long ts = static_cast<long long>(tile) * G, te = ts + G;
            const bool split = !(u0 <= ts && u1 >= te);
            if (NT == 1 && tile == tile_last && split && tbf == b && tnc > 1 && tnc - 1 <= PRE_PARTS) {
                const uint64_t t0 = global_timer_ns();
                while (true) {
                    if (__all_sync(0xFFFFFFFFu, ld_acquire_gpu_u32(&p.ctr[b]) == static_cast<unsigned>(tnc - 1))) {
                        npre = tnc - 1;
                        break;
                    }
                    if (mbar_try_wait(smem_addr(red_full), static_cast<uint32_t>(k & 1))) break;
                    if (global_timer_ns() - t0 > WAIT_LIMIT_NS) break;
                    __nanosleep(256);
                }
                float *dst = reinterpret_cast<float *>(smem + p.off_pre);
                for (int j = 0; j < npre; ++j) {
                    const float *src = p.part + static_cast<size_t>(b + 1 + j) * 2 * PART_FLOATS;
#pragma unroll
                    for (int h = 0; h < 2; ++h)
#pragma unroll
                        for (int q = 0; q < 2; ++q)
                            if (4 * q < T)
                                *reinterpret_cast<float4 *>(dst + (j * ROWS + lane + 32 * h) * 8 + 4 * q) =
                                    ldcg_f4(src + (lane + 32 * h) * TMAX + 4 * q);
                }
            }
            wait_or_flag(p, flag, smem_addr(red_full), static_cast<uint32_t>(k & 1));
            const bool complete = !split;
            // This CTA's sums of the group slots (fixed slot order) for rows
            // lane and lane+32 of every token, kept as v[t][h] in registers
            // for the tokens being processed (chunks of 4).
            // Split tiles: the tile's contributors are CTAs bf..bf+nc-1, and
            // bf finishes the tile.  bf's part is the end of its range, so it
            // comes to the tile last of its work; the others' parts are the
            // start of their ranges (or all of them), done early.  The others
            // publish their partials in the scratch area as [row][TMAX]
            // floats and count themselves in with a release add they do not
            // wait for; bf waits (acquire loads, bounded) until all nc - 1
            // are in, adds the contributions in CTA order -- its own from
            // shared memory, the others' with vectorised loads issued
            // together -- and resets the counter for the next launch.
            int bf = 0, nc = 1, me = 0;
            bool finish = true;
            const float *others[4] = {nullptr, nullptr, nullptr, nullptr};
            if (!complete) {
                bf = tbf;
                nc = tnc;
                me = b - bf;
                finish = me == 0;
                if (!finish) {
                    float *mine = p.part + (static_cast<size_t>(b) * 2 + (tile == tile_first ? 0 : 1)) * PART_FLOATS;
                    for (int t0 = 0; t0 < T; t0 += 4) {
#pragma unroll
                        for (int h = 0; h < 2; ++h) {
                            const int row = lane + 32 * h;
                            *reinterpret_cast<float4 *>(mine + row * TMAX + t0) = slot_sums4<NT, C::GPS>(red, t0, row, T);
                        }
                    }
                    __syncwarp();
                    if (lane == 0) red_add_release_gpu(&p.ctr[bf], 1u);
                } else if (npre == 0) {
                    const uint64_t t0 = global_timer_ns();
                    while (!__all_sync(0xFFFFFFFFu, ld_acquire_gpu_u32(&p.ctr[bf]) == static_cast<unsigned>(nc - 1))) {
                        if (global_timer_ns() - t0 > (*flag ? WAIT_LIMIT_AFTER_ERR_NS : WAIT_LIMIT_NS)) {
                            *flag = 1;
                            if (lane == 0) atomicOr(p.err, 2);
                            break;
                        }
                    }
                }
                if (finish) {
                    if (lane == 0) p.ctr[bf] = 0u;        // ready for the next launch
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        // partial slot 0 holds a CTA's first tile: every later
                        // contributor starts inside this tile; bf does when its
                        // range starts exactly at the tile
                        const int wb2 = (j > 0 || (first ? bf_firstA : u0 == ts)) ? 0 : 1;
                        others[j] = p.part + (static_cast<size_t>(bf + j) * 2 + wb2) * PART_FLOATS;
                    }
                }
            }
            const int32_t *ids = idbuf + kb * ROWS;
            const int id0 = HEAD ? ids[lane] : 0, id1 = HEAD ? ids[lane + 32] : 0;
            for (int t0 = 0; t0 < T && finish; t0 += 4) {
                float v[4][2];
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int row = lane + 32 * h;
                    const float4 o4 = slot_sums4<NT, C::GPS>(red, t0, row, T);
                    const float own[4] = {o4.x, o4.y, o4.z, o4.w};
                    if (complete) {
#pragma unroll
                        for (int j = 0; j < 4; ++j) v[j][h] = own[j];
                    } else {
                        // contributions in CTA order (the loads are independent of
                        // the sum, so they are all in flight together)
                        const float4 mine4 = make_float4(own[0], own[1], own[2], own[3]);
                        float4 acc4 = mine4;
#pragma unroll
                        for (int j = 0; j < 4; ++j)
                            if (j < nc) {
                                const float4 e = j == me ? mine4
                                                 : (NT == 1 && npre > 0) ? *reinterpret_cast<const float4 *>(
                                                       reinterpret_cast<const float *>(smem + p.off_pre) +
                                                       ((j - 1) * ROWS + row) * 8 + t0)
                                                 : ldcg_f4(others[j] + row * TMAX + t0);
                                if (j == 0) {
                                    acc4 = e;
                                } else {
                                    acc4.x += e.x;
                                    acc4.y += e.y;
                                    acc4.z += e.z;
                                    acc4.w += e.w;
                                }
                            }
                        for (int j = 4; j < nc; ++j) {      // more than 4 CTAs on one tile (small K)
                            float4 e = mine4;
                            if (j != me) {
                                const int bb = bf + j;
                                const int wb2 = (cta_start(bb, U, B) >= ts) ? 0 : 1;
                                e = ldcg_f4(p.part + (static_cast<size_t>(bb) * 2 + wb2) * PART_FLOATS + row * TMAX + t0);
                            }
                            acc4.x += e.x;
                            acc4.y += e.y;
                            acc4.z += e.z;
                            acc4.w += e.w;
                        }
                        v[0][h] = acc4.x;
                        v[1][h] = acc4.y;
                        v[2][h] = acc4.z;
                        v[3][h] = acc4.w;
                    }
                }
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int t = t0 + j;
                    if (t >= T) break;
                    if constexpr (!HEAD) {
#pragma unroll
                        for (int h = 0; h < 2; ++h) {
                            const long long rg = static_cast<long long>(tile) * ROWS + lane + 32 * h;
                            if (rg < p.n_rows) {
                                if (p.y32)
                                    p.y32[static_cast<size_t>(t) * p.n_rows + rg] = v[j][h];
                                else
                                    p.y[static_cast<size_t>(t) * p.n_rows + rg] =
                                        __bfloat16_as_ushort(__float2bfloat16_rn(v[j][h]));
                            }
                        }
                    } else {
                        const unsigned long long k0 = id0 >= 0 ? make_key(v[j][0], static_cast<uint32_t>(id0)) : 0ull;
                        const unsigned long long k1 = id1 >= 0 ? make_key(v[j][1], static_cast<uint32_t>(id1)) : 0ull;
                        const unsigned long long kk = k0 > k1 ? k0 : k1;
                        if (kk > bk[t]) bk[t] = kk;
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_addr(red_empty));     // red may be overwritten
            // Metadata of tile k+2 goes into the buffers tile k used.
            if (tile + 2 <= tile_last) {
                wait_or_flag(p, flag, smem_addr(&meta_empty[kb]), static_cast<uint32_t>((k >> 1) & 1));
                stage_tile_meta<HEAD, GATHER>(p, tile + 2, sbuf + kb * p.sbuf_bytes, idbuf + kb * ROWS,
                                              smem_addr(&meta_full[kb]), lane);
            }
        }
        if constexpr (HEAD) {
            // ================================================ grid argmax + verify
            __syncwarp();
            unsigned long long best = 0ull;    // lane t: best key of token t in this CTA
            if (lane < T) {
                const unsigned long long *col = reinterpret_cast<const unsigned long long *>(smem + p.off_bk) + lane;
                for (int l = 0; l < 32; ++l) {
                    const unsigned long long v = col[l * BK_STRIDE];
                    best = v > best ? v : best;
                }
            }
            head_grid_tail(p, best, lane, B);
        }
        return;
    }

    // ================================================================ consumers
    const int cw = warp;
    const int slot = cw % C::GPS;
    const int mset = cw / C::GPS;
    const int g = lane >> 2, c = lane & 3;

    // Lane-constant shared-memory offsets (within a stage / a scale buffer).
    constexpr int RSTEP = GATHER ? 16 * C::GROW : 16 * 64;   // next m16 tile
    constexpr int HSTEP = GATHER ? 8 * C::GROW : 8 * 64;     // row g + 8
    const int row0 = mset * C::R * 16 + g;                     // first row of this lane
    const uint32_t w_lane = GATHER ? static_cast<uint32_t>(row0 * C::GROW + slot * 64 + c * 16)
                                   : static_cast<uint32_t>(slot * (ROWS * 64) + row0 * 64 + c * 16);
    const uint32_t x_lane = XBF ? static_cast<uint32_t>(C::W_BYTES + slot * p.xslot_bytes + g * XROW_BYTES + c * 64)
                                : static_cast<uint32_t>(C::W_BYTES + slot * p.xslot_bytes + g * XSTR + c * 64);
    const uint32_t s_lane = static_cast<uint32_t>(row0 * G * 2);
    const uint32_t xzero_lane = smem_addr(smem + p.off_xzero) + static_cast<uint32_t>(c * 64);
    const uint32_t sbuf0 = smem_addr(sbuf);
    const uint32_t smem0 = smem_addr(smem);

    // Activations reach the B loads as rows of 16-byte chunks, each chunk
    // holding its 8 values in B-fragment order (x0,x4, x1,x5, x2,x6, x3,x7),
    // chunk index XOR-swizzled (chunk_slot) and rows padded to 16 (mod 128)
    // bytes, so that the B loads are conflict-free and need no byte permutes:
    // resident in shared memory for the whole kernel (XRES; row T is zeros,
    // read by the lanes of absent tokens), or as ready-made group blocks
    // copied into each stage (xprep_kernel; rows T..TP-1 are zeros).
    //
    // The rows are fp16, not bf16: row t holds x[t] * 2^s_t, with
    // s_t chosen so that the row's largest magnitude lands in [2^14, 2^15).
    // A bf16 value has 8 significant bits and fp16 11, so every element of
    // magnitude >= 2^-32 of the row maximum converts exactly (smaller ones
    // round to fp16 subnormals, an error below 2^-40 of the row maximum);
    // fp16 weights then dequantise with one shift per word instead of three
    // (dequant2_f16_lo/hi).  Products are exact in the fp32 accumulators and
    // a power-of-two scale commutes with fp32 rounding, so multiplying each
    // token's sums by 2^-s_t at the end of a tile gives exactly the sums of
    // the unscaled bf16 products.
    // chunk_slot(4c + m) * 16 = 64c + ((16m) ^ xsw): the m-dependent part is
    // a compile-time offset XOR one lane constant
    const uint32_t xsw = static_cast<uint32_t>((c & 2) * 16);
    uint32_t xr_lane = 0;
    // 2^-s of tokens 2c and 2c+1 (resident rows; streamed rows read
    // p.xinv at the end of each tile instead of holding 2*NT registers)
    float xinv[2] = {1.f, 1.f};
    if constexpr (XPREP) {
        pdl_wait_prior();              // p.xinv comes from the conversion kernel
    } else if constexpr (XRES) {
        pdl_wait_prior();                  // activations may come from the previous kernel
        // Token-major: the warps of token tt (wpt of them) load its row,
        // XB 16-byte chunks per thread in flight at once, and reduce the
        // row's largest |x| (bf16 bits) into xmax[tt]; after a barrier every
        // thread converts the chunks it holds to fp16 and stores them in
        // B-fragment order.  Rows longer than XB chunks per thread take two
        // passes over global memory (maximum, then conversion).
        uint8_t *xr = smem + p.off_xres;
        unsigned *xmax = reinterpret_cast<unsigned *>(smem + p.off_xsc);
        const int cpr = p.K / 8;                       // chunks per row
        const int wpt = NCW / T;                       // warps per token (T <= 8)
        const int tt = cw / wpt;                       // this warp's token
        const int nthr = wpt * 32;
        const int j0 = (cw - tt * wpt) * 32 + lane;
        const bool loader = tt < T;
        const uint4 *xrow = reinterpret_cast<const uint4 *>(p.x) + static_cast<size_t>(loader ? tt : 0) * cpr;
        uint8_t *xdst = xr + static_cast<size_t>(tt) * p.xres_stride;
        constexpr int XB = 10;
        const bool one_batch = cpr <= XB * nthr;
        uint4 r[XB];
        unsigned mx = 0u;
        for (int jb = j0; jb < cpr; jb += XB * nthr) {
#pragma unroll
            for (int u = 0; u < XB; ++u) {
                const int j = jb + u * nthr;
                r[u] = (loader && j < cpr) ? xrow[j] : make_uint4(0u, 0u, 0u, 0u);
            }
#pragma unroll
            for (int u = 0; u < XB; ++u) mx = max(mx, chunk_absmax(r[u]));
            if (one_batch) break;
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) mx = max(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, o));
        if (loader && lane == 0 && mx != 0u) atomicMax(&xmax[tt], mx);
        // row T: zeros, read by the lanes of absent tokens
        for (int i = cw * 32 + lane; i < cpr; i += NCW * 32)
            sts128(smem_addr(xr + static_cast<size_t>(T) * p.xres_stride + i * 16), make_uint4(0u, 0u, 0u, 0u));
        named_bar_sync(1, NCW * 32);
        if (loader) {
            const float sc = __uint_as_float(static_cast<uint32_t>(127 + xres_shift(xmax[tt])) << 23);
            for (int jb = j0; jb < cpr; jb += XB * nthr) {
                if (!one_batch) {
#pragma unroll
                    for (int u = 0; u < XB; ++u) {
                        const int j = jb + u * nthr;
                        r[u] = j < cpr ? xrow[j] : make_uint4(0u, 0u, 0u, 0u);
                    }
                }
#pragma unroll
                for (int u = 0; u < XB; ++u) {
                    const int j = jb + u * nthr;
                    if (j < cpr) sts128(smem_addr(xdst + ((j & ~15) + chunk_slot(j & 15)) * 16), chunk_to_f16(r[u], sc));
                }
            }
        }
        named_bar_sync(1, NCW * 32);
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const int tok = 2 * c + e;
            xinv[e] = tok < T ? __uint_as_float(static_cast<uint32_t>(127 - xres_shift(xmax[tok])) << 23) : 1.f;
        }
        xr_lane = smem_addr(xr) + static_cast<uint32_t>((g < T ? g : T) * p.xres_stride + c * 64);
    }

    float acc[C::R][NT][4];
#pragma unroll
    for (int r = 0; r < C::R; ++r)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[r][nt][e] = 0.f;
    // FMA: this lane's partial sums over its 32 columns of each group, for
    // rows g (h = 0) and g + 8 (h = 1) of each m16 tile and all 8 tokens
    float accf[FMA ? C::R : 1][2][8];
    if constexpr (FMA) {
#pragma unroll
        for (int r = 0; r < C::R; ++r)
#pragma unroll
            for (int h = 0; h < 2; ++h)
#pragma unroll
                for (int t = 0; t < 8; ++t) accf[r][h][t] = 0.f;
    }
    const uint32_t xr0 = XRES ? smem_addr(smem + p.off_xres) + static_cast<uint32_t>(c * 64) : 0u;

    int s = 0, grp = grp_first, rem = n_units, k = 0;
    uint32_t ph = 0;
    bool tile_start = true;
    while (rem > 0) {
        const int n = min(min(C::GPS, G - grp), rem);
        const int kb = k & 1;
        if (tile_start) {
            wait_or_flag(p, flag, smem_addr(&meta_full[kb]), static_cast<uint32_t>((k >> 1) & 1));
            tile_start = false;
        }
        wait_or_flag(p, flag, smem_addr(&full[s]), ph);
        if (slot < n) {
            const int gs = grp + slot;     // group within the row
            const uint32_t stage = smem0 + static_cast<uint32_t>(s * p.stage_bytes);
            const uint32_t wbase = stage + w_lane;
          if constexpr (FMA) {
            // Each lane dots its 32 columns (chunk c of the group) of rows g
            // and g + 8 of its m16 tiles with every token's resident row:
            // the levels (fp16, pairs (j, j+4) as the dequant yields them)
            // times the activations (fp16, stored in the same pairing), one
            // fp32-accumulating fma per weight and token.
            const uint32_t sbf = sbuf0 + kb * p.sbuf_bytes + s_lane + gs * 2;
#pragma unroll
            for (int r = 0; r < C::R; ++r) {
                const uint4 wa = lds128(wbase + r * RSTEP);
                const uint4 wb = lds128(wbase + r * RSTEP + HSTEP);
                float fs[2][8];
#pragma unroll
                for (int h = 0; h < 2; ++h)
#pragma unroll
                    for (int t = 0; t < 8; ++t) fs[h][t] = 0.f;
#pragma unroll
                for (int m = 0; m < 4; ++m) {
                    uint32_t lv[2][4];
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const uint4 &w4 = h ? wb : wa;
                        const uint32_t w = (m == 0) ? w4.x : (m == 1) ? w4.y : (m == 2) ? w4.z : w4.w;
                        lv[h][0] = dequant2_f16_lo(w);         // nibbles (0, 4)
                        lv[h][1] = dequant2_f16_hi(w);         // (1, 5)
                        lv[h][2] = dequant2_f16_lo(w >> 8);    // (2, 6)
                        lv[h][3] = dequant2_f16_hi(w >> 8);    // (3, 7)
                    }
#pragma unroll
                    for (int t = 0; t < 8; ++t) {
                        if (t >= T) break;
                        const uint4 v = lds128(xr0 + static_cast<uint32_t>(t * p.xres_stride + gs * 256) +
                                               ((16u * m) ^ xsw));
#pragma unroll
                        for (int h = 0; h < 2; ++h) {
                            float a = fs[h][t];
                            a = fma2_f16_f32(lv[h][0], v.x, a);
                            a = fma2_f16_f32(lv[h][1], v.y, a);
                            a = fma2_f16_f32(lv[h][2], v.z, a);
                            a = fma2_f16_f32(lv[h][3], v.w, a);
                            fs[h][t] = a;
                        }
                    }
                }
                const float s0 = bf16_bits_to_float(lds_u16(sbf + r * 16 * G * 2));
                const float s1 = bf16_bits_to_float(lds_u16(sbf + (r * 16 + 8) * G * 2));
#pragma unroll
                for (int t = 0; t < 8; ++t) {
                    accf[r][0][t] += s0 * fs[0][t];
                    accf[r][1][t] += s1 * fs[1][t];
                }
            }
          } else {
            uint4 wa[C::R], wb[C::R];
#pragma unroll
            for (int r = 0; r < C::R; ++r) {
                wa[r] = lds128(wbase + r * RSTEP);
                wb[r] = lds128(wbase + r * RSTEP + HSTEP);
            }
            float gacc[C::R][NT][4];     // first k-step writes, later ones accumulate

            const uint32_t xbase = XRES ? xr_lane + gs * 256
                                   : (XBF && g >= T) ? xzero_lane
                                                     : stage + x_lane;
#pragma unroll
            for (int m = 0; m < 4; ++m) {
                // B fragments: token (nt*8 + g), the 8 activations of word
                // (4c + m) of the group, paired (j, j+4) like the nibbles.
                // Token rows >= T are zeros.
                uint32_t bx[NT][4];
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    if constexpr (XBF) {
                        const uint4 v = lds128(xbase + m * 16);
                        bx[nt][0] = __byte_perm(v.x, v.z, 0x5410);   // (x0, x4)
                        bx[nt][1] = __byte_perm(v.x, v.z, 0x7632);   // (x1, x5)
                        bx[nt][2] = __byte_perm(v.y, v.w, 0x5410);   // (x2, x6)
                        bx[nt][3] = __byte_perm(v.y, v.w, 0x7632);   // (x3, x7)
                    } else {
                        const uint4 v = lds128(xbase + (XRES ? 0 : nt * 8 * XSTR) + ((16u * m) ^ xsw));
                        bx[nt][0] = v.x;
                        bx[nt][1] = v.y;
                        bx[nt][2] = v.z;
                        bx[nt][3] = v.w;
                    }
                }
#pragma unroll
                for (int r = 0; r < C::R; ++r) {
                    const uint32_t wA = (m == 0) ? wa[r].x : (m == 1) ? wa[r].y : (m == 2) ? wa[r].z : wa[r].w;
                    const uint32_t wB = (m == 0) ? wb[r].x : (m == 1) ? wb[r].y : (m == 2) ? wb[r].z : wb[r].w;
                    if constexpr (XBF) {
                        // bf16 activations: bf16 levels, three shifts per word
                        uint32_t a0 = dequant2(wA), a1 = dequant2(wB);
                        uint32_t a2 = dequant2(wA >> 4), a3 = dequant2(wB >> 4);
                        if (m == 0)
                            mma_bf16_16816_zc(gacc[r][0], a0, a1, a2, a3, bx[0][0], bx[0][1]);
                        else
                            mma_bf16_16816(gacc[r][0], a0, a1, a2, a3, bx[0][0], bx[0][1]);
                        a0 = dequant2(wA >> 8);
                        a1 = dequant2(wB >> 8);
                        a2 = dequant2(wA >> 12);
                        a3 = dequant2(wB >> 12);
                        mma_bf16_16816(gacc[r][0], a0, a1, a2, a3, bx[0][2], bx[0][3]);
                        continue;
                    }
                    // k-step 2m: nibble pairs (0,4) and (1,5); k-step 2m+1:
                    // pairs (2,6) and (3,7) of the word >> 8
                    uint32_t a0 = dequant2_f16_lo(wA), a1 = dequant2_f16_lo(wB);
                    uint32_t a2 = dequant2_f16_hi(wA), a3 = dequant2_f16_hi(wB);
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt) {
                        if (m == 0)
                            mma_f16_16816_zc(gacc[r][nt], a0, a1, a2, a3, bx[nt][0], bx[nt][1]);
                        else
                            mma_f16_16816(gacc[r][nt], a0, a1, a2, a3, bx[nt][0], bx[nt][1]);
                    }
                    const uint32_t wA8 = wA >> 8, wB8 = wB >> 8;
                    a0 = dequant2_f16_lo(wA8);
                    a1 = dequant2_f16_lo(wB8);
                    a2 = dequant2_f16_hi(wA8);
                    a3 = dequant2_f16_hi(wB8);
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt)
                        mma_f16_16816(gacc[r][nt], a0, a1, a2, a3, bx[nt][2], bx[nt][3]);
                }
            }
            // group scales of this lane's rows (staged in shared memory)
            const uint32_t sb = sbuf0 + kb * p.sbuf_bytes + s_lane + gs * 2;
#pragma unroll
            for (int r = 0; r < C::R; ++r) {
                const float s0 = bf16_bits_to_float(lds_u16(sb + r * 16 * G * 2));
                const float s1 = bf16_bits_to_float(lds_u16(sb + (r * 16 + 8) * G * 2));
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    acc[r][nt][0] += s0 * gacc[r][nt][0];
                    acc[r][nt][1] += s0 * gacc[r][nt][1];
                    acc[r][nt][2] += s1 * gacc[r][nt][2];
                    acc[r][nt][3] += s1 * gacc[r][nt][3];
                }
            }
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_addr(&empty[s]));
        if (++s == nst) { s = 0; ph ^= 1u; }
        rem -= n;
        grp += n;

        if (grp == G || rem == 0) {
            // End of this CTA's share of a tile: hand the partial sums over.
            if (lane == 0) mbar_arrive(smem_addr(&meta_empty[kb]));   // scales no longer read
            if constexpr (FMA) {
                // the four lanes of a row hold its four 32-column parts:
                // add them (xor 1, 2), then keep tokens 2c, 2c+1 in the
                // fragment layout the hand-off below expects
#pragma unroll
                for (int r = 0; r < C::R; ++r)
#pragma unroll
                    for (int h = 0; h < 2; ++h)
#pragma unroll
                        for (int t = 0; t < 8; ++t) {
                            float v = accf[r][h][t];
                            v += __shfl_xor_sync(0xFFFFFFFFu, v, 1);
                            v += __shfl_xor_sync(0xFFFFFFFFu, v, 2);
                            accf[r][h][t] = v;
                        }
#pragma unroll
                for (int r = 0; r < C::R; ++r) {
#pragma unroll
                    for (int h = 0; h < 2; ++h)
#pragma unroll
                        for (int e = 0; e < 2; ++e) {
                            float v = 0.f;
#pragma unroll
                            for (int cc = 0; cc < 4; ++cc)
                                if (c == cc) v = accf[r][h][2 * cc + e];
                            acc[r][0][2 * h + e] = v;
                        }
#pragma unroll
                    for (int h = 0; h < 2; ++h)
#pragma unroll
                        for (int t = 0; t < 8; ++t) accf[r][h][t] = 0.f;
                }
            }
            wait_or_flag(p, flag, smem_addr(red_empty), static_cast<uint32_t>((k & 1) ^ 1));
#pragma unroll
            for (int r = 0; r < C::R; ++r)
#pragma unroll
                for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                    for (int hh = 0; hh < 2; ++hh) {
                        // tokens 2c and 2c+1 of row g (+8): elements 2hh, 2hh+1
                        const int row = (mset * C::R + r) * 16 + g + 8 * hh;
                        const int tok = nt * 8 + 2 * c;
                        float v0 = acc[r][nt][2 * hh], v1 = acc[r][nt][2 * hh + 1];
                        if constexpr (XRES) {
                            v0 *= xinv[0];
                            v1 *= xinv[1];
                        } else if constexpr (!XBF) {
                            v0 *= __ldg(p.xinv + tok);
                            v1 *= __ldg(p.xinv + tok + 1);
                        }
                        *reinterpret_cast<float2 *>(red + red_index<NT, C::GPS>(slot, tok, row)) = make_float2(v0, v1);
                        acc[r][nt][2 * hh] = 0.f;
                        acc[r][nt][2 * hh + 1] = 0.f;
                    }
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_addr(red_full));
            ++k;
            grp = 0;
            tile_start = true;
        }
    }
}

}  // namespace sv
