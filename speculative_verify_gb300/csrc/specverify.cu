// specverify.cu -- the C ABI declared in include/specverify.h: argument
// checks, the per-device scratch area, launch configuration and dispatch to
// the sm_103a stream kernel (w4a16_stream.cuh).
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cstdint>
#include <cstdio>
#include <cstring>
#include <atomic>
#include <mutex>

#include "draft_list.cuh"
#include "hbm_read.cuh"
#include "rescore.cuh"
#include "specverify.h"
#include "w4a16_stream.cuh"
#include "w4a16_wide.cuh"
#include "w4a16_tc.cuh"

namespace sv {
namespace {

constexpr int MAX_DEVICES = 64;

// Room left for rescore_kernel's static shared memory under the opt-in limit.
constexpr int RS_STATIC_SMEM_SLACK = 10240;
constexpr size_t RS_SCRATCH_BYTES = static_cast<size_t>(RS_TMAX) * RS_KMAX * 8 + 256;

struct DeviceState {
    bool ready = false;
    int sms = 0;
    int smem_optin = 0;
    float *part = nullptr;
    float *wpart = nullptr;     // split-tile partials of the wide kernel, [sms][2][WIDE_PART_FLOATS]
    unsigned *ctr = nullptr;
    unsigned long long *keys = nullptr;
    unsigned *done = nullptr;
    int *err = nullptr;
    uint8_t *x16 = nullptr;     // streamed activations, X16_MAX_GROUPS x TMAX x XSTR bytes
    float *xinv = nullptr;      // [TMAX]
    int x16_max_groups = 0;
    // rescoring (rescore.cuh); the logits and candidate buffers grow on demand
    float *cand_lg = nullptr;             // [RS_TMAX][RS_KMAX] rescored logits
    int32_t *cand_id = nullptr;           // [RS_TMAX][RS_KMAX] their ids
    unsigned *rdone = nullptr;            // rescore_kernel's CTA counter, left at 0
    unsigned *sdone = nullptr;            // sample_kernel's CTA counter, left at 0
    int32_t *row_acc = nullptr;           // [RS_TMAX] per-row accept flags of the sampled verify
    int32_t *row_tok = nullptr;           // [RS_TMAX] per-row drawn tokens
    float *rs_logits = nullptr;           // [RS_TMAX][rs_v_cap]
    unsigned long long *rs_smax = nullptr;   // [RS_TMAX][rs_s_cap] slice maxima
    long long rs_v_cap = 0, rs_s_cap = 0;
    // When set, every launch first clears these bytes on its stream (the
    // allocation-free verify, whose counters are not guaranteed to be zero).
    void *clear_ptr = nullptr;
    size_t clear_bytes = 0;
};

// Activations of calls with more than one token tile (T > 8) are converted
// into a per-device buffer sized for K <= 128 * X16_MAX_GROUPS.
constexpr int X16_MAX_GROUPS = 1024;

DeviceState g_state[MAX_DEVICES];
std::mutex g_mu;
std::atomic<uint32_t> g_stall_ns{0};    // sv_debug_set_wait_stall
std::atomic<int> g_fma_consumers{0};     // sv_debug_set_fma_consumers
std::atomic<int> g_tcgen05{1};           // sv_debug_set_tcgen05

template <int NT, bool HEAD, bool GATHER, bool XRES, bool FMA = false>
cudaError_t raise_smem_limit(int bytes)
{
    return cudaFuncSetAttribute(w4a16_stream_kernel<NT, HEAD, GATHER, XRES, FMA>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
}

template <int NT, bool HEAD, int NCW>
cudaError_t raise_smem_limit_wide(int bytes)
{
    return cudaFuncSetAttribute(w4a16_wide_kernel<NT, HEAD, NCW>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                bytes);
}

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

int tensor_map_fn()
{
    if (g_encode) return SV_OK;
    void *fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess || !fn)
        return SV_ERR_CUDA;
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    return SV_OK;
}

// 2-D row-major tensor [rows][cols] of `esize`-byte elements; box = bc x br.
int encode_2d(CUtensorMap *m, CUtensorMapDataType dt, int esize, const void *base,
              unsigned long long cols, unsigned long long rows, unsigned bc, unsigned br,
              CUtensorMapSwizzle sw = CU_TENSOR_MAP_SWIZZLE_NONE)
{
    const cuuint64_t dims[2] = {cols, rows};
    const cuuint64_t strides[1] = {cols * static_cast<unsigned long long>(esize)};
    const cuuint32_t box[2] = {bc, br};
    const cuuint32_t estr[2] = {1, 1};
    CUresult r = g_encode(m, dt, 2, const_cast<void *>(base), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? SV_OK : SV_ERR_CUDA;
}

// Scratch layout (one cudaMalloc): part [sms][2][PART_FLOATS] fp32, then
// ctr [sms], keys [TMAX], done, err.  All counters start (and are left) at 0.
int device_state(DeviceState **out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return SV_ERR_CUDA;
    if (dev < 0 || dev >= MAX_DEVICES) return SV_ERR_DEVICE;
    std::lock_guard<std::mutex> lock(g_mu);
    DeviceState &st = g_state[dev];
    if (!st.ready) {
        cudaDeviceProp prop;
        if (cudaGetDeviceProperties(&prop, dev) != cudaSuccess) return SV_ERR_CUDA;
        if (prop.major != 10) return SV_ERR_DEVICE;
        int optin = 0;
        if (cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
            return SV_ERR_CUDA;
        const size_t part_bytes = static_cast<size_t>(prop.multiProcessorCount) * 2 * PART_FLOATS * sizeof(float);
        const size_t ctr_bytes = static_cast<size_t>(prop.multiProcessorCount) * sizeof(unsigned);
        const size_t keys_bytes = TMAX * sizeof(unsigned long long);
        const size_t x16_bytes = static_cast<size_t>(X16_MAX_GROUPS) * TMAX * XSTR;
        const size_t wpart_bytes = static_cast<size_t>(prop.multiProcessorCount) * 2 * WIDE_PART_FLOATS * sizeof(float);
        const size_t total = part_bytes + ctr_bytes + keys_bytes + 2 * sizeof(unsigned) + 256 + x16_bytes +
                             TMAX * sizeof(float) + 256 + RS_SCRATCH_BYTES + 256 + wpart_bytes;
        uint8_t *base = nullptr;
        if (cudaMalloc(&base, total) != cudaSuccess) {
            cudaGetLastError();
            return SV_ERR_NOMEM;
        }
        if (cudaMemset(base, 0, total) != cudaSuccess) {
            cudaFree(base);
            return SV_ERR_CUDA;
        }
        size_t off = 0;
        st.part = reinterpret_cast<float *>(base + off);
        off += part_bytes;
        off = (off + 255) & ~static_cast<size_t>(255);
        st.keys = reinterpret_cast<unsigned long long *>(base + off);
        off += keys_bytes;
        st.ctr = reinterpret_cast<unsigned *>(base + off);
        off += ctr_bytes;
        st.done = reinterpret_cast<unsigned *>(base + off);
        off += sizeof(unsigned);
        st.err = reinterpret_cast<int *>(base + off);
        off += sizeof(int);
        off = (off + 255) & ~static_cast<size_t>(255);
        st.x16 = base + off;
        off += x16_bytes;
        st.xinv = reinterpret_cast<float *>(base + off);
        off += TMAX * sizeof(float);
        off = (off + 255) & ~static_cast<size_t>(255);
        st.cand_lg = reinterpret_cast<float *>(base + off);
        st.cand_id = reinterpret_cast<int32_t *>(base + off + RS_TMAX * RS_KMAX * sizeof(float));
        st.rdone = reinterpret_cast<unsigned *>(base + off + RS_TMAX * RS_KMAX * 8);
        st.sdone = st.rdone + 1;
        st.row_acc = reinterpret_cast<int32_t *>(base + off + RS_TMAX * RS_KMAX * 8 + 16);
        st.row_tok = st.row_acc + RS_TMAX;
        off += RS_SCRATCH_BYTES;
        off = (off + 255) & ~static_cast<size_t>(255);
        st.wpart = reinterpret_cast<float *>(base + off);
        st.x16_max_groups = X16_MAX_GROUPS;
        cudaError_t e = cudaSuccess;
        e = e != cudaSuccess ? e : raise_smem_limit<1, false, false, false>(optin);
        e = e != cudaSuccess ? e : raise_smem_limit<1, false, false, true>(optin);
        e = e != cudaSuccess ? e : raise_smem_limit<2, false, false, false>(optin);
        e = e != cudaSuccess ? e : raise_smem_limit<4, false, false, false>(optin);
        e = e != cudaSuccess ? e : raise_smem_limit<1, true, false, false>(optin);
        e = e != cudaSuccess ? e : raise_smem_limit<1, true, false, true>(optin);
        e = e != cudaSuccess ? e : raise_smem_limit<2, true, false, false>(optin);
        e = e != cudaSuccess ? e : raise_smem_limit<4, true, false, false>(optin);
        e = e != cudaSuccess ? e : raise_smem_limit<1, true, true, false>(optin);
        e = e != cudaSuccess ? e : raise_smem_limit<1, true, true, true>(optin);
        e = e != cudaSuccess ? e : raise_smem_limit<2, true, true, false>(optin);
        e = e != cudaSuccess ? e : raise_smem_limit<4, true, true, false>(optin);
        e = e != cudaSuccess ? e : raise_smem_limit<1, false, false, true, true>(optin);
        e = e != cudaSuccess ? e : raise_smem_limit<1, true, false, true, true>(optin);
        e = e != cudaSuccess ? e : cudaFuncSetAttribute(hbm_read_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                        HR_NST * HR_STAGE + 2 * HR_NST * 8);
        e = e != cudaSuccess ? e : cudaFuncSetAttribute(w4a16_tc_kernel<false>,
                                                        cudaFuncAttributeMaxDynamicSharedMemorySize, optin);
        e = e != cudaSuccess ? e : cudaFuncSetAttribute(w4a16_tc_kernel<true>,
                                                        cudaFuncAttributeMaxDynamicSharedMemorySize, optin);
        e = e != cudaSuccess ? e : raise_smem_limit_wide<2, false, 8>(optin);
        e = e != cudaSuccess ? e : raise_smem_limit_wide<2, true, 8>(optin);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(rescore_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     optin - RS_STATIC_SMEM_SLACK);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(sample_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     RS_SEL_MAX * 8);
        if (e != cudaSuccess || tensor_map_fn() != SV_OK) {
            cudaFree(base);
            return SV_ERR_CUDA;
        }
        st.sms = prop.multiProcessorCount;
        st.smem_optin = optin;
        st.ready = true;
    }
    *out = &st;
    return SV_OK;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned4(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

// Shared-memory layout of one launch (offsets in bytes, 128-byte aligned):
// nst pipeline stages | resident activations (XRES) | scales of 2 tiles |
// token ids of 2 tiles | the consumers' partial sums of one tile | mbarriers
// and a flag.
template <int NT, bool HEAD, bool GATHER, bool XRES>
int plan_layout(Params &p, int smem_optin, int *smem_total)
{
    using C = Cfg<NT, GATHER, consumer_warps(NT, XRES, GATHER)>;
    auto up = [](int v, int a) { return (v + a - 1) / a * a; };
    p.xslot_bytes = NT > 1 ? C::TP * XSTR                 // one group block of xprep_kernel
                           : up(p.T * XROW_BYTES, 128);      // a bf16 activation box of the T rows
    p.stage_bytes = XRES ? C::W_BYTES : up(C::W_BYTES + C::GPS * p.xslot_bytes, 128);
    p.sbuf_bytes = up(ROWS * p.G * 2, 128);
    p.xres_stride = 2 * p.K + 16;                     // = 16 (mod 128)
    const int xres_bytes = XRES ? up((p.T + 1) * p.xres_stride, 128) : 0;
    const int ids_bytes = up(2 * ROWS * 4, 128);
    const int red_bytes = up(C::RED_FLOATS * 4, 128);
    const int bk_bytes = HEAD ? up(32 * BK_STRIDE * 8, 128) : 0;
    const int pre_bytes = NT == 1 ? PRE_PARTS * ROWS * 8 * 4 : 0;
    const int fixed = xres_bytes + 2 * p.sbuf_bytes + ids_bytes + red_bytes + 128 + pre_bytes + bk_bytes + 256 + 6 * 8 + 16;
    int nst = (smem_optin - fixed - 1024) / (p.stage_bytes + 16);
    if (nst > 8) nst = 8;
    if (nst < 2) return SV_ERR_SHAPE;
    p.nst = nst;
    int off = nst * p.stage_bytes;
    p.off_xres = off;
    off += xres_bytes;
    p.off_sbuf = off;
    off += 2 * p.sbuf_bytes;
    p.off_ids = off;
    off += ids_bytes;
    p.off_red = off;
    off += red_bytes;
    p.off_xsc = off;
    off += 128;
    p.off_pre = off;
    off += pre_bytes;
    p.off_bk = off;
    off += bk_bytes;
    p.off_xzero = off;
    off += 256;
    p.off_bars = off;
    off += (2 * nst + 6) * 8 + 16;       // barriers, the time-out flag, the test hook's barrier
    *smem_total = off;
    return off <= smem_optin ? SV_OK : SV_ERR_SHAPE;
}

// Resident activations pay off when they fit with at least 3 weight stages,
// and when each CTA's share is long enough (at least 10 stages of 8 units)
// to amortise converting them before its first stage: with shorter shares
// (the QKV and down GEMMs of a 27B-class layer) the bf16 rows copied into
// every stage are faster.
constexpr int XRES_MAX_BYTES = 100 * 1024;
constexpr int XRES_MIN_UNITS = 80;

template <int NT, bool HEAD, bool GATHER, bool XRES, bool FMA = false>
int launch(Params p, const DeviceState &st, cudaStream_t stream)
{
    // several token tiles: the activations go through the conversion buffer
    if (!XRES && NT > 1 && p.G > st.x16_max_groups) return SV_ERR_SHAPE;
    int smem = 0;
    int rc = plan_layout<NT, HEAD, GATHER, XRES>(p, st.smem_optin, &smem);
    if (rc != SV_OK) return rc;
    CUtensorMap tmW, tmX;
    std::memset(&tmW, 0, sizeof tmW);
    std::memset(&tmX, 0, sizeof tmX);
    if (!GATHER) {
        rc = encode_2d(&tmW, CU_TENSOR_MAP_DATA_TYPE_UINT32, 4, p.Wq,
                       static_cast<unsigned long long>(p.K / 8), static_cast<unsigned long long>(p.n_rows),
                       16, ROWS);
    } else {
        // gathered rows: boxes one row high, GPS groups wide (tile::gather4)
        rc = encode_2d(&tmW, CU_TENSOR_MAP_DATA_TYPE_UINT32, 4, p.Wq,
                       static_cast<unsigned long long>(p.K / 8), static_cast<unsigned long long>(p.V),
                       static_cast<unsigned>(Cfg<NT, GATHER, consumer_warps(NT, XRES, GATHER)>::GPS * 16), 1);
    }
    if (rc != SV_OK) return rc;
    if (!XRES && NT == 1) {
        // bf16 activations copied into every stage: the box is exactly T rows
        // high (boxes reaching past the tensor are much slower to fill); the
        // kernel zeroes the spare token rows of every stage once.
        rc = encode_2d(&tmX, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, p.x, static_cast<unsigned long long>(p.K),
                       static_cast<unsigned long long>(p.T), XBOX, static_cast<unsigned>(p.T));
        if (rc != SV_OK) return rc;
    }
    long long B = st.sms;
    if (B > p.U) B = p.U;
    p.part = st.part;
    p.ctr = st.ctr;
    p.keys = st.keys;
    p.done = st.done;
    p.err = st.err;
    p.stall_ns = g_stall_ns.load(std::memory_order_relaxed);
    // Programmatic dependent launch: each kernel may begin while the previous
    // kernel of the stream drains; it waits (griddepcontrol.wait) before it
    // touches anything that kernel could have written.
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    // Every check has passed: from here on work is enqueued.
    if (st.clear_bytes && cudaMemsetAsync(st.clear_ptr, 0, st.clear_bytes, stream) != cudaSuccess) {
        cudaGetLastError();
        return SV_ERR_CUDA;
    }
    if (!XRES && NT > 1) {
        // several token tiles: convert x into ready-made group blocks first
        p.x16 = st.x16;
        p.xinv = st.xinv;
        cfg.gridDim = dim3(static_cast<unsigned>(Cfg<NT, GATHER, consumer_warps(NT, XRES, GATHER)>::TP));
        cfg.blockDim = dim3(XP_THREADS);
        cfg.dynamicSmemBytes = 0;
        if (cudaLaunchKernelEx(&cfg, xprep_kernel<false>, p.x, p.T, p.K, Cfg<NT, GATHER, consumer_warps(NT, XRES, GATHER)>::TP, st.x16, st.xinv) !=
            cudaSuccess) {
            cudaGetLastError();
            return SV_ERR_CUDA;
        }
    }
    cfg.gridDim = dim3(static_cast<unsigned>(B));
    cfg.blockDim = dim3(static_cast<unsigned>((consumer_warps(NT, XRES, GATHER) + 2) * 32));
    cfg.dynamicSmemBytes = static_cast<size_t>(smem);
    if (cudaLaunchKernelEx(&cfg, w4a16_stream_kernel<NT, HEAD, GATHER, XRES, FMA>, p, tmW, tmX) != cudaSuccess) {
        cudaGetLastError();
        return SV_ERR_CUDA;
    }
    return SV_OK;
}

// Shared-memory layout of a wide launch (offsets in bytes, 128-byte
// aligned): nst stages (one group of the tile's packed weights + the
// group's activation block) | the two-slot scale ring | the head's per-warp
// key table | mbarriers, the time-out flag and the split-tile decision word.
template <int NT, bool HEAD, int NCW>
int plan_layout_wide(Params &p, int smem_optin, int *smem_total)
{
    constexpr int RT = wide_rt(NCW);
    p.xslot_bytes = 8 * NT * XSTR;
    p.stage_bytes = RT * 64 + p.xslot_bytes;              // a multiple of 128
    const int ring_bytes = 2 * RT * 16;
    const int kt_bytes = HEAD ? NCW * TMAX * 8 : 0;
    int nst = (smem_optin - ring_bytes - kt_bytes - 256) / p.stage_bytes;
    if (nst > 8) nst = 8;           // the scale ring's reuse rule needs at most 9 stages
    if (nst < 2) return SV_ERR_SHAPE;
    p.nst = nst;
    int off = nst * p.stage_bytes;
    p.off_sbuf = off;
    off += ring_bytes;
    p.off_bk = off;
    off += kt_bytes;
    p.off_bars = off;
    off += (2 * nst + 2) * 8;
    *smem_total = off;
    return off <= smem_optin ? SV_OK : SV_ERR_SHAPE;
}

template <int NT, bool HEAD, int NCW>
int launch_wide(Params p, const DeviceState &st, cudaStream_t stream)
{
    constexpr int RT = wide_rt(NCW);
    constexpr unsigned BOX_ROWS = RT < 256 ? RT : 256;
    if (p.G > st.x16_max_groups) return SV_ERR_SHAPE;
    int smem = 0;
    int rc = plan_layout_wide<NT, HEAD, NCW>(p, st.smem_optin, &smem);
    if (rc != SV_OK) return rc;
    CUtensorMap tmW, tmS;
    std::memset(&tmW, 0, sizeof tmW);
    std::memset(&tmS, 0, sizeof tmS);
    rc = encode_2d(&tmW, CU_TENSOR_MAP_DATA_TYPE_UINT32, 4, p.Wq, static_cast<unsigned long long>(p.K / 8),
                   static_cast<unsigned long long>(p.n_rows), 16, BOX_ROWS);
    if (rc != SV_OK) return rc;
    rc = encode_2d(&tmS, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, p.scales, static_cast<unsigned long long>(p.G),
                   static_cast<unsigned long long>(p.n_rows), 8, BOX_ROWS);
    if (rc != SV_OK) return rc;
    const long long tiles = (static_cast<long long>(p.n_rows) + RT - 1) / RT;
    p.U = tiles * p.G;
    long long B = st.sms;
    if (B > p.U) B = p.U;
    p.part = st.wpart;
    p.ctr = st.ctr;
    p.keys = st.keys;
    p.done = st.done;
    p.err = st.err;
    p.stall_ns = g_stall_ns.load(std::memory_order_relaxed);
    p.x16 = st.x16;
    p.xinv = st.xinv;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    // the activations, converted into ready-made group blocks first
    cfg.gridDim = dim3(static_cast<unsigned>(8 * NT));
    cfg.blockDim = dim3(XP_THREADS);
    cfg.dynamicSmemBytes = 0;
    if (cudaLaunchKernelEx(&cfg, xprep_kernel<false>, p.x, p.T, p.K, 8 * NT, st.x16, st.xinv) != cudaSuccess) {
        cudaGetLastError();
        return SV_ERR_CUDA;
    }
    cfg.gridDim = dim3(static_cast<unsigned>(B));
    cfg.blockDim = dim3(static_cast<unsigned>((NCW + 1) * 32));
    cfg.dynamicSmemBytes = static_cast<size_t>(smem);
    if (cudaLaunchKernelEx(&cfg, w4a16_wide_kernel<NT, HEAD, NCW>, p, tmW, tmS) != cudaSuccess) {
        cudaGetLastError();
        return SV_ERR_CUDA;
    }
    return SV_OK;
}

// The wide kernel (512-row tiles) serves calls with two token tiles
// (9 <= T <= 16) and at least two 512-row tiles per SM -- an lm_head-sized
// pass -- when the scales' rows are 16-byte multiples (G % 8 == 0, a TMA
// requirement of the scale boxes), the rows are contiguous (no vocab_map)
// and the device state has its partial-sum area.  Measured on GB300 at
// V = 248,320, K = 5,120: 4.05 TB/s at T = 16 against 3.47 for 64-row
// tiles.  Smaller calls, and four token tiles (T > 16, where the 512-row
// kernel's 168-register cap spills and runs 10 % slower), stay on the
// 64-row kernel; the 256-row variant measured slower everywhere.
// Shared-memory layout of a tcgen05 launch (offsets in bytes): nst stages
// of TC_GU x 16 KB (8 KB of packed weights and 8 KB of activations per
// group) from 0 -- 1024-byte aligned, as the swizzled weight boxes need |
// the head's two finished-tile buffers | the tokens' xinv, 32 floats |
// mbarriers, flag, tensor-memory address, the buffers' tile numbers.  (The
// scales go from global memory to the dequant and epilogue threads'
// registers, one 16-byte load per row and box.)
template <bool HEAD>
int plan_layout_tc(Params &p, int smem_optin, int *smem_total)
{
    const int tb_bytes = HEAD ? 2 * TC_TB_BYTES : 0;   // the head's two finished-tile buffers
    const int bar_bytes = 1024;              // mbarriers and flags, rounded up
    int nst = (smem_optin - tb_bytes - bar_bytes) / TC_STAGE;
    if (nst > TC_MAX_STAGES) nst = TC_MAX_STAGES;
    // a dequant warpgroup waits only for its own units' stages: with nst a
    // multiple of the warpgroups the previous load of a stage it waits on
    // was its own, so its parity wait cannot alias a phase
    nst -= nst % TC_NDQ;
    if (nst < 2) return SV_ERR_SHAPE;
    p.nst = nst;
    p.stage_bytes = TC_STAGE;
    p.xslot_bytes = TC_X_BYTES;
    int off = nst * TC_STAGE;
    p.off_sbuf = off;
    p.off_bk = off;                          // finished-tile buffers
    off += tb_bytes;
    p.off_xinv = off;
    off += 128;
    p.off_bars = off;
    off += (2 * nst + 2 * TC_NDQ * TC_NSLOT + 2 * TC_NB + 4 + 2) * 8 + 32;
    *smem_total = off;
    return off <= smem_optin ? SV_OK : SV_ERR_SHAPE;
}

template <bool HEAD>
int launch_tc(Params p, const DeviceState &st, cudaStream_t stream)
{
    if (p.G > st.x16_max_groups) return SV_ERR_SHAPE;
    int smem = 0;
    int rc = plan_layout_tc<HEAD>(p, st.smem_optin, &smem);
    if (rc != SV_OK) return rc;
    CUtensorMap tmW;
    std::memset(&tmW, 0, sizeof tmW);
    rc = encode_2d(&tmW, CU_TENSOR_MAP_DATA_TYPE_UINT32, 4, p.Wq, static_cast<unsigned long long>(p.K / 8),
                   static_cast<unsigned long long>(p.n_rows), 16, TC_RT, CU_TENSOR_MAP_SWIZZLE_64B);
    if (rc != SV_OK) return rc;
    const long long tiles = (static_cast<long long>(p.n_rows) + TC_RT - 1) / TC_RT;
    p.U = tiles * (p.G / TC_GU);             // a unit is TC_GU groups of one tile
    long long B = st.sms;
    if (B > p.U) B = p.U;
    p.part = st.wpart;
    p.ctr = st.ctr;
    p.keys = st.keys;
    p.done = st.done;
    p.err = st.err;
    p.stall_ns = g_stall_ns.load(std::memory_order_relaxed);
    p.x16 = st.x16;
    p.xinv = st.xinv;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    // the activations, converted into the tensor cores' K-major layout first
    cfg.gridDim = dim3(32);
    cfg.blockDim = dim3(XP_THREADS);
    cfg.dynamicSmemBytes = 0;
    if (cudaLaunchKernelEx(&cfg, xprep_kernel<true>, p.x, p.T, p.K, 32, st.x16, st.xinv) != cudaSuccess) {
        cudaGetLastError();
        return SV_ERR_CUDA;
    }
    cfg.gridDim = dim3(static_cast<unsigned>(B));
    cfg.blockDim = dim3(TC_WARPS * 32);
    cfg.dynamicSmemBytes = static_cast<size_t>(smem);
    if (cudaLaunchKernelEx(&cfg, w4a16_tc_kernel<HEAD>, p, tmW) != cudaSuccess) {
        cudaGetLastError();
        return SV_ERR_CUDA;
    }
    return SV_OK;
}

// The tcgen05 kernel serves four token tiles (17 <= T <= 32) of contiguous
// rows whose scale rows are 16-byte multiples and split into boxes of eight
// groups (G % 8 == 0), when the device state has its partial-sum area.
// sv_debug_set_tcgen05(0) selects the mma.sync kernel for comparison.
template <bool HEAD, bool GATHER>
bool use_tc(const Params &p, const DeviceState &st)
{
    return g_tcgen05.load(std::memory_order_relaxed) && !GATHER && st.wpart && p.T > 16 && (p.G % 8) == 0 &&
           !p.y32;
}

template <bool HEAD, bool GATHER>
bool use_wide(const Params &p, const DeviceState &st)
{
    if (GATHER || !st.wpart || p.T <= 8 || p.T > 16 || (p.G % 8) != 0) return false;
    const long long tiles512 = (static_cast<long long>(p.n_rows) + 511) / 512;
    return tiles512 >= 2LL * st.sms;
}

template <bool HEAD, bool GATHER>
int dispatch(Params &p, const DeviceState &st, cudaStream_t stream)
{
    if (use_tc<HEAD, GATHER>(p, st)) return launch_tc<HEAD>(p, st, stream);
    if (use_wide<HEAD, GATHER>(p, st)) return launch_wide<2, HEAD, 8>(p, st, stream);
    if (p.T <= 8) {
        if (static_cast<long long>(p.T + 1) * (2LL * p.K + 16) <= XRES_MAX_BYTES &&
            p.U >= static_cast<long long>(XRES_MIN_UNITS) * st.sms) {
            if constexpr (!GATHER)
                if (g_fma_consumers.load(std::memory_order_relaxed)) return launch<1, HEAD, false, true, true>(p, st, stream);
            return launch<1, HEAD, GATHER, true>(p, st, stream);
        }
        return launch<1, HEAD, GATHER, false>(p, st, stream);
    }
    if (p.T <= 16) return launch<2, HEAD, GATHER, false>(p, st, stream);
    return launch<4, HEAD, GATHER, false>(p, st, stream);
}

int check_common(const void *x, const void *Wq, const void *scales, int T, int K)
{
    if (!x || !Wq || !scales) return SV_ERR_NULL;
    if (T < 1 || T > TMAX || K < 128 || (K % 128) != 0) return SV_ERR_SHAPE;
    if (!aligned16(x) || !aligned16(Wq) || !aligned16(scales)) return SV_ERR_ALIGN;
    return SV_OK;
}

int check_head(const sv_bf16 *x, const uint32_t *Wq, const sv_bf16 *scales, int K, int T,
               const int32_t *vocab_map, int n_map, int V, int mode, const int32_t *drafts,
               int n_draft, int32_t *accept_len, int32_t *next_token, int32_t *ids, float *vals)
{
    int rc = check_common(x, Wq, scales, T, K);
    if (rc != SV_OK) return rc;
    if (V < 1) return SV_ERR_SHAPE;
    if (vocab_map) {
        if (n_map < 1 || n_map > V) return SV_ERR_SHAPE;
        if (!aligned4(vocab_map)) return SV_ERR_ALIGN;
    }
    if (mode == 0) {
        if (!accept_len || !next_token) return SV_ERR_NULL;
        if (n_draft > 0 && !drafts) return SV_ERR_NULL;
        if ((drafts && !aligned4(drafts)) || !aligned4(accept_len) || !aligned4(next_token))
            return SV_ERR_ALIGN;
    } else {
        if (!ids) return SV_ERR_NULL;
        if (!aligned4(ids) || (vals && !aligned4(vals))) return SV_ERR_ALIGN;
    }
    return SV_OK;
}

int check_batched(int n_draft, int n_streams)
{
    if (n_draft < 0 || n_draft > 31 || n_streams < 1) return SV_ERR_SHAPE;
    if (static_cast<long long>(n_streams) * (n_draft + 1) > TMAX) return SV_ERR_SHAPE;
    return SV_OK;
}

int check_gemm(const sv_bf16 *x, const uint32_t *Wq, const sv_bf16 *scales, int T, int K, int N, sv_bf16 *y)
{
    int rc = check_common(x, Wq, scales, T, K);
    if (rc != SV_OK) return rc;
    if (!y) return SV_ERR_NULL;
    if (N < 1) return SV_ERR_SHAPE;
    if (!aligned16(y)) return SV_ERR_ALIGN;
    return SV_OK;
}

int head_call(const sv_bf16 *x, const uint32_t *Wq, const sv_bf16 *scales, int K, int T,
              const int32_t *vocab_map, int n_map, int V, int mode, const int32_t *drafts,
              int n_draft, int n_streams, int32_t *accept_len, int32_t *next_token,
              int32_t *ids, float *vals, cudaStream_t stream, int flags = 0)
{
    int rc = check_head(x, Wq, scales, K, T, vocab_map, n_map, V, mode, drafts, n_draft, accept_len, next_token,
                        ids, vals);
    if (rc != SV_OK) return rc;
    DeviceState *st = nullptr;
    rc = device_state(&st);
    if (rc != SV_OK) return rc;
    Params p{};
    p.x = x;
    p.Wq = Wq;
    p.scales = scales;
    p.map = vocab_map;
    p.T = T;
    p.K = K;
    p.G = K / 128;
    p.n_rows = vocab_map ? n_map : V;
    p.V = V;
    const long long tiles = (static_cast<long long>(p.n_rows) + ROWS - 1) / ROWS;
    p.U = tiles * p.G;
    p.mode = mode;
    p.drafts = drafts;
    p.n_draft = n_draft;
    p.n_streams = n_streams;
    p.accept_len = accept_len;
    p.next_token = next_token;
    p.ids = ids;
    p.vals = vals;
    p.map_static = (vocab_map && (flags & SV_MAP_STATIC)) ? 1 : 0;
    return vocab_map ? dispatch<true, true>(p, *st, stream) : dispatch<true, false>(p, *st, stream);
}

// ----------------------------------------------------------------------------
// Top-k candidates of the int4 head rescored by the bf16 head (rescore.cuh):
// pass 1 is the head kernel as a GEMM with fp32 outputs, pass 2
// slicemax_kernel, pass 3 rescore_kernel.

// Passes 1 and 2 shared by the rescored and the sampled calls: the int4
// head's fp32 logits [T][V] into a per-device buffer, then every 128-row
// slice's largest key.  On success *cfg is set up for the next PDL launch
// on `stream` (block RS_THREADS) and *nS_out is the slice count.
int logits_and_slice_maxima(const sv_bf16 *x, const uint32_t *Wq, const sv_bf16 *scales, int K, int T, int V,
                            cudaStream_t stream, DeviceState **st_out, int *nS_out, cudaLaunchConfig_t *cfg,
                            cudaLaunchAttribute *attr)
{
    DeviceState *st = nullptr;
    int rc = device_state(&st);
    if (rc != SV_OK) return rc;
    const long long nS = (static_cast<long long>(V) + RS_SLICE - 1) / RS_SLICE;
    {
        std::lock_guard<std::mutex> lock(g_mu);
        if (V > st->rs_v_cap || nS > st->rs_s_cap) {
            // first call with a larger head on this device: (re)allocate
            if (cudaStreamSynchronize(stream) != cudaSuccess) return SV_ERR_CUDA;
            cudaFree(st->rs_logits);
            cudaFree(st->rs_smax);
            st->rs_logits = nullptr;
            st->rs_smax = nullptr;
            st->rs_v_cap = st->rs_s_cap = 0;
            if (cudaMalloc(&st->rs_logits, static_cast<size_t>(RS_TMAX) * V * sizeof(float)) != cudaSuccess ||
                cudaMalloc(&st->rs_smax, static_cast<size_t>(nS) * RS_TMAX * 8) != cudaSuccess) {
                cudaGetLastError();
                return SV_ERR_NOMEM;
            }
            st->rs_v_cap = V;
            st->rs_s_cap = nS;
        }
    }
    // pass 1: the int4 head's fp32 logits [T][V]
    Params p{};
    p.x = x;
    p.Wq = Wq;
    p.scales = scales;
    p.T = T;
    p.K = K;
    p.G = K / 128;
    p.n_rows = V;
    p.V = V;
    const long long tiles = (static_cast<long long>(V) + ROWS - 1) / ROWS;
    p.U = tiles * p.G;
    p.y32 = st->rs_logits;
    rc = dispatch<false, false>(p, *st, stream);
    if (rc != SV_OK) return rc;
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    *cfg = cudaLaunchConfig_t{};
    cfg->blockDim = dim3(RS_THREADS);
    cfg->stream = stream;
    cfg->attrs = attr;
    cfg->numAttrs = 1;
    // pass 2: every slice's largest key per row
    SliceMaxParams mp{};
    mp.logits = st->rs_logits;
    mp.T = T;
    mp.V = V;
    mp.nS = static_cast<int>(nS);
    mp.smax = st->rs_smax;
    cfg->gridDim = dim3(static_cast<unsigned>((nS + RS_WARPS - 1) / RS_WARPS));
    cfg->dynamicSmemBytes = 0;
    if (cudaLaunchKernelEx(cfg, slicemax_kernel, mp) != cudaSuccess) {
        cudaGetLastError();
        return SV_ERR_CUDA;
    }
    *st_out = st;
    *nS_out = static_cast<int>(nS);
    return SV_OK;
}

int rescored_call(const sv_bf16 *x, const uint32_t *Wq, const sv_bf16 *scales, const sv_bf16 *Wbf, int K, int T,
                  int top_k, int V, int mode, const int32_t *drafts, int n_draft, int32_t *accept_len,
                  int32_t *next_token, int32_t *ids, float *vals, cudaStream_t stream)
{
    int rc = check_common(x, Wq, scales, T, K);
    if (rc != SV_OK) return rc;
    if (!Wbf) return SV_ERR_NULL;
    if (!aligned16(Wbf)) return SV_ERR_ALIGN;
    if (T > RS_TMAX || V < 1 || top_k < 1 || top_k > RS_KMAX || top_k > V) return SV_ERR_SHAPE;
    if (mode == 0) {
        if (!accept_len || !next_token) return SV_ERR_NULL;
        if (n_draft > 0 && !drafts) return SV_ERR_NULL;
        if ((drafts && !aligned4(drafts)) || !aligned4(accept_len) || !aligned4(next_token)) return SV_ERR_ALIGN;
    } else {
        if (!ids) return SV_ERR_NULL;
        if (!aligned4(ids) || (vals && !aligned4(vals))) return SV_ERR_ALIGN;
    }
    {
        DeviceState *st0 = nullptr;
        rc = device_state(&st0);
        if (rc != SV_OK) return rc;
        const long long limit = st0->smem_optin - RS_STATIC_SMEM_SLACK;
        if (K > 65536 || RS_SEL_MAX * 8LL + 2LL * K > limit) return SV_ERR_SHAPE;
    }
    DeviceState *st = nullptr;
    int nS = 0;
    cudaLaunchConfig_t cfg;
    cudaLaunchAttribute attr[1];
    rc = logits_and_slice_maxima(x, Wq, scales, K, T, V, stream, &st, &nS, &cfg, attr);
    if (rc != SV_OK) return rc;
    // pass 3: selection, rescoring with the bf16 head, argmax, verify
    RescoreParams rp{};
    rp.x = x;
    rp.Wbf = Wbf;
    rp.logits = st->rs_logits;
    rp.smax = st->rs_smax;
    rp.nS = nS;
    rp.T = T;
    rp.K = K;
    rp.V = V;
    rp.k = top_k;
    rp.mode = mode;
    rp.drafts = drafts;
    rp.accept_len = accept_len;
    rp.next_token = next_token;
    rp.ids = ids;
    rp.vals = vals;
    rp.cand_lg = st->cand_lg;
    rp.cand_id = st->cand_id;
    rp.done = st->rdone;
    cfg.gridDim = dim3(static_cast<unsigned>((top_k + RS_PER_CTA - 1) / RS_PER_CTA), static_cast<unsigned>(T));
    cfg.dynamicSmemBytes = static_cast<size_t>(RS_SEL_MAX) * 8 + 2 * static_cast<size_t>(K);
    if (cudaLaunchKernelEx(&cfg, rescore_kernel, rp) != cudaSuccess) {
        cudaGetLastError();
        return SV_ERR_CUDA;
    }
    return SV_OK;
}

// Exact speculative sampling verify (mode 0) or the rows' sampling
// distributions (mode 1): passes 1 and 2 as above, then sample_kernel.
int sampled_call(const sv_bf16 *x, const uint32_t *Wq, const sv_bf16 *scales, int K, int T, int V,
                 float temperature, int top_k, float top_p, float min_p, int mode, const float *u,
                 const int32_t *drafts, int32_t *accept_len, int32_t *next_token, int32_t *out_ids,
                 float *out_probs, cudaStream_t stream)
{
    int rc = check_common(x, Wq, scales, T, K);
    if (rc != SV_OK) return rc;
    if (T > RS_TMAX || V < 1 || top_k > SAMPLE_KEEP) return SV_ERR_SHAPE;
    if (temperature != temperature || top_p != top_p || min_p != min_p || min_p > 1.f) return SV_ERR_SHAPE;
    if (mode == 0) {
        if (!u || !accept_len || !next_token) return SV_ERR_NULL;
        if (T > 1 && !drafts) return SV_ERR_NULL;
        if (!aligned4(u) || (drafts && !aligned4(drafts)) || !aligned4(accept_len) || !aligned4(next_token))
            return SV_ERR_ALIGN;
    } else {
        if (!out_ids || !out_probs) return SV_ERR_NULL;
        if (!aligned4(out_ids) || !aligned4(out_probs)) return SV_ERR_ALIGN;
    }
    DeviceState *st = nullptr;
    int nS = 0;
    cudaLaunchConfig_t cfg;
    cudaLaunchAttribute attr[1];
    rc = logits_and_slice_maxima(x, Wq, scales, K, T, V, stream, &st, &nS, &cfg, attr);
    if (rc != SV_OK) return rc;
    SampleParams sp{};
    sp.logits = st->rs_logits;
    sp.smax = st->rs_smax;
    sp.nS = nS;
    sp.T = T;
    sp.V = V;
    sp.temperature = temperature;
    sp.top_p = top_p;
    sp.min_p = min_p;
    sp.top_k = top_k;
    sp.mode = mode;
    sp.u = u;
    sp.drafts = drafts;
    sp.accept_len = accept_len;
    sp.next_token = next_token;
    sp.out_ids = out_ids;
    sp.out_probs = out_probs;
    sp.row_acc = st->row_acc;
    sp.row_tok = st->row_tok;
    sp.done = st->sdone;
    cfg.gridDim = dim3(static_cast<unsigned>(T));
    cfg.dynamicSmemBytes = static_cast<size_t>(RS_SEL_MAX) * 8;
    if (cudaLaunchKernelEx(&cfg, sample_kernel, sp) != cudaSuccess) {
        cudaGetLastError();
        return SV_ERR_CUDA;
    }
    return SV_OK;
}

// ----------------------------------------------------------------------------
// Allocation-free variant of the verify (lmhead_verify_noalloc).
//
// Its scratch -- split-tile partial sums, arrival counters, argmax keys --
// lives in the file-scope device array below instead of a cudaMalloc'd
// area, so the call never allocates.  The array is sized for at most
// NOALLOC_MAX_CTAS thread blocks (each keeps two 32-token partial tiles,
// 2.6 MB in all) plus the conversion buffer of calls with more than 7
// drafts (1.1 MB, K <= 16384); the call never launches more blocks than
// that.  Every device that loads this library holds the array (about
// 3.7 MB) until the process exits.

constexpr int NOALLOC_MAX_CTAS = 160;
constexpr size_t NOALLOC_PART_BYTES = static_cast<size_t>(NOALLOC_MAX_CTAS) * 2 * PART_FLOATS * sizeof(float);
constexpr size_t NOALLOC_CTR_OFF = NOALLOC_PART_BYTES;
constexpr size_t NOALLOC_KEYS_OFF = NOALLOC_CTR_OFF + 1024;                 // 160 counters, padded
constexpr size_t NOALLOC_DONE_OFF = NOALLOC_KEYS_OFF + TMAX * sizeof(unsigned long long);
constexpr size_t NOALLOC_ERR_OFF = NOALLOC_DONE_OFF + 256;
constexpr int NOALLOC_X16_GROUPS = 128;                                     // K <= 16384
constexpr size_t NOALLOC_XINV_OFF = NOALLOC_ERR_OFF + 256;
constexpr size_t NOALLOC_X16_OFF = NOALLOC_XINV_OFF + 256;
constexpr size_t NOALLOC_BYTES = NOALLOC_X16_OFF + static_cast<size_t>(NOALLOC_X16_GROUPS) * TMAX * XSTR;

static __device__ __align__(256) unsigned char g_noalloc_scratch[NOALLOC_BYTES];

DeviceState g_noalloc_state[MAX_DEVICES];

// Once per device, with that device current: resolve the array's device
// address (the array's name is only a host-side stand-in), and raise the
// shared-memory limit of the head kernels.  Nothing here allocates.
int noalloc_state(DeviceState **out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return SV_ERR_CUDA;
    if (dev < 0 || dev >= MAX_DEVICES) return SV_ERR_DEVICE;
    std::lock_guard<std::mutex> lock(g_mu);
    DeviceState &st = g_noalloc_state[dev];
    if (!st.ready) {
        int major = 0, sms = 0, optin = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
            return SV_ERR_CUDA;
        if (major != 10) return SV_ERR_DEVICE;
        unsigned char *base = nullptr;
        if (cudaGetSymbolAddress(reinterpret_cast<void **>(&base), g_noalloc_scratch) != cudaSuccess) {
            cudaGetLastError();
            return SV_ERR_CUDA;
        }
        cudaError_t e = cudaSuccess;
        e = e != cudaSuccess ? e : raise_smem_limit<1, true, false, false>(optin);
        e = e != cudaSuccess ? e : raise_smem_limit<1, true, false, true>(optin);
        e = e != cudaSuccess ? e : raise_smem_limit<2, true, false, false>(optin);
        e = e != cudaSuccess ? e : raise_smem_limit<4, true, false, false>(optin);
        e = e != cudaSuccess ? e : raise_smem_limit<1, true, true, false>(optin);
        e = e != cudaSuccess ? e : raise_smem_limit<1, true, true, true>(optin);
        e = e != cudaSuccess ? e : raise_smem_limit<2, true, true, false>(optin);
        e = e != cudaSuccess ? e : raise_smem_limit<4, true, true, false>(optin);
        if (e != cudaSuccess || tensor_map_fn() != SV_OK) {
            cudaGetLastError();
            return SV_ERR_CUDA;
        }
        st.part = reinterpret_cast<float *>(base);
        st.ctr = reinterpret_cast<unsigned *>(base + NOALLOC_CTR_OFF);
        st.keys = reinterpret_cast<unsigned long long *>(base + NOALLOC_KEYS_OFF);
        st.done = reinterpret_cast<unsigned *>(base + NOALLOC_DONE_OFF);
        st.err = reinterpret_cast<int *>(base + NOALLOC_ERR_OFF);
        st.xinv = reinterpret_cast<float *>(base + NOALLOC_XINV_OFF);
        st.x16 = base + NOALLOC_X16_OFF;
        st.x16_max_groups = NOALLOC_X16_GROUPS;
        st.sms = sms < NOALLOC_MAX_CTAS ? sms : NOALLOC_MAX_CTAS;
        st.smem_optin = optin;
        // the array keeps whatever the last call left: the counters, keys,
        // completion count and error word are cleared before every launch
        st.clear_ptr = st.ctr;
        st.clear_bytes = NOALLOC_XINV_OFF - NOALLOC_CTR_OFF;
        st.ready = true;
    }
    *out = &st;
    return SV_OK;
}

}  // namespace
}  // namespace sv

extern "C" {

int lmhead_verify_noalloc(const sv_bf16 *x, const uint32_t *Wq, const sv_bf16 *scales, int K,
                          const int32_t *drafts, int n_draft, const int32_t *vocab_map, int n_map, int V,
                          int32_t *accept_len, int32_t *next_token, sv_stream stream)
{
    using namespace sv;
    if (n_draft < 0 || n_draft > TMAX - 1) return SV_ERR_SHAPE;
    const int T = n_draft + 1;
    int rc = check_common(x, Wq, scales, T, K);
    if (rc != SV_OK) return rc;
    if (V < 1) return SV_ERR_SHAPE;
    if (vocab_map) {
        if (n_map < 1 || n_map > V) return SV_ERR_SHAPE;
        if (!aligned4(vocab_map)) return SV_ERR_ALIGN;
    }
    if (!accept_len || !next_token) return SV_ERR_NULL;
    if (n_draft > 0 && !drafts) return SV_ERR_NULL;
    if ((drafts && !aligned4(drafts)) || !aligned4(accept_len) || !aligned4(next_token))
        return SV_ERR_ALIGN;
    // more than 7 drafts: the activations go through the fixed conversion
    // buffer, sized for K <= 128 * NOALLOC_X16_GROUPS
    if (T > 8 && K / 128 > NOALLOC_X16_GROUPS) return SV_ERR_SHAPE;
    DeviceState *st = nullptr;
    rc = noalloc_state(&st);
    if (rc != SV_OK) return rc;
    const cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
    Params p{};
    p.x = x;
    p.Wq = Wq;
    p.scales = scales;
    p.map = vocab_map;
    p.T = T;
    p.K = K;
    p.G = K / 128;
    p.n_rows = vocab_map ? n_map : V;
    p.V = V;
    const long long tiles = (static_cast<long long>(p.n_rows) + ROWS - 1) / ROWS;
    p.U = tiles * p.G;
    p.mode = 0;
    p.drafts = drafts;
    p.n_draft = n_draft;
    p.n_streams = 1;
    p.accept_len = accept_len;
    p.next_token = next_token;
    return vocab_map ? dispatch<true, true>(p, *st, cs) : dispatch<true, false>(p, *st, cs);
}


int w4a16_gemm(const sv_bf16 *x, const uint32_t *Wq, const sv_bf16 *scales, int T, int K, int N,
               sv_bf16 *y, sv_stream stream)
{
    using namespace sv;
    int rc = check_gemm(x, Wq, scales, T, K, N, y);
    if (rc != SV_OK) return rc;
    DeviceState *st = nullptr;
    rc = device_state(&st);
    if (rc != SV_OK) return rc;
    Params p{};
    p.x = x;
    p.Wq = Wq;
    p.scales = scales;
    p.T = T;
    p.K = K;
    p.G = K / 128;
    p.n_rows = N;
    p.V = N;
    const long long tiles = (static_cast<long long>(N) + ROWS - 1) / ROWS;
    p.U = tiles * p.G;
    p.y = y;
    return dispatch<false, false>(p, *st, reinterpret_cast<cudaStream_t>(stream));
}

int lmhead_verify_batched(const sv_bf16 *x, const uint32_t *Wq, const sv_bf16 *scales, int K,
                          const int32_t *drafts, int n_draft, int n_streams,
                          const int32_t *vocab_map, int n_map, int V, int32_t *accept_len,
                          int32_t *next_token, sv_stream stream)
{
    const int rc = sv::check_batched(n_draft, n_streams);
    if (rc != SV_OK) return rc;
    return sv::head_call(x, Wq, scales, K, n_streams * (n_draft + 1), vocab_map, n_map, V, 0, drafts,
                         n_draft, n_streams, accept_len, next_token, nullptr, nullptr,
                         reinterpret_cast<cudaStream_t>(stream));
}

int lmhead_verify_ex(const sv_bf16 *x, const uint32_t *Wq, const sv_bf16 *scales, int K,
                     const int32_t *drafts, int n_draft, int n_streams,
                     const int32_t *vocab_map, int n_map, int V, int flags, int32_t *accept_len,
                     int32_t *next_token, sv_stream stream)
{
    if (flags & ~SV_MAP_STATIC) return SV_ERR_SHAPE;
    const int rc = sv::check_batched(n_draft, n_streams);
    if (rc != SV_OK) return rc;
    return sv::head_call(x, Wq, scales, K, n_streams * (n_draft + 1), vocab_map, n_map, V, 0, drafts,
                         n_draft, n_streams, accept_len, next_token, nullptr, nullptr,
                         reinterpret_cast<cudaStream_t>(stream), flags);
}

int sv_verify_cycle(const sv_gemm_call *gemms, int n_gemms, const sv_verify_call *verify, sv_stream stream)
{
    using namespace sv;
    if (n_gemms < 0 || n_gemms > SV_CYCLE_MAX_GEMMS || (n_gemms == 0 && !verify)) return SV_ERR_SHAPE;
    if (n_gemms > 0 && !gemms) return SV_ERR_NULL;
    // every argument first: on an error nothing is enqueued
    for (int i = 0; i < n_gemms; ++i) {
        const sv_gemm_call &g = gemms[i];
        const int rc = check_gemm(g.x, g.Wq, g.scales, g.T, g.K, g.N, g.y);
        if (rc != SV_OK) return rc;
    }
    if (verify) {
        const sv_verify_call &v = *verify;
        int rc = check_batched(v.n_draft, v.n_streams);
        if (rc != SV_OK) return rc;
        rc = check_head(v.x, v.Wq, v.scales, v.K, v.n_streams * (v.n_draft + 1), v.vocab_map, v.n_map, v.V, 0,
                        v.drafts, v.n_draft, v.accept_len, v.next_token, nullptr, nullptr);
        if (rc != SV_OK) return rc;
    }
    DeviceState *st = nullptr;
    int rc = device_state(&st);
    if (rc != SV_OK) return rc;
    for (int i = 0; i < n_gemms; ++i) {
        const sv_gemm_call &g = gemms[i];
        rc = w4a16_gemm(g.x, g.Wq, g.scales, g.T, g.K, g.N, g.y, stream);
        if (rc != SV_OK) return rc;
    }
    if (verify) {
        const sv_verify_call &v = *verify;
        rc = lmhead_verify_batched(v.x, v.Wq, v.scales, v.K, v.drafts, v.n_draft, v.n_streams, v.vocab_map,
                                   v.n_map, v.V, v.accept_len, v.next_token, stream);
    }
    return rc;
}

int lmhead_verify(const sv_bf16 *x, const uint32_t *Wq, const sv_bf16 *scales, int K,
                  const int32_t *drafts, int n_draft, const int32_t *vocab_map, int n_map, int V,
                  int32_t *accept_len, int32_t *next_token, sv_stream stream)
{
    return lmhead_verify_batched(x, Wq, scales, K, drafts, n_draft, 1, vocab_map, n_map, V,
                                 accept_len, next_token, stream);
}

int lmhead_argmax(const sv_bf16 *x, const uint32_t *Wq, const sv_bf16 *scales, int K, int T,
                  const int32_t *vocab_map, int n_map, int V, int32_t *ids, float *vals,
                  sv_stream stream)
{
    return sv::head_call(x, Wq, scales, K, T, vocab_map, n_map, V, 1, nullptr, 0, 0, nullptr,
                         nullptr, ids, vals, reinterpret_cast<cudaStream_t>(stream));
}

const char *sv_status_string(int status)
{
    switch (status) {
    case SV_OK: return "ok";
    case SV_ERR_NULL: return "a required pointer is NULL";
    case SV_ERR_SHAPE: return "a size is out of range or inconsistent";
    case SV_ERR_ALIGN: return "a pointer is not suitably aligned";
    case SV_ERR_CUDA: return "a CUDA call or kernel launch failed";
    case SV_ERR_NOMEM: return "the per-device scratch area could not be allocated";
    case SV_ERR_DEVICE: return "the current device is not a compute capability 10.x GPU";
    default: return "unknown status";
    }
}

int sv_last_device_error(int32_t *out)
{
    using namespace sv;
    if (!out) return SV_ERR_NULL;
    DeviceState *st = nullptr;
    int rc = device_state(&st);
    if (rc != SV_OK) return rc;
    int v = 0;
    if (cudaMemcpy(&v, st->err, sizeof v, cudaMemcpyDeviceToHost) != cudaSuccess) return SV_ERR_CUDA;
    if (cudaMemset(st->err, 0, sizeof v) != cudaSuccess) return SV_ERR_CUDA;
    if (v & SV_DEVERR_TIMEOUT) {
        // A run that gave up on a wait may have left the counters of the
        // scratch area (tile arrivals, argmax keys, CTA completions) out of
        // step; put them back to zero so that later calls start clean.
        const size_t n = reinterpret_cast<uint8_t *>(st->err) - reinterpret_cast<uint8_t *>(st->keys);
        if (cudaMemset(st->keys, 0, n) != cudaSuccess) return SV_ERR_CUDA;
        if (cudaMemset(st->rdone, 0, 2 * sizeof(unsigned)) != cudaSuccess) return SV_ERR_CUDA;
    }
    if (cudaDeviceSynchronize() != cudaSuccess) return SV_ERR_CUDA;
    *out = v;
    return SV_OK;
}

int sv_hbm_read(const void *src, size_t bytes, uint32_t *sink, sv_stream stream)
{
    using namespace sv;
    if (!src || !sink) return SV_ERR_NULL;
    if (bytes < 16 || (bytes % 16) != 0) return SV_ERR_SHAPE;
    if (!aligned16(src) || !aligned4(sink)) return SV_ERR_ALIGN;
    DeviceState *st = nullptr;
    int rc = device_state(&st);
    if (rc != SV_OK) return rc;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.stream = reinterpret_cast<cudaStream_t>(stream);
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cfg.gridDim = dim3(static_cast<unsigned>(st->sms));
    cfg.blockDim = dim3(64);
    cfg.dynamicSmemBytes = HR_NST * HR_STAGE + 2 * HR_NST * 8;
    if (cudaLaunchKernelEx(&cfg, hbm_read_kernel, static_cast<const uint8_t *>(src),
                           static_cast<unsigned long long>(bytes), sink, st->err) != cudaSuccess) {
        cudaGetLastError();
        return SV_ERR_CUDA;
    }
    return SV_OK;
}

int sv_debug_set_fma_consumers(int on)
{
    sv::g_fma_consumers.store(on ? 1 : 0, std::memory_order_relaxed);
    return SV_OK;
}

int sv_debug_set_tcgen05(int on)
{
    sv::g_tcgen05.store(on ? 1 : 0, std::memory_order_relaxed);
    return SV_OK;
}

int sv_debug_set_wait_stall(uint32_t ns)
{
    if (ns > 1000000000u) return SV_ERR_SHAPE;
    sv::g_stall_ns.store(ns, std::memory_order_relaxed);
    return SV_OK;
}

int lmhead_verify_rescored(const sv_bf16 *x, const uint32_t *Wq, const sv_bf16 *scales, const sv_bf16 *Wbf, int K,
                           const int32_t *drafts, int n_draft, int top_k, int V, int32_t *accept_len,
                           int32_t *next_token, sv_stream stream)
{
    if (n_draft < 0 || n_draft > sv::RS_TMAX - 1) return SV_ERR_SHAPE;
    return sv::rescored_call(x, Wq, scales, Wbf, K, n_draft + 1, top_k, V, 0, drafts, n_draft, accept_len,
                             next_token, nullptr, nullptr, reinterpret_cast<cudaStream_t>(stream));
}

int lmhead_argmax_rescored(const sv_bf16 *x, const uint32_t *Wq, const sv_bf16 *scales, const sv_bf16 *Wbf, int K,
                           int T, int top_k, int V, int32_t *ids, float *vals, sv_stream stream)
{
    return sv::rescored_call(x, Wq, scales, Wbf, K, T, top_k, V, 1, nullptr, 0, nullptr, nullptr, ids, vals,
                             reinterpret_cast<cudaStream_t>(stream));
}

int lmhead_verify_sampled(const sv_bf16 *x, const uint32_t *Wq, const sv_bf16 *scales, int K,
                          const int32_t *drafts, int n_draft, int V, float temperature, int top_k, float top_p,
                          float min_p, const float *u, int32_t *accept_len, int32_t *next_token, sv_stream stream)
{
    if (n_draft < 0 || n_draft > sv::RS_TMAX - 1) return SV_ERR_SHAPE;
    return sv::sampled_call(x, Wq, scales, K, n_draft + 1, V, temperature, top_k, top_p, min_p, 0, u, drafts,
                            accept_len, next_token, nullptr, nullptr, reinterpret_cast<cudaStream_t>(stream));
}

int lmhead_sampling_dist(const sv_bf16 *x, const uint32_t *Wq, const sv_bf16 *scales, int K, int T, int V,
                         float temperature, int top_k, float top_p, float min_p, int32_t *ids, float *probs,
                         sv_stream stream)
{
    return sv::sampled_call(x, Wq, scales, K, T, V, temperature, top_k, top_p, min_p, 1, nullptr, nullptr, nullptr,
                            nullptr, ids, probs, reinterpret_cast<cudaStream_t>(stream));
}

// ----------------------------------------------------------------------------
// Dynamic draft list (draft_list.cuh)

size_t draft_list_bytes(int V, int n_static, int cap)
{
    if (V < 1 || n_static < 1 || cap < 0 || static_cast<long long>(n_static) + cap > (1LL << 28)) return 0;
    return sv::draft_list_ids_offset(V) + 4 * (static_cast<size_t>(n_static) + cap);
}

int32_t *draft_list_ids(void *ws, int V)
{
    if (!ws || V < 1) return nullptr;
    return reinterpret_cast<int32_t *>(static_cast<uint8_t *>(ws) + sv::draft_list_ids_offset(V));
}

int draft_list_init(void *ws, const int32_t *static_ids, int n_static, int V, int cap, sv_stream stream)
{
    using namespace sv;
    if (!ws || !static_ids) return SV_ERR_NULL;
    if (draft_list_bytes(V, n_static, cap) == 0) return SV_ERR_SHAPE;
    if (!aligned16(ws) || !aligned4(static_ids)) return SV_ERR_ALIGN;
    const cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
    uint8_t *base = static_cast<uint8_t *>(ws);
    if (cudaMemsetAsync(base + sizeof(DraftListHeader), 0, 4 * draft_list_bitmap_words(V), cs) != cudaSuccess) {
        cudaGetLastError();
        return SV_ERR_CUDA;
    }
    const int n = n_static + cap;
    draft_list_init_kernel<<<(n + 255) / 256, 256, 0, cs>>>(base, static_ids, n_static, V, cap);
    if (cudaGetLastError() != cudaSuccess) return SV_ERR_CUDA;
    return SV_OK;
}

int draft_list_add(void *ws, const int32_t *tokens, int n_tokens, sv_stream stream)
{
    using namespace sv;
    if (!ws) return SV_ERR_NULL;
    if (n_tokens < 0) return SV_ERR_SHAPE;
    if (n_tokens == 0) return SV_OK;
    if (!tokens) return SV_ERR_NULL;
    if (!aligned16(ws) || !aligned4(tokens)) return SV_ERR_ALIGN;
    draft_list_add_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(static_cast<uint8_t *>(ws), tokens,
                                                                                n_tokens);
    if (cudaGetLastError() != cudaSuccess) return SV_ERR_CUDA;
    return SV_OK;
}

int draft_list_count(const void *ws, int32_t *out)
{
    using namespace sv;
    if (!ws || !out) return SV_ERR_NULL;
    const auto *h = static_cast<const DraftListHeader *>(ws);
    if (cudaMemcpy(out, &h->count, sizeof(int32_t), cudaMemcpyDeviceToHost) != cudaSuccess) {
        cudaGetLastError();
        return SV_ERR_CUDA;
    }
    return SV_OK;
}

}  // extern "C"
