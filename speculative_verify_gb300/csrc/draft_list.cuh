// draft_list.cuh -- list maintenance for the restricted draft head: a
// static list of token ids plus the tokens of the current sequence missing
// from it, added on the fly, at most `cap` of them (page "OpenJet Engine:
// CUDA LLM inference for Qwen3.8-27B", section "How it gets its speed";
// page "Tesla P100 (sm_60) llama.cpp patches for Qwen3.5/3.6-35B-A3B: ~2x
// decode and prompt processing over the shinbunbun baseline", sections
// "MTP draft vocabulary (patch 17)" and "The draft vocabulary file").
//
// Workspace (caller-owned device memory, 16-byte aligned):
//   DraftListHeader            32 bytes
//   bitmap  [ceil(V/32)] u32   membership of every id in the list (padded to 16 B)
//   ids     [n_static + cap]   the list: static ids, then added tokens, then
//                              copies of ids[0] in the unused slots
// The id array is a ready vocab_map of n_static + cap entries for the
// restricted head: a repeated id ties with itself and changes no argmax.
#pragma once

#include <cstdint>

namespace sv {

struct DraftListHeader {
    int32_t V, n_static, cap, count;
    int32_t pad[4];
};

__host__ __device__ inline size_t draft_list_bitmap_words(int V)
{
    return ((static_cast<size_t>(V) + 31) / 32 + 3) / 4 * 4;   // 16-byte multiple
}

__host__ __device__ inline size_t draft_list_ids_offset(int V)
{
    return sizeof(DraftListHeader) + 4 * draft_list_bitmap_words(V);
}

// Fill the header, the id array and the static ids' bits (the bitmap was
// zeroed on the stream before).  One thread per list entry.
__global__ void draft_list_init_kernel(uint8_t *ws, const int32_t *static_ids, int n_static, int V, int cap)
{
    DraftListHeader *h = reinterpret_cast<DraftListHeader *>(ws);
    uint32_t *bitmap = reinterpret_cast<uint32_t *>(ws + sizeof(DraftListHeader));
    int32_t *ids = reinterpret_cast<int32_t *>(ws + draft_list_ids_offset(V));
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i == 0) {
        h->V = V;
        h->n_static = n_static;
        h->cap = cap;
        h->count = 0;
    }
    if (i < n_static) {
        const int t = static_ids[i];
        ids[i] = t;
        if (t >= 0 && t < V) atomicOr(&bitmap[t >> 5], 1u << (t & 31));
    } else if (i < n_static + cap) {
        ids[i] = static_ids[0];
    }
}

// Append tokens[0..n) in order: a token in [0, V) whose bit is clear is
// written to the next free dynamic slot and its bit set, until cap tokens
// have been added.  One warp, 32 tokens per round: lanes holding the same
// token keep only the first, a ballot gives each new token its slot, so the
// result depends only on the token order.  Bitmap words are read through L2
// (they may have been set by this warp's atomics in an earlier round).
__global__ void draft_list_add_kernel(uint8_t *ws, const int32_t *tokens, int n)
{
    DraftListHeader *h = reinterpret_cast<DraftListHeader *>(ws);
    uint32_t *bitmap = reinterpret_cast<uint32_t *>(ws + sizeof(DraftListHeader));
    const int lane = threadIdx.x;
    const int V = h->V, n_static = h->n_static, cap = h->cap;
    int32_t *ids = reinterpret_cast<int32_t *>(ws + draft_list_ids_offset(V));
    int count = h->count;
    for (int base = 0; base < n && count < cap; base += 32) {
        const int i = base + lane;
        const int t = i < n ? tokens[i] : -1;
        const bool in_range = t >= 0 && t < V;
        const unsigned same = __match_any_sync(0xFFFFFFFFu, t);
        const bool first = (__ffs(same) - 1) == lane;
        bool fresh = false;
        if (in_range && first) fresh = ((__ldcg(&bitmap[t >> 5]) >> (t & 31)) & 1u) == 0u;
        const unsigned bal = __ballot_sync(0xFFFFFFFFu, fresh);
        const int pos = count + __popc(bal & ((1u << lane) - 1u));
        if (fresh && pos < cap) {
            ids[n_static + pos] = t;
            atomicOr(&bitmap[t >> 5], 1u << (t & 31));
        }
        count = min(cap, count + __popc(bal));
        __syncwarp();
    }
    if (lane == 0) h->count = count;
}

}  // namespace sv
