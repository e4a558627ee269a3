// Experts held in host memory, streamed into a pool of HBM weight slots on demand.
//
// Page "Data Flow", "Ring Buffer State Machine": expert weights live in a ring of slots keyed
// by (layer, expert); a slot stays valid with its expert identity after use, and a later
// request for the same key is a hit.  A miss takes an EMPTY slot, else the least recently
// used idle slot (never one the current pass reads); freshly loaded slots carry the new
// tick.  "Handling Misses": correctness never depends on the cache.  Page "Layer-Major
// Batched Prefill", "Retention, never replay": the reuse comes from keeping what was read.
//
// On GB300 the weights sit in Grace memory (pinned, so the GPU reads it directly over
// NVLink-C2C) and the slots in HBM.  Everything is decided on the device from the union that
// the union kernel left there, so a layer needs no host synchronisation:
//   stream_plan_kernel   one CTA: hits, idle slots ranked by (stamp, slot id), misses in
//                        union order take them; writes the union's slot ids (the FFN's
//                        expert ids into the pool) and the copy list
//   stream_copy_kernel   grid-stride over (copy, tensor, 32 KB piece): 16-byte loads from
//                        host memory, 8 per thread in flight, stores into the slot
// State buffer (int32): [0] tick, [1] n_keys, [2] n_slots, [3] 0, then slot_of[n_keys]
// (slot holding the key or -1), owner[n_slots] (key or -1), stamp[n_slots] (tick of the last
// use, -1 while empty).
#include "smoe_internal.cuh"

#include <algorithm>

namespace smoe {
namespace {

constexpr int kStateHeader = 4;
constexpr int kPlanThreads = kMaxExperts;   // one thread per union position and per slot
constexpr int kCopyThreads = 256;
constexpr int kCopyPer = 8;                  // 16-byte loads in flight per thread
constexpr int64_t kPiece = (int64_t)kCopyThreads * kCopyPer;   // 16-byte units per piece (32 KB)

__global__ void stream_init_kernel(int32_t* state, int n_keys, int n_slots) {
    const int64_t n = kStateHeader + (int64_t)n_keys + 2 * (int64_t)n_slots;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
        int32_t v = -1;
        if (i == 0 || i == 3) v = 0;
        else if (i == 1) v = n_keys;
        else if (i == 2) v = n_slots;
        state[i] = v;
    }
}

// Thread t: union position t (hit / miss) and slot t (idle rank).  Keys of one union are
// distinct and a slot's previous key is never in the union (it would have been a hit), so the
// writes of different threads touch different entries.
__global__ void __launch_bounds__(kPlanThreads) stream_plan_kernel(int32_t* __restrict__ state, int n_keys, int S,
                                                                   int key_base, int E,
                                                                   const int32_t* __restrict__ union_ids,
                                                                   const int32_t* __restrict__ n_union,
                                                                   int32_t* __restrict__ slot_ids,
                                                                   int32_t* __restrict__ copy_list,
                                                                   uint32_t* __restrict__ status) {
    __shared__ int in_use[kPlanThreads];    // slot read by a hit of this call
    __shared__ int stamp_s[kPlanThreads];
    __shared__ int cand[kPlanThreads];      // idle slots in eviction order
    __shared__ int is_miss[kPlanThreads];
    __shared__ int bad;
    int32_t* slot_of = state + kStateHeader;
    int32_t* owner = slot_of + n_keys;
    int32_t* stamp = owner + S;
    const int t = threadIdx.x;
    if (t == 0) bad = state[1] != n_keys || state[2] != S;
    in_use[t] = 0;
    is_miss[t] = 0;
    __syncthreads();
    const int nu = *n_union;
    if (nu < 0 || nu > E) bad = 1;   // (same value from every thread)
    __syncthreads();
    const int tick = state[0] + 1;
    int key = -1, hit = -1;
    if (!bad && t < nu) {
        const int e = union_ids[t];
        key = key_base + e;
        if (e < 0 || e >= E || key < 0 || key >= n_keys) {
            bad = 1;
        } else {
            hit = slot_of[key];
            if (hit >= S) bad = 1;
            else if (hit >= 0) in_use[hit] = 1;
            else is_miss[t] = 1;
        }
    }
    if (t < S) stamp_s[t] = stamp[t];
    __syncthreads();
    if (bad) {
        if (t == 0) {
            atomicOr(status, SMOE_FAULT_SLOT_POOL);
            copy_list[0] = 0;
        }
        if (t < E) slot_ids[t] = -1;   // the FFN flags and skips these experts
        return;
    }
    const bool idle = t < S && !in_use[t];
    if (idle) {   // rank among the idle slots by (stamp, slot id)
        const int mine = stamp_s[t];
        int r = 0;
        for (int s = 0; s < S; ++s)
            r += !in_use[s] && (stamp_s[s] < mine || (stamp_s[s] == mine && s < t));
        cand[r] = t;
    }
    const int n_idle = __syncthreads_count(idle);
    if (t < nu) {
        if (hit >= 0) {
            stamp[hit] = tick;
            slot_ids[t] = hit;
        } else {
            int m = 0;   // rank of this miss in union order
            for (int u = 0; u < t; ++u) m += is_miss[u];
            if (m < n_idle) {
                const int s = cand[m];
                const int old = owner[s];
                if (old >= 0 && old < n_keys) slot_of[old] = -1;
                owner[s] = key;
                slot_of[key] = s;
                stamp[s] = tick;
                slot_ids[t] = s;
                copy_list[1 + 2 * m] = key - key_base;
                copy_list[2 + 2 * m] = s;
            } else {   // fewer slots than the union needs (the host check prevents it)
                slot_ids[t] = -1;
                atomicOr(status, SMOE_FAULT_SLOT_POOL);
            }
        }
    }
    const int n_miss = __syncthreads_count(t < nu && hit < 0);
    if (t == 0) {
        copy_list[0] = n_miss < n_idle ? n_miss : n_idle;
        state[0] = tick;
    }
}

__global__ void __launch_bounds__(kCopyThreads) stream_copy_kernel(StreamCopyArgs a) {
    const int n = a.list[0];
    if (n < 0 || n > a.E) {
        if (blockIdx.x == 0 && threadIdx.x == 0) atomicOr(a.status, SMOE_FAULT_SLOT_POOL);
        return;
    }
    const int64_t total = (int64_t)n * a.pieces_per_copy;
    for (int64_t q = blockIdx.x; q < total; q += gridDim.x) {
        const int c = (int)(q / a.pieces_per_copy);
        int j = (int)(q - (int64_t)c * a.pieces_per_copy);
        int r = 0;
        while (r < a.n_regions - 1 && j >= a.region[r].pieces) j -= a.region[r++].pieces;
        const int e = a.list[1 + 2 * c], s = a.list[2 + 2 * c];
        if (e < 0 || e >= a.E || s < 0 || s >= a.S) {
            if (threadIdx.x == 0) atomicOr(a.status, SMOE_FAULT_SLOT_POOL);
            continue;
        }
        const StreamRegion& R = a.region[r];
        const uint4* src = R.src + (int64_t)e * R.n16 + (int64_t)j * kPiece;
        uint4* dst = R.dst + (int64_t)s * R.n16 + (int64_t)j * kPiece;
        const int64_t left = R.n16 - (int64_t)j * kPiece;
        uint4 v[kCopyPer];
#pragma unroll
        for (int k = 0; k < kCopyPer; ++k) {
            const int64_t i = (int64_t)k * kCopyThreads + threadIdx.x;
            if (i < left) v[k] = __ldg(src + i);
        }
#pragma unroll
        for (int k = 0; k < kCopyPer; ++k) {
            const int64_t i = (int64_t)k * kCopyThreads + threadIdx.x;
            if (i < left) dst[i] = v[k];
        }
    }
}

}  // namespace

size_t stream_state_words(int n_keys, int n_slots) {
    return (size_t)kStateHeader + (size_t)n_keys + 2 * (size_t)n_slots;
}

int64_t stream_pieces(int64_t n16) { return (n16 + kPiece - 1) / kPiece; }

cudaError_t launch_stream_init(int32_t* state, int n_keys, int n_slots, cudaStream_t stream) {
    const int64_t n = (int64_t)stream_state_words(n_keys, n_slots);
    const int blocks = (int)std::min<int64_t>((n + 255) / 256, 1024);
    stream_init_kernel<<<blocks, 256, 0, stream>>>(state, n_keys, n_slots);
    return cudaGetLastError();
}

cudaError_t launch_stream_plan(int32_t* state, int n_keys, int n_slots, int key_base, int E, const int32_t* union_ids,
                               const int32_t* n_union, int32_t* slot_ids, int32_t* copy_list, uint32_t* status,
                               cudaStream_t stream) {
    stream_plan_kernel<<<1, kPlanThreads, 0, stream>>>(state, n_keys, n_slots, key_base, E, union_ids, n_union,
                                                      slot_ids, copy_list, status);
    return cudaGetLastError();
}

cudaError_t launch_stream_copy(const StreamCopyArgs& a, cudaStream_t stream) {
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return cudaErrorInvalidDevice;
    stream_copy_kernel<<<sms * 8, kCopyThreads, 0, stream>>>(a);   // 8 CTAs of 256 per SM: 256 KB in flight
    return cudaGetLastError();
}

}  // namespace smoe
