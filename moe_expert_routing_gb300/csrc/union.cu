// Step 2, the expert union of a chunk and the per-expert token lists.
//
// Page "Layer-Major Batched Prefill", "The Inversion": the chunk's routed experts are
// deduplicated into a UNION; each union expert is then read once and applied to every
// token routed to it.  Page "SSD Streaming Expert Layers", "Execution Paths" (exact):
// deduplicate the routing indices; "Sorting and Compilation": the sorted gather that
// groups tokens by expert.
//
// Entirely on the device (no host synchronisation): histogram of expert ids -> exclusive
// scan over experts (union positions and list offsets) -> a stable scatter of the flat
// (token, rank) entries into the lists.  The scatter is stable in the flat order t*K + k,
// so each list is in ascending token order and the output is deterministic: within a
// 1024-entry chunk, equal ids are ranked with __match_any_sync inside each warp and a
// per-expert prefix over the 32 warps.
//   up to 128 entries:   union_warp_kernel, one warp, registers and shuffles only (decode)
//   up to 1024 entries:  union_kernel, one CTA
//   more:                chunk_hist_kernel (one CTA per 1024-entry chunk: per-chunk counts)
//                        -> chunk_scan_kernel (one CTA: union, list offsets, chunk bases)
//                        -> chunk_scatter_kernel (one CTA per chunk)
#include "union_block.cuh"

namespace smoe {
namespace {

constexpr int kThreads = 1024;
constexpr int kWarps = kThreads / 32;

// Up to 128 entries: one warp (union_of_warp); up to 1024: one CTA (union_of_block).
__global__ void __launch_bounds__(32) union_warp_kernel(const int32_t* __restrict__ idx, int BK, int E,
                                                        int32_t* __restrict__ union_ids,
                                                        int32_t* __restrict__ n_union,
                                                        int32_t* __restrict__ offsets,
                                                        int32_t* __restrict__ token_list,
                                                        int32_t* __restrict__ slot_list, int K,
                                                        uint32_t* __restrict__ status) {
    union_of_warp(idx, BK, E, union_ids, n_union, offsets, token_list, slot_list, K, status);
}

template <int THREADS>
__global__ void __launch_bounds__(THREADS) union_kernel(const int32_t* __restrict__ idx, int BK, int E,
                                                         int32_t* __restrict__ union_ids,
                                                         int32_t* __restrict__ n_union,
                                                         int32_t* __restrict__ offsets,
                                                         int32_t* __restrict__ token_list,
                                                         int32_t* __restrict__ slot_list, int K,
                                                         uint32_t* __restrict__ status) {
    union_of_block<THREADS>(idx, BK, E, union_ids, n_union, offsets, token_list, slot_list, K, status);
}


// Rank of entry i among the equal ids of its 1024-entry chunk (stable), with the per-expert
// prefix over the chunk's 32 warps; wcount[w][e] is scratch, zero on entry and on exit.
__device__ __forceinline__ int chunk_rank(int e, int E, int (*wcount)[kMaxExperts]) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const unsigned peers = __match_any_sync(0xffffffffu, e);
    const int rank = __popc(peers & ((1u << lane) - 1u));
    if (e >= 0 && rank == 0) wcount[warp][e] = __popc(peers);
    __syncthreads();
    for (int x = tid; x < E; x += kThreads) {
        int s = 0;
        for (int w = 0; w < kWarps; ++w) {
            const int cnt = wcount[w][x];
            wcount[w][x] = s;
            s += cnt;
        }
    }
    __syncthreads();
    return e >= 0 ? wcount[warp][e] + rank : 0;
}

// Per-chunk histogram; cnt[c][e] (E entries per chunk), bad[0] set on an id outside [0, E).
__global__ void __launch_bounds__(kThreads) chunk_hist_kernel(const int32_t* __restrict__ idx, int BK, int E,
                                                              int32_t* __restrict__ cnt, int32_t* __restrict__ bad) {
    __shared__ int count[kMaxExperts];
    const int tid = threadIdx.x;
    for (int e = tid; e < E; e += kThreads) count[e] = 0;
    __syncthreads();
    const int i = blockIdx.x * kThreads + tid;
    if (i < BK) {
        const int e = idx[i];
        if (e < 0 || e >= E) atomicOr(bad, 1);
        else atomicAdd(&count[e], 1);
    }
    __syncthreads();
    for (int e = tid; e < E; e += kThreads) cnt[(size_t)blockIdx.x * E + e] = count[e];
}

// Union and offsets from the per-chunk counts; cnt[c][e] is replaced by the first list
// position of chunk c's entries of expert e.
__global__ void __launch_bounds__(kThreads) chunk_scan_kernel(int32_t* __restrict__ cnt, int chunks, int E,
                                                              const int32_t* __restrict__ bad,
                                                              int32_t* __restrict__ union_ids,
                                                              int32_t* __restrict__ n_union,
                                                              int32_t* __restrict__ offsets,
                                                              uint32_t* __restrict__ status) {
    __shared__ int total[kMaxExperts];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (*bad) {
        if (tid == 0) {
            atomicOr(status, SMOE_FAULT_EXPERT_INDEX);
            *n_union = 0;
            offsets[0] = 0;
        }
        return;
    }
    for (int e = tid; e < E; e += kThreads) {
        int s = 0;
        for (int c = 0; c < chunks; ++c) s += cnt[(size_t)c * E + e];
        total[e] = s;
    }
    __syncthreads();
    __shared__ int list_off[kMaxExperts];
    if (warp == 0) {
        constexpr int PER = kMaxExperts / 32;
        int c[PER], used = 0, tot = 0;
#pragma unroll
        for (int j = 0; j < PER; ++j) {
            const int e = lane * PER + j;
            c[j] = (e < E) ? total[e] : 0;
            used += c[j] > 0;
            tot += c[j];
        }
        int used_incl = used, tot_incl = tot;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int a = __shfl_up_sync(0xffffffffu, used_incl, off);
            const int b = __shfl_up_sync(0xffffffffu, tot_incl, off);
            if (lane >= off) { used_incl += a; tot_incl += b; }
        }
        int u = used_incl - used, o = tot_incl - tot;
#pragma unroll
        for (int j = 0; j < PER; ++j) {
            const int e = lane * PER + j;
            if (e < E) {
                list_off[e] = o;
                if (c[j] > 0) {
                    union_ids[u] = e;
                    offsets[u] = o;
                    ++u;
                }
                o += c[j];
            }
        }
        if (lane == 31) {
            *n_union = u;
            offsets[u] = o;
        }
    }
    __syncthreads();
    for (int e = tid; e < E; e += kThreads) {
        int s = list_off[e];
        for (int c = 0; c < chunks; ++c) {
            const int n = cnt[(size_t)c * E + e];
            cnt[(size_t)c * E + e] = s;
            s += n;
        }
    }
}

__global__ void __launch_bounds__(kThreads) chunk_scatter_kernel(const int32_t* __restrict__ idx, int BK, int E,
                                                                 int K, const int32_t* __restrict__ base,
                                                                 const int32_t* __restrict__ bad,
                                                                 int32_t* __restrict__ token_list,
                                                                 int32_t* __restrict__ slot_list) {
    __shared__ int wcount[kWarps][kMaxExperts];
    if (*bad) return;
    const int tid = threadIdx.x;
    for (int j = tid; j < kWarps * kMaxExperts; j += kThreads) (&wcount[0][0])[j] = 0;
    __syncthreads();
    const int i = blockIdx.x * kThreads + tid;
    const int e = (i < BK) ? idx[i] : -1;
    const int r = chunk_rank(e, E, wcount);
    if (e >= 0) {
        const int pos = base[(size_t)blockIdx.x * E + e] + r;
        token_list[pos] = i / K;
        slot_list[pos] = i - (i / K) * K;
    }
}

// Routing of a shared expert stored as P slices: every token to every slice with weight 1.
// union_ids[p] = p, offsets[p] = p B, the list of slice p = tokens 0..B-1 in order with slot
// p, weights w[t][p] = 1.
__global__ void __launch_bounds__(256) all_slices_kernel(int B, int P, int32_t* __restrict__ union_ids,
                                                         int32_t* __restrict__ n_union, int32_t* __restrict__ offsets,
                                                         int32_t* __restrict__ token_list,
                                                         int32_t* __restrict__ slot_list, float* __restrict__ w) {
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i <= P) offsets[i] = i * B;
    if (i < P) union_ids[i] = i;
    if (i == 0) *n_union = P;
    if (i < B * P) {
        const int p = i / B, t = i - p * B;
        token_list[i] = t;
        slot_list[i] = p;
        w[(size_t)t * P + p] = 1.f;
    }
}

}  // namespace

int union_chunks(int BK) { return (BK + kThreads - 1) / kThreads; }

cudaError_t launch_all_slices(int B, int P, int32_t* union_ids, int32_t* n_union, int32_t* offsets,
                              int32_t* token_list, int32_t* slot_list, float* w, cudaStream_t stream) {
    const int n = B * P > P + 1 ? B * P : P + 1;
    all_slices_kernel<<<(n + 255) / 256, 256, 0, stream>>>(B, P, union_ids, n_union, offsets, token_list, slot_list,
                                                           w);
    return cudaGetLastError();
}

cudaError_t launch_union(const smoe_layer_desc& D, const int32_t* topk_idx, int B, int32_t* union_ids,
                         int32_t* n_union, int32_t* offsets, int32_t* token_list, int32_t* slot_list,
                         uint32_t* status, int32_t* scratch, cudaStream_t stream) {
    const int BK = B * D.top_k, E = D.num_experts;
    if (BK <= kThreads || !scratch) {
        if (BK <= 128)
            union_warp_kernel<<<1, 32, 0, stream>>>(topk_idx, BK, E, union_ids, n_union, offsets, token_list,
                                                    slot_list, D.top_k, status);
        else
            union_kernel<kThreads><<<1, kThreads, 0, stream>>>(topk_idx, BK, E, union_ids, n_union, offsets,
                                                               token_list, slot_list, D.top_k, status);
        return cudaGetLastError();
    }
    // scratch: [0] bad flag, then the per-chunk counts / bases [chunks][E]
    const int chunks = union_chunks(BK);
    int32_t* bad = scratch;
    int32_t* cnt = scratch + 1;
    cudaError_t e = cudaMemsetAsync(bad, 0, sizeof(int32_t), stream);
    if (e != cudaSuccess) return e;
    chunk_hist_kernel<<<chunks, kThreads, 0, stream>>>(topk_idx, BK, E, cnt, bad);
    chunk_scan_kernel<<<1, kThreads, 0, stream>>>(cnt, chunks, E, bad, union_ids, n_union, offsets, status);
    chunk_scatter_kernel<<<chunks, kThreads, 0, stream>>>(topk_idx, BK, E, D.top_k, cnt, bad, token_list, slot_list);
    return cudaGetLastError();
}

}  // namespace smoe
