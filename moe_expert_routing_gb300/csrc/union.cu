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
#include "smoe_internal.cuh"

namespace smoe {
namespace {

constexpr int kThreads = 1024;
constexpr int kWarps = kThreads / 32;

// Up to 128 entries: lane l holds entries l, l+32, l+64, l+96.  Every entry is compared with
// every other (one shuffle per source entry): less = entries with a smaller expert id (its
// expert's list offset), eqb = earlier entries with the same id; less + eqb is its position
// in the stable expert-major order, and eqb == 0 marks the first entry of its expert, which
// writes the union slot.  The union position of expert e is the number of distinct ids below
// e, read from a 256-bit set of the ids present (OR-reduced over the warp).
__global__ void __launch_bounds__(32) union_warp_kernel(const int32_t* __restrict__ idx, int BK, int E,
                                                        int32_t* __restrict__ union_ids,
                                                        int32_t* __restrict__ n_union,
                                                        int32_t* __restrict__ offsets,
                                                        int32_t* __restrict__ token_list,
                                                        int32_t* __restrict__ slot_list, int K,
                                                        uint32_t* __restrict__ status) {
    constexpr int PER = 4;
    constexpr int WORDS = kMaxExperts / 32;
    const int lane = threadIdx.x;
    int e[PER];
    bool bad = false;
#pragma unroll
    for (int j = 0; j < PER; ++j) {
        const int i = lane + 32 * j;
        e[j] = i < BK ? idx[i] : -1;
        if (i < BK && (e[j] < 0 || e[j] >= E)) bad = true;
    }
    if (__any_sync(0xffffffffu, bad)) {
        if (lane == 0) {
            atomicOr(status, SMOE_FAULT_EXPERT_INDEX);
            *n_union = 0;
            offsets[0] = 0;
        }
        return;
    }
    int less[PER], eqb[PER];
#pragma unroll
    for (int j = 0; j < PER; ++j) less[j] = eqb[j] = 0;
#pragma unroll
    for (int sj = 0; sj < PER; ++sj) {
        if (32 * sj >= BK) break;
        const int n = BK - 32 * sj < 32 ? BK - 32 * sj : 32;
        for (int s = 0; s < n; ++s) {
            const int es = __shfl_sync(0xffffffffu, e[sj], s);
            const int is = 32 * sj + s;
#pragma unroll
            for (int j = 0; j < PER; ++j) {
                less[j] += es < e[j];
                eqb[j] += es == e[j] && is < lane + 32 * j;
            }
        }
    }
    uint32_t present[WORDS];
    int nu = 0;
#pragma unroll
    for (int w = 0; w < WORDS; ++w) {
        uint32_t mine = 0;
#pragma unroll
        for (int j = 0; j < PER; ++j)
            if (lane + 32 * j < BK && (e[j] >> 5) == w) mine |= 1u << (e[j] & 31);
        present[w] = __reduce_or_sync(0xffffffffu, mine);
        nu += __popc(present[w]);
    }
#pragma unroll
    for (int j = 0; j < PER; ++j) {
        const int i = lane + 32 * j;
        if (i >= BK) continue;
        const int pos = less[j] + eqb[j];
        token_list[pos] = i / K;
        slot_list[pos] = i - (i / K) * K;
        if (eqb[j] == 0) {
            int u = 0;
#pragma unroll
            for (int w = 0; w < WORDS; ++w) {
                if (w < (e[j] >> 5)) u += __popc(present[w]);
                else if (w == (e[j] >> 5)) u += __popc(present[w] & ((1u << (e[j] & 31)) - 1u));
            }
            union_ids[u] = e[j];
            offsets[u] = less[j];
        }
    }
    if (lane == 0) {
        *n_union = nu;
        offsets[nu] = BK;
    }
}

template <int THREADS>
__global__ void __launch_bounds__(THREADS) union_kernel(const int32_t* __restrict__ idx, int BK, int E,
                                                         int32_t* __restrict__ union_ids,
                                                         int32_t* __restrict__ n_union,
                                                         int32_t* __restrict__ offsets,
                                                         int32_t* __restrict__ token_list,
                                                         int32_t* __restrict__ slot_list, int K,
                                                         uint32_t* __restrict__ status) {
    __shared__ int count[kMaxExperts];
    __shared__ int list_off[kMaxExperts];  // start of expert e's list
    __shared__ int running[kMaxExperts];   // entries of expert e placed so far
    __shared__ int chunk_base[kMaxExperts];
    constexpr int WARPS = THREADS / 32;
    __shared__ int wcount[WARPS][kMaxExperts];
    __shared__ int bad;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

    if (tid == 0) bad = 0;
    for (int e = tid; e < kMaxExperts; e += THREADS) {
        count[e] = 0;
        running[e] = 0;
    }
    for (int i = tid; i < WARPS * kMaxExperts; i += THREADS) (&wcount[0][0])[i] = 0;
    __syncthreads();

    // histogram + validation
    for (int i = tid; i < BK; i += THREADS) {
        const int e = idx[i];
        if (e < 0 || e >= E) bad = 1;
        else atomicAdd(&count[e], 1);
    }
    __syncthreads();
    if (bad) {
        if (tid == 0) {
            atomicOr(status, SMOE_FAULT_EXPERT_INDEX);
            *n_union = 0;
            offsets[0] = 0;
        }
        return;
    }

    // exclusive scans over experts (E <= 256) by warp 0: union positions and list offsets
    if (warp == 0) {
        constexpr int PER = kMaxExperts / 32;
        int c[PER], used = 0, tot = 0;
#pragma unroll
        for (int j = 0; j < PER; ++j) {
            const int e = lane * PER + j;
            c[j] = (e < E) ? count[e] : 0;
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

    // stable scatter, THREADS entries per round
    for (int base = 0; base < BK; base += THREADS) {
        const int i = base + tid;
        const int e = (i < BK) ? idx[i] : -1;
        const unsigned peers = __match_any_sync(0xffffffffu, e);
        const int rank = __popc(peers & ((1u << lane) - 1u));
        if (e >= 0 && rank == 0) wcount[warp][e] = __popc(peers);
        __syncthreads();
        for (int x = tid; x < E; x += THREADS) {
            int s = 0;
            for (int w = 0; w < WARPS; ++w) {
                const int cnt = wcount[w][x];
                wcount[w][x] = s;
                s += cnt;
            }
            chunk_base[x] = running[x];
            running[x] += s;
        }
        __syncthreads();
        if (e >= 0) {
            const int pos = list_off[e] + chunk_base[e] + wcount[warp][e] + rank;
            token_list[pos] = i / K;
            slot_list[pos] = i - (i / K) * K;
        }
        __syncthreads();
        for (int x = tid; x < E; x += THREADS)
            for (int w = 0; w < WARPS; ++w) wcount[w][x] = 0;
        __syncthreads();
    }
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
