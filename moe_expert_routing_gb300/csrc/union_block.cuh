// Step 2 inside one CTA: the expert union of a chunk and its per-expert token lists, as the
// device functions of the one-warp and one-CTA union kernels (union.cu).
//
// Page "Layer-Major Batched Prefill", "The Inversion": the chunk's routed experts are
// deduplicated into a UNION and every union expert is applied to each token routed to it.
// Outputs: union_ids (ascending expert ids), n_union, offsets (list start of each union
// position; offsets[n_union] = B*K), token_list / slot_list (each expert's entries in ascending
// token order, with the rank k of the expert in the token's top-k).  The order is stable in
// the flat entry order t*K + k, so the output is deterministic.  An id outside [0, E) sets
// SMOE_FAULT_EXPERT_INDEX and n_union = 0.
//
// The routing indices are read with ld.global.cg (L2, not the non-coherent path), so the
// functions also hold where the indices were written by other CTAs of the calling kernel.
#pragma once

#include "smoe_internal.cuh"

namespace smoe {
namespace {

// Up to 128 entries, one warp (lane = threadIdx.x & 31; the caller's other warps do not
// enter): lane l holds entries l, l+32, l+64, l+96.  Every entry is compared with every other
// (one shuffle per source entry): less = entries with a smaller expert id (its expert's list
// offset), eqb = earlier entries with the same id; less + eqb is its position in the stable
// expert-major order, and eqb == 0 marks the first entry of its expert, which writes the union
// slot.  The union position of expert e is the number of distinct ids below e, read from a
// 256-bit set of the ids present (OR-reduced over the warp).
__device__ __forceinline__ void union_of_warp(const int32_t* idx, int BK, int E, int32_t* union_ids,
                                              int32_t* n_union, int32_t* offsets, int32_t* token_list,
                                              int32_t* slot_list, int K, uint32_t* status) {
    constexpr int PER = 4;
    constexpr int WORDS = kMaxExperts / 32;
    const int lane = threadIdx.x & 31;
    int e[PER];
    bool bad = false;
#pragma unroll
    for (int j = 0; j < PER; ++j) {
        const int i = lane + 32 * j;
        e[j] = i < BK ? __ldcg(idx + i) : -1;
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

// Any number of entries, one CTA of THREADS threads (all of them enter): histogram of the
// ids, exclusive scans over the experts by warp 0 (union positions and list offsets), then a
// stable scatter, THREADS entries per round: within a round equal ids are ranked with
// __match_any_sync inside each warp and a per-expert prefix over the warps.
template <int THREADS>
__device__ __forceinline__ void union_of_block(const int32_t* idx, int BK, int E, int32_t* union_ids,
                                               int32_t* n_union, int32_t* offsets, int32_t* token_list,
                                               int32_t* slot_list, int K, uint32_t* status) {
    constexpr int WARPS = THREADS / 32;
    __shared__ int count[kMaxExperts];
    __shared__ int list_off[kMaxExperts];  // start of expert e's list
    __shared__ int running[kMaxExperts];   // entries of expert e placed so far
    __shared__ int chunk_base[kMaxExperts];
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
        const int e = __ldcg(idx + i);
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
        const int e = (i < BK) ? __ldcg(idx + i) : -1;
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

}  // namespace
}  // namespace smoe
