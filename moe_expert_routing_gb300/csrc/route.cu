// Step 1, exact routing: router gate matvec, softmax, top-k, norm_topk_prob.
//
// Page "Layer-Major Batched Prefill", "Choreography Per Chunk" step 5: the real router gate
// (an E x d_model matvec) evaluated on every token's hidden state, norm_topk_prob
// re-normalisation of the selected weights.  Page "Surface Scout", "The Model Config":
// norm_topk_prob re-normalises the top-k routing weights to sum 1.
//
// Two kernels:
//   gate_logits_kernel  logits[s][t][e] = sum over split s of W[e][i] * x[t][i] on the tensor
//                       cores: x is bf16 and every fp32 gate weight is split into three bf16
//                       terms (hi + mid + lo, exact up to the last bit), so mma.sync bf16 with
//                       fp32 accumulation gives fp32-accurate logits.  Split-K over d so that
//                       even a single token spreads the 2 MB gate read over ~100 SMs; the
//                       partials are summed in a fixed order by the top-k kernel, so results
//                       are deterministic.
//   topk_kernel         one CTA per token: sums the partials (+ bias) with one thread per
//                       expert, selects the experts of ranks 0..K-1 (descending logit, ties ->
//                       lower expert id; by parallel rank counting for small batches, by K
//                       rounds of a warp arg-max for large ones), softmax weights.
#include "smoe_internal.cuh"

#include <math.h>

namespace smoe {
namespace {

constexpr int kMaxSplits = 32;
constexpr int kExpertsPerCta = 128;   // 8 warps x 16 experts

__device__ __forceinline__ void mma_bf16(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};\n"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Two fp32 values -> three bf16x2 terms (hi, mid, lo) with hi + mid + lo == the values
// (the last bit of lo may round).
__device__ __forceinline__ void split3(float2 v, uint32_t& hi, uint32_t& mid, uint32_t& lo) {
    const __nv_bfloat162 h = __float22bfloat162_rn(v);
    const float2 r1 = make_float2(v.x - __low2float(h), v.y - __high2float(h));
    const __nv_bfloat162 m = __float22bfloat162_rn(r1);
    const float2 r2 = make_float2(r1.x - __low2float(m), r1.y - __high2float(m));
    const __nv_bfloat162 l = __float22bfloat162_rn(r2);
    hi = *reinterpret_cast<const uint32_t*>(&h);
    mid = *reinterpret_cast<const uint32_t*>(&m);
    lo = *reinterpret_cast<const uint32_t*>(&l);
}

// CTA: WARPS warps x 16 experts, 8*NT tokens, one k-split of kchunk inputs.  Warp: A = 16 gate
// rows (three bf16 terms), B = NT 8-token tiles of x, fp32 accumulators.  The loads of KB
// k-steps are issued together before their products, so a warp has KB steps of its weight
// and activation reads in flight (kchunk is a multiple of 16 * KB).
template <int NT, int KB, int WARPS>
__device__ __forceinline__ void gate_tile(const uint16_t* __restrict__ x, const float* __restrict__ W, int B, int E,
                                          int d, int kchunk, float* __restrict__ partial) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, c = lane & 3;
    const int e0 = blockIdx.y * (WARPS * 16) + warp * 16;
    if (e0 >= E) return;
    const int t0 = blockIdx.x * 8 * NT;
    const int k_begin = blockIdx.z * kchunk, k_end = k_begin + kchunk;
    const int ea = e0 + g, eb = e0 + g + 8;
    const float* wa = W + (size_t)(ea < E ? ea : 0) * d;
    const float* wb = W + (size_t)(eb < E ? eb : 0) * d;
    const uint16_t* xr[NT];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
        const int t = t0 + nt * 8 + g;
        xr[nt] = x + (size_t)(t < B ? t : 0) * d;
    }
    float acc[NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int i = 0; i < 4; ++i) acc[nt][i] = 0.f;
    for (int kb = k_begin; kb < k_end; kb += 16 * KB) {
        float2 wv[KB][4];
        uint32_t xv[KB][NT][2];
#pragma unroll
        for (int j = 0; j < KB; ++j) {
            const int k0 = kb + 16 * j + 2 * c, k1 = k0 + 8;
            wv[j][0] = __ldg(reinterpret_cast<const float2*>(wa + k0));
            wv[j][1] = __ldg(reinterpret_cast<const float2*>(wb + k0));
            wv[j][2] = __ldg(reinterpret_cast<const float2*>(wa + k1));
            wv[j][3] = __ldg(reinterpret_cast<const float2*>(wb + k1));
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                xv[j][nt][0] = __ldg(reinterpret_cast<const uint32_t*>(xr[nt] + k0));
                xv[j][nt][1] = __ldg(reinterpret_cast<const uint32_t*>(xr[nt] + k1));
            }
        }
#pragma unroll
        for (int j = 0; j < KB; ++j) {
            if (ea >= E) wv[j][0] = wv[j][2] = make_float2(0.f, 0.f);
            if (eb >= E) wv[j][1] = wv[j][3] = make_float2(0.f, 0.f);
            uint32_t a[3][4];   // [term][a0..a3]: rows g / g+8, k 2c.. / 2c+8..
            split3(wv[j][0], a[0][0], a[1][0], a[2][0]);
            split3(wv[j][1], a[0][1], a[1][1], a[2][1]);
            split3(wv[j][2], a[0][2], a[1][2], a[2][2]);
            split3(wv[j][3], a[0][3], a[1][3], a[2][3]);
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int term = 2; term >= 0; --term)   // small terms first
                    mma_bf16(acc[nt], a[term][0], a[term][1], a[term][2], a[term][3], xv[j][nt][0], xv[j][nt][1]);
        }
    }
    float* out = partial + (size_t)blockIdx.z * B * E;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int t = t0 + nt * 8 + 2 * c + (i & 1);
            const int e = (i & 2) ? eb : ea;
            if (t < B && e < E) out[(size_t)t * E + e] = acc[nt][i];
        }
}

template <int NT, int KB, int WARPS = 8>
__global__ void __launch_bounds__(32 * WARPS) gate_logits_kernel(const uint16_t* __restrict__ x,
                                                                 const float* __restrict__ W, int B, int E, int d,
                                                                 int kchunk, float* __restrict__ partial) {
    gate_tile<NT, KB, WARPS>(x, W, B, E, d, kchunk, partial);
}

// Large batches: the same tile with the CTA's 64 token rows staged in shared memory piece by
// piece (256 inputs at a time, cp.async), so the 8 warps read each activation once from
// global memory instead of once per warp.  Rows padded by 16 bytes: the 8 rows a fragment
// load touches fall in different banks.
constexpr int kPiece = 256;
constexpr int kPieceStride = kPiece + 8;   // bf16 elements per staged row

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(dst), "l"(src) : "memory");
}

template <int NT, int KB>
__global__ void __launch_bounds__(256) gate_logits_staged_kernel(const uint16_t* __restrict__ x,
                                                                 const float* __restrict__ W, int B, int E, int d,
                                                                 int kchunk, float* __restrict__ partial) {
    extern __shared__ __align__(16) uint16_t xs[];   // [8 NT rows][kPieceStride]
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, c = lane & 3;
    const int e0 = blockIdx.y * kExpertsPerCta + warp * 16;
    const int t0 = blockIdx.x * 8 * NT;
    const int k_begin = blockIdx.z * kchunk, k_end = k_begin + kchunk;
    const int ea = e0 + g, eb = e0 + g + 8;
    const float* wa = W + (size_t)(ea < E ? ea : 0) * d;
    const float* wb = W + (size_t)(eb < E ? eb : 0) * d;
    const uint32_t xs_base = static_cast<uint32_t>(__cvta_generic_to_shared(xs));
    float acc[NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int i = 0; i < 4; ++i) acc[nt][i] = 0.f;
    for (int kp = k_begin; kp < k_end; kp += kPiece) {
        // stage rows t0.., inputs kp..kp+255: 32 chunks of 16 bytes per row
        for (int i = threadIdx.x; i < 8 * NT * 32; i += 256) {
            const int row = i >> 5, ch = i & 31;
            const int t = t0 + row < B ? t0 + row : 0;
            cp_async16(xs_base + (uint32_t)(row * kPieceStride + ch * 8) * 2u, x + (size_t)t * d + kp + ch * 8);
        }
        asm volatile("cp.async.wait_all;\n" ::: "memory");
        __syncthreads();
        if (e0 < E) {
            // each piece accumulates on its own (48 MMAs), then adds into acc in IEEE fp32: the
            // tensor core's accumulation is not IEEE-rounded, and one chain over thousands of
            // inputs (a single split) drifts by ~1e-4 of the logit
            float pacc[NT][4];
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int i = 0; i < 4; ++i) pacc[nt][i] = 0.f;
            for (int kb = 0; kb < kPiece; kb += 16 * KB) {
                float2 wv[KB][4];
#pragma unroll
                for (int j = 0; j < KB; ++j) {
                    const int k0 = kp + kb + 16 * j + 2 * c, k1 = k0 + 8;
                    wv[j][0] = __ldg(reinterpret_cast<const float2*>(wa + k0));
                    wv[j][1] = __ldg(reinterpret_cast<const float2*>(wb + k0));
                    wv[j][2] = __ldg(reinterpret_cast<const float2*>(wa + k1));
                    wv[j][3] = __ldg(reinterpret_cast<const float2*>(wb + k1));
                }
#pragma unroll
                for (int j = 0; j < KB; ++j) {
                    if (ea >= E) wv[j][0] = wv[j][2] = make_float2(0.f, 0.f);
                    if (eb >= E) wv[j][1] = wv[j][3] = make_float2(0.f, 0.f);
                    uint32_t a[3][4];   // [term][a0..a3]: rows g / g+8, k 2c.. / 2c+8..
                    split3(wv[j][0], a[0][0], a[1][0], a[2][0]);
                    split3(wv[j][1], a[0][1], a[1][1], a[2][1]);
                    split3(wv[j][2], a[0][2], a[1][2], a[2][2]);
                    split3(wv[j][3], a[0][3], a[1][3], a[2][3]);
                    const int kk = kb + 16 * j + 2 * c;
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt) {
                        const uint16_t* xr = xs + (nt * 8 + g) * kPieceStride + kk;
                        const uint32_t b0 = *reinterpret_cast<const uint32_t*>(xr);
                        const uint32_t b1 = *reinterpret_cast<const uint32_t*>(xr + 8);
#pragma unroll
                        for (int term = 2; term >= 0; --term)   // small terms first
                            mma_bf16(pacc[nt], a[term][0], a[term][1], a[term][2], a[term][3], b0, b1);
                    }
                }
            }
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int i = 0; i < 4; ++i) acc[nt][i] += pacc[nt][i];
        }
        __syncthreads();   // the piece is consumed before the next one is staged
    }
    if (e0 >= E) return;
    float* out = partial + (size_t)blockIdx.z * B * E;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int t = t0 + nt * 8 + 2 * c + (i & 1);
            const int e = (i & 2) ? eb : ea;
            if (t < B && e < E) out[(size_t)t * E + e] = acc[nt][i];
        }
}

// Tokens per CTA tile of the router: 8-token tiles up to 64 tokens (many small CTAs spread the
// gate read widest; at 64 tokens one staged 64-token tile per split measured 4.8 us slower per
// layer), 64-token tiles with the activations staged in shared memory beyond.
int tile_tokens(int B) { return B <= 64 ? 8 : 64; }

// Selection and weights of one token by one warp, from its E logits in shared memory (and, with
// RANK, the experts of ranks 0..K+n_spec-1 already placed in by_rank): the max logit and, where
// needed, the full softmax denominator by butterflies; without RANK, K + n_spec rounds of a
// warp arg-max over lanes holding experts l, l+32, ...; lane k then holds rank k's expert and
// computes its weight.
template <bool RANK>
__device__ __forceinline__ void topk_select_warp(const float* logit, const int* by_rank, int t, int E, int K, int norm,
                                                 int32_t* __restrict__ idx_out, float* __restrict__ w_out,
                                                 int n_spec, int32_t* __restrict__ spec_idx,
                                                 float* __restrict__ spec_p) {
    const int lane = threadIdx.x & 31;
    const int ranks = K + n_spec;   // <= 32
    constexpr int PER = kMaxExperts / 32;
    float v[PER];   // lane l holds experts l, l+32, ...
    bool live[PER];
#pragma unroll
    for (int i = 0; i < PER; ++i) {
        live[i] = lane + 32 * i < E;
        v[i] = live[i] ? logit[lane + 32 * i] : 0.f;
    }
    // max logit over all experts and, where needed, the full softmax denominator (butterflies)
    float mx = -INFINITY;
#pragma unroll
    for (int i = 0; i < PER; ++i)
        if (live[i]) mx = fmaxf(mx, v[i]);
#pragma unroll
    for (int off = 16; off; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
    float z_all = 0.f;
    if (!norm || spec_p) {
#pragma unroll
        for (int i = 0; i < PER; ++i)
            if (live[i]) z_all += expf(v[i] - mx);
#pragma unroll
        for (int off = 16; off; off >>= 1) z_all += __shfl_xor_sync(0xffffffffu, z_all, off);
    }
    int sel_i = 0;   // lane k: the expert of rank k
    if (RANK) {
        sel_i = lane < ranks ? by_rank[lane] : 0;
    } else {
        for (int k = 0; k < ranks; ++k) {
            float bv = -INFINITY;
            int bi = 0x7fffffff;
#pragma unroll
            for (int i = 0; i < PER; ++i) {
                const int ex = lane + 32 * i;
                if (live[i] && (v[i] > bv || (v[i] == bv && ex < bi))) { bv = v[i]; bi = ex; }
            }
#pragma unroll
            for (int off = 16; off; off >>= 1) {
                const float ov = __shfl_xor_sync(0xffffffffu, bv, off);
                const int oi = __shfl_xor_sync(0xffffffffu, bi, off);
                if (ov > bv || (ov == bv && oi < bi)) { bv = ov; bi = oi; }
            }
            if (lane == k) sel_i = bi < E ? bi : 0;   // (no live finite logit left: NaN input)
            if ((bi & 31) == lane) {
#pragma unroll
                for (int i = 0; i < PER; ++i)
                    if (i == (bi >> 5)) live[i] = false;
            }
        }
    }
    const float p = (lane < ranks) ? expf(logit[sel_i] - mx) : 0.f;
    float z = (lane < K) ? p : 0.f;
    if (norm) {
#pragma unroll
        for (int off = 16; off; off >>= 1) z += __shfl_xor_sync(0xffffffffu, z, off);
    } else {
        z = z_all;
    }
    if (lane < K) {
        idx_out[(size_t)t * K + lane] = sel_i;
        w_out[(size_t)t * K + lane] = p / z;
    } else if (lane < ranks) {
        spec_idx[(size_t)t * n_spec + (lane - K)] = sel_i;
        if (spec_p) spec_p[(size_t)t * n_spec + (lane - K)] = p / z_all;
    }
}

// One CTA per token.  Thread e sums expert e's split-K partials in split order (all loads
// issued before the sum) and adds the bias.  The experts of ranks 0 .. K + n_spec - 1
// (descending logit, ties -> lower expert id) are then found either by counting every
// expert's rank in parallel (RANK: rank(e) = experts with a larger logit, or an equal logit
// and a lower id; quickest for small batches, where one CTA's latency is the cost) or by
// K + n_spec rounds of a warp arg-max over lanes holding experts l, l+32, ... (fewer
// instructions per token for large batches); both give the same experts in the same order.
// Warp 0 computes the softmax weights.  Ranks 0..K-1 are the routing, ranks
// K..K+n_spec-1 the ranked continuation (page "Data Flow", "Serial Step Trace": the gate
// matvec ranks top-(8+spec); ranks beyond 8 are the bets for the next token) with their
// full-softmax probabilities.
template <bool RANK>
__global__ void __launch_bounds__(kMaxExperts) topk_kernel(const float* __restrict__ partial, int splits,
                                                           const float* __restrict__ bias, int B, int E, int K,
                                                           int norm, int32_t* __restrict__ idx_out,
                                                           float* __restrict__ w_out, int n_spec,
                                                           int32_t* __restrict__ spec_idx,
                                                           float* __restrict__ spec_p) {
    __shared__ __align__(16) float logit[kMaxExperts];
    __shared__ int by_rank[kMaxRanks];
    const int t = blockIdx.x;
    const int e = threadIdx.x;
    const int ranks = K + n_spec;   // <= 32
    if (e < E) {
        float p[kMaxSplits];
#pragma unroll
        for (int sp = 0; sp < kMaxSplits; ++sp)
            if (sp < splits) p[sp] = __ldg(partial + ((size_t)sp * B + t) * E + e);
        float s = 0.f;
#pragma unroll
        for (int sp = 0; sp < kMaxSplits; ++sp)
            if (sp < splits) s += p[sp];
        if (bias) s += bias[e];
        logit[e] = s;
    }
    if (e < kMaxRanks) by_rank[e] = 0;   // (only a non-finite logit could leave a rank unfilled)
    __syncthreads();
    if (RANK && e < E) {
        const float v = logit[e];
        int r = 0;
        int j = 0;
        for (; j + 4 <= E; j += 4) {   // the whole row, four logits per (broadcast) load
            const float4 u = *reinterpret_cast<const float4*>(logit + j);
            r += (u.x > v) || (u.x == v && j < e);
            r += (u.y > v) || (u.y == v && j + 1 < e);
            r += (u.z > v) || (u.z == v && j + 2 < e);
            r += (u.w > v) || (u.w == v && j + 3 < e);
        }
        for (; j < E; ++j) r += (logit[j] > v) || (logit[j] == v && j < e);
        if (r < ranks) by_rank[r] = e;
    }
    __syncthreads();
    if (threadIdx.x >= 32) return;
    topk_select_warp<RANK>(logit, by_rank, t, E, K, norm, idx_out, w_out, n_spec, spec_idx, spec_p);
}

}  // namespace

// Split-K factor of the router for B tokens: the largest divisor s of d / quantum (a split
// keeps a multiple of 128 inputs, 8 k-steps of 16 per load batch, and for the staged
// large-batch kernel of 256, one staged piece) with s <= cap and at most ~4 CTAs per SM.
int route_splits_capped(int B, int E, int d, int cap) {
    const int bt = tile_tokens(B);
    const int tiles = ((B + bt - 1) / bt) * ((E + kExpertsPerCta - 1) / kExpertsPerCta);
    const int quantum = bt == 64 ? 256 : 128;
    const int q = d % quantum ? 1 : d / quantum;
    const int limit = cap > 0 && cap < kMaxSplits ? cap : kMaxSplits;
    int best = 1;
    for (int s = 1; s <= limit && s <= q; ++s)
        if (q % s == 0 && (s == 1 || s * tiles <= 4 * 152)) best = s;
    return best;
}

int route_splits(int B, int E, int d) { return route_splits_capped(B, E, d, 0); }

cudaError_t launch_route(const smoe_layer_desc& D, const uint16_t* x, const float* gate_w, const float* gate_bias,
                         int B, int32_t* topk_idx, float* topk_w, float* logits_ws, cudaStream_t stream,
                         int split_cap, int n_spec, int32_t* spec_idx, float* spec_p) {
    const int E = D.num_experts, d = D.d_model, K = D.top_k;
    const int S = route_splits_capped(B, E, d, split_cap);
    const int bt = tile_tokens(B);
    dim3 grid((B + bt - 1) / bt, (E + kExpertsPerCta - 1) / kExpertsPerCta, S);
    const int kchunk = d / S;   // a multiple of 128 (route_splits)
    if (bt == 8 && B <= 8) {
        // one token tile: CTAs of 2 warps (32 experts) spread the gate read over 4x the SMs
        dim3 g2(grid.x, (E + 31) / 32, S);
        gate_logits_kernel<1, 8, 2><<<g2, 64, 0, stream>>>(x, gate_w, B, E, d, kchunk, logits_ws);
    } else if (bt == 8) {
        gate_logits_kernel<1, 8><<<grid, 256, 0, stream>>>(x, gate_w, B, E, d, kchunk, logits_ws);
    } else {
        const int smem = 64 * kPieceStride * 2;   // 33 KB: below the default dynamic limit
        gate_logits_staged_kernel<8, 4><<<grid, 256, smem, stream>>>(x, gate_w, B, E, d, kchunk, logits_ws);
    }
    const int threads = (E + 31) / 32 * 32;
    (B <= 512 ? topk_kernel<true> : topk_kernel<false>)<<<B, threads, 0, stream>>>(
        logits_ws, S, gate_bias, B, E, K, D.norm_topk_prob, topk_idx, topk_w, n_spec, spec_idx, spec_p);
    return cudaGetLastError();
}

}  // namespace smoe
