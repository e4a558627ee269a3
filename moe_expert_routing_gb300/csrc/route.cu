// Step 1, exact routing: router gate matvec, softmax, top-k, norm_topk_prob.
//
// Page "Layer-Major Batched Prefill", "Choreography Per Chunk" step 5: the real router gate
// (an E x d_model matvec) evaluated on every token's hidden state, norm_topk_prob
// re-normalisation of the selected weights.  Page "Surface Scout", "The Model Config":
// norm_topk_prob re-normalises the top-k routing weights to sum 1.
//
// Two kernels:
//   gate_logits_kernel  fp32 SIMT tile GEMM, logits[s][t][e] = sum over split s of
//                       W[e][i] * x[t][i].  Split-K over d so that even a single token
//                       spreads the 2 MB gate read over ~100 SMs; partials are summed in a
//                       fixed order by the top-k kernel, so results are deterministic.
//   topk_kernel         one warp per token: sums the partials (+ bias), K rounds of a
//                       warp arg-max (ties -> lower expert id), softmax weights.
#include "smoe_internal.cuh"

#include <math.h>

namespace smoe {
namespace {

constexpr int BN = 64;   // experts per tile
constexpr int BK = 32;   // k per smem stage
constexpr int kMaxSplits = 16;

// BM tokens x 64 experts per CTA (BM = 16 for small batches, 64 otherwise); each of the
// 256 threads owns BM/16 tokens x 4 experts.
template <int BM>
__global__ void __launch_bounds__(256) gate_logits_kernel(const uint16_t* __restrict__ x,
                                                          const float* __restrict__ W, int B, int E, int d,
                                                          int kchunk, float* __restrict__ partial) {
    constexpr int TM = BM / 16;
    __shared__ float As[BK][BM + 4];
    __shared__ float Bs[BK][BN + 4];
    const int tid = threadIdx.x;
    const int t0 = blockIdx.x * BM, e0 = blockIdx.y * BN;
    const int k_begin = blockIdx.z * kchunk, k_end = k_begin + kchunk;
    const int tx = tid & 15, ty = tid >> 4;
    float acc[TM][4];
#pragma unroll
    for (int i = 0; i < TM; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;

    for (int k0 = k_begin; k0 < k_end; k0 += BK) {
        // x tile: BM tokens x 32 k bf16; each loading thread takes 8 consecutive k of one token
        if (tid < BM * 4) {
            const int r = tid >> 2, kk = (tid & 3) * 8;
            const int t = t0 + r;
            uint4 raw = make_uint4(0, 0, 0, 0);
            if (t < B) raw = *reinterpret_cast<const uint4*>(x + (size_t)t * d + k0 + kk);
            const uint32_t w4[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                As[kk + 2 * q][r] = bf16_bits_to_float(w4[q] & 0xFFFFu);
                As[kk + 2 * q + 1][r] = bf16_bits_to_float(w4[q] >> 16);
            }
        }
        {   // W tile: 64 experts x 32 k fp32; each thread 8 consecutive k of one expert
            const int r = tid >> 2, kk = (tid & 3) * 8;
            const int e = e0 + r;
            float4 a = make_float4(0.f, 0.f, 0.f, 0.f), b = a;
            if (e < E) {
                a = *reinterpret_cast<const float4*>(W + (size_t)e * d + k0 + kk);
                b = *reinterpret_cast<const float4*>(W + (size_t)e * d + k0 + kk + 4);
            }
            Bs[kk + 0][r] = a.x; Bs[kk + 1][r] = a.y; Bs[kk + 2][r] = a.z; Bs[kk + 3][r] = a.w;
            Bs[kk + 4][r] = b.x; Bs[kk + 5][r] = b.y; Bs[kk + 6][r] = b.z; Bs[kk + 7][r] = b.w;
        }
        __syncthreads();
#pragma unroll 8
        for (int kk = 0; kk < BK; ++kk) {
            float av[TM], bv[4];
#pragma unroll
            for (int i = 0; i < TM; ++i) av[i] = As[kk][ty * TM + i];
#pragma unroll
            for (int j = 0; j < 4; ++j) bv[j] = Bs[kk][tx * 4 + j];
#pragma unroll
            for (int i = 0; i < TM; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
        }
        __syncthreads();
    }
    float* out = partial + (size_t)blockIdx.z * B * E;
#pragma unroll
    for (int i = 0; i < TM; ++i) {
        const int t = t0 + ty * TM + i;
        if (t >= B) continue;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int e = e0 + tx * 4 + j;
            if (e < E) out[(size_t)t * E + e] = acc[i][j];
        }
    }
}

int tile_tokens(int B) { return B <= 256 ? 16 : 64; }

// One warp per token.  Lane l holds experts l, l+32, ... (E <= 256).
__global__ void __launch_bounds__(256) topk_kernel(const float* __restrict__ partial, int splits,
                                                   const float* __restrict__ bias, int B, int E, int K, int norm,
                                                   int32_t* __restrict__ idx_out, float* __restrict__ w_out) {
    const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (warp >= B) return;
    const int t = warp;
    constexpr int PER = kMaxExperts / 32;
    float v[PER];
    bool live[PER];
#pragma unroll
    for (int i = 0; i < PER; ++i) {
        const int e = lane + 32 * i;
        live[i] = e < E;
        float s = 0.f;
        if (live[i]) {
#pragma unroll 4
            for (int sp = 0; sp < splits; ++sp) s += __ldg(partial + ((size_t)sp * B + t) * E + e);
            if (bias) s += bias[e];
        }
        v[i] = s;
    }
    // max logit over all experts
    float mx = -INFINITY;
#pragma unroll
    for (int i = 0; i < PER; ++i)
        if (live[i]) mx = fmaxf(mx, v[i]);
#pragma unroll
    for (int off = 16; off; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
    // full softmax denominator (only needed without norm_topk_prob)
    float z_all = 0.f;
    if (!norm) {
#pragma unroll
        for (int i = 0; i < PER; ++i)
            if (live[i]) z_all += expf(v[i] - mx);
#pragma unroll
        for (int off = 16; off; off >>= 1) z_all += __shfl_xor_sync(0xffffffffu, z_all, off);
    }
    float sel_v = 0.f;   // lane k keeps the k-th selection
    int sel_i = 0;
    for (int k = 0; k < K; ++k) {
        float bv = -INFINITY;
        int bi = 0x7fffffff;
#pragma unroll
        for (int i = 0; i < PER; ++i) {
            const int e = lane + 32 * i;
            if (live[i] && (v[i] > bv || (v[i] == bv && e < bi))) { bv = v[i]; bi = e; }
        }
#pragma unroll
        for (int off = 16; off; off >>= 1) {
            const float ov = __shfl_xor_sync(0xffffffffu, bv, off);
            const int oi = __shfl_xor_sync(0xffffffffu, bi, off);
            if (ov > bv || (ov == bv && oi < bi)) { bv = ov; bi = oi; }
        }
        if (lane == k) { sel_v = bv; sel_i = bi; }
        if ((bi & 31) == lane) {
#pragma unroll
            for (int i = 0; i < PER; ++i)
                if (i == (bi >> 5)) live[i] = false;
        }
    }
    float p = (lane < K) ? expf(sel_v - mx) : 0.f;
    float z = p;
    if (norm) {
#pragma unroll
        for (int off = 16; off; off >>= 1) z += __shfl_xor_sync(0xffffffffu, z, off);
    } else {
        z = z_all;
    }
    if (lane < K) {
        idx_out[(size_t)t * K + lane] = sel_i;
        w_out[(size_t)t * K + lane] = p / z;
    }
}

}  // namespace

int route_splits(int B, int E, int d) {
    const int bm = tile_tokens(B);
    const int tiles = ((B + bm - 1) / bm) * ((E + BN - 1) / BN);
    const int target = 2 * 152;
    int s = 1;
    while (s < kMaxSplits && s * tiles < target && (d / (2 * s)) % BK == 0 && d / (2 * s) >= 128) s *= 2;
    return s;
}

cudaError_t launch_route(const smoe_layer_desc& D, const uint16_t* x, const float* gate_w, const float* gate_bias,
                         int B, int32_t* topk_idx, float* topk_w, float* logits_ws, cudaStream_t stream) {
    const int E = D.num_experts, d = D.d_model, K = D.top_k;
    const int S = route_splits(B, E, d);
    const int bm = tile_tokens(B);
    dim3 grid((B + bm - 1) / bm, (E + BN - 1) / BN, S);
    if (bm == 16) gate_logits_kernel<16><<<grid, 256, 0, stream>>>(x, gate_w, B, E, d, d / S, logits_ws);
    else gate_logits_kernel<64><<<grid, 256, 0, stream>>>(x, gate_w, B, E, d, d / S, logits_ws);
    const int warps_per_block = 8;
    topk_kernel<<<(B + warps_per_block - 1) / warps_per_block, 32 * warps_per_block, 0, stream>>>(
        logits_ws, S, gate_bias, B, E, K, D.norm_topk_prob, topk_idx, topk_w);
    return cudaGetLastError();
}

}  // namespace smoe
