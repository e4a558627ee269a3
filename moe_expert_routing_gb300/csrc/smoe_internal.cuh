// Internal declarations of libsmoe (not part of the C ABI).
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <cuda_fp16.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "../../include/smoe.h"

namespace smoe {

constexpr int kGroup = 64;          // quantisation group along the input axis
constexpr int kMaxExperts = 256;    // union kernel keeps per-expert counters in shared memory
constexpr int kMaxTopK = 16;

// ----------------------------------------------------------------------------- workspace
// The caller's workspace is carved into these regions (each 256-byte aligned).
struct WsLayout {
    size_t status;        // uint32 status word (first 256 bytes)
    size_t logits;        // fp32 [splits, B, E]: split-K partial router logits
    size_t topk_idx;      // int32 [B, K]   (used when the caller passes no routing buffers)
    size_t topk_w;        // fp32  [B, K]
    size_t union_ids;     // int32 [E]
    size_t n_union;       // int32 [1]
    size_t offsets;       // int32 [E + 1]
    size_t token_list;    // int32 [B * K]
    size_t slot_list;     // int32 [B * K]
    size_t xg;            // fp16 [B * K, d]: gathered, pair-permuted expert inputs (odd inputs / 16)
    size_t sx;            // fp32 [B * K, d / 64]: per-group sums of the inputs
    size_t h;             // fp16 [B * K, 2F]: SwiGLU activations as hi | lo terms, pair-permuted
    size_t sh;            // fp32 [B * K, F / 64]: per-group sums of the activations
    size_t s16x;          // fp16 [2][B * K, d / 64]: input group sums as hi and lo planes
    size_t s16h;          // fp16 [2][B * K, F / 64]: activation group sums as hi and lo planes
    size_t y;             // fp32 [B * K, d]: weighted expert outputs w[t,k] y_k, row t*K + k
    size_t entl;          // int32 [B * K]: entry t*K + k of list position p (-1: index rejected)
    size_t wl;            // fp32 [B * K]: routing weight w[t,k] of list position p
    size_t ticket;        // int32 [2 + E]: work queues of the expert passes and per-expert counts
    size_t uscratch;      // int32 [1 + chunks * E]: the union's per-chunk counts (B * K > 1024)
    size_t total;
};

// Descriptor validation shared by every entry point (SMOE_OK, INVALID_ARG or UNSUPPORTED).
smoe_status check_desc(const smoe_layer_desc* D);
int route_splits(int B, int E, int d);
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder();
WsLayout ws_layout(const smoe_layer_desc& D, int max_tokens);

template <class T>
inline T* ws_ptr(void* ws, size_t off) { return reinterpret_cast<T*>(static_cast<char*>(ws) + off); }

// ----------------------------------------------------------------------------- launchers
// Each returns cudaGetLastError() after enqueueing its kernel(s) on `stream`.
// split_cap > 0 limits the number of split-K partials (callers with a fixed scratch size).
// n_spec > 0: also the ranks K..K+n_spec-1 (ids into spec_idx [B, n_spec], full-softmax
// probabilities into spec_p unless NULL); K + n_spec <= kMaxRanks.
constexpr int kMaxRanks = 32;
cudaError_t launch_route(const smoe_layer_desc& D, const uint16_t* x, const float* gate_w,
                         const float* gate_bias, int B, int32_t* topk_idx, float* topk_w,
                         float* logits_ws, cudaStream_t stream, int split_cap = 0, int n_spec = 0,
                         int32_t* spec_idx = nullptr, float* spec_p = nullptr);

// scratch: int32 [1 + union_chunks(B*K) * E] for batches of more than 1024 entries (may be
// NULL for smaller ones)
int union_chunks(int BK);
cudaError_t launch_union(const smoe_layer_desc& D, const int32_t* topk_idx, int B, int32_t* union_ids,
                         int32_t* n_union, int32_t* offsets, int32_t* token_list, int32_t* slot_list,
                         uint32_t* status, int32_t* scratch, cudaStream_t stream);

// Every token to every one of P slices with weight 1 (the routing of a shared expert).
cudaError_t launch_all_slices(int B, int P, int32_t* union_ids, int32_t* n_union, int32_t* offsets,
                              int32_t* token_list, int32_t* slot_list, float* w, cudaStream_t stream);

// Expert weights as the FFN kernels consume them.  The packed words are read through TMA
// tensor maps: 2-D u32 views [rows, in/8] of each weight tensor, box 32 words (4 groups) x
// 128 rows (gate, up) or 256 rows (down), 128-byte swizzle.  Fused gate_up: map_gate == map_up over the gate_up tensor, the up rows
// of expert e start at e * 2F + F (u_row_offset = F).
struct FfnPointers {
    CUtensorMap map_gate, map_up, map_down;
    CUtensorMap tc_gate, tc_up, tc_down;   // the same views, boxes of 64 (gate, up) / 128 (down) rows
    // scale / bias tables of the expert passes: bf16 [rows, in/64], box 8 groups x 128 rows
    // (gate, up) or 256 rows (down); see encode_group_map
    CUtensorMap map_sg, map_bg, map_su, map_bu, map_sd, map_bd;
    // the gate/up views and tables again with boxes of 192 rows (a gate/up launch with 12
    // consumer warps); set when ffn_dim is a multiple of 192 (wide)
    bool wide;
    CUtensorMap wide_gate, wide_up, wide_sg, wide_bg, wide_su, wide_bu;
    const uint16_t* sg; const uint16_t* bg; int64_t g_rows_per_expert;
    const uint16_t* su; const uint16_t* bu; int64_t u_rows_per_expert; int64_t u_row_offset;
    const uint16_t* sd; const uint16_t* bd;
};

// The tensor-core path reads the packed weights through maps with 128-byte rows (4 groups)
// and boxes of 64 rows (gate, up) or 128 rows (down).
struct FfnTcWeights {
    CUtensorMap map_gate, map_up, map_down;
    const uint16_t* sg; const uint16_t* bg; int64_t g_rows;
    const uint16_t* su; const uint16_t* bu; int64_t u_rows; int64_t u_off;
    const uint16_t* sd; const uint16_t* bd;
};

// Experts with at least this many list entries take the tcgen05 path (when the shape allows).
constexpr int kTcMinTokens = 32;
bool tc_path_supported(const smoe_layer_desc& D);
cudaError_t launch_ffn_tc(const smoe_layer_desc& D, const FfnTcWeights& W, int B, int pass,
                          const int32_t* union_ids, const int32_t* n_union, const int32_t* offsets,
                          const int32_t* token_list, const int32_t* slot_list, void* ws, const WsLayout& L,
                          int tc_min, int sms, cudaStream_t stream);

// all_tokens: every expert of the call holds all B tokens (the slices of a shared expert), so
// the tensor-core path is worth launching whenever B reaches its threshold.
// x_next (optional): after the combine, x_next = bf16(norm(residual)) as launch_rmsnorm computes
// it (eps, center), fused into the combine kernel for d_model <= 4096.
struct NextNorm {
    uint16_t* x_next = nullptr;
    float eps = 0.f;
    int center = 0;
};
cudaError_t launch_ffn(const smoe_layer_desc& D, const FfnPointers& W, const uint16_t* x, int B,
                       const int32_t* union_ids, const int32_t* n_union, const int32_t* offsets,
                       const int32_t* token_list, const int32_t* slot_list, const float* topk_w,
                       float* residual, void* ws, const WsLayout& L, cudaStream_t stream, bool all_tokens = false,
                       const NextNorm& next = NextNorm());

cudaError_t launch_rmsnorm(const float* h, float eps, int center, int B, int d, uint16_t* x_out,
                           cudaStream_t stream);

// ----------------------------------------------------------------------------- streamed experts
// One weight tensor of a layer for the slot copy: expert e's part starts at src + e * n16 in
// host memory (device-accessible address), slot s's at dst + s * n16 in the pool; n16 =
// 16-byte units per expert, pieces = 32 KB pieces per expert.
struct StreamRegion {
    const uint4* src;
    uint4* dst;
    int64_t n16;
    int pieces;
};
constexpr int kStreamRegions = 9;   // separate layout: 3 projections x (words, scales, biases)
struct StreamCopyArgs {
    StreamRegion region[kStreamRegions];
    int n_regions;
    int pieces_per_copy;            // sum of the regions' pieces
    const int32_t* list;            // [0] n, then (expert, slot) pairs
    int E;                          // experts of the layer (host tensors)
    int S;                          // slots of the pool
    uint32_t* status;
};
size_t stream_state_words(int n_keys, int n_slots);
int64_t stream_pieces(int64_t n16);
cudaError_t launch_stream_init(int32_t* state, int n_keys, int n_slots, cudaStream_t stream);
cudaError_t launch_stream_plan(int32_t* state, int n_keys, int n_slots, int key_base, int E, const int32_t* union_ids,
                               const int32_t* n_union, int32_t* slot_ids, int32_t* copy_list, uint32_t* status,
                               cudaStream_t stream);
cudaError_t launch_stream_copy(const StreamCopyArgs& a, cudaStream_t stream);

// ----------------------------------------------------------------------------- device helpers
__device__ __forceinline__ float bf16_bits_to_float(uint32_t bits16) {
    return __uint_as_float(bits16 << 16);
}

// Sum of v over a CTA of 512 threads (warp butterflies, then the 16 warp sums in warp order),
// returned to every thread; red: 16 floats of shared memory.  The RMS-norm kernels use it so
// that a norm fused into another kernel gives the standalone norm's results bit for bit.
__device__ __forceinline__ float block_sum512(float v, float* red) {
#pragma unroll
    for (int off = 16; off; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
    __syncthreads();
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
    __syncthreads();
    float tot = 0.f;
#pragma unroll
    for (int w = 0; w < 16; ++w) tot += red[w];
    return tot;
}

}  // namespace smoe
