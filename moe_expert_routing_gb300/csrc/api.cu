// libsmoe C ABI: argument validation, workspace layout and the kernel sequence of a layer.
// Declarations and the contract of every call are in include/smoe.h.
#include "smoe_internal.cuh"

#include <cudaTypedefs.h>
#include <stddef.h>

#include <algorithm>

namespace smoe {
namespace {

constexpr size_t kAlign = 256;

size_t align_up(size_t v) { return (v + kAlign - 1) & ~(kAlign - 1); }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

// Descriptor checks shared by every call.  INVALID_ARG for values that make no sense,
// UNSUPPORTED for sensible shapes the kernels do not handle.
smoe_status check_desc(const smoe_layer_desc* D) {
    if (!D) return SMOE_ERR_INVALID_ARG;
    if (D->d_model <= 0 || D->num_experts <= 0 || D->top_k <= 0 || D->ffn_dim <= 0 || D->group_size <= 0)
        return SMOE_ERR_INVALID_ARG;
    if (D->top_k > D->num_experts) return SMOE_ERR_INVALID_ARG;
    if (D->layout != SMOE_LAYOUT_SEPARATE && D->layout != SMOE_LAYOUT_FUSED_GATE_UP) return SMOE_ERR_INVALID_ARG;
    if (D->norm_topk_prob != 0 && D->norm_topk_prob != 1) return SMOE_ERR_INVALID_ARG;
    if (D->group_size != kGroup) return SMOE_ERR_UNSUPPORTED;
    // 256 or a multiple of 512: the scale rows are 8 bytes or a multiple of 16 (TMA strides)
    if ((D->d_model % 512 && D->d_model != 256) || (D->ffn_dim % 512 && D->ffn_dim != 256))
        return SMOE_ERR_UNSUPPORTED;
    if (D->num_experts > kMaxExperts || D->top_k > kMaxTopK) return SMOE_ERR_UNSUPPORTED;
    if ((int64_t)D->d_model * D->ffn_dim > (int64_t)1 << 30) return SMOE_ERR_UNSUPPORTED;
    return SMOE_OK;
}

namespace {

smoe_status check_ws(const smoe_layer_desc& D, int B, void* ws, size_t ws_bytes, WsLayout* L) {
    if (!ws || (reinterpret_cast<uintptr_t>(ws) & (kAlign - 1))) return SMOE_ERR_WORKSPACE;
    *L = ws_layout(D, B);
    if (ws_bytes < L->total) return SMOE_ERR_WORKSPACE;
    return SMOE_OK;
}

// 2-D u32 view [rows, in/8] of a packed weight tensor; box 32 words (4 groups) x box_rows,
// 128-byte swizzle.
bool encode_weight_map(CUtensorMap* map, const uint32_t* words, int64_t rows, int64_t in, int box_rows) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
    if (!enc) return false;
    cuuint64_t dims[2] = {(cuuint64_t)(in / 8), (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)(in / 2)};
    cuuint32_t box[2] = {32, (cuuint32_t)box_rows};
    cuuint32_t estr[2] = {1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT32, 2, const_cast<uint32_t*>(words), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 2-D bf16 view of a scale or bias tensor [rows, G] (G = in / 64 groups per row) for the
// per-stage tables of the expert passes: box 8 groups x box_rows rows.  With G == 4 a row
// is 8 bytes and the tensor is viewed as [rows / 2, 8] with box_rows / 2 rows, which lands
// in shared memory as the same [box_rows][4] table.
bool encode_group_map(CUtensorMap* map, const uint16_t* p, int64_t rows, int64_t in, int box_rows) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
    if (!enc) return false;
    const int64_t G = in / kGroup;
    const bool packed = G == 4;
    cuuint64_t dims[2] = {(cuuint64_t)(packed ? 8 : G), (cuuint64_t)(packed ? rows / 2 : rows)};
    cuuint64_t strides[1] = {(cuuint64_t)((packed ? 8 : G) * 2)};
    cuuint32_t box[2] = {8, (cuuint32_t)(packed ? box_rows / 2 : box_rows)};
    cuuint32_t estr[2] = {1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t*>(p), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Device-accessible address of memory the streamed-expert copy touches: pinned (registered)
// host memory (read over NVLink-C2C / PCIe), device or managed memory; NULL otherwise.
const void* device_view(const void* p) {
    if (!p) return nullptr;
    cudaPointerAttributes at{};
    if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
        (void)cudaGetLastError();
        return nullptr;
    }
    if (at.type == cudaMemoryTypeHost || at.type == cudaMemoryTypeDevice || at.type == cudaMemoryTypeManaged)
        return at.devicePointer;
    return nullptr;
}

// The tensors of one layer's experts as (host tensor, pool tensor, bytes per expert), in the
// order of smoe_expert_weights' layout: words, scales, biases of each projection.
int expert_tensors(const smoe_layer_desc& D, const smoe_expert_weights& H, const smoe_expert_weights& P,
                   const void* (&src)[kStreamRegions], void* (&dst)[kStreamRegions], int64_t (&bytes)[kStreamRegions]) {
    const int64_t d = D.d_model, F = D.ffn_dim;
    int n = 0;
    auto add = [&](const void* s, const void* t, int64_t rows, int64_t in) {
        src[n] = s; dst[n] = const_cast<void*>(t); bytes[n] = rows * in / 2; ++n;                  // packed words
    };
    auto add_g = [&](const void* s, const void* t, int64_t rows, int64_t in) {
        src[n] = s; dst[n] = const_cast<void*>(t); bytes[n] = rows * (in / kGroup) * 2; ++n;      // bf16 per group
    };
    if (D.layout == SMOE_LAYOUT_SEPARATE) {
        add(H.w_gate, P.w_gate, F, d); add_g(H.s_gate, P.s_gate, F, d); add_g(H.b_gate, P.b_gate, F, d);
        add(H.w_up, P.w_up, F, d);     add_g(H.s_up, P.s_up, F, d);     add_g(H.b_up, P.b_up, F, d);
    } else {
        add(H.w_gate_up, P.w_gate_up, 2 * F, d);
        add_g(H.s_gate_up, P.s_gate_up, 2 * F, d);
        add_g(H.b_gate_up, P.b_gate_up, 2 * F, d);
    }
    add(H.w_down, P.w_down, d, F); add_g(H.s_down, P.s_down, d, F); add_g(H.b_down, P.b_down, d, F);
    return n;
}

smoe_status check_weights(const smoe_layer_desc& D, const smoe_expert_weights* W, FfnPointers* P) {
    if (!W) return SMOE_ERR_INVALID_ARG;
    const int64_t F = D.ffn_dim, d = D.d_model, E = D.num_experts;
    const bool sep = D.layout == SMOE_LAYOUT_SEPARATE;
    // pointers and alignment first: nothing touches CUDA before the arguments are known good
    if (!W->w_down || !W->s_down || !W->b_down) return SMOE_ERR_INVALID_ARG;
    if (sep && (!W->w_up || !W->s_up || !W->b_up || !W->w_gate || !W->s_gate || !W->b_gate))
        return SMOE_ERR_INVALID_ARG;
    if (!sep && (!W->w_gate_up || !W->s_gate_up || !W->b_gate_up)) return SMOE_ERR_INVALID_ARG;
    if (!aligned16(W->w_down) || !aligned16(W->s_down) || !aligned16(W->b_down)) return SMOE_ERR_UNSUPPORTED;
    if (sep && (!aligned16(W->w_up) || !aligned16(W->s_up) || !aligned16(W->b_up) || !aligned16(W->w_gate) ||
                !aligned16(W->s_gate) || !aligned16(W->b_gate)))
        return SMOE_ERR_UNSUPPORTED;
    if (!sep && (!aligned16(W->w_gate_up) || !aligned16(W->s_gate_up) || !aligned16(W->b_gate_up)))
        return SMOE_ERR_UNSUPPORTED;
    P->sd = W->s_down; P->bd = W->b_down;
    if (sep) {
        P->sg = W->s_gate; P->bg = W->b_gate; P->g_rows_per_expert = F;
        P->su = W->s_up;   P->bu = W->b_up;   P->u_rows_per_expert = F; P->u_row_offset = 0;
    } else {
        // per expert 2F rows: gate rows 0..F-1, up rows F..2F-1
        P->sg = W->s_gate_up; P->bg = W->b_gate_up; P->g_rows_per_expert = 2 * F;
        P->su = W->s_gate_up; P->bu = W->b_gate_up; P->u_rows_per_expert = 2 * F; P->u_row_offset = F;
    }
    if (!encode_weight_map(&P->map_down, W->w_down, E * d, F, 256)) return SMOE_ERR_CUDA;
    if (!encode_weight_map(&P->tc_down, W->w_down, E * d, F, 128)) return SMOE_ERR_CUDA;
    if (!encode_group_map(&P->map_sd, W->s_down, E * d, F, 256) || !encode_group_map(&P->map_bd, W->b_down, E * d, F, 256))
        return SMOE_ERR_CUDA;
    if (sep) {
        if (!encode_weight_map(&P->map_gate, W->w_gate, E * F, d, 128)) return SMOE_ERR_CUDA;
        if (!encode_weight_map(&P->map_up, W->w_up, E * F, d, 128)) return SMOE_ERR_CUDA;
        if (!encode_weight_map(&P->tc_gate, W->w_gate, E * F, d, 64)) return SMOE_ERR_CUDA;
        if (!encode_weight_map(&P->tc_up, W->w_up, E * F, d, 64)) return SMOE_ERR_CUDA;
        if (!encode_group_map(&P->map_sg, W->s_gate, E * F, d, 128) || !encode_group_map(&P->map_bg, W->b_gate, E * F, d, 128) ||
            !encode_group_map(&P->map_su, W->s_up, E * F, d, 128) || !encode_group_map(&P->map_bu, W->b_up, E * F, d, 128))
            return SMOE_ERR_CUDA;
    } else {
        if (!encode_weight_map(&P->map_gate, W->w_gate_up, E * 2 * F, d, 128)) return SMOE_ERR_CUDA;
        if (!encode_weight_map(&P->tc_gate, W->w_gate_up, E * 2 * F, d, 64)) return SMOE_ERR_CUDA;
        P->map_up = P->map_gate;
        P->tc_up = P->tc_gate;
        if (!encode_group_map(&P->map_sg, W->s_gate_up, E * 2 * F, d, 128) ||
            !encode_group_map(&P->map_bg, W->b_gate_up, E * 2 * F, d, 128))
            return SMOE_ERR_CUDA;
        P->map_su = P->map_sg;
        P->map_bu = P->map_bg;
    }
    P->wide = F % 192 == 0;
    if (P->wide) {
        const uint32_t* wg = sep ? W->w_gate : W->w_gate_up;
        const uint32_t* wu = sep ? W->w_up : W->w_gate_up;
        const uint16_t* sg = sep ? W->s_gate : W->s_gate_up;
        const uint16_t* bg = sep ? W->b_gate : W->b_gate_up;
        const uint16_t* su = sep ? W->s_up : W->s_gate_up;
        const uint16_t* bu = sep ? W->b_up : W->b_gate_up;
        const int64_t rows = sep ? E * F : E * 2 * F;
        if (!encode_weight_map(&P->wide_gate, wg, rows, d, 192) || !encode_weight_map(&P->wide_up, wu, rows, d, 192) ||
            !encode_group_map(&P->wide_sg, sg, rows, d, 192) || !encode_group_map(&P->wide_bg, bg, rows, d, 192) ||
            !encode_group_map(&P->wide_su, su, rows, d, 192) || !encode_group_map(&P->wide_bu, bu, rows, d, 192))
            return SMOE_ERR_CUDA;
    }
    return SMOE_OK;
}

smoe_status cuda_status(cudaError_t e) { return e == cudaSuccess ? SMOE_OK : SMOE_ERR_CUDA; }

}  // namespace

// cuTensorMapEncodeTiled through the runtime's driver entry point (no link-time libcuda).
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = []() {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            p = nullptr;
        return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }();
    return fn;
}

WsLayout ws_layout(const smoe_layer_desc& D, int max_tokens) {
    const size_t B = max_tokens > 0 ? (size_t)max_tokens : 1, E = D.num_experts, K = D.top_k;
    const size_t d = D.d_model, F = D.ffn_dim, BK = B * K;
    // max over b <= B of splits(b) * b; splits(b) is constant between multiples of 8
    size_t max_split_rows = 0;
    for (size_t b = 8; b < B + 8; b += 8) {
        const size_t bb = b < B ? b : B;
        const size_t v = (size_t)route_splits((int)bb, (int)E, (int)d) * bb;
        if (v > max_split_rows) max_split_rows = v;
    }
    WsLayout L{};
    size_t o = 0;
    auto take = [&](size_t bytes) { const size_t at = o; o = align_up(o + bytes); return at; };
    L.status = take(4);
    L.logits = take(max_split_rows * E * 4);
    L.topk_idx = take(BK * 4);
    L.topk_w = take(BK * 4);
    L.union_ids = take(E * 4);
    L.n_union = take(4);
    L.offsets = take((E + 1) * 4);
    L.token_list = take(BK * 4);
    L.slot_list = take(BK * 4);
    L.xg = take(BK * d * 2);
    L.sx = take(BK * (d / kGroup) * 4);
    L.h = take(BK * 2 * F * 2);
    L.sh = take(BK * (F / kGroup) * 4);
    L.s16x = take(2 * BK * (d / kGroup) * 2);
    L.s16h = take(2 * BK * (F / kGroup) * 2);
    L.y = take(BK * d * 4);
    L.entl = take(BK * 4);
    L.wl = take(BK * 4);
    L.ticket = take((E + 2) * 4);
    L.uscratch = take((1 + (size_t)union_chunks((int)BK) * E) * 4);
    L.total = o;
    return L;
}

}  // namespace smoe

using namespace smoe;

extern "C" {

size_t smoe_workspace_bytes(const smoe_layer_desc* desc, int32_t max_tokens) {
    if (check_desc(desc) != SMOE_OK || max_tokens < 0) return 0;
    return ws_layout(*desc, max_tokens).total;
}

smoe_status smoe_route(const smoe_layer_desc* desc, const uint16_t* x, const float* gate_w, const float* gate_bias,
                       int32_t B, int32_t* topk_idx, float* topk_w, void* workspace, size_t workspace_bytes,
                       void* stream) {
    smoe_status st = check_desc(desc);
    if (st != SMOE_OK) return st;
    if (B < 0) return SMOE_ERR_INVALID_ARG;
    if (B == 0) return SMOE_OK;
    if (!x || !gate_w || !topk_idx || !topk_w) return SMOE_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(gate_w)) return SMOE_ERR_UNSUPPORTED;
    WsLayout L;
    if ((st = check_ws(*desc, B, workspace, workspace_bytes, &L)) != SMOE_OK) return st;
    return cuda_status(launch_route(*desc, x, gate_w, gate_bias, B, topk_idx, topk_w,
                                    ws_ptr<float>(workspace, L.logits), static_cast<cudaStream_t>(stream)));
}

smoe_status smoe_route_ranked(const smoe_layer_desc* desc, const uint16_t* x, const float* gate_w,
                              const float* gate_bias, int32_t B, int32_t n_spec, int32_t* topk_idx, float* topk_w,
                              int32_t* spec_idx, float* spec_p, void* workspace, size_t workspace_bytes,
                              void* stream) {
    smoe_status st = check_desc(desc);
    if (st != SMOE_OK) return st;
    if (B < 0 || n_spec < 0) return SMOE_ERR_INVALID_ARG;
    const int ranks = desc->top_k + n_spec;
    if (ranks > desc->num_experts || ranks > kMaxRanks) return SMOE_ERR_INVALID_ARG;
    if (n_spec > 0 && !spec_idx) return SMOE_ERR_INVALID_ARG;
    if (B == 0) return SMOE_OK;
    if (!x || !gate_w || !topk_idx || !topk_w) return SMOE_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(gate_w)) return SMOE_ERR_UNSUPPORTED;
    WsLayout L;
    if ((st = check_ws(*desc, B, workspace, workspace_bytes, &L)) != SMOE_OK) return st;
    return cuda_status(launch_route(*desc, x, gate_w, gate_bias, B, topk_idx, topk_w,
                                    ws_ptr<float>(workspace, L.logits), static_cast<cudaStream_t>(stream), 0,
                                    n_spec, n_spec > 0 ? spec_idx : nullptr, n_spec > 0 ? spec_p : nullptr));
}

smoe_status smoe_expert_union(const smoe_layer_desc* desc, const int32_t* topk_idx, int32_t B, int32_t* union_ids,
                              int32_t* n_union, int32_t* offsets, int32_t* token_list, int32_t* slot_list,
                              void* workspace, size_t workspace_bytes, void* stream) {
    smoe_status st = check_desc(desc);
    if (st != SMOE_OK) return st;
    if (B < 0) return SMOE_ERR_INVALID_ARG;
    if (!topk_idx || !union_ids || !n_union || !offsets || !token_list || !slot_list) return SMOE_ERR_INVALID_ARG;
    WsLayout L;
    if ((st = check_ws(*desc, B, workspace, workspace_bytes, &L)) != SMOE_OK) return st;
    return cuda_status(launch_union(*desc, topk_idx, B, union_ids, n_union, offsets, token_list, slot_list,
                                    ws_ptr<uint32_t>(workspace, L.status), ws_ptr<int32_t>(workspace, L.uscratch),
                                    static_cast<cudaStream_t>(stream)));
}

smoe_status smoe_moe_ffn_batch(const smoe_layer_desc* desc, const smoe_expert_weights* weights, const uint16_t* x,
                               int32_t B, const int32_t* union_ids, const int32_t* n_union, const int32_t* offsets,
                               const int32_t* token_list, const int32_t* slot_list, const float* topk_w,
                               float* residual, void* workspace, size_t workspace_bytes, void* stream) {
    smoe_status st = check_desc(desc);
    if (st != SMOE_OK) return st;
    if (B < 0) return SMOE_ERR_INVALID_ARG;
    if (B == 0) return SMOE_OK;
    if (!x || !union_ids || !n_union || !offsets || !token_list || !slot_list || !topk_w || !residual)
        return SMOE_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(residual)) return SMOE_ERR_UNSUPPORTED;
    FfnPointers P{};
    if ((st = check_weights(*desc, weights, &P)) != SMOE_OK) return st;
    WsLayout L;
    if ((st = check_ws(*desc, B, workspace, workspace_bytes, &L)) != SMOE_OK) return st;
    return cuda_status(launch_ffn(*desc, P, x, B, union_ids, n_union, offsets, token_list, slot_list, topk_w,
                                  residual, workspace, L, static_cast<cudaStream_t>(stream)));
}

smoe_status smoe_moe_ffn_batch_norm(const smoe_layer_desc* desc, const smoe_expert_weights* weights,
                                    const uint16_t* x, int32_t B, const int32_t* union_ids, const int32_t* n_union,
                                    const int32_t* offsets, const int32_t* token_list, const int32_t* slot_list,
                                    const float* topk_w, float* residual, float eps, int32_t center,
                                    uint16_t* x_next, void* workspace, size_t workspace_bytes, void* stream) {
    smoe_status st = check_desc(desc);
    if (st != SMOE_OK) return st;
    if (B < 0 || !(eps >= 0.f) || (center != 0 && center != 1)) return SMOE_ERR_INVALID_ARG;
    if (B == 0) return SMOE_OK;
    if (!x || !union_ids || !n_union || !offsets || !token_list || !slot_list || !topk_w || !residual || !x_next)
        return SMOE_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(residual) || (reinterpret_cast<uintptr_t>(x_next) & 7u))
        return SMOE_ERR_UNSUPPORTED;
    FfnPointers P{};
    if ((st = check_weights(*desc, weights, &P)) != SMOE_OK) return st;
    WsLayout L;
    if ((st = check_ws(*desc, B, workspace, workspace_bytes, &L)) != SMOE_OK) return st;
    NextNorm next;
    next.x_next = x_next;
    next.eps = eps;
    next.center = center;
    return cuda_status(launch_ffn(*desc, P, x, B, union_ids, n_union, offsets, token_list, slot_list, topk_w,
                                  residual, workspace, L, static_cast<cudaStream_t>(stream), false, next));
}

smoe_status smoe_moe_layer(const smoe_layer_desc* desc, const smoe_expert_weights* weights, const uint16_t* x,
                           const float* gate_w, const float* gate_bias, int32_t B, float* residual,
                           int32_t* topk_idx, float* topk_w, void* workspace, size_t workspace_bytes, void* stream) {
    smoe_status st = check_desc(desc);
    if (st != SMOE_OK) return st;
    if (B < 0) return SMOE_ERR_INVALID_ARG;
    if (B == 0) return SMOE_OK;
    if (!x || !gate_w || !residual) return SMOE_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(gate_w) || !aligned16(residual)) return SMOE_ERR_UNSUPPORTED;
    FfnPointers P{};
    if ((st = check_weights(*desc, weights, &P)) != SMOE_OK) return st;
    WsLayout L;
    if ((st = check_ws(*desc, B, workspace, workspace_bytes, &L)) != SMOE_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int32_t* idx = topk_idx ? topk_idx : ws_ptr<int32_t>(workspace, L.topk_idx);
    float* w = topk_w ? topk_w : ws_ptr<float>(workspace, L.topk_w);
    int32_t* uid = ws_ptr<int32_t>(workspace, L.union_ids);
    int32_t* nu = ws_ptr<int32_t>(workspace, L.n_union);
    int32_t* off = ws_ptr<int32_t>(workspace, L.offsets);
    int32_t* tl = ws_ptr<int32_t>(workspace, L.token_list);
    int32_t* sl = ws_ptr<int32_t>(workspace, L.slot_list);
    cudaError_t e = launch_route(*desc, x, gate_w, gate_bias, B, idx, w, ws_ptr<float>(workspace, L.logits), s);
    if (e == cudaSuccess)
        e = launch_union(*desc, idx, B, uid, nu, off, tl, sl, ws_ptr<uint32_t>(workspace, L.status),
                         ws_ptr<int32_t>(workspace, L.uscratch), s);
    if (e == cudaSuccess) e = launch_ffn(*desc, P, x, B, uid, nu, off, tl, sl, w, residual, workspace, L, s);
    return cuda_status(e);
}

smoe_status smoe_shared_expert_ffn(const smoe_layer_desc* desc, const smoe_expert_weights* weights, const uint16_t* x,
                                   int32_t B, float* residual, void* workspace, size_t workspace_bytes, void* stream) {
    smoe_status st = check_desc(desc);
    if (st != SMOE_OK) return st;
    if (desc->num_experts != desc->top_k || B < 0) return SMOE_ERR_INVALID_ARG;
    if (B == 0) return SMOE_OK;
    if (!x || !residual) return SMOE_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(residual)) return SMOE_ERR_UNSUPPORTED;
    FfnPointers P{};
    if ((st = check_weights(*desc, weights, &P)) != SMOE_OK) return st;
    WsLayout L;
    if ((st = check_ws(*desc, B, workspace, workspace_bytes, &L)) != SMOE_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int32_t* uid = ws_ptr<int32_t>(workspace, L.union_ids);
    int32_t* nu = ws_ptr<int32_t>(workspace, L.n_union);
    int32_t* off = ws_ptr<int32_t>(workspace, L.offsets);
    int32_t* tl = ws_ptr<int32_t>(workspace, L.token_list);
    int32_t* sl = ws_ptr<int32_t>(workspace, L.slot_list);
    float* w = ws_ptr<float>(workspace, L.topk_w);
    cudaError_t e = launch_all_slices(B, desc->num_experts, uid, nu, off, tl, sl, w, s);
    if (e == cudaSuccess) e = launch_ffn(*desc, P, x, B, uid, nu, off, tl, sl, w, residual, workspace, L, s, true);
    return cuda_status(e);
}

smoe_status smoe_rmsnorm_bf16(const float* h, float eps, int32_t center, int32_t B, int32_t d, uint16_t* x_out,
                              void* stream) {
    if (B < 0 || d <= 0 || !(eps >= 0.f) || (center != 0 && center != 1)) return SMOE_ERR_INVALID_ARG;
    if (B == 0) return SMOE_OK;
    if (!h || !x_out) return SMOE_ERR_INVALID_ARG;
    if (d % 4 || !aligned16(h) || (reinterpret_cast<uintptr_t>(x_out) & 7u)) return SMOE_ERR_UNSUPPORTED;
    return cuda_status(launch_rmsnorm(h, eps, center, B, d, x_out, static_cast<cudaStream_t>(stream)));
}

size_t smoe_stream_state_bytes(int32_t n_keys, int32_t n_slots) {
    if (n_keys <= 0 || n_slots <= 0 || n_slots > kMaxExperts) return 0;
    return stream_state_words(n_keys, n_slots) * sizeof(int32_t);
}

smoe_status smoe_stream_init(void* state, int32_t n_keys, int32_t n_slots, void* stream) {
    if (!state || n_keys <= 0 || n_slots <= 0 || (reinterpret_cast<uintptr_t>(state) & 3u)) return SMOE_ERR_INVALID_ARG;
    if (n_slots > kMaxExperts) return SMOE_ERR_UNSUPPORTED;
    return cuda_status(launch_stream_init(static_cast<int32_t*>(state), n_keys, n_slots,
                                          static_cast<cudaStream_t>(stream)));
}

smoe_status smoe_stream_plan(const smoe_layer_desc* desc, int32_t B, int32_t key_base, const int32_t* union_ids,
                             const int32_t* n_union, void* state, int32_t n_keys, int32_t n_slots, int32_t* slot_ids,
                             int32_t* copy_list, void* workspace, size_t workspace_bytes, void* stream) {
    smoe_status st = check_desc(desc);
    if (st != SMOE_OK) return st;
    if (B < 0 || n_keys <= 0 || n_slots <= 0 || key_base < 0) return SMOE_ERR_INVALID_ARG;
    if (n_slots > kMaxExperts) return SMOE_ERR_UNSUPPORTED;
    if ((int64_t)key_base + desc->num_experts > n_keys) return SMOE_ERR_INVALID_ARG;
    // every union fits: at most min(B * top_k, num_experts) experts, all held at once
    const int64_t need = std::min<int64_t>((int64_t)B * desc->top_k, desc->num_experts);
    if (n_slots < need) return SMOE_ERR_INVALID_ARG;
    if (B == 0) return SMOE_OK;
    if (!union_ids || !n_union || !state || !slot_ids || !copy_list || (reinterpret_cast<uintptr_t>(state) & 3u))
        return SMOE_ERR_INVALID_ARG;
    WsLayout L;
    if ((st = check_ws(*desc, B, workspace, workspace_bytes, &L)) != SMOE_OK) return st;
    return cuda_status(launch_stream_plan(static_cast<int32_t*>(state), n_keys, n_slots, key_base, desc->num_experts,
                                          union_ids, n_union, slot_ids, copy_list,
                                          ws_ptr<uint32_t>(workspace, L.status), static_cast<cudaStream_t>(stream)));
}

smoe_status smoe_stream_copy(const smoe_layer_desc* desc, const smoe_expert_weights* host_weights,
                             const smoe_expert_weights* pool_weights, int32_t n_slots, const int32_t* copy_list,
                             void* workspace, size_t workspace_bytes, void* stream) {
    smoe_status st = check_desc(desc);
    if (st != SMOE_OK) return st;
    if (!host_weights || !pool_weights || !copy_list || n_slots <= 0) return SMOE_ERR_INVALID_ARG;
    if (n_slots > kMaxExperts) return SMOE_ERR_UNSUPPORTED;
    const void* src[kStreamRegions];
    void* dst[kStreamRegions];
    int64_t bytes[kStreamRegions];
    const int n = expert_tensors(*desc, *host_weights, *pool_weights, src, dst, bytes);
    for (int r = 0; r < n; ++r) {
        if (!src[r] || !dst[r]) return SMOE_ERR_INVALID_ARG;
        if (!aligned16(src[r]) || !aligned16(dst[r]) || bytes[r] % 16) return SMOE_ERR_UNSUPPORTED;
    }
    WsLayout L;
    if ((st = check_ws(*desc, 1, workspace, workspace_bytes, &L)) != SMOE_OK) return st;
    StreamCopyArgs a{};
    a.n_regions = n;
    a.pieces_per_copy = 0;
    for (int r = 0; r < n; ++r) {
        // host tensors must be pinned (or device / managed) memory: the kernel reads them directly
        const void* s = device_view(src[r]);
        const void* t = device_view(dst[r]);
        if (!s || !t) return SMOE_ERR_UNSUPPORTED;
        a.region[r].src = static_cast<const uint4*>(s);
        a.region[r].dst = static_cast<uint4*>(const_cast<void*>(t));
        a.region[r].n16 = bytes[r] / 16;
        a.region[r].pieces = (int)stream_pieces(bytes[r] / 16);
        a.pieces_per_copy += a.region[r].pieces;
    }
    a.list = copy_list;
    a.E = desc->num_experts;
    a.S = n_slots;
    a.status = ws_ptr<uint32_t>(workspace, L.status);
    return cuda_status(launch_stream_copy(a, static_cast<cudaStream_t>(stream)));
}

smoe_status smoe_clear_device_status(void* workspace, void* stream) {
    if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & (kAlign - 1))) return SMOE_ERR_WORKSPACE;
    return cuda_status(cudaMemsetAsync(workspace, 0, sizeof(uint32_t), static_cast<cudaStream_t>(stream)));
}

smoe_status smoe_read_device_status(void* workspace, void* stream, uint32_t* bits_out) {
    if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & (kAlign - 1))) return SMOE_ERR_WORKSPACE;
    uint32_t bits = 0;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (cudaMemcpyAsync(&bits, workspace, sizeof(bits), cudaMemcpyDeviceToHost, s) != cudaSuccess)
        return SMOE_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return SMOE_ERR_CUDA;
    if (bits_out) *bits_out = bits;
    return bits ? SMOE_ERR_DEVICE_FAULT : SMOE_OK;
}

const char* smoe_status_string(smoe_status status) {
    switch (status) {
        case SMOE_OK: return "ok";
        case SMOE_ERR_INVALID_ARG: return "invalid argument";
        case SMOE_ERR_UNSUPPORTED: return "unsupported shape or alignment";
        case SMOE_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
        case SMOE_ERR_CUDA: return "CUDA runtime error";
        case SMOE_ERR_DEVICE_FAULT: return "device reported a fault (see status bits)";
    }
    return "unknown status";
}

}  // extern "C"
