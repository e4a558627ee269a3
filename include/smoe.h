/*
 * smoe.h -- C ABI of libsmoe, the GB300 (sm_103a) per-layer MoE block.
 *
 * One MoE layer of exact-routing, layer-major batched prefill and decode, in four steps:
 *   1. route   router gate matvec on each token's hidden state, softmax, top-k and
 *              norm_topk_prob re-normalisation
 *              (page "Layer-Major Batched Prefill", "Choreography Per Chunk" step 5;
 *               page "Surface Scout", "The Model Config": norm_topk_prob)
 *   2. union   the chunk's routed experts deduplicated into a union, with a per-expert
 *              token list        (page "Layer-Major Batched Prefill", "The Inversion")
 *   3. FFN     each union expert applied once to all of its tokens:
 *              y = down(silu(gate(x)) * up(x)) on 4-bit affine, group-64 weights
 *              (page "SSD Streaming Expert Layers", "Math Contract" and "Quantized Layout";
 *               "Layer-Major Batched Prefill", "Choreography Per Chunk" step 6)
 *   4. combine residual[t] += sum_k w[t][k] * y_{idx[t][k]}(x[t])
 *              (page "Data Flow", "Serial Step Trace", FFN block: outputs x routing
 *               weights into the residual)
 *
 * Conventions for every call
 *   - All data pointers are DEVICE pointers unless stated otherwise; the caller owns every
 *     buffer, including the workspace.  The library never allocates or frees memory and
 *     keeps no state between calls other than per-device attributes it caches once.
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL = legacy default stream).
 *     Nothing is read back to the host: counts such as the union size stay on the device.
 *     Only smoe_read_device_status synchronises.
 *   - Argument errors are found on the host before anything is launched: the call returns
 *     an error status and enqueues nothing.  Faults found on the device (an expert index
 *     outside [0, E), a value outside the fp16 range of the tensor-core operands) set bits in
 *     the status word kept at the start of the workspace; the kernels then skip the bad work
 *     and return, they never trap.  smoe_read_device_status reports them.
 *   - bf16 values are passed as uint16_t bit patterns.
 *   - Supported shapes: group_size 64; d_model and ffn_dim each 256 or a multiple of 512
 *     (a row of scales or biases is 8 bytes or a multiple of 16); 1 <= top_k
 *     <= 16; top_k <= num_experts <= 256.  Weight, scale, bias, x and residual pointers
 *     16-byte aligned.  Other shapes return SMOE_ERR_UNSUPPORTED.
 */
#ifndef SMOE_H
#define SMOE_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define SMOE_API __attribute__((visibility("default")))
#else
#define SMOE_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    SMOE_OK = 0,
    SMOE_ERR_INVALID_ARG = 1,   /* NULL pointer, negative size, inconsistent descriptor   */
    SMOE_ERR_UNSUPPORTED = 2,   /* shape or alignment outside what the kernels support   */
    SMOE_ERR_WORKSPACE = 3,     /* workspace NULL, misaligned or smaller than required   */
    SMOE_ERR_CUDA = 4,          /* a CUDA runtime call failed (launch or synchronise)    */
    SMOE_ERR_DEVICE_FAULT = 5   /* the device status word has a fault bit set           */
} smoe_status;

typedef enum {
    SMOE_LAYOUT_SEPARATE = 0,       /* up, gate, down as three tensors                  */
    SMOE_LAYOUT_FUSED_GATE_UP = 1   /* gate_up [E, 2F, d/8]: per expert, gate rows
                                       0..F-1 on top, up rows F..2F-1 below ("Math
                                       Contract", fused gate+up; "Why Whole-Layer Loading
                                       Is Also Fast": per-expert interleave)             */
} smoe_layout;

/* Device status bits (smoe_read_device_status). */
#define SMOE_FAULT_EXPERT_INDEX 0x1u  /* a routed expert id outside [0, num_experts)      */
#define SMOE_FAULT_FP16_RANGE   0x2u  /* an input x, one of its 64-group sums or a SwiGLU
                                         activation silu(g) * v is outside the fp16 range
                                         (or not finite); the outputs are then not
                                         meaningful                                        */
#define SMOE_FAULT_TIMEOUT      0x4u  /* a bounded wait for an async weight copy gave up   */
#define SMOE_FAULT_TOKEN_INDEX  0x8u  /* a token list entry outside [0, B) or a slot list
                                         entry outside [0, top_k): row 0 is read in its
                                         place, the entry's output is dropped and the
                                         residual is not meaningful                         */
#define SMOE_FAULT_SLOT_POOL    0x10u /* a streamed-expert plan or copy entry out of range */

/* Layer descriptor: the subset of the model config the MoE block needs
 * (page "Surface Scout", "The Model Config": d_model, ffn_dim, max_experts_per_layer,
 * norm_topk_prob).  top_k is the number of routed experts per token. */
typedef struct {
    int32_t d_model;
    int32_t num_experts;
    int32_t top_k;
    int32_t ffn_dim;
    int32_t group_size;      /* must be 64 */
    int32_t norm_topk_prob;  /* 1: top-k weights re-normalised to sum 1; 0: full softmax p */
    int32_t layout;          /* smoe_layout */
} smoe_layer_desc;

/* Expert weights of one layer ("SSD Streaming Expert Layers", "Quantized Layout"):
 *   packed words u32 [E, out, in/8], element i of a row = bits 4*(i%8).. of word i/8
 *   scales, biases bf16 [E, out, in/64];  weight = scale * q + bias
 * up/gate: out = ffn_dim, in = d_model;  down: out = d_model, in = ffn_dim.
 * SEPARATE layout uses w_up/w_gate (+ scales, biases) and leaves the gate_up fields NULL;
 * FUSED_GATE_UP uses w_gate_up/s_gate_up/b_gate_up [E, 2*ffn_dim, ...] and leaves the
 * up/gate fields NULL.  The down fields are always used.  Device pointers, read only. */
typedef struct {
    const uint32_t* w_up;      const uint16_t* s_up;      const uint16_t* b_up;
    const uint32_t* w_gate;    const uint16_t* s_gate;    const uint16_t* b_gate;
    const uint32_t* w_gate_up; const uint16_t* s_gate_up; const uint16_t* b_gate_up;
    const uint32_t* w_down;    const uint16_t* s_down;    const uint16_t* b_down;
} smoe_expert_weights;

/* Bytes of device workspace the calls below need for up to `max_tokens` tokens per call
 * (0 on an invalid descriptor).  The workspace must be 256-byte aligned.  Its first 256
 * bytes hold the device status word; the caller clears it with smoe_clear_device_status
 * once after allocation (and after reading a fault). */
SMOE_API size_t smoe_workspace_bytes(const smoe_layer_desc* desc, int32_t max_tokens);

/* Step 1, exact routing.
 *   x        bf16 [B, d_model], row-major: the tokens' hidden states
 *   gate_w   fp32 [num_experts, d_model], row-major: router gate
 *   gate_bias fp32 [num_experts] added to the logits, or NULL
 *   topk_idx int32 [B, top_k] out: experts by descending probability, equal
 *            probabilities ordered by the lower expert id
 *   topk_w   fp32 [B, top_k] out: routing weights (softmax of the logits; with
 *            norm_topk_prob, divided by the sum over the selected experts)
 * Logits accumulate in fp32.  B == 0 is a no-op. */
SMOE_API smoe_status smoe_route(const smoe_layer_desc* desc, const uint16_t* x, const float* gate_w,
                       const float* gate_bias, int32_t B, int32_t* topk_idx, float* topk_w,
                       void* workspace, size_t workspace_bytes, void* stream);

/* Step 1 with the ranking continued past top_k (page "Data Flow", "Serial Step Trace": the
 * exact gate matvec yields a ranked top-(8 + spec); the ranks beyond 8 are the bets
 * prefetched for the next token).  topk_idx / topk_w as smoe_route (bit-identical), plus
 *   n_spec   number of further ranks, 0 <= n_spec, top_k + n_spec <= min(num_experts, 32)
 *   spec_idx int32 [B, n_spec] out: the experts of ranks top_k .. top_k + n_spec - 1, in
 *            rank order (same ordering rule as topk_idx)
 *   spec_p   fp32 [B, n_spec] out, or NULL: their probabilities under the softmax over all
 *            num_experts logits (not renormalised)
 * n_spec == 0 is smoe_route.  Errors as smoe_route; SMOE_ERR_INVALID_ARG for an n_spec out
 * of range or a NULL spec_idx with n_spec > 0. */
SMOE_API smoe_status smoe_route_ranked(const smoe_layer_desc* desc, const uint16_t* x, const float* gate_w,
                       const float* gate_bias, int32_t B, int32_t n_spec, int32_t* topk_idx,
                       float* topk_w, int32_t* spec_idx, float* spec_p, void* workspace,
                       size_t workspace_bytes, void* stream);

/* Step 2, the expert union of a chunk.
 *   topk_idx   int32 [B, top_k] in
 *   union_ids  int32 [num_experts] out: ascending routed expert ids, first n_union valid
 *   n_union    int32 [1] out
 *   offsets    int32 [num_experts + 1] out: entries offsets[u]..offsets[u+1]-1 of
 *              token_list/slot_list belong to union_ids[u]; offsets[n_union] = B*top_k
 *   token_list int32 [B*top_k] out: token rows, ascending within each expert
 *   slot_list  int32 [B*top_k] out: rank k of that expert in the token's top-k
 * An id outside [0, num_experts) sets SMOE_FAULT_EXPERT_INDEX and n_union = 0. */
SMOE_API smoe_status smoe_expert_union(const smoe_layer_desc* desc, const int32_t* topk_idx, int32_t B,
                              int32_t* union_ids, int32_t* n_union, int32_t* offsets,
                              int32_t* token_list, int32_t* slot_list,
                              void* workspace, size_t workspace_bytes, void* stream);

/* Steps 3 + 4: every union expert applied once to its token list, outputs weighted by
 * topk_w and added to the residual in rank order k = 0..top_k-1: the down projection's epilogue
 * stores each slot already weighted, w[t][k] * y_k (fp32 product), and one reduction per row adds
 * the top_k weighted slots into residual[t] in rank order (deterministic).
 *   x         bf16 [B, d_model] (the same rows that were routed)
 *   union ... slot_list: as produced by smoe_expert_union
 *   topk_w    fp32 [B, top_k]
 *   residual  fp32 [B, d_model], updated in place
 * Dequantised weights, x and the SwiGLU activation are fp16 on the tensor cores with fp32
 * accumulation. */
SMOE_API smoe_status smoe_moe_ffn_batch(const smoe_layer_desc* desc, const smoe_expert_weights* weights,
                               const uint16_t* x, int32_t B, const int32_t* union_ids,
                               const int32_t* n_union, const int32_t* offsets,
                               const int32_t* token_list, const int32_t* slot_list,
                               const float* topk_w, float* residual,
                               void* workspace, size_t workspace_bytes, void* stream);

/* Steps 3 + 4 followed by the norm that feeds the next block (page "Data Flow", "Serial Step
 * Trace": the hidden state is RMS-normed before every FFN block): smoe_moe_ffn_batch, then
 *   x_next = bf16(norm(residual))  exactly as smoe_rmsnorm_bf16(residual, eps, center) computes it
 * (bit for bit), in the same kernel as the weighted combine (d_model <= 4096; wider rows run the
 * standalone norm after the combine).
 *   x_next  bf16 [B, d_model] out, 8-byte aligned; it may be the same buffer as x, which is no
 *           longer read when x_next is written
 *   eps, center  as smoe_rmsnorm_bf16
 * Other arguments and errors as smoe_moe_ffn_batch; SMOE_ERR_INVALID_ARG for a NULL x_next, a
 * negative eps or center outside {0, 1}.  After a routing fault (SMOE_FAULT_EXPERT_INDEX) the
 * residual is left unchanged and x_next is not meaningful. */
SMOE_API smoe_status smoe_moe_ffn_batch_norm(const smoe_layer_desc* desc, const smoe_expert_weights* weights,
                                             const uint16_t* x, int32_t B, const int32_t* union_ids,
                                             const int32_t* n_union, const int32_t* offsets,
                                             const int32_t* token_list, const int32_t* slot_list,
                                             const float* topk_w, float* residual, float eps, int32_t center,
                                             uint16_t* x_next, void* workspace, size_t workspace_bytes,
                                             void* stream);

/* The shared expert (page "Data Flow", "Serial Step Trace": the shared expert FFN runs on
 * every token and residual += shared_out + routed_out; page "Surface Scout", "The Model
 * Config": shared_expert_ffn_dim, 0 when the model has none): residual += down(silu(gate x)
 * * up x) for all B tokens, with no routing weight.
 * Layout: a shared expert of ffn width P * F is passed as P column slices of width F, slice
 * p holding FFN columns pF .. pF + F - 1: desc->num_experts = desc->top_k = P (P <= 16),
 * desc->ffn_dim = F, and the weight tensors [P, ...] of smoe_expert_weights (gate / up rows
 * pF.., down input columns pF..; separate or fused layout as desc->layout says).  Since
 * SwiGLU acts column by column, the sum of the slices' outputs is the whole expert's; the
 * slices give the down projection P times the output tiles.  The call routes every token
 * to every slice with weight 1 in the workspace (sized by smoe_workspace_bytes(desc, B)),
 * runs steps 3 + 4 and adds the slices' outputs in slice order.  desc->norm_topk_prob is
 * ignored.  Errors as smoe_moe_ffn_batch; SMOE_ERR_INVALID_ARG if num_experts != top_k. */
SMOE_API smoe_status smoe_shared_expert_ffn(const smoe_layer_desc* desc, const smoe_expert_weights* weights,
                                            const uint16_t* x, int32_t B, float* residual, void* workspace,
                                            size_t workspace_bytes, void* stream);

/* The whole MoE block (steps 1-4) for B tokens: residual += MoE(x).
 * topk_idx / topk_w may be NULL (the routing then lives in the workspace only) or device
 * buffers [B, top_k] that receive it. */
SMOE_API smoe_status smoe_moe_layer(const smoe_layer_desc* desc, const smoe_expert_weights* weights,
                           const uint16_t* x, const float* gate_w, const float* gate_bias,
                           int32_t B, float* residual, int32_t* topk_idx, float* topk_w,
                           void* workspace, size_t workspace_bytes, void* stream);

/* Chaining glue between stacked layers (page "Data Flow", "Serial Step Trace": RMS norm
 * before the FFN block), unit norm weight:
 *   c = center ? mean_i h[t][i] : 0
 *   x_out[t][i] = bf16( (h[t][i] - c) / sqrt(mean_i (h[t][i] - c)^2 + eps) )
 *   h fp32 [B, d], x_out bf16 [B, d].  fp32 arithmetic, bf16 round to nearest even.
 * center = 0 is the pages' RMS norm; center = 1 first removes the row mean.  Synthetic
 * expert weights with q uniform on 0..15 and bias -8 scale have mean -scale/2, so every layer
 * output carries a per-token common mode; chained through a plain RMS norm it turns the next
 * layer's inputs into same-sign vectors that route to ever fewer experts.  Removing the row
 * mean keeps the chained inputs zero-mean, as real hidden states are. */
SMOE_API smoe_status smoe_rmsnorm_bf16(const float* h, float eps, int32_t center, int32_t B, int32_t d,
                                       uint16_t* x_out, void* stream);

/* ---- Experts streamed from host memory into a pool of HBM slots ------------------------
 * Page "Data Flow", "Ring Buffer State Machine": the expert weights live in a ring of slots
 * keyed by (layer, expert); a slot keeps its expert after use and a later request for the same
 * key is a hit; a miss takes an EMPTY slot, else the least recently used idle slot (never one
 * the current pass reads), and a freshly loaded slot carries the new tick.  "Handling Misses":
 * correctness never depends on the cache.  Page "Layer-Major Batched Prefill", "Retention,
 * never replay": reuse comes from keeping what was read, never from guessing.
 * Here the layers' expert tensors stay in pinned host memory (on GB300: Grace memory, read by
 * the GPU over NVLink-C2C) and a pool of n_slots experts lives in HBM.  Per layer, after
 * smoe_expert_union:
 *   smoe_stream_plan  -> slot_ids (the union's experts as slots of the pool) + copy_list
 *   smoe_stream_copy  -> the missed experts' bytes from host memory into their slots
 *   smoe_moe_ffn_batch with a pool descriptor (num_experts = n_slots), the pool tensors and
 *                       slot_ids as union_ids: the same results, bit for bit, as the
 *                       resident layer
 * Everything is decided on the device (no host synchronisation); calls on one state must be
 * ordered on one stream.
 *
 * State: int32 [4 + n_keys + 2 * n_slots] device buffer of smoe_stream_state_bytes(n_keys,
 * n_slots) bytes (0 for invalid sizes), set up by smoe_stream_init and owned by the caller.  A
 * key is key_base + expert (for instance layer * num_experts + expert); n_slots <= 256. */
SMOE_API size_t smoe_stream_state_bytes(int32_t n_keys, int32_t n_slots);

/* Empty pool: no key resident, every slot empty, tick 0 (asynchronous). */
SMOE_API smoe_status smoe_stream_init(void* state, int32_t n_keys, int32_t n_slots, void* stream);

/* Residency plan of one layer call.  The tick advances by one; every union expert that a slot
 * holds is a hit and its slot is re-stamped; the misses, in union order, take the idle slots
 * (slots no hit of this call uses) in order of (stamp, slot id) -- empty slots first, then the
 * least recently used, slots of equal stamp lowest id first -- evicting their previous keys.
 *   union_ids, n_union  as produced by smoe_expert_union for desc, B
 *   slot_ids   int32 [num_experts]: slot of union position u (u < n_union)
 *   copy_list  int32 [1 + 2 * num_experts]: [0] = number of misses m, then m pairs (expert,
 *              slot) in union order, the input of smoe_stream_copy
 * SMOE_ERR_INVALID_ARG if key_base + num_experts > n_keys or n_slots < min(B * top_k,
 * num_experts) (a union must fit).  A union id outside [0, num_experts) or a state set up for
 * other sizes sets SMOE_FAULT_SLOT_POOL, slot_ids -1 and no copies.  workspace: the layer's
 * (status word). */
SMOE_API smoe_status smoe_stream_plan(const smoe_layer_desc* desc, int32_t B, int32_t key_base,
                                      const int32_t* union_ids, const int32_t* n_union, void* state,
                                      int32_t n_keys, int32_t n_slots, int32_t* slot_ids, int32_t* copy_list,
                                      void* workspace, size_t workspace_bytes, void* stream);

/* Copy the experts of copy_list from the layer's tensors into their pool slots.
 *   host_weights  the layer's [num_experts, ...] tensors (layout of desc) in pinned host memory
 *                 (or device / managed memory); the GPU reads them directly
 *   pool_weights  device tensors of the same layout with n_slots experts: slot s of a tensor
 *                 holds the bytes of the copied expert's row block
 *   copy_list     as written by smoe_stream_plan
 * SMOE_ERR_UNSUPPORTED for unaligned tensors or host memory the GPU cannot address
 * (unregistered pageable memory).  An entry outside range sets SMOE_FAULT_SLOT_POOL and is
 * skipped.  workspace: the layer's (status word). */
SMOE_API smoe_status smoe_stream_copy(const smoe_layer_desc* desc, const smoe_expert_weights* host_weights,
                                      const smoe_expert_weights* pool_weights, int32_t n_slots,
                                      const int32_t* copy_list, void* workspace, size_t workspace_bytes,
                                      void* stream);

/* Step 1 without a workspace, for callers that cannot allocate device memory (a plugin
 * inside a host application that owns the device-memory budget, or a latency-critical loop
 * that cannot risk the device-wide synchronisation of a cudaMalloc).  The pages have no
 * counterpart: it is an addition of this library.  Arguments and results are those of
 * smoe_route; the split-K scratch is a fixed 4 MiB device array inside the library (held by
 * every GPU that loads it until the process exits).  A call needs B * num_experts <= 2^20
 * (B <= 8192 at 128 experts) and returns SMOE_ERR_UNSUPPORTED beyond that, without launching.
 * Up to B = 256 at 128 experts the results equal smoe_route's; beyond, fewer split-K partials
 * fit and the logits differ from smoe_route's by fp32 summation order only.  The first call
 * on a device looks up the array's address (cudaGetSymbolAddress) with that device current:
 * make it before any stream capture.  The address is kept per CUDA context; after a device
 * reset the next call is a first call again.  All calls share the array: calls that overlap
 * on the GPU race and must be ordered by the caller.  Argument errors as smoe_route (no
 * workspace errors).  Allocates nothing. */
SMOE_API smoe_status smoe_route_noalloc(const smoe_layer_desc* desc, const uint16_t* x, const float* gate_w,
                                        const float* gate_bias, int32_t B, int32_t* topk_idx, float* topk_w,
                                        void* stream);

/* Zero the device status word (asynchronous). */
SMOE_API smoe_status smoe_clear_device_status(void* workspace, void* stream);

/* Synchronise `stream` and read the device status word.  SMOE_OK if it is zero, else
 * SMOE_ERR_DEVICE_FAULT with the bits stored to *bits_out (may be NULL). */
SMOE_API smoe_status smoe_read_device_status(void* workspace, void* stream, uint32_t* bits_out);

/* Static description of a status code. */
SMOE_API const char* smoe_status_string(smoe_status status);

#ifdef __cplusplus
}
#endif
#endif /* SMOE_H */
