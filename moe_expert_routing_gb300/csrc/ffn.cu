// Steps 3 + 4: each union expert applied once to its token list, then the weighted combine.
//
// Page "SSD Streaming Expert Layers", "Math Contract": y = down(silu(gate(x)) * up(x));
// "Quantized Layout": packed u32 [E, out, in/8] 4-bit affine weights, bf16 scales and
// biases per group of 64 inputs.  Page "Layer-Major Batched Prefill", "Choreography Per
// Chunk" step 6: a two-pass token-batch dispatch per claimed expert (gate/up, then down),
// one dequantisation stream for all of the expert's tokens.  Page "Data Flow", "Serial
// Step Trace": expert outputs times routing weights are added into the residual.
//
// Kernels (all on one stream, no host synchronisation; union size and counts are read
// on the device):
//   gather_kernel      x rows of every (expert, token) entry -> fp16, pair-permuted,
//                      with per-64-group sums (xg, sx)
//   ffn_expert_kernel  the experts with few tokens, persistent: gate/up projections + SwiGLU,
//                      128 or 192 h columns of one expert per tile, writing h (fp16, pair-
//                      permuted) and its per-group sums; the down projection, 256 output rows
//                      of one expert per tile, writing the weighted slots of y.  One launch per
//                      pass (static tile order), or both passes in one launch for long
//                      prompts (a device-side queue)
//   combine_kernel     residual[t] += sum_k w[t][k] * y[t*K + k], k in rank order
//
// The pass kernels are persistent and warp-specialised: one producer warp streams, for
// every tile and every 256-input k-slice, the packed weight rows and the activation rows
// (TMA, 128-byte swizzle), the activations' group sums and the rows' scales and biases (TMA)
// into a shared-memory ring; eight (or, for 192-column gate/up tiles, twelve) consumer warps
// decode and multiply.
// Full/empty mbarriers hand the stages back and forth, so the weight stream never drains
// between tiles and the consumers never wait on a global load.
//
// Tensor-core use in the bandwidth-bound regime.  With a handful of tokens per expert the
// work is a stream of 4-bit weights that must be decoded faster than HBM delivers them;
// FFMA dot products would cost ~5 issue slots per weight.  Instead each consumer warp turns
// nibbles straight into A-fragment registers of mma.sync.m16n8k16 and lets the tensor core
// do the multiply-adds:
//   * a u32 word holds nibbles n0..n7.  w & 0x000F000F is the fp16 pair (n0, n4) * 2^-24
//     (fp16 subnormals, exact); w & 0x00F000F0 is (n1, n5) * 16 * 2^-24; the same masks on
//     w >> 8 give n2/n6 and n3/n7: five integer ops per eight weights and no offset to take
//     back out.  The activations at odd positions within every 8 inputs are stored divided
//     by 16 (exact), so 16 q x/16 = q x.  (Measured on GB300: mma.sync multiplies subnormal
//     fp16 operands exactly and accumulates them to ~3e-6 of the result.)
//   * the mma contraction order is free, so the k axis is permuted: within every 8 inputs
//     the activations are stored as (x0,x4,x1,x5,x2,x6,x3,x7), which makes each decoded
//     pair line up with one B-fragment register.
//   * each mma covers 16 inputs of ONE group, so the affine map is applied after the mma,
//     in fp32:  sum_i (s q_i + b) x_i = (s * 2^24) * C + b * S,  C = mma result,
//     S = sum of the group's activations; weights are never rounded.  Both terms are fp32
//     FMAs per group.
//   * the down projection's input h = silu(g) * up is carried as two fp16 terms, hi + lo
//     (lo = the rounding remainder), and both are multiplied: h keeps ~22 bits.
#include "smoe_internal.cuh"

#include <cuda.h>
#include <math.h>

#include <algorithm>
#include <atomic>

namespace smoe {
namespace {

__device__ __forceinline__ void mma16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};\n"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Exact fp16 pairs of the nibbles of a word w (w8 = w >> 8), as subnormals (units of 2^-24):
//   even(w) = (n0, n4),  odd(w) = 16 (n1, n5),  even(w8) = (n2, n6),  odd(w8) = 16 (n3, n7).
__device__ __forceinline__ uint32_t nib_even(uint32_t w) { return w & 0x000F000Fu; }
__device__ __forceinline__ uint32_t nib_odd(uint32_t w) { return w & 0x00F000F0u; }


// storage slot of logical element m (0..7) inside an 8-element chunk: (0,4,1,5,2,6,3,7)
__device__ __forceinline__ int perm8(int m) { return 2 * (m & 3) + (m >> 2); }

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n" ::"r"(bar), "r"(bytes) : "memory");
}

// Bounded wait on an mbarrier phase: true when the phase completed, false after ~0.5 s.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity) {
    uint64_t t0 = 0;
    for (uint32_t i = 0;; ++i) {
        uint32_t ok;
        asm volatile(
            "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
            : "=r"(ok)
            : "r"(bar), "r"(parity)
            : "memory");
        if (ok) return true;
        if ((i & 1023) == 0) {
            uint64_t now;
            asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(now));
            if (i == 0) t0 = now;
            else if (now - t0 > 500000000ull) return false;
        }
    }
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];\n" ::"r"(
            dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
        : "memory");
}




__device__ __forceinline__ void prefetch_l2(const void* p, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;\n" ::"l"(p), "r"(bytes) : "memory");
}

__device__ __forceinline__ uint2 lds_u2(uint32_t a) {
    uint2 v;
    asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];\n" : "=r"(v.x), "=r"(v.y) : "r"(a));
    return v;
}

__device__ __forceinline__ uint4 lds_u4(uint32_t a) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];\n" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(a));
    return v;
}


// ----------------------------------------------------------------------------- gather
// One warp per segment of 32 x U 8-element chunks of a list entry p: xg[p] = pair-permuted
// fp16(x[token_list[p]]) with the odd elements of every 8 divided by 16; sx[p][g] = sum of the
// values the stored halves stand for in group g (8 consecutive lanes hold a group's chunks),
// also as fp16 hi and lo planes s16[0|1][p][g].  The first segment's warp also writes the
// entry's output row t*K + k (entl[p], -1 for a token or slot index out of range, flagged) and
// routing weight (wl[p]), so the down passes read both by list position.  The warp issues all U of its loads before
// converting, so the kernel streams instead of waiting on one dependent load chain per 16
// bytes; small batches use U = 1 (more warps), large ones U = 16 (fewer index loads).
template <int U>
__global__ void __launch_bounds__(256) gather_kernel(const uint16_t* __restrict__ x, int d, int B,
                                                     const int32_t* __restrict__ n_union,
                                                     const int32_t* __restrict__ offsets,
                                                     const int32_t* __restrict__ token_list,
                                                     const int32_t* __restrict__ slot_list,
                                                     const float* __restrict__ topk_w, int K,
                                                     int32_t* __restrict__ entl, float* __restrict__ wl,
                                                     uint32_t* __restrict__ status,
                                                     __half* __restrict__ xg, float* __restrict__ sx,
                                                     __half* __restrict__ s16, int BK, int32_t* __restrict__ ticket,
                                                     int n_ticket) {
    if (blockIdx.x == 0)   // work queue of the expert passes that follow
        for (int i = threadIdx.x; i < n_ticket; i += blockDim.x) ticket[i] = 0;
    const int lane = threadIdx.x & 31;
    const int cpr = d / 8;   // 8-element chunks per row, a multiple of 32
    const int G = d / kGroup;
    const int segs = (cpr + 32 * U - 1) / (32 * U);   // warps per row
    int wg = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    // the warp's first entry's token is loaded alongside the list length (lists hold BK entries)
    const int t_first = wg / segs < BK ? token_list[wg / segs] : -1;
    const int total = offsets[*n_union];
    for (bool first = true; wg < total * segs; wg += (gridDim.x * blockDim.x) >> 5, first = false) {
        const int p = wg / segs, seg = wg - p * segs;
        int t = first ? t_first : token_list[p];
        if (seg == 0 && lane == 0) {   // the entry's output row and routing weight
            const int k = slot_list[p];
            const bool ok = t >= 0 && t < B && k >= 0 && k < K;
            entl[p] = ok ? t * K + k : -1;
            wl[p] = ok ? topk_w[(size_t)t * K + k] : 0.f;
            if (!ok && t >= 0 && t < B) atomicOr(status, SMOE_FAULT_TOKEN_INDEX);   // slot out of range
        }
        if (t < 0 || t >= B) {   // a caller-supplied list that does not match B: flag, use row 0
            if (lane == 0) atomicOr(status, SMOE_FAULT_TOKEN_INDEX);
            t = 0;
        }
        const uint4* xr = reinterpret_cast<const uint4*>(x + (size_t)t * d);
        uint4* orow = reinterpret_cast<uint4*>(xg + (size_t)p * d);
        {
            const int base = seg * 32 * U;
            uint4 raw[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int ch = base + u * 32 + lane;
                raw[u] = ch < cpr ? __ldg(xr + ch) : make_uint4(0, 0, 0, 0);
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int ch = base + u * 32 + lane;   // warp-uniform validity: cpr % 32 == 0
                if (ch >= cpr) break;
                const uint32_t wv[4] = {raw[u].x, raw[u].y, raw[u].z, raw[u].w};
                __half hv[8];
                float sa = 0.f;
                float vmax = 0.f;
#pragma unroll
                for (int m = 0; m < 8; ++m) {
                    const float v = bf16_bits_to_float((m & 1) ? (wv[m >> 1] >> 16) : (wv[m >> 1] & 0xFFFFu));
                    const __half h = __float2half_rn((m & 1) ? v * 0.0625f : v);
                    hv[perm8(m)] = h;
                    sa += (m & 1) ? __half2float(h) * 16.f : __half2float(h);
                    vmax = fmaxf(vmax, fabsf(v));
                }
                uint4 o;
                o.x = (uint32_t)__half_as_ushort(hv[0]) | ((uint32_t)__half_as_ushort(hv[1]) << 16);
                o.y = (uint32_t)__half_as_ushort(hv[2]) | ((uint32_t)__half_as_ushort(hv[3]) << 16);
                o.z = (uint32_t)__half_as_ushort(hv[4]) | ((uint32_t)__half_as_ushort(hv[5]) << 16);
                o.w = (uint32_t)__half_as_ushort(hv[6]) | ((uint32_t)__half_as_ushort(hv[7]) << 16);
                orow[ch] = o;
#pragma unroll
                for (int off = 1; off < 8; off <<= 1) sa += __shfl_xor_sync(0xffffffffu, sa, off);
                // an input (or a group sum, which the tensor cores take as fp16) outside the fp16
                // range, or not finite (fmaxf drops NaN, the sum keeps it)
                if (__any_sync(0xffffffffu, !(vmax <= 65504.f) || !(fabsf(sa) <= 65504.f)) && lane == 0)
                    atomicOr(status, SMOE_FAULT_FP16_RANGE);
                if ((lane & 7) == 0) {
                    const size_t i = (size_t)p * G + ch / 8;
                    sx[i] = sa;
                    const __half hh = __float2half_rn(sa);   // hi and lo planes for the tensor-core path
                    s16[i] = hh;
                    s16[(size_t)BK * G + i] = __float2half_rn(sa - __half2float(hh));
                }
            }
        }
    }
}

// ----------------------------------------------------------------------------- expert passes
constexpr int kConsumerWarps = 8;                           // down and both-pass launches; gate/up: 8 or 12
constexpr int kMailbox = 4;                                // finished gate/up tiles awaiting publication

// Which passes a launch of the expert-pass kernel runs.
constexpr int kGateUp = 1, kDown = 2, kBoth = 3;
constexpr bool has_publisher(int mode) { return mode == kBoth; }
constexpr bool gate_up_only(int mode) { return mode == kGateUp; }
constexpr bool down_only(int mode) { return mode == kDown; }
constexpr bool claims(int mode) { return mode == kBoth; }   // atomic queue, down tiles wait per expert
// NW consumer warps + a producer warp (+ a publisher warp when both passes share a launch)
constexpr int pass_threads(int mode, int nw) { return 32 * (nw + 1 + has_publisher(mode)); }
constexpr int kTokChunk = 16;              // tokens per pass over the weights (or 8, see StageCfg)

// One ring stage: packed weights | activation boxes (4, or 4 hi + 4 lo; one row per token of
// the chunk) | scales | biases | activation group sums fp32 [chunk tokens][4 groups]; a
// 1024-byte multiple.  The scale and bias tables hold, per weight row, the 8 groups of the
// 16-byte-aligned window that contains the stage's 4 groups ([rows][8] bf16), or with 4 groups
// per row ([rows][4]) the whole row.  CH tokens per chunk (a pass over the weights): 16, or for
// a down-only launch whose experts average at most 4 tokens 8 (8-row boxes).  As many stages
// as fit, up to 4: 4 for 8-warp gate/up and for 8-token down chunks, 3 for 12-warp gate/up
// (stages of 1.5x the rows) and for 16-token down chunks (a down-only launch with many tokens
// per expert, and the both-pass launch).
// A tile holds 32 NW weight rows (gate/up: 16 NW gate rows above 16 NW up rows; down: 32 NW
// output rows), consumer warp w taking rows 16w.. and 16 NW + 16w.. (gate/up) or 32w.. (down).
constexpr int kMaxDynSmem = 227 * 1024 - 3072;   // the rest of a CTA's 227 KB holds the static arrays
template <int MODE, int CH, int NW>
struct StageCfg {
    static constexpr int kRows = 32 * NW;                            // weight rows of a tile
    static constexpr int kWBytes = kRows * 128;                      // kRows x 32 u32 words (4 groups)
    static constexpr int kSbBytes = kRows * 16;                      // kRows x up to 8 bf16 (scales or biases)
    static constexpr int kChunk = CH;                                // tokens per pass over the weights
    static constexpr int kBox = kChunk * 128;                        // one activation box: CH rows x 64 fp16
    static constexpr int kXOff = kWBytes;
    static constexpr int kSOff = kXOff + (gate_up_only(MODE) ? 4 : 8) * kBox;
    static constexpr int kBOff = kSOff + kSbBytes;
    static constexpr int kSumOff = kBOff + kSbBytes;
    static constexpr int kSumBytes = kChunk * 4 * 4;
    static constexpr int kBytes = (kSumOff + kSumBytes + 1023) / 1024 * 1024;
    static constexpr int kFit = (kMaxDynSmem - 1024) / kBytes;
    static constexpr int kCount = kFit < 4 ? kFit : 4;
    static constexpr int kSmem = kCount * kBytes + 1024;
    // TMA bytes of a pass's stage, without the scale / bias tables
    static constexpr int tx(int pass) { return kWBytes + (pass ? 8 : 4) * kBox + kSumBytes; }
};
static_assert(StageCfg<kGateUp, 16, 8>::kCount == 4 && StageCfg<kDown, 8, 8>::kCount == 4, "ring depth");
static_assert(StageCfg<kDown, 16, 8>::kCount == 3 && StageCfg<kBoth, 16, 8>::kCount == 3, "ring depth");
static_assert(StageCfg<kGateUp, 16, 12>::kCount == 3, "ring depth (12 consumer warps: stages of 1.5x the work)");
static_assert(StageCfg<kGateUp, 16, 8>::kSmem <= kMaxDynSmem && StageCfg<kDown, 8, 8>::kSmem <= kMaxDynSmem &&
                  StageCfg<kDown, 16, 8>::kSmem <= kMaxDynSmem && StageCfg<kBoth, 16, 8>::kSmem <= kMaxDynSmem &&
                  StageCfg<kGateUp, 16, 12>::kSmem <= kMaxDynSmem,
              "expert pass shared memory");


struct PassArgs {
    int64_t wrow0;        // pass 0: gate rows per expert in map_w0; pass 1: d
    int64_t wrow1;        // pass 0: up rows per expert in map_w1
    int64_t woff1;        // pass 0: first up row inside an expert block (0 or F)
    const uint16_t* s0; const uint16_t* b0;   // scales/biases of map_w0 rows
    const uint16_t* s1; const uint16_t* b1;   // scales/biases of map_w1 rows
    int kdim;             // contraction length (d for pass 0, F for pass 1)
    int F, d, K, E, B;
    int tiles_per_expert;
    int tc_min;           // experts with at least this many entries belong to the tensor-core path (0: none)
    const int32_t* union_ids; const int32_t* n_union; const int32_t* offsets;
    const int32_t* token_list; const int32_t* slot_list;
    __half* h_out; float* hsum_out;   // pass 0 outputs
    float* y_out;                     // pass 1 output [B*K, d]: w[t,k] y_k(x_t), the weighted slot
    const int32_t* entl;              // output row t*K + k of list position p (-1: rejected)
    const float* wl;                  // routing weight of list position p
    uint32_t* status;
};

struct Tile {
    bool ok;              // indices valid
    bool mine;            // handled by this kernel (not by the tensor-core path)
    int e, p0, p1, row;   // row: first h column (pass 0) or output row (pass 1) of the tile
};

// One 256-input k-slice (4 groups) of a consumer warp: two 16-row m-tiles against NT
// 8-token n-tiles.  wb0/wb1: shared addresses of the m-tiles' first rows; xs: the activation
// boxes (4, or with LO 4 hi + 4 lo); sc/bi: the stage's bf16 scales / biases of rows g and
// g+8 of each m-tile ([m][row], 4 groups each); sums: the stage's activation group sums.
// Per group: acc += (scale * 2^24) * C + bias * S, C the exact mma result in units of 2^-24
// and S the tokens' group sums.
// PK (with LO, NT = 1, at most 4 tokens): the hi and lo terms share one 8-column n-tile,
// columns 0-3 the hi terms of tokens 0-3 and columns 4-7 their lo terms, so each k-step is
// one mma instead of two.  The lo columns get no bias term (S = 0 there: the group sum
// already covers hi + lo); the caller adds column j + 4 into column j at the end.
template <int NT, bool LO, bool PK, int XB>
__device__ __forceinline__ void consume_stage(float (&acc)[2][NT][4], uint32_t wb0, uint32_t wb1, uint32_t xs,
                                              const uint2 (&sc)[2][2], const uint2 (&bi)[2][2], uint32_t sums,
                                              int g, int c) {
    static_assert(!PK || (LO && NT == 1), "packed hi/lo columns: down pass, one n-tile");
    static_assert(NT * 8 * 128 <= XB, "the chunk's tokens fit the activation box");
    constexpr int NB = (LO && !PK) ? 2 : 1;   // activation terms per input (separate n-tiles)
    float4 S[NT][2];                 // group sums of tokens 2c and 2c+1 of each n-tile, 4 groups
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
        if (PK && c >= 2) {   // lo columns
            S[nt][0] = S[nt][1] = make_float4(0.f, 0.f, 0.f, 0.f);
            continue;
        }
        const uint4 v0 = lds_u4(sums + (uint32_t)(nt * 8 + 2 * c) * 16u);
        const uint4 v1 = lds_u4(sums + (uint32_t)(nt * 8 + 2 * c + 1) * 16u);
        S[nt][0] = make_float4(__uint_as_float(v0.x), __uint_as_float(v0.y), __uint_as_float(v0.z),
                               __uint_as_float(v0.w));
        S[nt][1] = make_float4(__uint_as_float(v1.x), __uint_as_float(v1.y), __uint_as_float(v1.z),
                               __uint_as_float(v1.w));
    }
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        uint32_t bf[NT][NB][8];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            // B row g of the n-tile: token row r of box hl; packed: token g & 3 of the hi (g < 4)
            // or lo (g >= 4) boxes.  The 128-byte swizzle XORs chunks with the row's low bits.
            const int r = PK ? (g & 3) : nt * 8 + g;
            const int sw = r & 7;
#pragma unroll
            for (int hl = 0; hl < NB; ++hl) {
                const int box = PK ? (g >> 2) * 4 + q : hl * 4 + q;
                const uint32_t rb = xs + box * XB + r * 128;
                const uint4 v0 = lds_u4(rb + (((2 * c) ^ sw) << 4));
                const uint4 v1 = lds_u4(rb + (((2 * c + 1) ^ sw) << 4));
                bf[nt][hl][0] = v0.x; bf[nt][hl][1] = v0.y; bf[nt][hl][2] = v0.z; bf[nt][hl][3] = v0.w;
                bf[nt][hl][4] = v1.x; bf[nt][hl][5] = v1.y; bf[nt][hl][6] = v1.z; bf[nt][hl][7] = v1.w;
            }
        }
        const uint32_t off = (uint32_t)g * 128u + ((uint32_t)((2 * q + (c >> 1)) ^ g) << 4) + ((c & 1) << 3);
#pragma unroll
        for (int m = 0; m < 2; ++m) {
            const uint32_t wb = m ? wb1 : wb0;
            const uint2 wl = lds_u2(wb + off);
            const uint2 wh = lds_u2(wb + 8 * 128 + off);
            float ct[NT][4];
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int i = 0; i < 4; ++i) ct[nt][i] = 0.f;
#pragma unroll
            for (int h = 0; h < 2; ++h) {   // word 2c (h = 0) and word 2c+1 (h = 1) of the group
                const uint32_t Wl = h ? wl.y : wl.x, Wh = h ? wh.y : wh.x;
                const uint32_t Wl8 = __umulhi(Wl, 0x01000000u), Wh8 = __umulhi(Wh, 0x01000000u);   // >> 8 on the FMA pipe
                const uint32_t e0 = nib_even(Wl), e1 = nib_even(Wh), o0 = nib_odd(Wl), o1 = nib_odd(Wh);
                const uint32_t f0 = nib_even(Wl8), f1 = nib_even(Wh8), p0 = nib_odd(Wl8), p1 = nib_odd(Wh8);
                // step 2h: pairs of n0/n4 and n1/n5; step 2h+1: pairs of n2/n6 and n3/n7
#pragma unroll
                for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                    for (int hl = 0; hl < NB; ++hl) {
                        mma16816(ct[nt], e0, e1, o0, o1, bf[nt][hl][4 * h], bf[nt][hl][4 * h + 1]);
                        mma16816(ct[nt], f0, f1, p0, p1, bf[nt][hl][4 * h + 2], bf[nt][hl][4 * h + 3]);
                    }
            }
            // scale and bias of this group: rows g (lo) and g+8 (hi); C is in units of 2^-24
            const uint32_t swl = (q < 2) ? sc[m][0].x : sc[m][0].y, swh = (q < 2) ? sc[m][1].x : sc[m][1].y;
            const uint32_t bwl = (q < 2) ? bi[m][0].x : bi[m][0].y, bwh = (q < 2) ? bi[m][1].x : bi[m][1].y;
            const float slo = __uint_as_float((q & 1) ? (swl & 0xFFFF0000u) : (swl * 65536u)) * 16777216.f;
            const float shi = __uint_as_float((q & 1) ? (swh & 0xFFFF0000u) : (swh * 65536u)) * 16777216.f;
            const float blo = __uint_as_float((q & 1) ? (bwl & 0xFFFF0000u) : (bwl * 65536u));
            const float bhi = __uint_as_float((q & 1) ? (bwh & 0xFFFF0000u) : (bwh * 65536u));
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                const float s0 = q == 0 ? S[nt][0].x : q == 1 ? S[nt][0].y : q == 2 ? S[nt][0].z : S[nt][0].w;
                const float s1 = q == 0 ? S[nt][1].x : q == 1 ? S[nt][1].y : q == 2 ? S[nt][1].z : S[nt][1].w;
                acc[m][nt][0] = fmaf(slo, ct[nt][0], fmaf(blo, s0, acc[m][nt][0]));
                acc[m][nt][1] = fmaf(slo, ct[nt][1], fmaf(blo, s1, acc[m][nt][1]));
                acc[m][nt][2] = fmaf(shi, ct[nt][2], fmaf(bhi, s0, acc[m][nt][2]));
                acc[m][nt][3] = fmaf(shi, ct[nt][3], fmaf(bhi, s1, acc[m][nt][3]));
            }
        }
    }
}

struct Ring {
    uint32_t buf, full, empty;   // shared addresses: stage 0, full[0], empty[0] (8 bytes apart)
};

// All consumer warps of a chunk: stream the k-slices, then the pass epilogue.
// Finished gate/up tiles go to the publisher warp through a small mailbox ring: slot k % 4
// holds the union slot of the k-th finished tile (-1: no more), full/empty mbarriers.
struct Mailbox {
    int* uu;                // [kMailbox]
    uint32_t full, empty;   // shared addresses of full[0], empty[0] (8 bytes apart)
    uint32_t k;             // posts so far (consumer thread 0)
};

// Consumer thread 0: hand the k-th entry to the publisher (bounded wait for a free slot).
__device__ __forceinline__ bool mailbox_post(Mailbox& M, int uu) {
    const uint32_t slot = M.k % kMailbox;
    if (M.k >= kMailbox && !mbar_wait(M.empty + 8 * slot, ((M.k / kMailbox) - 1) & 1u)) return false;
    M.uu[slot] = uu;
    mbar_arrive(M.full + 8 * slot);   // release: the consumers' stores before it (named barrier)
    ++M.k;
    return true;
}

// Pass 0, the tile's last chunk (done_uu >= 0): after the named barrier that ends the
// epilogue, every consumer thread's h and group-sum stores happen before consumer thread 0
// posts the tile to the publisher, which makes them visible device-wide and counts the tile
// for the expert's down tiles.  Publishing from a warp of its own keeps the fence's wait for
// outstanding stores off the consumers.
template <int NT, int PASS, int MODE, int CH, int NW, bool PK = false>
__device__ __forceinline__ void consume_chunk(const PassArgs& a, const Ring& R, uint32_t& it, bool& poisoned,
                                              const Tile& T, int pc, int n, int warp, int lane, float* red,
                                              int done_uu, Mailbox& M) {
    using C = StageCfg<MODE, CH, NW>;
    const int g = lane >> 2, c = lane & 3;
    const int nst = a.kdim / kGroup / 4;
    float acc[2][NT][4];
#pragma unroll
    for (int m = 0; m < 2; ++m)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int i = 0; i < 4; ++i) acc[m][nt][i] = 0.f;

    // the m-tiles' first rows inside a stage (weight box and scale / bias tables)
    uint32_t wrow_off0, wrow_off1;
    int lrow0, lrow1;
    if (PASS == 0) {
        lrow0 = warp * 16;               // gate rows 16w.. of the tile
        lrow1 = 16 * NW + warp * 16;     // up rows
    } else {
        lrow0 = warp * 32;
        lrow1 = warp * 32 + 16;
    }
    wrow_off0 = (uint32_t)lrow0 * 128u;
    wrow_off1 = (uint32_t)lrow1 * 128u;
    // pass 1: output row t*K + k (-1 past the chunk or for an index the gather rejected) and
    // routing weight of this thread's output columns, loaded before the k loop and first used
    // after it
    int ent[NT][2];
    float wgt[NT][2];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            const int slot = nt * 8 + 2 * c + j;
            ent[nt][j] = -1;
            wgt[nt][j] = 0.f;
            if (PASS == 1 && slot < n) {
                ent[nt][j] = a.entl[pc + slot];
                wgt[nt][j] = a.wl[pc + slot];
            }
        }
    const bool packed = a.kdim / kGroup == 4;   // tables [256][4]: the whole row
    const uint32_t rs = packed ? 8u : 16u;
    auto tab_off = [&](int st) { return packed ? 0u : (uint32_t)(st & 1) * 8u; };
    for (int st = 0; st < nst; ++st) {
        const uint32_t slot = it % C::kCount;
        const uint32_t parity = (it / C::kCount) & 1u;
        if (!poisoned && !mbar_wait(R.full + 8 * slot, parity)) {
            poisoned = true;
            if (lane == 0) atomicOr(a.status, SMOE_FAULT_TIMEOUT);
        }
        const uint32_t base = R.buf + slot * C::kBytes;
        // this stage's 4 groups in the tables: row stride rs, at byte tab_off inside a row
        const uint32_t ts = base + C::kSOff + tab_off(st), tb = base + C::kBOff + tab_off(st);
        uint2 sc[2][2], bi[2][2];
        sc[0][0] = lds_u2(ts + (uint32_t)(lrow0 + g) * rs);
        sc[0][1] = lds_u2(ts + (uint32_t)(lrow0 + g + 8) * rs);
        sc[1][0] = lds_u2(ts + (uint32_t)(lrow1 + g) * rs);
        sc[1][1] = lds_u2(ts + (uint32_t)(lrow1 + g + 8) * rs);
        bi[0][0] = lds_u2(tb + (uint32_t)(lrow0 + g) * rs);
        bi[0][1] = lds_u2(tb + (uint32_t)(lrow0 + g + 8) * rs);
        bi[1][0] = lds_u2(tb + (uint32_t)(lrow1 + g) * rs);
        bi[1][1] = lds_u2(tb + (uint32_t)(lrow1 + g + 8) * rs);
        consume_stage<NT, PASS == 1, PK, C::kBox>(acc, base + wrow_off0, base + wrow_off1, base + C::kXOff, sc, bi,
                                     base + C::kSumOff, g, c);
        __syncwarp();   // the warp's reads of the slot, then one arrival for the warp
        if (lane == 0) mbar_arrive(R.empty + 8 * slot);
        ++it;
    }

    if (PASS == 0) {
        // h = silu(gate) * up as two fp16 terms hi + lo, pair-permuted columns [0, F) and
        // [F, 2F), odd columns of every 8 divided by 16; per 64-column group the sum of the
        // values the stored halves stand for
        float hs[NT][2];   // [nt][token 2c / 2c+1]
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            hs[nt][0] = hs[nt][1] = 0.f;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float gv = acc[0][nt][i], uv = acc[1][nt][i];
                const float hv = gv / (1.f + expf(-gv)) * uv;
                const int slot = nt * 8 + 2 * c + (i & 1);
                const int j = T.row + warp * 16 + g + ((i & 2) ? 8 : 0);
                const bool odd = j & 1;   // same parity as g
                const float hsv = odd ? hv * 0.0625f : hv;
                const __half hh = __float2half_rn(hsv);
                const __half hl = __float2half_rn(hsv - __half2float(hh));
                if (slot < n) {
                    if (!(fabsf(hv) <= 65504.f)) atomicOr(a.status, SMOE_FAULT_FP16_RANGE);
                    __half* row = a.h_out + (size_t)(pc + slot) * (2 * a.F);
                    const int col = (j & ~7) + perm8(j & 7);
                    row[col] = hh;
                    row[a.F + col] = hl;
                }
                const float stood = __half2float(hh) + __half2float(hl);
                hs[nt][i & 1] += odd ? stood * 16.f : stood;
            }
#pragma unroll
            for (int q = 0; q < 2; ++q) {
                float v = hs[nt][q];
                v += __shfl_xor_sync(0xffffffffu, v, 4);
                v += __shfl_xor_sync(0xffffffffu, v, 8);
                v += __shfl_xor_sync(0xffffffffu, v, 16);
                hs[nt][q] = v;
            }
        }
        if (g == 0) {
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                red[warp * 16 + nt * 8 + 2 * c] = hs[nt][0];
                red[warp * 16 + nt * 8 + 2 * c + 1] = hs[nt][1];
            }
        }
        asm volatile("bar.sync 1, %0;\n" ::"r"(32 * NW) : "memory");
        const int tid = warp * 32 + lane;
        if (tid < 4 * NW) {
            // 16 NW columns = NW / 4 groups of 64 columns, four warps each
            const int grp = tid >> 4, slot = tid & 15;
            if (slot < n) {
                const float s = red[(4 * grp) * 16 + slot] + red[(4 * grp + 1) * 16 + slot] +
                                red[(4 * grp + 2) * 16 + slot] + red[(4 * grp + 3) * 16 + slot];
                a.hsum_out[(size_t)(pc + slot) * (a.F / kGroup) + T.row / kGroup + grp] = s;
            }
        }
        asm volatile("bar.sync 1, %0;\n" ::"r"(32 * NW) : "memory");
        // every consumer thread's h / sum stores happen before this point (named barrier);
        // the fence makes them visible device-wide before the count
        if (done_uu >= 0 && tid == 0 && !mailbox_post(M, done_uu)) atomicOr(a.status, SMOE_FAULT_TIMEOUT);
    } else {
        if (PK) {   // lo columns 4-7 (lanes c = 2, 3) into hi columns 0-3 (lanes c = 0, 1)
#pragma unroll
            for (int m = 0; m < 2; ++m)
#pragma unroll
                for (int i = 0; i < 4; ++i) acc[m][0][i] += __shfl_xor_sync(0xffffffffu, acc[m][0][i], 2);
        }
#pragma unroll
        for (int m = 0; m < 2; ++m)
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int e = ent[nt][i & 1];
                    if (e < 0) continue;
                    const int r = T.row + warp * 32 + m * 16 + g + ((i & 2) ? 8 : 0);
                    a.y_out[(size_t)e * a.d + r] = acc[m][nt][i] * wgt[nt][i & 1];
                }
    }
}

// The expert passes as persistent kernels with a device-side work queue.  Work items, in this
// order: the gate/up tiles (16 NW h columns of one union expert: consumer warp w takes gate and
// up rows 16w..16w+15; NW = 8, or 12 where ffn_dim is a multiple of 192 and the tiles fill the
// SMs twice: three consumer warps per scheduler instead of two hide more of each warp's
// latency), then the down tiles (256 output rows of one union expert: consumer warp w takes
// rows 32w..32w+31), expert-major.  A launch runs the gate/up items, the down
// items, or both (MODE).  The producer thread takes the next item with an atomic ticket, so
// CTAs that draw long items (experts with many tokens) do not hold up the rest.  With both
// passes in one launch, items are claimed in order and every item a CTA waits for has been
// claimed by a running CTA: a down tile waits (bounded) until all gate/up tiles of its expert
// have been published, which lets the down tiles of finished experts fill the SMs while the
// last gate/up tiles run, with no grid-wide barrier.  The item of every ring stage travels
// with it in shared memory; an item < 0 tells the consumers to stop.
struct FusedArgs {
    PassArgs p[2];
    int32_t* ticket;      // [0]: next item of a gate/up or both-pass launch; [1]: next item of a
                          // down launch; [2 + u]: published gate/up tiles of union expert u
};

// OR of v over the NW consumer warps' threads (named barrier 1).
template <int NW>
__device__ __forceinline__ bool consumers_any(bool v) {
    uint32_t r;
    asm volatile(
        "{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n bar.red.or.pred q, 1, %2, p;\n selp.u32 %0, 1, 0, q;\n}\n"
        : "=r"(r)
        : "r"((uint32_t)v), "r"(32 * NW)
        : "memory");
    return r != 0;
}

__device__ __forceinline__ int ld_acquire(const int32_t* p) {
    int v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];\n" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// Bounded wait (~0.5 s) until *p >= target.
__device__ __forceinline__ bool wait_count(const int32_t* p, int target) {
    uint64_t t0 = 0;
    for (uint32_t i = 0;; ++i) {
        if (ld_acquire(p) >= target) return true;
        uint64_t now;
        asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(now));
        if (i == 0) t0 = now;
        else if (now - t0 > 500000000ull) return false;
        __nanosleep(256);
    }
}

__device__ __forceinline__ int ld_relaxed(const int32_t* p) {
    int v;
    asm volatile("ld.relaxed.gpu.global.b32 %0, [%1];\n" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// A claimed work item and the global values it needs, loaded as soon as the item is known
// and used one item later (so the producer does not wait on their latency).
struct Claim {
    int item, pass, j, uu;   // item, its pass, index inside the pass, union slot of the expert
    int e, p0, p1;           // expert id and its token-list range
    int done;                // pass 1: finished gate/up tiles of the expert when loaded
};

__device__ __forceinline__ Claim claim_item(const FusedArgs& f, int item, int n0, int n_items) {
    Claim c{};
    c.item = item;
    if (item >= n_items) return c;
    c.pass = item >= n0;
    c.j = c.pass ? item - n0 : item;
    c.uu = c.j / (c.pass ? f.p[1].tiles_per_expert : f.p[0].tiles_per_expert);
    c.e = f.p[0].union_ids[c.uu];
    c.p0 = f.p[0].offsets[c.uu];
    c.p1 = f.p[0].offsets[c.uu + 1];
    if (c.pass) c.done = ld_relaxed(f.ticket + 2 + c.uu);
    return c;
}

template <int MODE, int CH, int NW>
__global__ void __launch_bounds__(pass_threads(MODE, NW), 1)
    ffn_expert_kernel(const __grid_constant__ CUtensorMap map_gate, const __grid_constant__ CUtensorMap map_up,
                     const __grid_constant__ CUtensorMap map_down, const __grid_constant__ CUtensorMap map_xg,
                     const __grid_constant__ CUtensorMap map_h, const __grid_constant__ CUtensorMap map_sx,
                     const __grid_constant__ CUtensorMap map_sh, const __grid_constant__ CUtensorMap map_sg,
                     const __grid_constant__ CUtensorMap map_su, const __grid_constant__ CUtensorMap map_bg,
                     const __grid_constant__ CUtensorMap map_bu, const __grid_constant__ CUtensorMap map_sd,
                     const __grid_constant__ CUtensorMap map_bd, FusedArgs f) {
    using C = StageCfg<MODE, CH, NW>;
    static_assert(NW % 4 == 0 && (NW == kConsumerWarps || gate_up_only(MODE)), "consumer warps");
    extern __shared__ uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t bars[2 * C::kCount];
    // per stage: item (< 0: stop), chunk start, and the decoded tile (expert, list range, row)
    __shared__ int slot_meta[C::kCount][6];
    __shared__ float red[NW * 16];
    __shared__ __align__(8) uint64_t mbars[2 * kMailbox];
    __shared__ int mail[kMailbox];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    Ring R;
    R.buf = smem_addr(smem);
    R.full = smem_addr(&bars[0]);
    R.empty = smem_addr(&bars[C::kCount]);
    Mailbox M;
    M.uu = mail;
    M.full = smem_addr(&mbars[0]);
    M.empty = smem_addr(&mbars[kMailbox]);
    M.k = 0;
    if (threadIdx.x == 0) {
        for (int s = 0; s < C::kCount; ++s) {
            mbar_init(R.full + 8 * s, 1);
            mbar_init(R.empty + 8 * s, NW);   // one arrival per consumer warp
        }
        for (int s = 0; s < kMailbox; ++s) {
            mbar_init(M.full + 8 * s, 1);
            mbar_init(M.empty + 8 * s, 1);
        }
        asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
    }
    __syncthreads();

    const int nu = *f.p[0].n_union;
    const int t0 = f.p[0].tiles_per_expert, n0 = nu * t0;
    const int first_item = down_only(MODE) ? n0 : 0;
    const int n_items = gate_up_only(MODE) ? n0 : n0 + nu * f.p[1].tiles_per_expert;
    int32_t* queue = f.ticket + (down_only(MODE) ? 1 : 0);
    uint32_t it = 0;
    bool poisoned = false;

    if (has_publisher(MODE) && warp == NW + 1) {
        // ---------------------------------------------------------------- publisher (one thread)
        if (lane == 0) {
            for (uint32_t k = 0;; ++k) {
                const uint32_t slot = k % kMailbox;
                if (!mbar_wait(M.full + 8 * slot, (k / kMailbox) & 1u)) {
                    atomicOr(f.p[0].status, SMOE_FAULT_TIMEOUT);
                    break;
                }
                const int uu = *reinterpret_cast<volatile int*>(&mail[slot]);
                if (uu < 0) break;
                __threadfence();                 // the tile's h / sums before the count
                atomicAdd(f.ticket + 2 + uu, 1);
                mbar_arrive(M.empty + 8 * slot);
            }
        }
        return;
    }

    if (warp == NW) {
        // ---------------------------------------------------------------- producer (one thread)
        if (lane == 0) {
            // tickets run two items ahead and the globals of an item are loaded one item ahead,
            // so no latency of the queue sits between the stages of consecutive items
            // one-pass launches: static round-robin (uniform items, no queue latency); both
            // passes: the ordered queue that makes the cross-CTA waits safe
            int sk = 0;
            auto take = [&]() { return claims(MODE) ? atomicAdd(queue, 1) : (int)(blockIdx.x + gridDim.x * sk++); };
            Claim cur = claim_item(f, first_item + take(), n0, n_items);
            int next_item = first_item + take();
            for (;;) {
                const int item = cur.item;
                if (item >= n_items || poisoned) break;
                const int after_next = first_item + take();
                const Claim nxt = claim_item(f, next_item, n0, n_items);
                const PassArgs& a = cur.pass ? f.p[1] : f.p[0];
                Tile T;
                T.e = cur.e;
                T.p0 = cur.p0;
                T.p1 = cur.p1;
                T.row = (cur.j - cur.uu * a.tiles_per_expert) * (cur.pass ? 32 * NW : 16 * NW);
                T.ok = T.e >= 0 && T.e < a.E && T.p0 >= 0 && T.p1 >= T.p0 && T.p1 <= a.B * a.K;
                T.mine = a.tc_min <= 0 || T.p1 - T.p0 < a.tc_min;
                if (!T.ok) atomicOr(a.status, SMOE_FAULT_EXPERT_INDEX);
                if (T.ok && T.mine) {
                    if (claims(MODE) && cur.pass == 1) {
                        // every gate/up tile of this expert has published h and its group sums
                        // (an acquire load, not a fence: a fence would also wait for this
                        // thread's copies in flight)
                        if (!(cur.done >= t0 && ld_acquire(f.ticket + 2 + cur.uu) >= t0) &&
                            !wait_count(f.ticket + 2 + cur.uu, t0)) {
                            poisoned = true;
                            atomicOr(a.status, SMOE_FAULT_TIMEOUT);
                            break;
                        }
                        asm volatile("fence.proxy.async.global;\n" ::: "memory");   // h is read by TMA
                    }
                    const int G = a.kdim / kGroup, nst = G / 4;
                    const bool packed = G == 4;
                    const uint32_t rs = packed ? 8u : 16u;
                    const uint32_t tx = (uint32_t)C::tx(cur.pass) + 2u * (uint32_t)C::kRows * rs;
                    // first rows of the tile in the weight maps
                    const int64_t r0 = (int64_t)T.e * a.wrow0 + T.row;
                    const int64_t r1 = cur.pass == 0 ? (int64_t)T.e * a.wrow1 + a.woff1 + T.row : r0;
                    // the tile's scale / bias rows into L2 ahead of the table copies
                    const uint32_t bytes = (uint32_t)((cur.pass ? 32 * NW : 16 * NW) * G * 2);
                    prefetch_l2(a.s0 + r0 * G, bytes); prefetch_l2(a.b0 + r0 * G, bytes);
                    if (cur.pass == 0) { prefetch_l2(a.s1 + r1 * G, bytes); prefetch_l2(a.b1 + r1 * G, bytes); }
                    const int ty0 = (int)(packed ? r0 / 2 : r0), ty1 = (int)(packed ? r1 / 2 : r1);
                    for (int pc = T.p0; pc < T.p1 && !poisoned; pc += C::kChunk) {
                        for (int st = 0; st < nst; ++st) {
                            const uint32_t slot = it % C::kCount;
                            if (it >= C::kCount && !mbar_wait(R.empty + 8 * slot, ((it / C::kCount) - 1) & 1u)) {
                                poisoned = true;
                                atomicOr(a.status, SMOE_FAULT_TIMEOUT);
                                break;
                            }
                            const uint32_t base = R.buf + slot * C::kBytes;
                            const uint32_t full = R.full + 8 * slot;
                            slot_meta[slot][0] = item;
                            slot_meta[slot][1] = pc;
                            slot_meta[slot][2] = T.e;
                            slot_meta[slot][3] = T.p0;
                            slot_meta[slot][4] = T.p1;
                            slot_meta[slot][5] = T.row;
                            mbar_expect_tx(full, tx);
                            const int tx0 = packed ? 0 : (st * 4) & ~7;   // 16-byte window of the stage's groups
                            if (gate_up_only(MODE) || (MODE == kBoth && cur.pass == 0)) {
                                tma_load_2d(base, &map_gate, st * 32, (int)r0, full);
                                tma_load_2d(base + 16 * NW * 128, &map_up, st * 32, (int)r1, full);
                                tma_load_2d(base + C::kSOff, &map_sg, tx0, ty0, full);
                                tma_load_2d(base + C::kSOff + 16 * NW * rs, &map_su, tx0, ty1, full);
                                tma_load_2d(base + C::kBOff, &map_bg, tx0, ty0, full);
                                tma_load_2d(base + C::kBOff + 16 * NW * rs, &map_bu, tx0, ty1, full);
#pragma unroll
                                for (int q = 0; q < 4; ++q)
                                    tma_load_2d(base + C::kXOff + q * C::kBox, &map_xg, (st * 4 + q) * 64, pc,
                                                full);
                                tma_load_2d(base + C::kSumOff, &map_sx, st * 4, pc, full);
                            } else if (!gate_up_only(MODE)) {
                                tma_load_2d(base, &map_down, st * 32, (int)r0, full);
                                tma_load_2d(base + C::kSOff, &map_sd, tx0, ty0, full);
                                tma_load_2d(base + C::kBOff, &map_bd, tx0, ty0, full);
#pragma unroll
                                for (int q = 0; q < 4; ++q) {   // h hi, then its lo terms (columns F..)
                                    tma_load_2d(base + C::kXOff + q * C::kBox, &map_h, (st * 4 + q) * 64, pc, full);
                                    tma_load_2d(base + C::kXOff + (4 + q) * C::kBox, &map_h,
                                                a.F + (st * 4 + q) * 64, pc, full);
                                }
                                tma_load_2d(base + C::kSumOff, &map_sh, st * 4, pc, full);
                            }
                            ++it;
                        }
                    }
                }
                cur = nxt;
                next_item = after_next;
            }
            if (!poisoned) {
                // end of work: a stage with item -1 and no copies
                const uint32_t slot = it % C::kCount;
                if (it >= C::kCount && !mbar_wait(R.empty + 8 * slot, ((it / C::kCount) - 1) & 1u)) {
                    poisoned = true;
                    atomicOr(f.p[0].status, SMOE_FAULT_TIMEOUT);
                } else {
                    slot_meta[slot][0] = -1;
                    mbar_arrive(R.full + 8 * slot);
                }
            }
            // drain: every issued stage has landed before the CTA may exit
            if (poisoned) {
                const uint32_t first = it > C::kCount ? it - C::kCount : 0;
                for (uint32_t i = first; i < it; ++i) mbar_wait(R.full + 8 * (i % C::kCount), (i / C::kCount) & 1u);
            }
        }
        return;
    }

    // -------------------------------------------------------------------- consumers
    for (;;) {
        const uint32_t slot = it % C::kCount;
        // launches with gate/up tiles: all consumer threads take the same decision, so that
        // they run the same chunks and meet at the same named barriers; a down-only launch has
        // none, and each warp decides for itself (no cross-warp sync per chunk)
        const bool late = !mbar_wait(R.full + 8 * slot, (it / C::kCount) & 1u);
        if (down_only(MODE) ? __any_sync(0xffffffffu, late) : consumers_any<NW>(late)) {
            if (threadIdx.x == 0) atomicOr(f.p[0].status, SMOE_FAULT_TIMEOUT);
            break;
        }
        const volatile int* meta = slot_meta[slot];
        const int item = meta[0];
        if (item < 0) break;
        const int pc = meta[1];
        Tile T;
        T.ok = T.mine = true;
        T.e = meta[2];
        T.p0 = meta[3];
        T.p1 = meta[4];
        T.row = meta[5];
        const int n = min(C::kChunk, T.p1 - pc);
        const bool gate_up = gate_up_only(MODE) || (MODE == kBoth && item < n0);
        if constexpr (!down_only(MODE)) {
            if (gate_up) {
                // both passes in this launch: publish the tile after its last chunk
                const int done_uu = has_publisher(MODE) && pc + C::kChunk >= T.p1 ? item / t0 : -1;
                if (n <= 8) consume_chunk<1, 0, MODE, CH, NW>(f.p[0], R, it, poisoned, T, pc, n, warp, lane, red, done_uu, M);
                else consume_chunk<2, 0, MODE, CH, NW>(f.p[0], R, it, poisoned, T, pc, n, warp, lane, red, done_uu, M);
            }
        }
        if constexpr (!gate_up_only(MODE)) {
            if (!gate_up) {
                if (n <= 4)
                    consume_chunk<1, 1, MODE, CH, NW, true>(f.p[1], R, it, poisoned, T, pc, n, warp, lane, red, -1, M);
                else if constexpr (CH <= 8)   // chunks of at most 8 tokens
                    consume_chunk<1, 1, MODE, CH, NW>(f.p[1], R, it, poisoned, T, pc, n, warp, lane, red, -1, M);
                else if (n <= 8)
                    consume_chunk<1, 1, MODE, CH, NW>(f.p[1], R, it, poisoned, T, pc, n, warp, lane, red, -1, M);
                else consume_chunk<2, 1, MODE, CH, NW>(f.p[1], R, it, poisoned, T, pc, n, warp, lane, red, -1, M);
            }
        }
        if (poisoned) break;
    }
    // no more tiles to publish
    if (has_publisher(MODE) && threadIdx.x == 0 && !mailbox_post(M, -1)) atomicOr(f.p[0].status, SMOE_FAULT_TIMEOUT);
}

// ----------------------------------------------------------------------------- combine
// The down passes' epilogues store every slot already weighted (w[t,k] y_k, the weighted half
// of the combine); this is the deterministic rank-order reduction that adds a token's K
// weighted slots into its residual row: residual[t] += sum_k (w y)_k in rank order k = 0..K-1.
// Skipped entirely (residual untouched) when the union did not cover all B*K entries, i.e.
// after a flagged routing fault.  A thread issues the loads of up to 8 slots (and the union
// check) together before its rank-ordered chain of adds, so it waits on one L2 round trip
// instead of one per slot.
__global__ void __launch_bounds__(256) combine_kernel(const float* __restrict__ y,
                                                      const int32_t* __restrict__ n_union,
                                                      const int32_t* __restrict__ offsets, int B, int K, int d,
                                                      float* __restrict__ residual) {
    const size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;   // float4 index
    const size_t n4 = (size_t)B * d / 4;
    if (i >= n4) return;
    const int covered = offsets[*n_union];
    const int t = (int)(i / (d / 4));
    const int c4 = (int)(i - (size_t)t * (d / 4));
    const float4* yt = reinterpret_cast<const float4*>(y + (size_t)t * K * d) + c4;
    float4 acc = reinterpret_cast<float4*>(residual)[i];
    for (int k0 = 0; k0 < K; k0 += 8) {
        float4 v[8];
#pragma unroll
        for (int j = 0; j < 8; ++j)
            if (k0 + j < K) v[j] = yt[(size_t)(k0 + j) * (d / 4)];
#pragma unroll
        for (int j = 0; j < 8; ++j)
            if (k0 + j < K) {
                acc.x += v[j].x;
                acc.y += v[j].y;
                acc.z += v[j].z;
                acc.w += v[j].w;
            }
    }
    if (covered != B * K) return;
    reinterpret_cast<float4*>(residual)[i] = acc;
}

// The combine followed by the norm that feeds the next block, one CTA of 512 threads per token
// row (d <= 4096: a thread holds up to 2 float4 of the row): residual[t] += sum_k (w y)_k (the
// combine_kernel's rank-ordered chain of adds), then x_next[t] = bf16(norm(residual[t])) with
// rmsnorm_bf16_kernel's loop order and reductions, so both outputs equal combine_kernel +
// rmsnorm_bf16_kernel bit for bit.  After a flagged routing fault (the union did not cover all
// B*K entries) neither residual nor x_next is written.
__global__ void __launch_bounds__(512) combine_norm_kernel(const float* __restrict__ y,
                                                           const int32_t* __restrict__ n_union,
                                                           const int32_t* __restrict__ offsets, int B, int K, int d,
                                                           float* __restrict__ residual, float eps, int center,
                                                           uint16_t* __restrict__ x_next) {
    __shared__ float red[16];
    const int t = blockIdx.x;
    const int n4 = d / 4;   // <= 1024
    const bool covered = offsets[*n_union] == B * K;
    float4* row = reinterpret_cast<float4*>(residual + (size_t)t * d);
    float4 v[2];
#pragma unroll
    for (int j = 0; j < 2; ++j) {
        const int i = threadIdx.x + 512 * j;
        if (i >= n4) break;
        const float4* yt = reinterpret_cast<const float4*>(y + (size_t)t * K * d) + i;
        float4 acc = row[i];
        for (int k0 = 0; k0 < K; k0 += 8) {
            float4 yv[8];
#pragma unroll
            for (int q = 0; q < 8; ++q)
                if (k0 + q < K) yv[q] = yt[(size_t)(k0 + q) * n4];
#pragma unroll
            for (int q = 0; q < 8; ++q)
                if (k0 + q < K) {
                    acc.x += yv[q].x;
                    acc.y += yv[q].y;
                    acc.z += yv[q].z;
                    acc.w += yv[q].w;
                }
        }
        v[j] = acc;
    }
    if (!covered) return;   // the same decision in every thread of the CTA
#pragma unroll
    for (int j = 0; j < 2; ++j)
        if (threadIdx.x + 512 * j < n4) row[threadIdx.x + 512 * j] = v[j];
    float mean = 0.f;
    if (center) {
        float s = 0.f;
#pragma unroll
        for (int j = 0; j < 2; ++j)
            if (threadIdx.x + 512 * j < n4) s += (v[j].x + v[j].y) + (v[j].z + v[j].w);
        mean = block_sum512(s, red) / (float)d;
    }
    float ss = 0.f;
#pragma unroll
    for (int j = 0; j < 2; ++j)
        if (threadIdx.x + 512 * j < n4) {
            const float a = v[j].x - mean, b = v[j].y - mean, c = v[j].z - mean, e = v[j].w - mean;
            ss = fmaf(a, a, ss);
            ss = fmaf(b, b, ss);
            ss = fmaf(c, c, ss);
            ss = fmaf(e, e, ss);
        }
    const float tot = block_sum512(ss, red);
    const float inv = 1.0f / sqrtf(tot / (float)d + eps);
    uint2* out = reinterpret_cast<uint2*>(x_next + (size_t)t * d);
#pragma unroll
    for (int j = 0; j < 2; ++j)
        if (threadIdx.x + 512 * j < n4) {
            const uint32_t a = __bfloat16_as_ushort(__float2bfloat16_rn((v[j].x - mean) * inv));
            const uint32_t b = __bfloat16_as_ushort(__float2bfloat16_rn((v[j].y - mean) * inv));
            const uint32_t c = __bfloat16_as_ushort(__float2bfloat16_rn((v[j].z - mean) * inv));
            const uint32_t e = __bfloat16_as_ushort(__float2bfloat16_rn((v[j].w - mean) * inv));
            out[threadIdx.x + 512 * j] = make_uint2(a | (b << 16), c | (e << 16));
        }
}

}  // namespace

// 2-D tensor map over a row-major buffer [rows, cols] of `esize`-byte elements.
static bool encode_map_2d(CUtensorMap* map, const void* base, CUtensorMapDataType dt, int esize, int64_t rows,
                          int64_t cols, int box_cols, int box_rows, CUtensorMapSwizzle swz) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
    if (!enc) return false;
    cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)(cols * esize)};
    cuuint32_t box[2] = {(cuuint32_t)box_cols, (cuuint32_t)box_rows};
    cuuint32_t estr[2] = {1, 1};
    return enc(map, dt, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

cudaError_t launch_ffn(const smoe_layer_desc& D, const FfnPointers& W, const uint16_t* x, int B,
                       const int32_t* union_ids, const int32_t* n_union, const int32_t* offsets,
                       const int32_t* token_list, const int32_t* slot_list, const float* topk_w,
                       float* residual, void* ws, const WsLayout& L, cudaStream_t stream, bool all_tokens,
                       const NextNorm& next) {
    const int d = D.d_model, F = D.ffn_dim, K = D.top_k, E = D.num_experts;
    const int BK = B * K;
    const int max_u = BK < E ? BK : E;
    __half* xg = ws_ptr<__half>(ws, L.xg);
    float* sx = ws_ptr<float>(ws, L.sx);
    __half* h = ws_ptr<__half>(ws, L.h);
    float* sh = ws_ptr<float>(ws, L.sh);
    float* y = ws_ptr<float>(ws, L.y);
    uint32_t* status = ws_ptr<uint32_t>(ws, L.status);

    // per device: dynamic shared memory above 48 KB is opted into once; SM count cached
    static std::atomic<uint64_t> attr_done{0};
    static int sm_count[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return cudaErrorInvalidDevice;
    const uint64_t bit = 1ull << (dev & 63);
    if (!(attr_done.load() & bit)) {
        cudaError_t e = cudaFuncSetAttribute(ffn_expert_kernel<kGateUp, 16, 8>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             StageCfg<kGateUp, 16, 8>::kSmem);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(ffn_expert_kernel<kGateUp, 16, 12>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     StageCfg<kGateUp, 16, 12>::kSmem);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(ffn_expert_kernel<kDown, 8, 8>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     StageCfg<kDown, 8, 8>::kSmem);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(ffn_expert_kernel<kDown, 16, 8>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     StageCfg<kDown, 16, 8>::kSmem);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(ffn_expert_kernel<kBoth, 16, 8>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     StageCfg<kBoth, 16, 8>::kSmem);
        if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sm_count[dev & 63], cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return e;
        attr_done.fetch_or(bit);
    }
    const int sms = sm_count[dev & 63] > 0 ? sm_count[dev & 63] : 1;

    // experts with many tokens go to the tcgen05 path; with fewer than 256 tokens in the chunk
    // a routed expert rarely reaches the threshold, so the extra launches are skipped (the
    // slices of a shared expert hold every token and take it from kTcMinTokens tokens on)
    const int tc_min = (tc_path_supported(D) && (B >= 256 || (all_tokens && B >= kTcMinTokens))) ? kTcMinTokens : 0;
    const bool both = tc_min > 0;
    // tokens per down chunk: 8 while the experts average at most 4 tokens (then nearly all have
    // at most 8, and the smaller stages make a 4-stage ring), else 16
    const int ch_dn = !both && (int64_t)BK <= 4 * (int64_t)E ? 8 : kTokChunk;

    // activation / group-sum maps over this call's workspace rows, one box row per chunk token
    CUtensorMap map_xg, map_h, map_sx, map_sh;
    if (!encode_map_2d(&map_xg, xg, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, BK, d, 64, kTokChunk,
                       CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_map_2d(&map_h, h, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, BK, 2 * F, 64, ch_dn,
                       CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_map_2d(&map_sx, sx, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, BK, d / kGroup, 4, kTokChunk,
                       CU_TENSOR_MAP_SWIZZLE_NONE) ||
        !encode_map_2d(&map_sh, sh, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, BK, F / kGroup, 4, ch_dn,
                       CU_TENSOR_MAP_SWIZZLE_NONE))
        return cudaErrorInvalidValue;

    int32_t* ticket = ws_ptr<int32_t>(ws, L.ticket);
    // warps: one per 256 elements of a row for small batches, one per 4096 for large ones
    const bool big = BK > 4096;
    const int segs = (d / 8 + 32 * (big ? 16 : 1) - 1) / (32 * (big ? 16 : 1));
    const int gather_blocks = std::max(1, std::min((BK * segs + 7) / 8, sms * 16));
    (big ? gather_kernel<16> : gather_kernel<1>)<<<gather_blocks, 256, 0, stream>>>(x, d, B, n_union, offsets,
                                                                                     token_list, slot_list, topk_w, K,
                                                                                     ws_ptr<int32_t>(ws, L.entl),
                                                                                     ws_ptr<float>(ws, L.wl), status,
                                                                          xg, sx, ws_ptr<__half>(ws, L.s16x), BK,
                                                                          ticket, E + 2);

    FfnTcWeights TW{};
    TW.map_gate = W.tc_gate; TW.map_up = W.tc_up; TW.map_down = W.tc_down;
    TW.sg = W.sg; TW.bg = W.bg; TW.g_rows = W.g_rows_per_expert;
    TW.su = W.su; TW.bu = W.bu; TW.u_rows = W.u_rows_per_expert; TW.u_off = W.u_row_offset;
    TW.sd = W.sd; TW.bd = W.bd;

    PassArgs a{};
    a.wrow0 = W.g_rows_per_expert; a.wrow1 = W.u_rows_per_expert; a.woff1 = W.u_row_offset;
    a.s0 = W.sg; a.b0 = W.bg; a.s1 = W.su; a.b1 = W.bu;
    a.kdim = d; a.F = F; a.d = d; a.K = K; a.E = E; a.B = B;
    // gate/up tiles of 16 NW h columns: 12 consumer warps (192 columns) where ffn_dim allows it and
    // the tiles fill the SMs at least twice, else 8 (128 columns); the both-pass launch takes 8
    const int nw_gu = !both && W.wide && (int64_t)max_u * (F / 192) >= 2 * (int64_t)sms ? 12 : kConsumerWarps;
    a.tiles_per_expert = F / (16 * nw_gu);
    a.tc_min = tc_min;
    a.union_ids = union_ids; a.n_union = n_union; a.offsets = offsets;
    a.token_list = token_list; a.slot_list = slot_list;
    a.h_out = h; a.hsum_out = sh; a.y_out = y; a.status = status;
    a.entl = ws_ptr<int32_t>(ws, L.entl); a.wl = ws_ptr<float>(ws, L.wl);
    PassArgs b = a;
    b.wrow0 = d; b.wrow1 = d; b.woff1 = 0;
    b.s0 = W.sd; b.b0 = W.bd; b.s1 = W.sd; b.b1 = W.bd;
    b.kdim = F;
    b.tiles_per_expert = d / 256;
    FusedArgs fa{};
    fa.p[0] = a;
    fa.p[1] = b;
    fa.ticket = ticket;
    const int t0 = a.tiles_per_expert, t1 = b.tiles_per_expert;

    if (both) {
        // long prompts: experts with a few tokens each run both passes from one queue
        const int grid = std::min(sms, max_u * (t0 + t1));
        ffn_expert_kernel<kBoth, 16, 8><<<grid, pass_threads(kBoth, 8), StageCfg<kBoth, 16, 8>::kSmem, stream>>>(
            W.map_gate, W.map_up, W.map_down, map_xg, map_h, map_sx, map_sh, W.map_sg, W.map_su, W.map_bg, W.map_bu,
            W.map_sd, W.map_bd, fa);
    } else {
        if (nw_gu == 12)
            ffn_expert_kernel<kGateUp, 16, 12><<<std::min(sms, max_u * t0), pass_threads(kGateUp, 12),
                                                StageCfg<kGateUp, 16, 12>::kSmem, stream>>>(
                W.wide_gate, W.wide_up, W.map_down, map_xg, map_h, map_sx, map_sh, W.wide_sg, W.wide_su, W.wide_bg,
                W.wide_bu, W.map_sd, W.map_bd, fa);
        else
            ffn_expert_kernel<kGateUp, 16, 8><<<std::min(sms, max_u * t0), pass_threads(kGateUp, 8),
                                               StageCfg<kGateUp, 16, 8>::kSmem, stream>>>(
                W.map_gate, W.map_up, W.map_down, map_xg, map_h, map_sx, map_sh, W.map_sg, W.map_su, W.map_bg,
                W.map_bu, W.map_sd, W.map_bd, fa);
        const int g1 = std::min(sms, max_u * t1);
        if (ch_dn == 8)
            ffn_expert_kernel<kDown, 8, 8><<<g1, pass_threads(kDown, 8), StageCfg<kDown, 8, 8>::kSmem, stream>>>(
                W.map_gate, W.map_up, W.map_down, map_xg, map_h, map_sx, map_sh, W.map_sg, W.map_su, W.map_bg,
                W.map_bu, W.map_sd, W.map_bd, fa);
        else
            ffn_expert_kernel<kDown, 16, 8><<<g1, pass_threads(kDown, 8), StageCfg<kDown, 16, 8>::kSmem, stream>>>(
                W.map_gate, W.map_up, W.map_down, map_xg, map_h, map_sx, map_sh, W.map_sg, W.map_su, W.map_bg,
                W.map_bu, W.map_sd, W.map_bd, fa);
    }
    if (both) {
        for (int pass = 0; pass < 2; ++pass) {
            cudaError_t e = launch_ffn_tc(D, TW, B, pass, union_ids, n_union, offsets, token_list, slot_list, ws, L,
                                          tc_min, sms, stream);
            if (e != cudaSuccess) return e;
        }
    }

    if (next.x_next && d <= 4096) {
        combine_norm_kernel<<<B, 512, 0, stream>>>(y, n_union, offsets, B, K, d, residual, next.eps,
                                                   next.center, next.x_next);
        return cudaGetLastError();
    }
    const size_t n4 = (size_t)B * d / 4;
    combine_kernel<<<(unsigned)((n4 + 255) / 256), 256, 0, stream>>>(y, n_union, offsets, B, K, d,
                                                                      residual);
    if (next.x_next) {   // wider rows: the standalone norm after the combine
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
        return launch_rmsnorm(residual, next.eps, next.center, B, d, next.x_next, stream);
    }
    return cudaGetLastError();
}

}  // namespace smoe
