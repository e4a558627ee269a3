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
//   ffn_pass_kernel<0> gate/up projections + SwiGLU, 128 h columns of one expert per tile;
//                      writes h (fp16, pair-permuted) and its per-group sums
//   ffn_pass_kernel<1> down projection, 256 output rows of one expert per tile; writes y
//   combine_kernel     residual[t] += sum_k w[t][k] * y[t*K + k], k in rank order
//
// The pass kernels are persistent and warp-specialised: one producer warp streams, for
// every tile and every 256-input k-slice, the packed weight rows and the activation rows
// (TMA, 128-byte swizzle), the activations' group sums and the rows' scales and biases (TMA)
// into a shared-memory ring; eight consumer warps decode and multiply.
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
// One thread per 8-element chunk of a list entry p: xg[p] = pair-permuted fp16(x[token_list[p]])
// with the odd elements of every 8 divided by 16; sx[p][g] = sum of the values the stored
// halves stand for in group g (8 consecutive lanes hold a group), also as fp16 hi and lo
// planes s16[0|1][p][g].
__global__ void __launch_bounds__(256) gather_kernel(const uint16_t* __restrict__ x, int d, int B,
                                                     const int32_t* __restrict__ n_union,
                                                     const int32_t* __restrict__ offsets,
                                                     const int32_t* __restrict__ token_list,
                                                     uint32_t* __restrict__ status,
                                                     __half* __restrict__ xg, float* __restrict__ sx,
                                                     __half* __restrict__ s16, int BK) {
    const int cpr = d / 8;   // chunks per row, a multiple of 32: a warp never spans two rows
    const size_t gid = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int p = (int)(gid / cpr), ch = (int)(gid - (size_t)p * cpr);
    const int lane = threadIdx.x & 31;
    const int total = offsets[*n_union];
    if (p >= total) return;
    int t = token_list[p];
    if (t < 0 || t >= B) {   // a caller-supplied list that does not match B: flag, use row 0
        if (lane == 0) atomicOr(status, SMOE_FAULT_TOKEN_INDEX);
        t = 0;
    }
    const uint4 raw = __ldg(reinterpret_cast<const uint4*>(x + (size_t)t * d) + ch);
    const uint32_t wv[4] = {raw.x, raw.y, raw.z, raw.w};
    __half hv[8];
    float sa = 0.f;
#pragma unroll
    for (int m = 0; m < 8; ++m) {
        const float v = bf16_bits_to_float((m & 1) ? (wv[m >> 1] >> 16) : (wv[m >> 1] & 0xFFFFu));
        const __half h = __float2half_rn((m & 1) ? v * 0.0625f : v);
        hv[perm8(m)] = h;
        sa += (m & 1) ? __half2float(h) * 16.f : __half2float(h);
    }
    uint4 o;
    o.x = (uint32_t)__half_as_ushort(hv[0]) | ((uint32_t)__half_as_ushort(hv[1]) << 16);
    o.y = (uint32_t)__half_as_ushort(hv[2]) | ((uint32_t)__half_as_ushort(hv[3]) << 16);
    o.z = (uint32_t)__half_as_ushort(hv[4]) | ((uint32_t)__half_as_ushort(hv[5]) << 16);
    o.w = (uint32_t)__half_as_ushort(hv[6]) | ((uint32_t)__half_as_ushort(hv[7]) << 16);
    reinterpret_cast<uint4*>(xg + (size_t)p * d)[ch] = o;
#pragma unroll
    for (int off = 1; off < 8; off <<= 1) sa += __shfl_xor_sync(0xffffffffu, sa, off);
    if ((lane & 7) == 0) {
        const size_t i = (size_t)p * (d / kGroup) + ch / 8;
        sx[i] = sa;
        const __half hh = __float2half_rn(sa);   // hi and lo planes for the tensor-core path
        s16[i] = hh;
        s16[(size_t)BK * (d / kGroup) + i] = __float2half_rn(sa - __half2float(hh));
    }
}

// ----------------------------------------------------------------------------- expert passes
constexpr int kConsumerWarps = 8;
constexpr int kPassThreads = 32 * (kConsumerWarps + 1);   // + one producer warp
constexpr int kWBytes = 256 * 128;         // 256 weight rows x 32 u32 words (4 groups)
constexpr int kXBoxBytes = 16 * 128;       // 16 activation rows x 64 fp16 (one group)
constexpr int kTokChunk = 16;              // tokens per pass over the weights
constexpr int kSbBytes = 256 * 16;         // 256 rows x up to 8 bf16 (a table of scales or biases)

// One ring stage: packed weights | activation boxes (4, or 4 hi + 4 lo) | scales | biases |
// activation group sums fp32 [16 tokens][4 groups]; a 1024-byte multiple.  The scale and
// bias tables hold, per weight row, the 8 groups of the 16-byte-aligned window that
// contains the stage's 4 groups ([256][8] bf16), or with 4 groups per row ([256][4]) the
// whole row.
template <int PASS>
struct PassCfg {
    static constexpr int kStages = PASS ? 3 : 4;
    static constexpr int kXBoxes = PASS ? 8 : 4;
    static constexpr int kXOff = kWBytes;
    static constexpr int kSOff = kXOff + kXBoxes * kXBoxBytes;
    static constexpr int kBOff = kSOff + kSbBytes;
    static constexpr int kSumOff = kBOff + kSbBytes;
    static constexpr int kSumBytes = kTokChunk * 4 * 4;
    static constexpr int kStageBytes = (kSumOff + kSumBytes + 1023) / 1024 * 1024;
    static constexpr int kTx = kWBytes + kXBoxes * kXBoxBytes + kSumBytes;   // TMA bytes of a stage
                                                                              // (without the tables)
    static constexpr int kSmem = kStages * kStageBytes + 1024;
};
static_assert(PassCfg<0>::kSmem <= 227 * 1024 - 2048, "pass 0 shared memory");
static_assert(PassCfg<1>::kSmem <= 227 * 1024 - 2048, "pass 1 shared memory");

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
    float* y_out;                     // pass 1 output [B*K, d]
    uint32_t* status;
};

struct Tile {
    bool ok;              // indices valid
    bool mine;            // handled by this kernel (not by the tensor-core path)
    int e, p0, p1, row;   // row: first h column (pass 0) or output row (pass 1) of the tile
};

__device__ __forceinline__ Tile decode_tile(const PassArgs& a, int t, int pass_rows) {
    Tile T;
    const int u = t / a.tiles_per_expert;
    T.row = (t - u * a.tiles_per_expert) * pass_rows;
    T.e = a.union_ids[u];
    T.p0 = a.offsets[u];
    T.p1 = a.offsets[u + 1];
    T.ok = T.e >= 0 && T.e < a.E && T.p0 >= 0 && T.p1 >= T.p0 && T.p1 <= a.B * a.K;
    T.mine = a.tc_min <= 0 || T.p1 - T.p0 < a.tc_min;
    return T;
}

// One 256-input k-slice (4 groups) of a consumer warp: two 16-row m-tiles against NT
// 8-token n-tiles.  wb0/wb1: shared addresses of the m-tiles' first rows; xs: the activation
// boxes (4, or with LO 4 hi + 4 lo); sc/bi: the stage's bf16 scales / biases of rows g and
// g+8 of each m-tile ([m][row], 4 groups each); sums: the stage's activation group sums.
// Per group: acc += (scale * 2^24) * C + bias * S, C the exact mma result in units of 2^-24
// and S the tokens' group sums.
template <int NT, bool LO>
__device__ __forceinline__ void consume_stage(float (&acc)[2][NT][4], uint32_t wb0, uint32_t wb1, uint32_t xs,
                                              const uint2 (&sc)[2][2], const uint2 (&bi)[2][2], uint32_t sums,
                                              int g, int c) {
    constexpr int NB = LO ? 2 : 1;   // activation terms per input
    float4 S[NT][2];                 // group sums of tokens 2c and 2c+1 of each n-tile, 4 groups
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
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
            const int r = nt * 8 + g;
#pragma unroll
            for (int hl = 0; hl < NB; ++hl) {
                const uint32_t rb = xs + (hl * 4 + q) * kXBoxBytes + r * 128;
                const uint4 v0 = lds_u4(rb + (((2 * c) ^ g) << 4));
                const uint4 v1 = lds_u4(rb + (((2 * c + 1) ^ g) << 4));
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
template <int NT, int PASS>
__device__ __forceinline__ void consume_chunk(const PassArgs& a, const Ring& R, uint32_t& it, bool& poisoned,
                                              const Tile& T, int pc, int n, int warp, int lane, float* red) {
    using C = PassCfg<PASS>;
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
        lrow0 = warp * 16;          // gate rows 16w.. of the tile
        lrow1 = 128 + warp * 16;    // up rows
    } else {
        lrow0 = warp * 32;
        lrow1 = warp * 32 + 16;
    }
    wrow_off0 = (uint32_t)lrow0 * 128u;
    wrow_off1 = (uint32_t)lrow1 * 128u;
    const bool packed = a.kdim / kGroup == 4;   // tables [256][4]: the whole row
    const uint32_t rs = packed ? 8u : 16u;
    auto tab_off = [&](int st) { return packed ? 0u : (uint32_t)(st & 1) * 8u; };
    for (int st = 0; st < nst; ++st) {
        const uint32_t slot = it % C::kStages;
        const uint32_t parity = (it / C::kStages) & 1u;
        if (!poisoned && !mbar_wait(R.full + 8 * slot, parity)) {
            poisoned = true;
            if (lane == 0) atomicOr(a.status, SMOE_FAULT_TIMEOUT);
        }
        const uint32_t base = R.buf + slot * C::kStageBytes;
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
        consume_stage<NT, PASS == 1>(acc, base + wrow_off0, base + wrow_off1, base + C::kXOff, sc, bi,
                                     base + C::kSumOff, g, c);
        mbar_arrive(R.empty + 8 * slot);   // this thread is done reading the slot
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
        asm volatile("bar.sync 1, %0;\n" ::"r"(32 * kConsumerWarps) : "memory");
        const int tid = warp * 32 + lane;
        if (tid < 32) {
            const int half = tid >> 4, slot = tid & 15;   // 128 columns = two 64-column groups
            if (slot < n) {
                const float s = red[(4 * half) * 16 + slot] + red[(4 * half + 1) * 16 + slot] +
                                red[(4 * half + 2) * 16 + slot] + red[(4 * half + 3) * 16 + slot];
                a.hsum_out[(size_t)(pc + slot) * (a.F / kGroup) + T.row / kGroup + half] = s;
            }
        }
        asm volatile("bar.sync 1, %0;\n" ::"r"(32 * kConsumerWarps) : "memory");
    } else {
#pragma unroll
        for (int m = 0; m < 2; ++m)
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int slot = nt * 8 + 2 * c + (i & 1);
                    if (slot >= n) continue;
                    const int p = pc + slot;
                    const int t = a.token_list[p], k = a.slot_list[p];
                    if (t < 0 || t >= a.B || k < 0 || k >= a.K) continue;   // flagged by the gather
                    const int r = T.row + warp * 32 + m * 16 + g + ((i & 2) ? 8 : 0);
                    a.y_out[((size_t)t * a.K + k) * a.d + r] = acc[m][nt][i];
                }
    }
}

// PASS 0: tile = 128 h columns of one expert (consumer warp w: gate and up rows 16w..16w+15).
// PASS 1: tile = 256 down rows of one expert (consumer warp w: rows 32w..32w+31).
// Tiles t = blockIdx.x, blockIdx.x + gridDim.x, ... over n_union * tiles_per_expert.
// Producer warp (lane 0): the TMA copies of a stage (weights, activations, group sums, and
// the scale and bias tables: map_sc0 / map_bi0 rows of map_w0, map_sc1 / map_bi1 rows of
// map_w1).
template <int PASS>
__global__ void __launch_bounds__(kPassThreads, 1)
    ffn_pass_kernel(const __grid_constant__ CUtensorMap map_w0, const __grid_constant__ CUtensorMap map_w1,
                    const __grid_constant__ CUtensorMap map_x, const __grid_constant__ CUtensorMap map_s,
                    const __grid_constant__ CUtensorMap map_sc0, const __grid_constant__ CUtensorMap map_sc1,
                    const __grid_constant__ CUtensorMap map_bi0, const __grid_constant__ CUtensorMap map_bi1,
                    PassArgs a) {
    using C = PassCfg<PASS>;
    extern __shared__ uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t bars[2 * C::kStages];
    __shared__ float red[kConsumerWarps * 16];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int pass_rows = PASS == 0 ? 128 : 256;
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    Ring R;
    R.buf = smem_addr(smem);
    R.full = smem_addr(&bars[0]);
    R.empty = smem_addr(&bars[C::kStages]);
    if (threadIdx.x == 0) {
        for (int s = 0; s < C::kStages; ++s) {
            mbar_init(R.full + 8 * s, 1);   // TMA arrive + one cp.async arrive per producer lane
            mbar_init(R.empty + 8 * s, 32 * kConsumerWarps);
        }
        asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
    }
    __syncthreads();

    const int n_tiles = *a.n_union * a.tiles_per_expert;
    const int G = a.kdim / kGroup, nst = G / 4;
    uint32_t it = 0;
    bool poisoned = false;

    if (warp == kConsumerWarps) {
        // ---------------------------------------------------------------- producer (one thread)
        if (lane == 0) {
            const bool packed = G == 4;
            const uint32_t rs = packed ? 8u : 16u;
            const uint32_t tx = C::kTx + 2u * 256u * rs;
            for (int t = blockIdx.x; t < n_tiles; t += gridDim.x) {
                const Tile T = decode_tile(a, t, pass_rows);
                if (!T.ok || !T.mine) continue;
                // first rows of the tile in map_w0 and (pass 0) map_w1
                const int64_t r0 = (int64_t)T.e * a.wrow0 + T.row;
                const int64_t r1 = PASS == 0 ? (int64_t)T.e * a.wrow1 + a.woff1 + T.row : r0;
                // the tile's scale / bias rows into L2 ahead of the table copies
                const uint32_t bytes = (uint32_t)(pass_rows * G * 2);
                prefetch_l2(a.s0 + r0 * G, bytes); prefetch_l2(a.b0 + r0 * G, bytes);
                if (PASS == 0) { prefetch_l2(a.s1 + r1 * G, bytes); prefetch_l2(a.b1 + r1 * G, bytes); }
                const int ty0 = (int)(packed ? r0 / 2 : r0), ty1 = (int)(packed ? r1 / 2 : r1);
                for (int pc = T.p0; pc < T.p1; pc += kTokChunk) {
                    for (int st = 0; st < nst; ++st) {
                        const uint32_t slot = it % C::kStages;
                        if (it >= C::kStages && !poisoned &&
                            !mbar_wait(R.empty + 8 * slot, ((it / C::kStages) - 1) & 1u)) {
                            poisoned = true;
                            atomicOr(a.status, SMOE_FAULT_TIMEOUT);
                        }
                        const uint32_t base = R.buf + slot * C::kStageBytes;
                        const uint32_t full = R.full + 8 * slot;
                        if (!poisoned) {
                            mbar_expect_tx(full, tx);
                            const int tx0 = packed ? 0 : (st * 4) & ~7;   // 16-byte window of the stage's groups
                            if (PASS == 0) {
                                tma_load_2d(base, &map_w0, st * 32, (int)r0, full);
                                tma_load_2d(base + 128 * 128, &map_w1, st * 32, (int)r1, full);
                                tma_load_2d(base + C::kSOff, &map_sc0, tx0, ty0, full);
                                tma_load_2d(base + C::kSOff + 128 * rs, &map_sc1, tx0, ty1, full);
                                tma_load_2d(base + C::kBOff, &map_bi0, tx0, ty0, full);
                                tma_load_2d(base + C::kBOff + 128 * rs, &map_bi1, tx0, ty1, full);
                            } else {
                                tma_load_2d(base, &map_w0, st * 32, (int)r0, full);
                                tma_load_2d(base + C::kSOff, &map_sc0, tx0, ty0, full);
                                tma_load_2d(base + C::kBOff, &map_bi0, tx0, ty0, full);
                            }
#pragma unroll
                            for (int q = 0; q < 4; ++q)
                                tma_load_2d(base + C::kXOff + q * kXBoxBytes, &map_x, (st * 4 + q) * 64, pc, full);
                            if (PASS == 1) {   // lo terms of h: columns F.. of the same rows
#pragma unroll
                                for (int q = 0; q < 4; ++q)
                                    tma_load_2d(base + C::kXOff + (4 + q) * kXBoxBytes, &map_x,
                                                a.F + (st * 4 + q) * 64, pc, full);
                            }
                            tma_load_2d(base + C::kSumOff, &map_s, st * 4, pc, full);
                        }
                        ++it;
                    }
                }
            }
            // drain: every issued stage has landed before the CTA may exit
            if (poisoned) {
                const uint32_t first = it > C::kStages ? it - C::kStages : 0;
                for (uint32_t i = first; i < it; ++i) mbar_wait(R.full + 8 * (i % C::kStages), (i / C::kStages) & 1u);
            }
        }
        return;
    }

    // -------------------------------------------------------------------- consumers
    for (int t = blockIdx.x; t < n_tiles; t += gridDim.x) {
        const Tile T = decode_tile(a, t, pass_rows);
        if (!T.ok) {
            if (warp == 0 && lane == 0) atomicOr(a.status, SMOE_FAULT_EXPERT_INDEX);
            continue;
        }
        if (!T.mine) continue;
        for (int pc = T.p0; pc < T.p1; pc += kTokChunk) {
            const int n = min(kTokChunk, T.p1 - pc);
            if (n <= 8) consume_chunk<1, PASS>(a, R, it, poisoned, T, pc, n, warp, lane, red);
            else consume_chunk<2, PASS>(a, R, it, poisoned, T, pc, n, warp, lane, red);
        }
    }
}

// ----------------------------------------------------------------------------- combine
// Skipped entirely (residual untouched) when the union did not cover all B*K entries, i.e.
// after a flagged routing fault.
__global__ void __launch_bounds__(256) combine_kernel(const float* __restrict__ y, const float* __restrict__ w,
                                                      const int32_t* __restrict__ n_union,
                                                      const int32_t* __restrict__ offsets, int B, int K, int d,
                                                      float* __restrict__ residual) {
    const size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;   // float4 index
    const size_t n4 = (size_t)B * d / 4;
    if (i >= n4) return;
    if (offsets[*n_union] != B * K) return;
    const int t = (int)(i / (d / 4));
    const int c4 = (int)(i - (size_t)t * (d / 4));
    float4 acc = reinterpret_cast<float4*>(residual)[i];
    for (int k = 0; k < K; ++k) {
        const float wk = w[(size_t)t * K + k];
        const float4 v = reinterpret_cast<const float4*>(y + ((size_t)t * K + k) * d)[c4];
        acc.x = fmaf(wk, v.x, acc.x);
        acc.y = fmaf(wk, v.y, acc.y);
        acc.z = fmaf(wk, v.z, acc.z);
        acc.w = fmaf(wk, v.w, acc.w);
    }
    reinterpret_cast<float4*>(residual)[i] = acc;
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
                       float* residual, void* ws, const WsLayout& L, cudaStream_t stream) {
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
        cudaError_t e =
            cudaFuncSetAttribute(ffn_pass_kernel<0>, cudaFuncAttributeMaxDynamicSharedMemorySize, PassCfg<0>::kSmem);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(ffn_pass_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, PassCfg<1>::kSmem);
        if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sm_count[dev & 63], cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return e;
        attr_done.fetch_or(bit);
    }
    const int sms = sm_count[dev & 63] > 0 ? sm_count[dev & 63] : 1;

    // activation / group-sum maps over this call's workspace rows
    CUtensorMap map_xg, map_h, map_sx, map_sh;
    if (!encode_map_2d(&map_xg, xg, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, BK, d, 64, 16, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_map_2d(&map_h, h, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, BK, 2 * F, 64, 16,
                       CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_map_2d(&map_sx, sx, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, BK, d / kGroup, 4, kTokChunk,
                       CU_TENSOR_MAP_SWIZZLE_NONE) ||
        !encode_map_2d(&map_sh, sh, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, BK, F / kGroup, 4, kTokChunk,
                       CU_TENSOR_MAP_SWIZZLE_NONE))
        return cudaErrorInvalidValue;

    const size_t chunks = (size_t)BK * (d / 8);
    gather_kernel<<<(unsigned)((chunks + 255) / 256), 256, 0, stream>>>(x, d, B, n_union, offsets, token_list, status,
                                                                          xg, sx, ws_ptr<__half>(ws, L.s16x), BK);

    // experts with many tokens go to the tcgen05 path; with fewer than 256 tokens in the chunk
    // an expert rarely reaches the threshold, so the extra launches are skipped
    const int tc_min = (tc_path_supported(D) && B >= 256) ? kTcMinTokens : 0;
    FfnTcWeights TW{};
    TW.pm_gate = W.pm_gate; TW.pm_up = W.pm_up; TW.pm_down = W.pm_down;
    TW.sg = W.sg; TW.bg = W.bg; TW.g_rows = W.g_rows_per_expert;
    TW.su = W.su; TW.bu = W.bu; TW.u_rows = W.u_rows_per_expert; TW.u_off = W.u_row_offset;
    TW.sd = W.sd; TW.bd = W.bd;

    PassArgs a{};
    a.wrow0 = W.g_rows_per_expert; a.wrow1 = W.u_rows_per_expert; a.woff1 = W.u_row_offset;
    a.s0 = W.sg; a.b0 = W.bg; a.s1 = W.su; a.b1 = W.bu;
    a.kdim = d; a.F = F; a.d = d; a.K = K; a.E = E; a.B = B;
    a.tiles_per_expert = F / 128;
    a.tc_min = tc_min;
    a.union_ids = union_ids; a.n_union = n_union; a.offsets = offsets;
    a.token_list = token_list; a.slot_list = slot_list;
    a.h_out = h; a.hsum_out = sh; a.y_out = y; a.status = status;
    const int grid0 = std::min(sms, max_u * a.tiles_per_expert);
    ffn_pass_kernel<0><<<grid0, kPassThreads, PassCfg<0>::kSmem, stream>>>(W.map_gate, W.map_up, map_xg, map_sx,
                                                                            W.map_sg, W.map_su, W.map_bg, W.map_bu, a);
    if (tc_min > 0) {
        cudaError_t e = launch_ffn_tc(D, TW, B, 0, union_ids, n_union, offsets, token_list, slot_list, ws, L, tc_min,
                                      sms, stream);
        if (e != cudaSuccess) return e;
    }

    PassArgs b = a;
    b.wrow0 = d; b.wrow1 = d; b.woff1 = 0;
    b.s0 = W.sd; b.b0 = W.bd; b.s1 = W.sd; b.b1 = W.bd;
    b.kdim = F;
    b.tiles_per_expert = d / 256;
    const int grid1 = std::min(sms, max_u * b.tiles_per_expert);
    ffn_pass_kernel<1><<<grid1, kPassThreads, PassCfg<1>::kSmem, stream>>>(W.map_down, W.map_down, map_h, map_sh,
                                                                            W.map_sd, W.map_sd, W.map_bd, W.map_bd, b);
    if (tc_min > 0) {
        cudaError_t e = launch_ffn_tc(D, TW, B, 1, union_ids, n_union, offsets, token_list, slot_list, ws, L, tc_min,
                                      sms, stream);
        if (e != cudaSuccess) return e;
    }

    const size_t n4 = (size_t)B * d / 4;
    combine_kernel<<<(unsigned)((n4 + 255) / 256), 256, 0, stream>>>(y, topk_w, n_union, offsets, B, K, d,
                                                                      residual);
    return cudaGetLastError();
}

}  // namespace smoe
