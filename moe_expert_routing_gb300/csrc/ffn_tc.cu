// Expert FFN for experts with many tokens: tcgen05 (5th-generation tensor core) GEMM tiles.
//
// Same math as ffn.cu (page "SSD Streaming Expert Layers", "Math Contract" and "Quantized
// Layout"), for union experts whose token list is long enough (long prompts with hot
// experts) that the contraction is a real dense GEMM: per expert, D[rows, tokens] =
// W[rows, k] X[k, tokens], W dequantised from 4-bit affine groups of 64.
//
// Exact fp16 weights.  w = s q + b = s (q - 8) + (b + 8 s).  s is bf16 (8-bit significand)
// and q - 8 a 4-bit signed integer, so s (q - 8) has at most 11 significant bits and is
// exactly an fp16 number within fp16's normal range (scales from 2^-14 up; smaller ones round
// among the subnormals); the rest, eps = b + 8 s, depends only on (row, group).  Hence
//   sum_i w_i x_i = sum_i [s (q_i - 8)]_fp16 x_i  +  sum_g eps_g S_g,   S_g = sum_{i in g} x_i,
// the first term one long fp16 contraction with fp32 accumulation in tensor memory, the
// second a small [rows x groups] x [groups x tokens] product that runs as one extra k-stage
// (eps as fp16, S as an fp16 hi + lo pair).
//
// Tile per CTA: 128 weight rows (UMMA M = 128) x 192 tokens (UMMA N); k in stages of one
// 64-input group.  The dequantised weights (the A operand) go from registers straight into
// tensor memory and the MMAs read them there, so shared memory carries only the packed
// weights and the activations (the B operand): two shared-memory rings (see TcCfg).
// Tensor memory (512 columns): two accumulator buffers of 192 columns (one tile's epilogue
// overlaps the next tile's MMAs) and a ring of 4 A stages of 32 columns (128 rows x 64 fp16).
// Warp roles (one CTA per SM, persistent over the work items):
//   warp 0      producer of the packed weight rows (TMA)
//   warp 1      TMEM owner; lane 0 issues tcgen05.mma and tcgen05.commit
//   warps 2-9   dequantisers, one A row per thread and half of its group: packed nibbles ->
//               fp16 s (q - 8) -> tcgen05.st into the row's TMEM lane
//   warps 10-13 epilogue: tcgen05.ld of the accumulators -> SwiGLU (pass 0) or y (pass 1)
//   warp 14     producer of the activation rows (B operand, TMA)
// Every mbarrier wait is bounded.  Pass 0's epilogue stages
// h through shared memory for 16-byte stores and also writes the per-group sums of h that
// pass 1's eps stage needs.
//
// Activation layouts are those of ffn.cu (pair-permuted k within every 8 inputs, odd
// inputs stored divided by 16); the dequantisers write the weights in the same k order and
// multiply the odd ones by 16, which the fp16 format absorbs exactly.
#include "smoe_internal.cuh"

#include <cuda.h>
#include <math.h>

#include <algorithm>
#include <atomic>

namespace smoe {
namespace {

constexpr int TC_M = 128;                    // weight rows per tile (UMMA M, one TMEM lane each)
constexpr int TC_N = 192;                    // tokens per tile (UMMA N; 64 / 128 for an expert's last short tile)
constexpr int TC_BOX_ROWS = 64;              // token rows per activation box
constexpr int TC_P_BYTES = TC_M * 128;       // packed slot: 128 rows x 32 words (4 stages), SW128
constexpr int TC_BOX_BYTES = TC_BOX_ROWS * 128;   // one activation box: 64 token rows x 64 fp16, SW128 K-major
constexpr int TC_B_BYTES = (TC_N / TC_BOX_ROWS) * TC_BOX_BYTES;   // one B sub-tile: 192 token rows
constexpr int TC_H_STRIDE = 33;             // pass 0 epilogue staging: 64 h columns x 32 tokens fp32,
constexpr int TC_H_BYTES = 64 * TC_H_STRIDE * 4;   // column-major, padded (conflict-free both ways)
constexpr int TC_THREADS = 480;
constexpr uint32_t TC_TMEM_COLS = 512;       // 2 accumulator buffers of TC_N columns + the A ring
constexpr int TC_A_GROUPS = 4;               // A ring in tensor memory: 4 groups (32 columns each)
constexpr uint32_t TC_A_COL = 2 * TC_N;      // first TMEM column of the A ring
static_assert(TC_A_COL + 32 * TC_A_GROUPS <= TC_TMEM_COLS, "tensor memory columns");

// Per-pass stage shapes.  A stage is 8 MMAs (k = 16 each) over two B sub-tiles: gate/up takes
// two input groups per stage (x of group 2j and 2j + 1 against their own A columns), down one
// group (h hi and h lo against the same A columns); the last stage of a tile is the eps stage
// (S hi and S lo against eps).  Issuing 8 MMAs per pair of barrier waits and commits keeps
// the single issuing thread ahead of the tensor core.  Two shared-memory rings: B slots (kB,
// two sub-tiles each) and packed-weight slots (kP, each 4 groups of 128-byte rows).  Packed
// slots are freed by the dequantisers once they have consumed them, so the packed stream runs
// ahead of the MMAs; B slots are freed by the MMAs.  The A operand never passes through
// shared memory.
template <int PASS>
struct TcCfg {
    static constexpr int kGps = PASS ? 1 : 2;                 // groups per main stage
    static constexpr int kKa = TC_A_GROUPS / kGps;            // A stages in tensor memory
    static constexpr int kB = 3;
    static constexpr int kP = 3;
    static constexpr int kNb = 2;                             // B sub-tiles per stage (8 MMAs)
    static constexpr int kBSlot = kNb * TC_B_BYTES;
    static constexpr int kOffB = 0;
    static constexpr int kOffP = kOffB + kB * kBSlot;
    static constexpr int kOffStage = kOffP + kP * TC_P_BYTES;   // epilogue staging
    static constexpr int kSmem = kOffStage + (PASS ? 0 : TC_H_BYTES) + 1024;
    static constexpr int kCorr = 1;                           // eps stage
};
static_assert(TcCfg<0>::kSmem <= 227 * 1024 - 7168, "pass 0 shared memory");
static_assert(TcCfg<1>::kSmem <= 227 * 1024 - 7168, "pass 1 shared memory");
static_assert(TcCfg<0>::kNb == 2 && TcCfg<1>::kNb == 2, "a stage is 4 k steps x 2 sub-tiles = 8 MMAs (umma_stage8)");

// ----------------------------------------------------------------------------- PTX helpers
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
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
// Bounded wait (~0.5 s): true when the phase with this parity completed.
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
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;\n" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;\n" ::: "memory"); }

// Shared-memory matrix descriptor: K-major operand, 128-byte swizzle, 8-row groups 1024 B
// apart; start address advanced by 32 B per 16-element k step inside the swizzle atom.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t addr) {
    uint64_t d = (uint64_t)((addr & 0x3FFFFu) >> 4);
    d |= (uint64_t)1 << 16;            // leading byte offset (unused for swizzled K-major)
    d |= (uint64_t)(1024 >> 4) << 32;  // stride byte offset: next 8-row group
    d |= (uint64_t)1 << 46;            // descriptor version
    d |= (uint64_t)2 << 61;            // 128-byte swizzle
    return d;
}

// Instruction descriptor, kind::f16: fp16 A and B, fp32 D, both K-major, M = 128, N = n.
__host__ __device__ constexpr uint32_t idesc_f16(int n) {
    return (1u << 4) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(TC_M >> 4) << 24);
}

// The A operand comes from tensor memory: lane i holds row i, two fp16 k-elements per 32-bit
// column (lower k in the low half), 8 columns per 16-element k step.
// One pipeline stage: 8 MMAs with the A operand in tensor memory (a[m], b[m] for m = 0..7, the
// first one initialising D when accumulate is 0) and the commits of the stage's B and A slots,
// in one asm block.  Issued back to back like this, 8 MMAs of N = 192 cost the issuing thread
// less time than the tensor core takes to run them, so work queues up ahead of the tensor core;
// as separate statements, each with its own predicate, every MMA took the thread longer than
// the tensor core did.
__device__ __forceinline__ void umma_stage8(uint32_t d_tmem, const uint32_t (&a)[8], const uint64_t (&b)[8],
                                            uint32_t idesc, uint32_t accumulate, uint32_t bar_b, uint32_t bar_a) {
    asm volatile(
        "{\n .reg .pred p, q;\n setp.ne.b32 p, %18, 0;\n setp.eq.b32 q, %18, %18;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %9, %17, p;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], [%2], %10, %17, q;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], [%3], %11, %17, q;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], [%4], %12, %17, q;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], [%5], %13, %17, q;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], [%6], %14, %17, q;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], [%7], %15, %17, q;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], [%8], %16, %17, q;\n"
        " tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%19];\n"
        " tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%20];\n}\n" ::"r"(d_tmem),
        "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(a[4]), "r"(a[5]), "r"(a[6]), "r"(a[7]), "l"(b[0]), "l"(b[1]),
        "l"(b[2]), "l"(b[3]), "l"(b[4]), "l"(b[5]), "l"(b[6]), "l"(b[7]), "r"(idesc), "r"(accumulate), "r"(bar_b),
        "r"(bar_a)
        : "memory");
}
__device__ __forceinline__ void umma_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n" ::"r"(bar)
                 : "memory");
}

// 32 consecutive fp32 columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;\n" ::: "memory");
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// 32 consecutive 32-bit columns of this thread's TMEM lane from v (not waited for).
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&v)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
        "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};\n" ::"r"(taddr),
        "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]), "r"(v[9]),
        "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]), "r"(v[16]), "r"(v[17]), "r"(v[18]),
        "r"(v[19]), "r"(v[20]), "r"(v[21]), "r"(v[22]), "r"(v[23]), "r"(v[24]), "r"(v[25]), "r"(v[26]), "r"(v[27]),
        "r"(v[28]), "r"(v[29]), "r"(v[30]), "r"(v[31])
        : "memory");
}

// OR of v over the 128 epilogue threads (named barrier 2), so that they all take the same
// branch around the named barriers that follow.
__device__ __forceinline__ bool epilogue_any(bool v) {
    uint32_t r;
    asm volatile(
        "{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n bar.red.or.pred q, 2, 128, p;\n selp.u32 %0, 1, 0, q;\n}\n"
        : "=r"(r)
        : "r"((uint32_t)v)
        : "memory");
    return r != 0;
}

__device__ __forceinline__ uint32_t h2u(__half2 h) { return *reinterpret_cast<uint32_t*>(&h); }
__device__ __forceinline__ __half2 u2h(uint32_t u) { return *reinterpret_cast<__half2*>(&u); }

// storage slot of logical element m (0..7) inside an 8-element chunk: (0,4,1,5,2,6,3,7)
__device__ __forceinline__ int perm8(int m) { return 2 * (m & 3) + (m >> 2); }

// One packed word (8 nibbles of a row) -> 8 fp16 weights s (q - 8) in storage order, odd
// elements times 16 (exact): (n0, n4), 16 (n1, n5), (n2, n6), 16 (n3, n7).
__device__ __forceinline__ uint4 dequant_word(uint32_t w, __half2 s2) {
    const __half2 o1 = u2h(0x64086408u);   // 1032 = 1024 + 8
    const __half2 o2 = u2h(0x64806480u);   // 1152 = 1024 + 16 * 8
    const uint32_t w8 = w >> 8;
    uint4 r;
    r.x = h2u(__hmul2(__hsub2(u2h((w & 0x000F000Fu) | 0x64006400u), o1), s2));
    r.y = h2u(__hmul2(__hsub2(u2h((w & 0x00F000F0u) | 0x64006400u), o2), s2));
    r.z = h2u(__hmul2(__hsub2(u2h((w8 & 0x000F000Fu) | 0x64006400u), o1), s2));
    r.w = h2u(__hmul2(__hsub2(u2h((w8 & 0x00F000F0u) | 0x64006400u), o2), s2));
    return r;
}

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];\n" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
    return v;
}

struct TcArgs {
    int64_t wrow0, wrow1, woff1;      // rows per expert (map_w0 / map_w1), first up row inside an expert
    const uint16_t* s0; const uint16_t* b0;   // scales / biases of map_w0 rows
    const uint16_t* s1; const uint16_t* b1;   // scales / biases of map_w1 rows (pass 0 up)
    int kdim, F, d, K, E, B;
    int m_tiles;                      // 128-row tiles per expert (pass 0: 64 h columns, gate and up rows)
    int tc_min;                       // experts with at least this many entries take this path
    const int32_t* union_ids; const int32_t* n_union; const int32_t* offsets;
    const int32_t* token_list; const int32_t* slot_list;
    __half* h_out;                    // pass 0: [B*K, 2F] hi | lo
    __half* hsum_out;                 // pass 0: group sums of h, fp16 planes [2][B*K, F/64]
    float* y_out;                     // pass 1: [B*K, d], each slot weighted: w[t,k] y_k
    const int32_t* entl;              // output row t*K + k of list position p (-1: rejected)
    const float* wl;                  // routing weight of list position p
    uint32_t* status;
};

struct Item {
    int e, p0, n, mt, nt;             // expert, first list entry, entries, row tile, token tile
};

// Work items: for every union expert with n >= tc_min, m_tiles x ceil(n / TC_N) tiles.  The
// per-expert prefix (up to 256 experts) is built by warp 0 in shared memory, next to copies of
// the union ids and list offsets (pref[0..nu], uid = pref + kMaxExperts + 1, off = uid +
// kMaxExperts + 1), so the per-tile decoding in every role reads shared memory only.
__device__ int build_items(const TcArgs& a, int* pref) {
    __shared__ int total;
    int* uid = pref + kMaxExperts + 1;
    int* off = uid + kMaxExperts + 1;
    {
        const int nu = *a.n_union;
        for (int u = threadIdx.x; u <= nu; u += blockDim.x) {
            off[u] = a.offsets[u];
            if (u < nu) uid[u] = a.union_ids[u];
        }
    }
    if (threadIdx.x < 32) {
        const int nu = *a.n_union;
        int run = 0;
        for (int base = 0; base < nu; base += 32) {
            const int u = base + threadIdx.x;
            int cnt = 0;
            if (u < nu) {
                const int n = a.offsets[u + 1] - a.offsets[u];
                if (n >= a.tc_min) cnt = a.m_tiles * ((n + TC_N - 1) / TC_N);
            }
            int incl = cnt;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const int v = __shfl_up_sync(0xffffffffu, incl, off);
                if ((int)threadIdx.x >= off) incl += v;
            }
            if (u < nu) pref[u] = run + incl - cnt;
            run += __shfl_sync(0xffffffffu, incl, 31);
        }
        if (threadIdx.x == 0) {
            total = run;
            pref[nu] = run;
        }
    }
    __syncthreads();
    return total;
}

__device__ __forceinline__ Item decode_item(const TcArgs& a, const int* pref, int t) {
    const int nu = *a.n_union;
    int lo = 0, hi = nu;   // largest u with pref[u] <= t
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (pref[mid] <= t) lo = mid;
        else hi = mid;
    }
    // skip experts with no items (pref[u] == pref[u+1])
    while (lo + 1 < nu && pref[lo + 1] <= t) ++lo;
    const int* uid = pref + kMaxExperts + 1;
    const int* off = uid + kMaxExperts + 1;
    Item it;
    it.e = uid[lo];
    it.p0 = off[lo];
    it.n = off[lo + 1] - it.p0;
    const int r = t - pref[lo];
    it.nt = r / a.m_tiles;
    it.mt = r - it.nt * a.m_tiles;
    return it;
}

template <int PASS>
__global__ void __launch_bounds__(TC_THREADS, 1)
    ffn_tc_kernel(const __grid_constant__ CUtensorMap map_w0, const __grid_constant__ CUtensorMap map_w1,
                  const __grid_constant__ CUtensorMap map_b, const __grid_constant__ CUtensorMap map_shi,
                  const __grid_constant__ CUtensorMap map_slo, TcArgs a) {
    using C = TcCfg<PASS>;
    extern __shared__ uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t full_p[C::kP], empty_p[C::kP], full_b[C::kB], empty_b[C::kB];
    __shared__ __align__(8) uint64_t empty_a[C::kKa];
    __shared__ __align__(8) uint64_t acc_full[2], acc_empty[2];
    __shared__ __align__(8) uint64_t mma_drain;   // commit of every MMA the issuer launched
    __shared__ uint32_t tmem_base_sh;
    __shared__ int pref[3 * (kMaxExperts + 1)];   // item prefix, union ids, list offsets
    __shared__ __align__(16) int ent_sh[2][TC_N];   // pass 1: output row t*K + k of each column (-1: none)
    __shared__ __align__(16) float w_sh[2][TC_N];   // pass 1: routing weight of each column
    __shared__ float gsum_sh[4][32];   // pass 0 epilogue: partial group sums [column quarter][token]

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    const int G = a.kdim / kGroup;     // <= 64, a multiple of 8
    const int n_main = G / C::kGps;    // main stages
    const int n_st = n_main + C::kCorr;
    constexpr int kSps = 4 / C::kGps;  // main stages per packed slot

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::kP; ++s) {
            mbar_init(smem_u32(&full_p[s]), 1);
            mbar_init(smem_u32(&empty_p[s]), 8);     // every dequantiser warp has consumed the slot
        }
        for (int s = 0; s < C::kB; ++s) {
            // the stage's activation copies (one arrival with their byte count) and its
            // dequantised A (one arrival per warp of the stage's dequantiser set): the MMA
            // issuer waits on one barrier per stage
            mbar_init(smem_u32(&full_b[s]), 1 + 4);
            mbar_init(smem_u32(&empty_b[s]), 1);     // tcgen05.commit of the stage's MMAs
        }
        for (int s = 0; s < C::kKa; ++s) {
            mbar_init(smem_u32(&empty_a[s]), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(smem_u32(&acc_full[b]), 1);
            mbar_init(smem_u32(&acc_empty[b]), 4);   // one arrival per epilogue warp
        }
        mbar_init(smem_u32(&mma_drain), 1);
        asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;\n" ::"r"(
                         smem_u32(&tmem_base_sh)),
                     "r"(TC_TMEM_COLS)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_base_sh;
    const int n_items = build_items(a, pref);
    bool poisoned = false;
    auto fail = [&](bool ok) {
        if (!ok && !poisoned) {
            poisoned = true;
            atomicOr(a.status, SMOE_FAULT_TIMEOUT);
        }
    };

    if (warp == 0) {
        // ------------------------------------------------------------------ packed-weight producer
        if (lane == 0) {
            uint32_t ip = 0;
            for (int t = blockIdx.x; t < n_items && !poisoned; t += gridDim.x) {
                const Item I = decode_item(a, pref, t);
                for (int st = 0; st < G; st += 4, ++ip) {   // one slot per 4 groups
                    const uint32_t s = ip % C::kP;
                    if (ip >= (uint32_t)C::kP) fail(mbar_wait(smem_u32(&empty_p[s]), ((ip / C::kP) - 1) & 1u));
                    if (poisoned) break;
                    const uint32_t slot = sbase + C::kOffP + s * TC_P_BYTES;
                    const uint32_t bar = smem_u32(&full_p[s]);
                    mbar_expect_tx(bar, TC_P_BYTES);
                    if (PASS == 0) {
                        const int j0 = I.mt * 64;   // 64 h columns: gate rows, then up rows
                        tma_load_2d(slot, &map_w0, st * 8, (int)(I.e * a.wrow0 + j0), bar);
                        tma_load_2d(slot + 64 * 128, &map_w1, st * 8, (int)(I.e * a.wrow1 + a.woff1 + j0), bar);
                    } else {
                        tma_load_2d(slot, &map_w0, st * 8, (int)(I.e * a.wrow0 + I.mt * TC_M), bar);
                    }
                }
            }
            // the copies issued into the last kP slots land (bounded waits) before the CTA may
            // exit and release its shared memory, also when another role gave up early
            for (uint32_t i = ip > (uint32_t)C::kP ? ip - C::kP : 0u; i < ip; ++i)
                mbar_wait(smem_u32(&full_p[i % C::kP]), (i / C::kP) & 1u);
        }
    } else if (warp == 14) {
        // ------------------------------------------------------------------ activation producer
        if (lane == 0) {
            uint32_t ib = 0;
            for (int t = blockIdx.x; t < n_items && !poisoned; t += gridDim.x) {
                const Item I = decode_item(a, pref, t);
                const int tok0 = I.p0 + I.nt * TC_N;
                const int boxes = (min(TC_N, I.n - I.nt * TC_N) + TC_BOX_ROWS - 1) / TC_BOX_ROWS;   // boxes of this tile
                for (int st = 0; st < n_st; ++st, ++ib) {
                    const uint32_t s = ib % C::kB;
                    if (ib >= (uint32_t)C::kB) fail(mbar_wait(smem_u32(&empty_b[s]), ((ib / C::kB) - 1) & 1u));
                    if (poisoned) break;
                    const uint32_t bar = smem_u32(&full_b[s]);
                    mbar_expect_tx(bar, (uint32_t)(C::kNb * boxes * TC_BOX_BYTES));
#pragma unroll
                    for (int sub = 0; sub < C::kNb; ++sub) {
                        const uint32_t dst = sbase + C::kOffB + s * C::kBSlot + sub * TC_B_BYTES;
                        for (int bx = 0; bx < boxes; ++bx) {
                            const int y = tok0 + bx * TC_BOX_ROWS;
                            const uint32_t d = dst + bx * TC_BOX_BYTES;
                            if (st < n_main)   // x of groups 2st, 2st+1, or h hi (sub 0) and h lo (sub 1)
                                tma_load_2d(d, &map_b, PASS ? (sub ? a.F : 0) + st * 64 : (2 * st + sub) * 64, y, bar);
                            else   // eps stage: S hi, S lo
                                tma_load_2d(d, sub ? &map_slo : &map_shi, 0, y, bar);
                        }
                    }
                }
            }
            // as above: the issued activation copies land before the exit
            for (uint32_t i = ib > (uint32_t)C::kB ? ib - C::kB : 0u; i < ib; ++i)
                mbar_wait(smem_u32(&full_b[i % C::kB]), (i / C::kB) & 1u);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            uint32_t tile = 0, s = 0, sa = 0, ph_b = 0;
            const uint64_t bdesc0 = sw128_desc(sbase + C::kOffB);
            for (int t = blockIdx.x; t < n_items; t += gridDim.x, ++tile) {
                const Item I = decode_item(a, pref, t);
                const int ntok = min(TC_N, I.n - I.nt * TC_N);
                const uint32_t idesc = idesc_f16((ntok + TC_BOX_ROWS - 1) / TC_BOX_ROWS * TC_BOX_ROWS);
                const uint32_t buf = tile & 1u;
                if (tile >= 2 && !poisoned) fail(mbar_wait(smem_u32(&acc_empty[buf]), ((tile >> 1) - 1) & 1u));
                tc_fence_after();
                const uint32_t d_tmem = tmem + buf * TC_N;
                for (int st = 0; st < n_st; ++st) {
                    if (!poisoned) fail(mbar_wait(smem_u32(&full_b[s]), ph_b));   // activations and A
                    if (!poisoned) {
                        tc_fence_after();
                        const uint32_t a_tmem = tmem + TC_A_COL + sa * 32u * C::kGps;
                        const bool two = PASS == 0 && st < n_main;   // sub-tile b against A group b
                        const uint64_t bd0 = bdesc0 + (uint64_t)((s * (uint32_t)C::kBSlot) >> 4);
                        uint32_t av[8];
                        uint64_t bv[8];
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk) {
#pragma unroll
                            for (int b = 0; b < C::kNb; ++b) {
                                av[kk * 2 + b] = a_tmem + (two ? 32u * b : 0u) + kk * 8u;
                                bv[kk * 2 + b] = bd0 + (uint64_t)((b * TC_B_BYTES + kk * 32) >> 4);
                            }
                        }
                        // the MMAs, then the commits: B slot and dequantised slot free once they finish
                        umma_stage8(d_tmem, av, bv, idesc, st > 0 ? 1u : 0u, smem_u32(&empty_b[s]),
                                    smem_u32(&empty_a[sa]));
                    }
                    if (++s == (uint32_t)C::kB) { s = 0; ph_b ^= 1u; }
                    if (++sa == (uint32_t)C::kKa) sa = 0;
                }
                if (!poisoned) umma_commit(smem_u32(&acc_full[buf]));   // accumulators of this tile ready
            }
            // every MMA this thread issued has completed (and stopped reading tensor and shared
            // memory) before the CTA releases them, also when another role gave up early
            umma_commit(smem_u32(&mma_drain));
            mbar_wait(smem_u32(&mma_drain), 0u);
        }
    } else if (warp < 10) {
        // ------------------------------------------------------------------ dequantisers
        // Two sets of 4 warps take alternate A stages (set = stage parity), 128 threads per
        // stage, one A row each.  A warp reaches only its own quarter of the TMEM lanes
        // (warp % 4), so thread -> row r = 32 (warp % 4) + lane; it writes the row's 64 weights
        // of each group of the stage (32 TMEM columns per group).
        const int r = 32 * (warp & 3) + lane;
        const uint32_t set = (uint32_t)(warp - 2) >> 2;
        const uint32_t lane_base = (uint32_t)(32 * (warp & 3)) << 16;
        uint32_t it = 0, ip = 0;   // stages (A ring), packed slots (4 groups each)
        for (int ti = blockIdx.x; ti < n_items; ti += gridDim.x) {
            const Item I = decode_item(a, pref, ti);
            // source row of A row r
            int64_t src;
            const uint16_t *sp, *bp;
            uint32_t prow;   // packed row inside the packed slot
            if (PASS == 0) {
                const int i = r >> 1;   // h column offset inside the tile; odd A rows are up rows
                const bool up = r & 1;
                src = up ? (int64_t)I.e * a.wrow1 + a.woff1 + I.mt * 64 + i : (int64_t)I.e * a.wrow0 + I.mt * 64 + i;
                sp = up ? a.s1 : a.s0;
                bp = up ? a.b1 : a.b0;
                prow = (up ? 64 : 0) + i;
            } else {
                src = (int64_t)I.e * a.wrow0 + I.mt * TC_M + r;
                sp = a.s0;
                bp = a.b0;
                prow = r;
            }
            const uint4* srow = reinterpret_cast<const uint4*>(sp + src * G);   // 8 bf16 per uint4
            const uint4* brow = reinterpret_cast<const uint4*>(bp + src * G);
            uint4 scl = __ldg(srow), scl_next = G > 8 ? __ldg(srow + 1) : make_uint4(0, 0, 0, 0);
            for (int st = 0; st < n_st; ++st, ++it) {
                const uint32_t sa = it % C::kKa;
                const int g0 = st * C::kGps;              // first group of a main stage
                if (st < n_main && (g0 & 7) == 0 && g0 > 0) {   // scales of groups g0 .. g0 + 7
                    scl = scl_next;
                    if (g0 + 8 < G) scl_next = __ldg(srow + (g0 >> 3) + 1);
                }
                const uint32_t ipc = ip;                  // packed slot of this stage
                const uint32_t sp_ = ipc % C::kP;
                if (st < n_main && st % kSps == kSps - 1) ++ip;   // every thread tracks the packed slots
                if ((it & 1u) != set) continue;           // the other set's stage
                // main stage: per group g the row's 8 packed words (chunks 2q, 2q+1 of the 128-byte
                // row, q = g % 4, swizzled by row & 7), read before the A stage is waited for
                uint4 w[C::kGps][2];
#pragma unroll
                for (int gi = 0; gi < C::kGps; ++gi) w[gi][0] = w[gi][1] = make_uint4(0, 0, 0, 0);
                if (st < n_main) {
                    if (!poisoned) fail(mbar_wait(smem_u32(&full_p[sp_]), (ipc / C::kP) & 1u));
                    if (!poisoned) {
                        const uint32_t pk = sbase + C::kOffP + sp_ * TC_P_BYTES + prow * 128u;
#pragma unroll
                        for (int gi = 0; gi < C::kGps; ++gi) {
                            const uint32_t q2 = (uint32_t)((g0 + gi) & 3) * 2u;
                            w[gi][0] = lds128(pk + ((q2 ^ (prow & 7u)) << 4));
                            w[gi][1] = lds128(pk + (((q2 + 1u) ^ (prow & 7u)) << 4));
                        }
                    }
                }
                if (it >= (uint32_t)C::kKa && !poisoned)
                    fail(mbar_wait(smem_u32(&empty_a[sa]), ((it / C::kKa) - 1) & 1u));
                // tcgen05.st is warp-collective: the warp takes one decision
                const bool skip = __any_sync(0xffffffffu, poisoned);
                if (!skip) {
                    tc_fence_after();   // the MMAs that read this stage before (commit) -> the stores
                    const uint32_t acol = tmem + lane_base + TC_A_COL + sa * 32u * C::kGps;
                    if (st < n_main) {
#pragma unroll
                        for (int gi = 0; gi < C::kGps; ++gi) {   // group g0 + gi -> 32 columns
                            const int g = g0 + gi;
                            const uint32_t wsel = (uint32_t)(g & 7) >> 1;   // selects, not a local-memory index
                            const uint32_t sw = wsel == 0 ? scl.x : wsel == 1 ? scl.y : wsel == 2 ? scl.z : scl.w;
                            const float sf = __uint_as_float((g & 1) ? (sw & 0xFFFF0000u) : (sw << 16));
                            const __half2 s2 = __float2half2_rn(sf);   // exact: bf16 -> fp16
                            const uint32_t wv[8] = {w[gi][0].x, w[gi][0].y, w[gi][0].z, w[gi][0].w,
                                                    w[gi][1].x, w[gi][1].y, w[gi][1].z, w[gi][1].w};
                            uint32_t v[32];
#pragma unroll
                            for (int c = 0; c < 8; ++c) {   // word c -> 8 inputs = 4 columns
                                const uint4 q = dequant_word(wv[c], s2);
                                v[4 * c] = q.x; v[4 * c + 1] = q.y; v[4 * c + 2] = q.z; v[4 * c + 3] = q.w;
                            }
                            tmem_st32(acol + 32u * gi, v);
                        }
                    } else {
                        // eps = b + 8 s for the row's G groups (zero beyond G), natural group order:
                        // chunk c = groups 8c .. 8c + 7
                        uint32_t v[32];
#pragma unroll
                        for (int c = 0; c < 8; ++c) {
                            uint32_t hv[4] = {0u, 0u, 0u, 0u};
                            if (c < G / 8) {
                                const uint4 es = __ldg(srow + c), eb = __ldg(brow + c);
                                const uint32_t sw[4] = {es.x, es.y, es.z, es.w};
                                const uint32_t bw[4] = {eb.x, eb.y, eb.z, eb.w};
#pragma unroll
                                for (int q = 0; q < 4; ++q) {
                                    const float e0 = fmaf(8.f, __uint_as_float(sw[q] << 16), __uint_as_float(bw[q] << 16));
                                    const float e1 = fmaf(8.f, __uint_as_float(sw[q] & 0xFFFF0000u),
                                                          __uint_as_float(bw[q] & 0xFFFF0000u));
                                    hv[q] = h2u(__floats2half2_rn(e0, e1));
                                }
                            }
                            v[4 * c] = hv[0]; v[4 * c + 1] = hv[1]; v[4 * c + 2] = hv[2]; v[4 * c + 3] = hv[3];
                        }
                        tmem_st32(acol, v);
                    }
                    asm volatile("tcgen05.wait::st.sync.aligned;\n" ::: "memory");
                    tc_fence_before();   // the stores -> the MMA issuer, through the arrival below
                }
                // one arrival per warp, after all lanes' stores completed
                __syncwarp();
                if (st < n_main && st % kSps >= kSps - 2 && lane == 0)   // this set's last stage of the slot
                    mbar_arrive(smem_u32(&empty_p[sp_]));
                if (lane == 0) {
                    // A of stage it is in place.  Stage it's barrier slot last served stage
                    // it - kB; with an A ring at least as deep as the activation ring (the down
                    // pass: 4 A stages, 3 activation slots) this set can run far enough ahead of
                    // the MMA issuer to arrive while that phase is still open, so it first waits
                    // (bounded) for it; with fewer A stages (gate/up: 2), reaching stage it at all
                    // means the issuer has passed stage it - 2, so that phase is complete.
                    if (C::kKa >= C::kB && it >= (uint32_t)C::kB && !poisoned)
                        fail(mbar_wait(smem_u32(&full_b[it % C::kB]), ((it / C::kB) - 1) & 1u));
                    mbar_arrive(smem_u32(&full_b[it % C::kB]));
                }
            }
        }
    } else {
        // ------------------------------------------------------------------ epilogue
        const int q = warp & 3;                  // TMEM lane quarter of this warp
        const int et = threadIdx.x - 320;        // 0..127
        const int lr = q * 32 + lane;            // accumulator row (TMEM lane) of this thread
        float* hsm = reinterpret_cast<float*>(smem + C::kOffStage);   // pass 0: [64 cols][33]
        uint32_t tile = 0;
        for (int t = blockIdx.x; t < n_items; t += gridDim.x, ++tile) {
            const Item I = decode_item(a, pref, t);
            const uint32_t buf = tile & 1u;
            const int tok0 = I.p0 + I.nt * TC_N;
            const int ntok = min(TC_N, I.n - I.nt * TC_N);
            // output row and routing weight of the tile's entries (pass 1)
            if (PASS == 1) {
                for (int j = et; j < TC_N; j += 128) {
                    ent_sh[buf][j] = j < ntok ? a.entl[tok0 + j] : -1;
                    w_sh[buf][j] = j < ntok ? a.wl[tok0 + j] : 0.f;
                }
                asm volatile("bar.sync 2, 128;\n" ::: "memory");
            }
            if (!poisoned) fail(mbar_wait(smem_u32(&acc_full[buf]), (tile >> 1) & 1u));
            poisoned = epilogue_any(poisoned);
            tc_fence_after();
            if (!poisoned) {
#pragma unroll 1
                for (int c0 = 0; c0 < TC_N; c0 += 32) {
                    if (c0 >= ntok) break;
                    float v[32];
                    tmem_ld32(tmem + ((uint32_t)(q * 32) << 16) + buf * TC_N + c0, v);
                    if (PASS == 0) {
                        // lanes 2i (gate) and 2i+1 (up) of h column i; the even lane takes tokens
                        // 0..15 of the chunk, the odd lane tokens 16..31
                        const bool odd_lane = lane & 1;
                        const int hc = lr >> 1;   // 0..63
#pragma unroll
                        for (int k = 0; k < 16; ++k) {
                            const float mine = v[odd_lane ? k : 16 + k];   // value the partner needs
                            const float other = __shfl_xor_sync(0xffffffffu, mine, 1);
                            const float g = odd_lane ? other : v[k];
                            const float u = odd_lane ? v[16 + k] : other;
                            const int tk = (odd_lane ? 16 : 0) + k;
                            const float hv = g / (1.f + expf(-g)) * u;
                            if (c0 + tk < ntok && !(fabsf(hv) <= 65504.f)) atomicOr(a.status, SMOE_FAULT_FP16_RANGE);
                            hsm[hc * TC_H_STRIDE + tk] = hv;
                        }
                        asm volatile("bar.sync 2, 128;\n" ::: "memory");
                        // 32 tokens x 64 columns: thread -> (token et & 31, columns 16 (et >> 5) .. + 16)
                        const int tk = et & 31, cq = et >> 5;
                        const bool valid = c0 + tk < ntok;
                        float gs = 0.f;
#pragma unroll
                        for (int half = 0; half < 2; ++half) {
                            const int cb = cq * 16 + half * 8;   // first column of this 8-chunk
                            __half hh[8], hl[8];
#pragma unroll
                            for (int e = 0; e < 8; ++e) {
                                const float hv = hsm[(cb + e) * TC_H_STRIDE + tk];
                                const float hs = (e & 1) ? hv * 0.0625f : hv;   // odd columns / 16
                                const __half h1 = __float2half_rn(hs);
                                const __half h2 = __float2half_rn(hs - __half2float(h1));
                                hh[perm8(e)] = h1;
                                hl[perm8(e)] = h2;
                                const float stood = __half2float(h1) + __half2float(h2);
                                gs += (e & 1) ? stood * 16.f : stood;
                            }
                            if (valid) {
                                const int j = I.mt * 64 + cb;   // first h column of the chunk
                                __half* rowp = a.h_out + (size_t)(tok0 + c0 + tk) * (2 * a.F) + j;
                                *reinterpret_cast<uint4*>(rowp) = *reinterpret_cast<const uint4*>(hh);
                                *reinterpret_cast<uint4*>(rowp + a.F) = *reinterpret_cast<const uint4*>(hl);
                            }
                        }
                        gsum_sh[cq][tk] = gs;   // the group's 4 column quarters, summed by warp 0
                        asm volatile("bar.sync 2, 128;\n" ::: "memory");
                        if (cq == 0 && valid) {
                            const float g4 = gsum_sh[0][tk] + gsum_sh[1][tk] + gsum_sh[2][tk] + gsum_sh[3][tk];
                            const int Gh = a.F / kGroup;
                            const size_t i = (size_t)(tok0 + c0 + tk) * Gh + I.mt;   // 64 columns = group mt
                            const __half sh = __float2half_rn(g4);
                            a.hsum_out[i] = sh;
                            a.hsum_out[(size_t)a.B * a.K * Gh + i] = __float2half_rn(g4 - __half2float(sh));
                        }
                    } else {
                        // output row r of the 32 columns' entries (-1 past the tile's tokens), their
                        // rows and weights read 4 columns at a time
                        float* yr = a.y_out + (I.mt * TC_M + lr);
                        const int4* ep = reinterpret_cast<const int4*>(&ent_sh[buf][c0]);
                        const float4* wp = reinterpret_cast<const float4*>(&w_sh[buf][c0]);
#pragma unroll
                        for (int k4 = 0; k4 < 8; ++k4) {
                            const int4 e4 = ep[k4];
                            const float4 w4 = wp[k4];
                            if (e4.x >= 0) yr[(size_t)e4.x * a.d] = v[4 * k4] * w4.x;
                            if (e4.y >= 0) yr[(size_t)e4.y * a.d] = v[4 * k4 + 1] * w4.y;
                            if (e4.z >= 0) yr[(size_t)e4.z * a.d] = v[4 * k4 + 2] * w4.z;
                            if (e4.w >= 0) yr[(size_t)e4.w * a.d] = v[4 * k4 + 3] * w4.w;
                        }
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&acc_empty[buf]));
        }
    }

    // all roles done; the accumulators are no longer read: release the tensor memory
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;\n" ::"r"(tmem), "r"(TC_TMEM_COLS)
                     : "memory");
}

bool encode_map(CUtensorMap* map, const void* base, CUtensorMapDataType dt, int esize, int64_t rows, int64_t cols,
                int box_cols, int box_rows, CUtensorMapSwizzle swz) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
    if (!enc) return false;
    cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)(cols * esize)};
    cuuint32_t box[2] = {(cuuint32_t)box_cols, (cuuint32_t)box_rows};
    cuuint32_t estr[2] = {1, 1};
    return enc(map, dt, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

bool tc_path_supported(const smoe_layer_desc& D) {
    // one eps stage covers up to 64 groups: d_model, ffn_dim <= 4096
    return D.d_model % 512 == 0 && D.ffn_dim % 512 == 0 && D.d_model <= 4096 && D.ffn_dim <= 4096;
}

cudaError_t launch_ffn_tc(const smoe_layer_desc& D, const FfnTcWeights& W, int B, int pass,
                          const int32_t* union_ids, const int32_t* n_union, const int32_t* offsets,
                          const int32_t* token_list, const int32_t* slot_list, void* ws, const WsLayout& L,
                          int tc_min, int sms, cudaStream_t stream) {
    const int d = D.d_model, F = D.ffn_dim, K = D.top_k, E = D.num_experts;
    const int BK = B * K;
    static std::atomic<uint64_t> attr_done{0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return cudaErrorInvalidDevice;
    const uint64_t bit = 1ull << (dev & 63);
    if (!(attr_done.load() & bit)) {
        cudaError_t e =
            cudaFuncSetAttribute(ffn_tc_kernel<0>, cudaFuncAttributeMaxDynamicSharedMemorySize, TcCfg<0>::kSmem);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(ffn_tc_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, TcCfg<1>::kSmem);
        if (e != cudaSuccess) return e;
        attr_done.fetch_or(bit);
    }
    __half* xg = ws_ptr<__half>(ws, L.xg);
    __half* h = ws_ptr<__half>(ws, L.h);
    __half* sxh = ws_ptr<__half>(ws, L.s16x);
    __half* shh = ws_ptr<__half>(ws, L.s16h);
    const int Gx = d / kGroup, Gh = F / kGroup;

    TcArgs a{};
    a.kdim = pass == 0 ? d : F;
    a.F = F; a.d = d; a.K = K; a.E = E; a.B = B;
    a.tc_min = tc_min;
    a.union_ids = union_ids; a.n_union = n_union; a.offsets = offsets;
    a.token_list = token_list; a.slot_list = slot_list;
    a.entl = ws_ptr<int32_t>(ws, L.entl); a.wl = ws_ptr<float>(ws, L.wl);
    a.h_out = h; a.hsum_out = shh; a.y_out = ws_ptr<float>(ws, L.y);
    a.status = ws_ptr<uint32_t>(ws, L.status);
    CUtensorMap mb, mshi, mslo;
    if (pass == 0) {
        a.wrow0 = W.g_rows; a.wrow1 = W.u_rows; a.woff1 = W.u_off;
        a.s0 = W.sg; a.b0 = W.bg; a.s1 = W.su; a.b1 = W.bu;
        a.m_tiles = F / 64;
        if (!encode_map(&mb, xg, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, BK, d, 64, TC_BOX_ROWS, CU_TENSOR_MAP_SWIZZLE_128B) ||
            !encode_map(&mshi, sxh, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, BK, Gx, 64, TC_BOX_ROWS, CU_TENSOR_MAP_SWIZZLE_128B) ||
            !encode_map(&mslo, sxh + (size_t)BK * Gx, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, BK, Gx, 64, TC_BOX_ROWS,
                        CU_TENSOR_MAP_SWIZZLE_128B))
            return cudaErrorInvalidValue;
        const int grid = std::max(1, std::min(sms, E * a.m_tiles * ((BK + TC_N - 1) / TC_N)));
        ffn_tc_kernel<0><<<grid, TC_THREADS, TcCfg<0>::kSmem, stream>>>(W.map_gate, W.map_up, mb, mshi, mslo, a);
    } else {
        const size_t nw = (size_t)BK * Gh;
        a.wrow0 = d; a.wrow1 = d; a.woff1 = 0;
        a.s0 = W.sd; a.b0 = W.bd; a.s1 = W.sd; a.b1 = W.bd;
        a.m_tiles = d / TC_M;
        if (!encode_map(&mb, h, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, BK, 2 * F, 64, TC_BOX_ROWS, CU_TENSOR_MAP_SWIZZLE_128B) ||
            !encode_map(&mshi, shh, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, BK, Gh, 64, TC_BOX_ROWS, CU_TENSOR_MAP_SWIZZLE_128B) ||
            !encode_map(&mslo, shh + nw, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, BK, Gh, 64, TC_BOX_ROWS,
                        CU_TENSOR_MAP_SWIZZLE_128B))
            return cudaErrorInvalidValue;
        const int grid = std::max(1, std::min(sms, E * a.m_tiles * ((BK + TC_N - 1) / TC_N)));
        ffn_tc_kernel<1><<<grid, TC_THREADS, TcCfg<1>::kSmem, stream>>>(W.map_down, W.map_down, mb, mshi, mslo, a);
    }
    return cudaGetLastError();
}

}  // namespace smoe
