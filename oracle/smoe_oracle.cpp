// Oracle for the per-layer MoE block: a plain, slow, CPU implementation in double precision.
//
// TEST INFRASTRUCTURE ONLY.  This file is the yardstick the CUDA library is checked
// against; it is called from the tests, from the package's smoke check and from the
// benchmark's CPU-baseline leg, never from the product path.  It shares no code, header,
// table or helper with the CUDA library.
//
// What it computes, per layer, follows the pages' statement of the problem:
//   * dequantisation of 4-bit affine, group-64 weights packed u32 [E, out, in/8] with
//     bf16 scales/biases [E, out, in/64]           (page "SSD Streaming Expert Layers",
//                                                     section "Quantized Layout")
//   * exact routing: gate matvec on the hidden state, softmax, top-k, norm_topk_prob
//     re-normalisation                             (page "Layer-Major Batched Prefill",
//                                                     "Choreography Per Chunk" step 5;
//                                                     page "Surface Scout", "The Model Config")
//   * the union of the chunk's experts with a per-expert token list
//                                                   (page "Layer-Major Batched Prefill",
//                                                     "The Inversion")
//   * the SwiGLU expert FFN down(silu(gate(x)) * up(x)) (page "SSD Streaming Expert Layers",
//                                                     "Math Contract")
//   * the routing-weighted sum of expert outputs added to the residual
//                                                   (page "Data Flow", "Serial Step Trace",
//                                                     FFN block)
//   * RMSNorm with unit weight between chained layers (page "Data Flow", "Serial Step Trace")
//
// Readings where the pages are silent (the plainest reading the rest of the pages supports):
//   nibble i of a row lives in word i/8 at bits 4*(i%8) (low nibble first);
//   w = scale * q + bias;  top-k ordered by probability descending, equal values by the
//   lower expert id; selection by logit (softmax is strictly increasing, so the order by
//   probability equals the order by logit); routing weights kept in double and reported as
//   fp32; expert outputs summed in rank order k = 0..K-1.
//
// Parity pins (what ties this file to something other than itself) live in
// tests/test_oracle_pins.py: hand-packed dequantisation fixtures, closed-form FFN and
// routing cases, brute-force union and top-k on tiny inputs, token-major == layer-major,
// fused layout == separate layout.
//
// Build: g++ -O2 -std=c++17 -ffp-contract=off -fPIC -shared -pthread (no fused multiply-add
// contraction, so every sum is the plain sequence of IEEE operations written here).

#include <cmath>
#include <cstdint>
#include <cstring>
#include <algorithm>
#include <atomic>
#include <set>
#include <thread>
#include <vector>

namespace {

float bf16_to_float(uint16_t v) {
    uint32_t bits = static_cast<uint32_t>(v) << 16;
    float f;
    std::memcpy(&f, &bits, 4);
    return f;
}

// round-to-nearest-even of a double to bf16 (via the exact double value, one rounding)
uint16_t double_to_bf16(double v) {
    if (std::isnan(v)) return 0x7FC0;
    // The nearest bf16 is found by exact comparison in double: bf16 values are exactly
    // representable in double.
    float f = static_cast<float>(v);  // candidate near v (may be off by double rounding)
    uint32_t bits;
    std::memcpy(&bits, &f, 4);
    uint32_t lo = bits & 0xFFFF0000u;           // truncate towards zero in magnitude
    uint32_t hi = lo + 0x00010000u;             // next bf16 away from zero
    float flo, fhi;
    std::memcpy(&flo, &lo, 4);
    std::memcpy(&fhi, &hi, 4);
    double dlo = flo, dhi = fhi;
    double elo = std::fabs(v - dlo), ehi = std::fabs(dhi - v);
    // pick nearest; ties to even (even = low mantissa bit of bf16 is zero)
    uint32_t pick;
    if (elo < ehi) pick = lo;
    else if (ehi < elo) pick = hi;
    else pick = ((lo >> 16) & 1u) ? hi : lo;
    return static_cast<uint16_t>(pick >> 16);
}

struct Desc {
    int32_t d_model, num_experts, top_k, ffn_dim, group_size, norm_topk_prob, layout;
};

struct Weights {
    // separate layout (layout == 0)
    const uint32_t* w_up; const uint16_t* s_up; const uint16_t* b_up;
    const uint32_t* w_gate; const uint16_t* s_gate; const uint16_t* b_gate;
    // fused layout (layout == 1): per expert 2F rows, gate rows 0..F-1, up rows F..2F-1
    const uint32_t* w_gate_up; const uint16_t* s_gate_up; const uint16_t* b_gate_up;
    // down projection, both layouts
    const uint32_t* w_down; const uint16_t* s_down; const uint16_t* b_down;
};

// Dequantise `rows` rows of `in` inputs: w[o][i] = s[o][i/g] * q[o][i] + b[o][i/g] in fp32.
// The product of an 8-bit-significand bf16 and a 4-bit integer is exact in fp32, so the
// only rounding is at the add.
void dequant_rows(const uint32_t* q, const uint16_t* s, const uint16_t* b, int64_t rows, int64_t in,
                  int32_t g, float* out) {
    const int64_t words = in / 8, groups = in / g;
    for (int64_t o = 0; o < rows; ++o) {
        for (int64_t i = 0; i < in; ++i) {
            uint32_t word = q[o * words + i / 8];
            uint32_t nib = (word >> (4 * (i % 8))) & 0xFu;
            float sc = bf16_to_float(s[o * groups + i / g]);
            float bi = bf16_to_float(b[o * groups + i / g]);
            float prod = sc * static_cast<float>(nib);
            out[o * in + i] = prod + bi;
        }
    }
}

// One expert, dequantised once: gate [F][d], up [F][d], down [d][F] in fp32.
struct DenseExpert {
    std::vector<float> gate, up, down;
};

void dequant_expert(const Desc& D, const Weights& W, int32_t e, DenseExpert& X) {
    const int64_t d = D.d_model, F = D.ffn_dim, g = D.group_size;
    X.gate.resize(F * d);
    X.up.resize(F * d);
    X.down.resize(d * F);
    if (D.layout == 0) {
        dequant_rows(W.w_gate + e * F * (d / 8), W.s_gate + e * F * (d / g), W.b_gate + e * F * (d / g), F, d, g,
                     X.gate.data());
        dequant_rows(W.w_up + e * F * (d / 8), W.s_up + e * F * (d / g), W.b_up + e * F * (d / g), F, d, g,
                     X.up.data());
    } else {
        const uint32_t* wq = W.w_gate_up + e * 2 * F * (d / 8);
        const uint16_t* ws = W.s_gate_up + e * 2 * F * (d / g);
        const uint16_t* wb = W.b_gate_up + e * 2 * F * (d / g);
        dequant_rows(wq, ws, wb, F, d, g, X.gate.data());                                        // rows 0..F-1
        dequant_rows(wq + F * (d / 8), ws + F * (d / g), wb + F * (d / g), F, d, g, X.up.data()); // rows F..2F-1
    }
    dequant_rows(W.w_down + e * d * (F / 8), W.s_down + e * d * (F / g), W.b_down + e * d * (F / g), d, F, g,
                 X.down.data());
}

// y = down( silu(gate x) * up x ), all sums in double, in index order.
void expert_apply(const Desc& D, const DenseExpert& X, const uint16_t* x_row, double* y) {
    const int64_t d = D.d_model, F = D.ffn_dim;
    std::vector<double> xv(d), h(F);
    for (int64_t i = 0; i < d; ++i) xv[i] = bf16_to_float(x_row[i]);
    for (int64_t j = 0; j < F; ++j) {
        double gs = 0.0, us = 0.0;
        const float* gr = &X.gate[j * d];
        const float* ur = &X.up[j * d];
        for (int64_t i = 0; i < d; ++i) {
            gs += static_cast<double>(gr[i]) * xv[i];
            us += static_cast<double>(ur[i]) * xv[i];
        }
        double silu = gs / (1.0 + std::exp(-gs));
        h[j] = silu * us;
    }
    for (int64_t r = 0; r < d; ++r) {
        double acc = 0.0;
        const float* dr = &X.down[r * F];
        for (int64_t j = 0; j < F; ++j) acc += static_cast<double>(dr[j]) * h[j];
        y[r] = acc;
    }
}

template <class Fn>
void parallel_for(int64_t n, int32_t threads, Fn fn) {
    if (threads <= 1 || n <= 1) {
        for (int64_t i = 0; i < n; ++i) fn(i);
        return;
    }
    std::atomic<int64_t> next(0);
    std::vector<std::thread> pool;
    int32_t nt = static_cast<int32_t>(std::min<int64_t>(threads, n));
    for (int32_t t = 0; t < nt; ++t)
        pool.emplace_back([&]() {
            for (int64_t i = next.fetch_add(1); i < n; i = next.fetch_add(1)) fn(i);
        });
    for (auto& th : pool) th.join();
}

bool desc_ok(const Desc& D) {
    return D.d_model > 0 && D.num_experts > 0 && D.top_k > 0 && D.top_k <= D.num_experts && D.ffn_dim > 0 &&
           D.group_size > 0 && D.d_model % D.group_size == 0 && D.ffn_dim % D.group_size == 0 &&
           D.group_size % 8 == 0 && (D.layout == 0 || D.layout == 1);
}

}  // namespace

extern "C" {

int oracle_hardware_threads() { return static_cast<int>(std::thread::hardware_concurrency()); }

// Dequantise rows x in of one projection (pointers already at the wanted expert/row).
int oracle_dequant(const uint32_t* q, const uint16_t* s, const uint16_t* b, int64_t rows, int64_t in, int32_t g,
                   float* out) {
    if (!q || !s || !b || !out || rows < 0 || in <= 0 || g <= 0 || in % g || g % 8) return 1;
    dequant_rows(q, s, b, rows, in, g, out);
    return 0;
}

// Router logits in double: l[t][e] = sum_i W[e][i] * x[t][i] (+ bias[e]).
int oracle_logits(const uint16_t* x, const float* W, const float* bias, int32_t B, int32_t d, int32_t E,
                  double* logits) {
    if (!x || !W || !logits || B < 0 || d <= 0 || E <= 0) return 1;
    for (int32_t t = 0; t < B; ++t)
        for (int32_t e = 0; e < E; ++e) {
            double acc = 0.0;
            for (int32_t i = 0; i < d; ++i)
                acc += static_cast<double>(W[static_cast<int64_t>(e) * d + i]) *
                       static_cast<double>(bf16_to_float(x[static_cast<int64_t>(t) * d + i]));
            if (bias) acc += static_cast<double>(bias[e]);
            logits[static_cast<int64_t>(t) * E + e] = acc;
        }
    return 0;
}

// Top-k routing from logits: softmax p over all E, the K largest p (ties -> lower id),
// weights p_k (norm_topk_prob = 0) or p_k / sum of the K selected p (norm_topk_prob = 1).
int oracle_topk(const double* logits, int32_t B, int32_t E, int32_t K, int32_t norm, int32_t* idx, double* w64,
                float* w32) {
    if (!logits || !idx || B < 0 || E <= 0 || K <= 0 || K > E) return 1;
    std::vector<int32_t> order(E);
    std::vector<double> p(E);
    for (int32_t t = 0; t < B; ++t) {
        const double* l = logits + static_cast<int64_t>(t) * E;
        double mx = l[0];
        for (int32_t e = 1; e < E; ++e) mx = std::max(mx, l[e]);
        double z = 0.0;
        for (int32_t e = 0; e < E; ++e) {
            p[e] = std::exp(l[e] - mx);
            z += p[e];
        }
        for (int32_t e = 0; e < E; ++e) p[e] /= z;
        for (int32_t e = 0; e < E; ++e) order[e] = e;
        std::stable_sort(order.begin(), order.end(), [&](int32_t a, int32_t b) { return l[a] > l[b]; });
        double sel = 0.0;
        for (int32_t k = 0; k < K; ++k) sel += p[order[k]];
        for (int32_t k = 0; k < K; ++k) {
            double wk = norm ? p[order[k]] / sel : p[order[k]];
            idx[static_cast<int64_t>(t) * K + k] = order[k];
            if (w64) w64[static_cast<int64_t>(t) * K + k] = wk;
            if (w32) w32[static_cast<int64_t>(t) * K + k] = static_cast<float>(wk);
        }
    }
    return 0;
}

// Expert union and per-expert token lists.
// union_ids[u]: the u-th smallest routed expert id, u < n_union; offsets[u]..offsets[u+1]
// delimit its entries in token_list/slot_list (ascending token; slot = rank k of that
// expert in the token's top-k).  Returns 2 if an index is outside [0, E).
int oracle_union(const int32_t* idx, int32_t B, int32_t K, int32_t E, int32_t* union_ids, int32_t* n_union,
                 int32_t* offsets, int32_t* token_list, int32_t* slot_list) {
    if (!idx || !union_ids || !n_union || !offsets || !token_list || !slot_list || B < 0 || K <= 0 || E <= 0)
        return 1;
    for (int64_t i = 0; i < static_cast<int64_t>(B) * K; ++i)
        if (idx[i] < 0 || idx[i] >= E) return 2;
    std::set<int32_t> uni(idx, idx + static_cast<int64_t>(B) * K);
    int32_t u = 0, pos = 0;
    offsets[0] = 0;
    for (int32_t e : uni) {
        union_ids[u] = e;
        for (int32_t t = 0; t < B; ++t)
            for (int32_t k = 0; k < K; ++k)
                if (idx[static_cast<int64_t>(t) * K + k] == e) {
                    token_list[pos] = t;
                    slot_list[pos] = k;
                    ++pos;
                }
        offsets[++u] = pos;
    }
    *n_union = u;
    return 0;
}

// Expert outputs for a list of tokens of one expert: y[n][d] in double.
int oracle_expert_ffn(const Desc* D, const Weights* W, int32_t expert, const uint16_t* x, const int32_t* tokens,
                      int32_t n, double* y) {
    if (!D || !W || !x || (n > 0 && (!tokens || !y)) || !desc_ok(*D) || expert < 0 || expert >= D->num_experts)
        return 1;
    DenseExpert X;
    dequant_expert(*D, *W, expert, X);
    for (int32_t j = 0; j < n; ++j)
        expert_apply(*D, X, x + static_cast<int64_t>(tokens[j]) * D->d_model, y + static_cast<int64_t>(j) * D->d_model);
    return 0;
}

// The whole MoE block for B tokens given their routing (idx, w64):
//   out[t] = residual[t] + sum_{k=0..K-1} w[t][k] * y_{idx[t][k]}(x[t])   (double, rank order)
// mode 0 = layer-major (union, each union expert dequantised once and applied to its token
// list), mode 1 = token-major (each token, each of its K experts).  y_slots [B][K][d]
// (optional) receives the unweighted expert outputs.  Rows listed in `rows` (count n_rows,
// NULL = all) are the only ones computed in token-major mode.
int oracle_moe_combine(const Desc* D, const Weights* W, const uint16_t* x, int32_t B, const int32_t* idx,
                       const double* w64, const float* residual, float* out, double* out64, int32_t mode,
                       int32_t threads, double* y_slots, const int32_t* rows, int32_t n_rows) {
    if (!D || !W || !x || !idx || !w64 || !residual || !desc_ok(*D) || B < 0) return 1;
    const int32_t K = D->top_k, E = D->num_experts;
    const int64_t d = D->d_model;
    for (int64_t i = 0; i < static_cast<int64_t>(B) * K; ++i)
        if (idx[i] < 0 || idx[i] >= E) return 2;
    std::vector<int32_t> row_list;
    if (rows) row_list.assign(rows, rows + n_rows);
    else for (int32_t t = 0; t < B; ++t) row_list.push_back(t);
    std::vector<double> ys(static_cast<size_t>(B) * K * d, 0.0);
    if (mode == 0) {
        std::vector<int32_t> uid(E), off(E + 1), tl(static_cast<size_t>(B) * K + 1), sl(static_cast<size_t>(B) * K + 1);
        int32_t nu = 0;
        if (oracle_union(idx, B, K, E, uid.data(), &nu, off.data(), tl.data(), sl.data())) return 2;
        std::vector<char> want(B, rows ? 0 : 1);
        for (int32_t t : row_list) want[t] = 1;
        parallel_for(nu, threads, [&](int64_t u) {
            DenseExpert X;
            dequant_expert(*D, *W, uid[u], X);
            for (int32_t p = off[u]; p < off[u + 1]; ++p) {
                if (!want[tl[p]]) continue;
                expert_apply(*D, X, x + tl[p] * d, &ys[(static_cast<size_t>(tl[p]) * K + sl[p]) * d]);
            }
        });
    } else {
        parallel_for(static_cast<int64_t>(row_list.size()), threads, [&](int64_t r) {
            int32_t t = row_list[r];
            for (int32_t k = 0; k < K; ++k) {
                DenseExpert X;
                dequant_expert(*D, *W, idx[static_cast<int64_t>(t) * K + k], X);
                expert_apply(*D, X, x + t * d, &ys[(static_cast<size_t>(t) * K + k) * d]);
            }
        });
    }
    for (int32_t t : row_list)
        for (int64_t r = 0; r < d; ++r) {
            double acc = residual[t * d + r];
            for (int32_t k = 0; k < K; ++k)
                acc += w64[static_cast<int64_t>(t) * K + k] * ys[(static_cast<size_t>(t) * K + k) * d + r];
            if (out) out[t * d + r] = static_cast<float>(acc);
            if (out64) out64[t * d + r] = acc;
        }
    if (y_slots)
        for (int32_t t : row_list)
            std::memcpy(y_slots + static_cast<size_t>(t) * K * d, &ys[static_cast<size_t>(t) * K * d],
                        sizeof(double) * K * d);
    return 0;
}

// x_out[t] = bf16( (h[t] - c) / sqrt(mean_i (h[t][i] - c)^2 + eps) ), unit norm weight,
// c = row mean when center != 0 else 0; double inside.
int oracle_rmsnorm_bf16(const float* h, int32_t B, int32_t d, double eps, int32_t center, uint16_t* x_out) {
    if (!h || !x_out || B < 0 || d <= 0) return 1;
    for (int32_t t = 0; t < B; ++t) {
        const float* row = h + static_cast<int64_t>(t) * d;
        double c = 0.0;
        if (center) {
            for (int32_t i = 0; i < d; ++i) c += row[i];
            c /= d;
        }
        double ss = 0.0;
        for (int32_t i = 0; i < d; ++i) {
            double v = row[i] - c;
            ss += v * v;
        }
        double inv = 1.0 / std::sqrt(ss / d + eps);
        for (int32_t i = 0; i < d; ++i)
            x_out[static_cast<int64_t>(t) * d + i] = double_to_bf16((row[i] - c) * inv);
    }
    return 0;
}

// bf16 rounding of doubles (exposed so tests can pin it against hand values).
int oracle_to_bf16(const double* v, int64_t n, uint16_t* out) {
    if (!v || !out || n < 0) return 1;
    for (int64_t i = 0; i < n; ++i) out[i] = double_to_bf16(v[i]);
    return 0;
}

}  // extern "C"
