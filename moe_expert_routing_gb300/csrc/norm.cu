// Chaining glue between stacked MoE layers: RMSNorm with unit weight, output bf16, optionally
// of the mean-centred row.  Page "Data Flow", "Serial Step Trace": an RMS norm produces the
// normed hidden state that the FFN block (router gate and experts) consumes.
#include "smoe_internal.cuh"

namespace smoe {
namespace {

// One CTA of 512 threads per row, float4 loads; the row mean (if centring) and the sum of
// squares are reduced across the CTA in fp32 (block_sum512).
__global__ void __launch_bounds__(512) rmsnorm_bf16_kernel(const float* __restrict__ h, float eps, int center, int d,
                                                           uint16_t* __restrict__ x_out) {
    __shared__ float red[16];
    const int t = blockIdx.x;
    const float4* row = reinterpret_cast<const float4*>(h + (size_t)t * d);
    float mean = 0.f;
    if (center) {
        float s = 0.f;
        for (int i = threadIdx.x; i < d / 4; i += blockDim.x) {
            const float4 v = row[i];
            s += (v.x + v.y) + (v.z + v.w);
        }
        mean = block_sum512(s, red) / (float)d;
    }
    float ss = 0.f;
    for (int i = threadIdx.x; i < d / 4; i += blockDim.x) {
        const float4 v = row[i];
        const float a = v.x - mean, b = v.y - mean, c = v.z - mean, e = v.w - mean;
        ss = fmaf(a, a, ss);
        ss = fmaf(b, b, ss);
        ss = fmaf(c, c, ss);
        ss = fmaf(e, e, ss);
    }
    const float tot = block_sum512(ss, red);
    const float inv = 1.0f / sqrtf(tot / (float)d + eps);
    uint2* out = reinterpret_cast<uint2*>(x_out + (size_t)t * d);
    for (int i = threadIdx.x; i < d / 4; i += blockDim.x) {
        const float4 v = row[i];
        const uint32_t a = __bfloat16_as_ushort(__float2bfloat16_rn((v.x - mean) * inv));
        const uint32_t b = __bfloat16_as_ushort(__float2bfloat16_rn((v.y - mean) * inv));
        const uint32_t c = __bfloat16_as_ushort(__float2bfloat16_rn((v.z - mean) * inv));
        const uint32_t e = __bfloat16_as_ushort(__float2bfloat16_rn((v.w - mean) * inv));
        out[i] = make_uint2(a | (b << 16), c | (e << 16));
    }
}

}  // namespace

cudaError_t launch_rmsnorm(const float* h, float eps, int center, int B, int d, uint16_t* x_out,
                           cudaStream_t stream) {
    rmsnorm_bf16_kernel<<<B, 512, 0, stream>>>(h, eps, center, d, x_out);
    return cudaGetLastError();
}

}  // namespace smoe
