// The RMS norm that closes a residual-norm call, as a launch of its own: one CTA per row of h.
//
// The residual-norm entry point follows a projection with the next layer's RMS norm ("plan.rs", `Fold` with `Norm`,
// `gemv_norm_epilogue`: out = h / sqrt(mean(h^2) + eps) * gamma).  The product's last CTA can run the norm itself
// (finish_norm, the one-launch fold), but that one CTA's pass over every row is then the call's tail at any m; so
// the product writes h and this kernel, chained by programmatic dependent launch, spreads the rows over CTAs.  The
// arithmetic is finish_norm's: fp32 sums of squares in a fixed order, rstd = 1 / sqrtf(ss / N + eps), (h * rstd) *
// gamma rounded to bf16, and the quantized form taken from those bf16 values by the rule of q8_quantize_act.
#include <cuda_bf16.h>
#include <stdint.h>

#include "q8_device.cuh"
#include "q8_launch.h"

namespace q8 {
namespace {

constexpr int kNormThreads = 256;
constexpr int kNormKept = 4;  // 16-byte chunks of h a thread keeps in registers between its two passes

// Four columns n = 4j .. 4j + 3 of row r: the bf16 output and, with the quantized form, the codes and the 32-column
// block's scale.  All 32 lanes of the warp call it together (the block amax is a shuffle over eight lanes).
__device__ __forceinline__ void norm_emit(const NormRows &a, int r, const float4 hv, int j, int chunks, float rs) {
    const bool live = j < chunks;  // eight consecutive lanes (one block) are live or not together: chunks % 8 == 0
    const int n = 4 * j;
    float g[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) g[e] = live && n + e < a.N ? a.gamma[n + e] : 0.0f;
    const __nv_bfloat16 b0 = __float2bfloat16_rn(n < a.N ? hv.x * rs * g[0] : 0.0f);
    const __nv_bfloat16 b1 = __float2bfloat16_rn(n + 1 < a.N ? hv.y * rs * g[1] : 0.0f);
    const __nv_bfloat16 b2 = __float2bfloat16_rn(n + 2 < a.N ? hv.z * rs * g[2] : 0.0f);
    const __nv_bfloat16 b3 = __float2bfloat16_rn(n + 3 < a.N ? hv.w * rs * g[3] : 0.0f);
    if (a.ybf && live) {
        const uint32_t lo = (uint32_t)__bfloat16_as_ushort(b0) | ((uint32_t)__bfloat16_as_ushort(b1) << 16);
        const uint32_t hi = (uint32_t)__bfloat16_as_ushort(b2) | ((uint32_t)__bfloat16_as_ushort(b3) << 16);
        *reinterpret_cast<uint2 *>(a.ybf + (size_t)r * a.Np + n) = make_uint2(lo, hi);
    }
    if (!a.yq) return;  // uniform across the launch
    const float v0 = __bfloat162float(b0), v1 = __bfloat162float(b1);
    const float v2 = __bfloat162float(b2), v3 = __bfloat162float(b3);
    uint32_t mx = max(max(__float_as_uint(v0) & 0x7FFFFFFFu, __float_as_uint(v1) & 0x7FFFFFFFu),
                      max(__float_as_uint(v2) & 0x7FFFFFFFu, __float_as_uint(v3) & 0x7FFFFFFFu));
#pragma unroll
    for (int o = 1; o < 8; o <<= 1) mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    const float d = act_scale(mx), inv = act_inv(d);
    const uint32_t codes = act_code(v0, d, inv, mx) | (act_code(v1, d, inv, mx) << 8) |
                           (act_code(v2, d, inv, mx) << 16) | (act_code(v3, d, inv, mx) << 24);
    if (live) {
        *reinterpret_cast<uint32_t *>(a.yq + (size_t)r * a.Np + n) = codes;
        if ((j & 7) == 0) a.yd[(size_t)r * (a.Np / kBlock) + j / 8] = d;
    }
}

// Thread t takes the 16-byte chunks t, t + 256, ... of its CTA's row: the first kNormKept of them stay in registers
// for the second pass, any further ones are read again.  The sum of squares goes lane order within a thread, a fixed
// shuffle tree within a warp and warp order across the CTA, so a row's rstd does not depend on the launch.
__global__ void __launch_bounds__(kNormThreads) norm_rows_kernel(NormRows a) {
    // h is written by the product launch this one follows: wait for all of it.  Then let the next launch in the stream
    // start its own prologue (its weight prefetch), since it too waits for this grid before reading what we write.
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int r = blockIdx.x;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int chunks = a.Np / 4;
    const float4 *hr = reinterpret_cast<const float4 *>(a.h + (size_t)r * a.Np);
    float4 kept[kNormKept];
#pragma unroll
    for (int i = 0; i < kNormKept; ++i) {
        const int j = threadIdx.x + i * kNormThreads;
        kept[i] = j < chunks ? __ldcg(hr + j) : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    }
    float ss = 0.0f;
#pragma unroll
    for (int i = 0; i < kNormKept; ++i) {
        ss = fmaf(kept[i].x, kept[i].x, ss);
        ss = fmaf(kept[i].y, kept[i].y, ss);
        ss = fmaf(kept[i].z, kept[i].z, ss);
        ss = fmaf(kept[i].w, kept[i].w, ss);
    }
    for (int j = threadIdx.x + kNormKept * kNormThreads; j < chunks; j += kNormThreads) {
        const float4 v = __ldcg(hr + j);
        ss = fmaf(v.x, v.x, ss);
        ss = fmaf(v.y, v.y, ss);
        ss = fmaf(v.z, v.z, ss);
        ss = fmaf(v.w, v.w, ss);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    __shared__ float wsum[kNormThreads / 32];
    if (lane == 0) wsum[warp] = ss;
    __syncthreads();
    float tot = 0.0f;
#pragma unroll
    for (int w = 0; w < kNormThreads / 32; ++w) tot += wsum[w];
    const float rs = 1.0f / sqrtf(tot / (float)a.N + a.eps);
    // Second pass, warp-uniform: a warp's iteration covers the 32 consecutive chunks j0 .. j0 + 31.
#pragma unroll
    for (int i = 0; i < kNormKept; ++i) {
        const int j0 = warp * 32 + i * kNormThreads;
        if (j0 < chunks) norm_emit(a, r, kept[i], j0 + lane, chunks, rs);
    }
    for (int j0 = warp * 32 + kNormKept * kNormThreads; j0 < chunks; j0 += kNormThreads) {
        const int j = j0 + lane;
        const float4 v = j < chunks ? __ldcg(hr + j) : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        norm_emit(a, r, v, j, chunks, rs);
    }
}

}  // namespace

cudaError_t launch_norm_rows(const NormRows &a, int m, cudaStream_t stream, bool pdl) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)m, 1, 1);
    cfg.blockDim = dim3(kNormThreads, 1, 1);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    if (pdl) {
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
    }
    return cudaLaunchKernelEx(&cfg, norm_rows_kernel, a);
}

}  // namespace q8
