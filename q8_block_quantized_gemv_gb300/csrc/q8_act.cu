// The quantized form of an activation: int8 codes and one fp32 scale per 32 values of a row ("plan.rs", `QBLOCK`
// and `Buffer::quantized`), by the rule stated with q8_quantize_act in q8_gemv.h (the weight rule of "from_q8.rs"
// `quantize` taken in fp32).
#include <stdint.h>

#include "../../include/q8_gemv.h"
#include "q8_launch.h"

namespace q8 {
void set_last_cuda_error(int e);  // q8_host.cpp
}

namespace {

// One thread per 8 values (16 bytes of bf16).  The four threads of a 32-value block are one quad of a warp (K is a
// multiple of 32, so blocks never straddle rows), and the block's amax is a two-step shuffle reduction over the
// magnitudes' bit patterns (ordered as the values are; inf and NaN above every finite value).
__global__ void quantize_act_kernel(const uint4 *__restrict__ x, uint2 *__restrict__ xq, float *__restrict__ xd,
                                    long long chunks) {
    const long long id = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    const bool live = id < chunks;  // a quad is live or dead as a whole (chunks % 4 == 0)
    const uint4 v = live ? x[id] : make_uint4(0u, 0u, 0u, 0u);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    float f[8];
    uint32_t mx = 0u;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const uint32_t lo = w[k] << 16, hi = w[k] & 0xFFFF0000u;
        f[2 * k] = __uint_as_float(lo);
        f[2 * k + 1] = __uint_as_float(hi);
        mx = max(mx, max(lo & 0x7FFFFFFFu, hi & 0x7FFFFFFFu));
    }
    mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
    mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
    if (!live) return;
    const float d = q8::act_scale(mx), inv = q8::act_inv(d);
    uint32_t codes[2] = {0u, 0u};
#pragma unroll
    for (int j = 0; j < 8; ++j) codes[j / 4] |= q8::act_code(f[j], d, inv, mx) << (8 * (j % 4));
    xq[id] = make_uint2(codes[0], codes[1]);
    if ((id & 3) == 0) xd[id >> 2] = d;
}

}  // namespace

extern "C" int64_t q8_act_bytes(int m, int K) {
    if (m < 1 || K <= 0 || K % Q8_BLOCK != 0) return -1;
    return (int64_t)m * K + (int64_t)m * (K / Q8_BLOCK) * 4;
}

extern "C" q8_status q8_quantize_act(const void *x, void *xa, int m, int K, q8_stream_t stream) {
    if (!x || !xa) return Q8_ERR_ARG;
    const int64_t bytes = q8_act_bytes(m, K);
    if (bytes < 0) return Q8_ERR_SHAPE;
    if (((uintptr_t)x & 15) || ((uintptr_t)xa & 15)) return Q8_ERR_ALIGN;
    const uintptr_t x0 = (uintptr_t)x, a0 = (uintptr_t)xa;
    const uintptr_t xn = (uintptr_t)((long long)m * K * 2);
    if (x0 < a0 + (uintptr_t)bytes && a0 < x0 + xn) return Q8_ERR_ARG;
    const long long chunks = (long long)m * K / 8;
    const int threads = 256;
    const long long blocks = (chunks + threads - 1) / threads;
    if (blocks > 0x7FFFFFFFLL) return Q8_ERR_SHAPE;
    unsigned char *base = static_cast<unsigned char *>(xa);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)blocks, 1, 1);
    cfg.blockDim = dim3(threads, 1, 1);
    cfg.stream = (cudaStream_t)stream;
    cudaError_t e = cudaLaunchKernelEx(&cfg, quantize_act_kernel, static_cast<const uint4 *>(x),
                                       reinterpret_cast<uint2 *>(base),
                                       reinterpret_cast<float *>(base + (long long)m * K), chunks);
    if (e != cudaSuccess) {
        q8::set_last_cuda_error((int)e);
        return Q8_ERR_CUDA;
    }
    return Q8_OK;
}
