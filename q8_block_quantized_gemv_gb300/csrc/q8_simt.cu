// CUDA-core Q8_0 GEMV: every thread holds V adjacent output columns for all M rows in fp32 registers.
//
// A warp reads one weight row at a time, 32 * V contiguous bytes (16-byte, 8-byte or 4-byte vector loads per lane,
// bypassing L1), converts each int8 to fp32 exactly, and accumulates x[r, k] * q[k, n] for every row r.  After each
// 32-row block the lane sums are multiplied by the block's scale and added into the carry ("from_q8.rs", module doc:
// per block, int8 rows are contracted lane by lane, then each column's sum is scaled into the carry).  For M >= 8 the
// per-block partials would not fit in registers, so the scale is applied to each value first (x * (q * s), the
// order of the `q8_fold` stage body); both orders give the same real number and stay within the error bound.
#include "q8_launch.h"

namespace q8 {

template <int M, int V, bool ARGMAX>
__global__ void __launch_bounds__(kThreads, 2) simt_kernel(const Args a) {
    using VT = typename Vec<V>::T;
    constexpr int NW = V / 4;  // 32-bit words of a lane's row segment
    constexpr int TC = simt_tile(V);
    constexpr bool kScaleFirst = M >= 8;
    extern __shared__ __align__(16) float smem[];

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int cl = lane * V;                       // first column of this lane within the tile
    const int col = blockIdx.x * TC + cl;          // ... within the weight
    int b0, b1;
    warp_blocks(a, warp, b0, b1);

    float acc[M][V];
#pragma unroll
    for (int r = 0; r < M; ++r)
#pragma unroll
        for (int v = 0; v < V; ++v) acc[r][v] = 0.0f;

    if (col < a.Np) {
        for (int b = b0; b < b1; ++b) {
            const int8_t *qb = a.q + (size_t)b * kBlock * a.Np + col;
            const uint16_t *xb = a.x + (size_t)b * kBlock;
            float sc[V];
#pragma unroll
            for (int v4 = 0; v4 < V / 4; ++v4) {
                uint4 t;
                ld_stream(t, a.s + (size_t)b * a.Np + col + 4 * v4);
                sc[4 * v4 + 0] = __uint_as_float(t.x);
                sc[4 * v4 + 1] = __uint_as_float(t.y);
                sc[4 * v4 + 2] = __uint_as_float(t.z);
                sc[4 * v4 + 3] = __uint_as_float(t.w);
            }
            constexpr int PM = kScaleFirst ? 1 : M, PV = kScaleFirst ? 1 : V;
            float p[PM][PV];  // the block's lane sums (unused when the scale goes first)
#pragma unroll
            for (int r = 0; r < PM; ++r)
#pragma unroll
                for (int v = 0; v < PV; ++v) p[r][v] = 0.0f;
#pragma unroll
            for (int ch = 0; ch < 4; ++ch) {  // four chunks of 8 rows
                VT w[8];
#pragma unroll
                for (int j = 0; j < 8; ++j) ld_stream(w[j], qb + (size_t)(8 * ch + j) * a.Np);
                uint4 xr[M];
#pragma unroll
                for (int r = 0; r < M; ++r)
                    xr[r] = __ldg(reinterpret_cast<const uint4 *>(xb + (size_t)r * a.K + 8 * ch));
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    float xv[M];
#pragma unroll
                    for (int r = 0; r < M; ++r) {
                        const uint32_t pair = word_of(xr[r], j >> 1);
                        xv[r] = (j & 1) ? bf16_hi(pair) : bf16_lo(pair);
                    }
#pragma unroll
                    for (int wi = 0; wi < NW; ++wi) {
                        const uint32_t u = word_of(w[j], wi) ^ 0x80808080u;
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const int v = 4 * wi + e;
                            const float f = q8_to_f32(u, e);
                            if constexpr (kScaleFirst) {
                                const float fs = f * sc[v];
#pragma unroll
                                for (int r = 0; r < M; ++r) acc[r][v] = fmaf(xv[r], fs, acc[r][v]);
                            } else {
#pragma unroll
                                for (int r = 0; r < M; ++r) p[r][v] = fmaf(xv[r], f, p[r][v]);
                            }
                        }
                    }
                }
            }
            if constexpr (!kScaleFirst) {
#pragma unroll
                for (int r = 0; r < M; ++r)
#pragma unroll
                    for (int v = 0; v < V; ++v) acc[r][v] = fmaf(sc[v], p[r][v], acc[r][v]);
            }
        }
    }

    float *red = smem + warp * M * TC;
#pragma unroll
    for (int r = 0; r < M; ++r)
#pragma unroll
        for (int v4 = 0; v4 < V / 4; ++v4)
            *reinterpret_cast<float4 *>(red + r * TC + cl + 4 * v4) =
                make_float4(acc[r][4 * v4], acc[r][4 * v4 + 1], acc[r][4 * v4 + 2], acc[r][4 * v4 + 3]);
    __syncthreads();
    finish<M, TC, ARGMAX>(a, smem);
}

template <int M, int V>
static cudaError_t launch_mv(const Args &a, bool argmax, cudaStream_t st) {
    constexpr int TC = simt_tile(V);
    constexpr int smem = finish_smem_bytes(M, TC);
    return argmax ? launch_tiles(simt_kernel<M, V, true>, a, TC, smem, st)
                  : launch_tiles(simt_kernel<M, V, false>, a, TC, smem, st);
}

bool simt_has(int m, int V) {
    switch (m) {
        case 1: case 2: return V == 16 || V == 8 || V == 4;
        case 3: return V == 8 || V == 4;
        case 4: case 8: return V == 4;
        default: return false;
    }
}

cudaError_t launch_simt(const Args &a, int V, bool argmax, cudaStream_t st) {
    switch (a.m * 100 + V) {
        case 116: return launch_mv<1, 16>(a, argmax, st);
        case 108: return launch_mv<1, 8>(a, argmax, st);
        case 104: return launch_mv<1, 4>(a, argmax, st);
        case 216: return launch_mv<2, 16>(a, argmax, st);
        case 208: return launch_mv<2, 8>(a, argmax, st);
        case 204: return launch_mv<2, 4>(a, argmax, st);
        case 308: return launch_mv<3, 8>(a, argmax, st);
        case 304: return launch_mv<3, 4>(a, argmax, st);
        case 404: return launch_mv<4, 4>(a, argmax, st);
        case 804: return launch_mv<8, 4>(a, argmax, st);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace q8
