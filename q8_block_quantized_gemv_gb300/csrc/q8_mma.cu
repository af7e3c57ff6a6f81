// Tensor-core Q8_0 GEMV for batches: the weight tile is the MMA's A operand, the activations its B operand.
//
// One bf16 m16n8k16 MMA multiplies 16 weight columns (the MMA's rows) by up to 8 activation rows (its columns) over
// 16 weight rows.  The MMA's K order and row order are free relabelings of the weight's rows and columns, chosen so
// that each lane's operands come straight from its own loads:
//   - lane (g, t) = (lane / 4, lane % 4) loads V adjacent columns (V bytes) of 4 adjacent weight rows 4t .. 4t+3 of a
//     16-row step; MMA reduction index 2t, 2t+1, 2t+8, 2t+9 is weight row 4t, 4t+1, 4t+2, 4t+3;
//   - MMA row g of the MMA for column pair p is weight column g*V + 2p, MMA row g+8 is column g*V + 2p + 1;
//   - the B fragment of lane (g, t) is then 4 consecutive activations x[8*tile + g][4t .. 4t+3], one 8-byte load.
// Each int8 is converted exactly to bf16 (|q| <= 127 needs 8 significant bits, bf16 has 8).  Every product of a bf16
// activation and an int8 value is exact; the MMA sums the block's 32 products in fp32 into a fresh accumulator, and
// the block's sum is then multiplied by its scale and added into an fp32 carry on the CUDA cores ("from_q8.rs", module
// doc: int8 rows are contracted lane by lane, and each column's block sums are scaled and accumulated in fp32).
#include "q8_launch.h"

namespace q8 {

__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                               uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// NT tiles of 8 activation rows (m <= 8 * NT), V columns per lane, TC = 8 * V columns per CTA.
template <int NT, int V, bool ARGMAX>
__global__ void __launch_bounds__(kThreads, 2) mma_kernel(const Args a) {
    using VT = typename Vec<V>::T;
    constexpr int NW = V / 4;
    constexpr int NP = V / 2;  // column pairs = MMAs per 16-row step and row tile
    constexpr int TC = mma_tile(V);
    constexpr int MR = 8 * NT;
    extern __shared__ __align__(16) float smem[];

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, t = lane & 3;
    const int cl = g * V;
    const int col = blockIdx.x * TC + cl;
    int b0, b1;
    warp_blocks(a, warp, b0, b1);

    float acc[NT][NP][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int p = 0; p < NP; ++p)
#pragma unroll
            for (int i = 0; i < 4; ++i) acc[nt][p][i] = 0.0f;

    // Activation rows this lane feeds to the MMA (rows at or past m read as zeros).
    const uint16_t *xrow[NT];
    bool xlive[NT];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
        const int r = 8 * nt + g;
        xlive[nt] = r < a.m;
        xrow[nt] = a.x + (size_t)(xlive[nt] ? r : 0) * a.K + 4 * t;
    }

    // Every lane runs the loop (mma.sync needs the whole warp); lanes past the last column load zeros.
    const bool live = col < a.Np;
    for (int b = b0; b < b1; ++b) {
        float d[NT][NP][4];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int p = 0; p < NP; ++p)
#pragma unroll
                for (int i = 0; i < 4; ++i) d[nt][p][i] = 0.0f;
#pragma unroll
        for (int step = 0; step < 2; ++step) {
            const int k0 = b * kBlock + 16 * step + 4 * t;
            VT w[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                w[j] = VT{};
                if (live) ld_stream(w[j], a.q + (size_t)(k0 + j) * a.Np + col);
            }
            uint32_t bx[NT][2];
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                uint2 xv = make_uint2(0u, 0u);
                if (xlive[nt]) xv = __ldg(reinterpret_cast<const uint2 *>(xrow[nt] + b * kBlock + 16 * step));
                bx[nt][0] = xv.x;
                bx[nt][1] = xv.y;
            }
#pragma unroll
            for (int wi = 0; wi < NW; ++wi) {
                const uint32_t u0 = word_of(w[0], wi) ^ 0x80808080u;
                const uint32_t u1 = word_of(w[1], wi) ^ 0x80808080u;
                const uint32_t u2 = word_of(w[2], wi) ^ 0x80808080u;
                const uint32_t u3 = word_of(w[3], wi) ^ 0x80808080u;
                uint32_t lo[4], hi[4];  // per column: rows (4t, 4t+1) and (4t+2, 4t+3) as bf16 pairs
                lo[0] = q8x2_to_bf16x2<0>(u0, u1, kMagicPair);
                lo[1] = q8x2_to_bf16x2<1>(u0, u1, kMagicPair);
                lo[2] = q8x2_to_bf16x2<2>(u0, u1, kMagicPair);
                lo[3] = q8x2_to_bf16x2<3>(u0, u1, kMagicPair);
                hi[0] = q8x2_to_bf16x2<0>(u2, u3, kMagicPair);
                hi[1] = q8x2_to_bf16x2<1>(u2, u3, kMagicPair);
                hi[2] = q8x2_to_bf16x2<2>(u2, u3, kMagicPair);
                hi[3] = q8x2_to_bf16x2<3>(u2, u3, kMagicPair);
#pragma unroll
                for (int h = 0; h < 2; ++h) {  // the two column pairs of this word
                    const int p = 2 * wi + h;
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt)
                        mma_bf16_16816(d[nt][p], lo[2 * h], lo[2 * h + 1], hi[2 * h], hi[2 * h + 1], bx[nt][0],
                                       bx[nt][1]);
                }
            }
        }
        float sc[V];
#pragma unroll
        for (int v4 = 0; v4 < V / 4; ++v4) {
            uint4 tt = make_uint4(0u, 0u, 0u, 0u);
            if (live) ld_stream(tt, a.s + (size_t)b * a.Np + col + 4 * v4);
            sc[4 * v4 + 0] = __uint_as_float(tt.x);
            sc[4 * v4 + 1] = __uint_as_float(tt.y);
            sc[4 * v4 + 2] = __uint_as_float(tt.z);
            sc[4 * v4 + 3] = __uint_as_float(tt.w);
        }
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int p = 0; p < NP; ++p) {
                acc[nt][p][0] = fmaf(sc[2 * p], d[nt][p][0], acc[nt][p][0]);
                acc[nt][p][1] = fmaf(sc[2 * p], d[nt][p][1], acc[nt][p][1]);
                acc[nt][p][2] = fmaf(sc[2 * p + 1], d[nt][p][2], acc[nt][p][2]);
                acc[nt][p][3] = fmaf(sc[2 * p + 1], d[nt][p][3], acc[nt][p][3]);
            }
    }

    // D fragment: element 0/1 -> activation rows 2t, 2t+1 of MMA row g (column cl + 2p); 2/3 -> the same rows of
    // MMA row g + 8 (column cl + 2p + 1).
    float *red = smem + warp * MR * TC;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int p = 0; p < NP; ++p) {
            const int r = 8 * nt + 2 * t;
            const int c = cl + 2 * p;
            *reinterpret_cast<float2 *>(red + r * TC + c) = make_float2(acc[nt][p][0], acc[nt][p][2]);
            *reinterpret_cast<float2 *>(red + (r + 1) * TC + c) = make_float2(acc[nt][p][1], acc[nt][p][3]);
        }
    __syncthreads();
    finish<MR, TC, ARGMAX>(a, smem);
}

template <int NT, int V>
static cudaError_t launch_nv(const Args &a, bool argmax, cudaStream_t st) {
    constexpr int TC = mma_tile(V);
    constexpr int smem = finish_smem_bytes(8 * NT, TC);
    return argmax ? launch_tiles(mma_kernel<NT, V, true>, a, TC, smem, st)
                  : launch_tiles(mma_kernel<NT, V, false>, a, TC, smem, st);
}

bool mma_has(int m, int V) {
    if (m < 1 || m > 16) return false;
    return m <= 8 ? (V == 16 || V == 8) : V == 8;
}

cudaError_t launch_mma(const Args &a, int V, bool argmax, cudaStream_t st) {
    const int nt = a.m <= 8 ? 1 : 2;
    switch (nt * 100 + V) {
        case 116: return launch_nv<1, 16>(a, argmax, st);
        case 108: return launch_nv<1, 8>(a, argmax, st);
        case 208: return launch_nv<2, 8>(a, argmax, st);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace q8
