// Q8_0 GEMV over the tiled weight storage: every warp streams its own contiguous run of weight units.
//
// The tiled storage (q8_tile) keeps every 32-row x 128-column block of the weight as one contiguous 4 KB unit, in
// MMA-fragment order: the unit is eight 512-byte segments (16-row step s = 0, 1; row group j = 0..3), and in segment
// (s, j) lane L = 4g + t of a warp finds its 16 bytes at L * 16: weight row 16s + 4t + j, columns 16g .. 16g + 15 of
// the tile.  The scales of the unit follow in their own storage, 128 fp32 in column order.  So one warp instruction
// copies 512 contiguous bytes, and the units of a column tile follow each other along K: a warp that owns a run of K
// blocks of one tile reads one contiguous range of memory.
//
// A CTA owns one 128-column tile and a range of its K blocks (split across a thread-block cluster when N is too
// narrow to fill the SMs); its eight warps split that range into contiguous runs.  Each warp keeps a private ring of
// three stages in shared memory, filled with cp.async (16 bytes a lane, bypassing L1): it issues block i + 2 while
// it computes block i, so about two units per warp -- 150 KB per SM -- are in flight without holding registers.  Per
// block a lane converts its 4 x 16 int8 values exactly to bf16 pairs, runs the 8 (or 16) bf16 m16n8k16 MMAs of the
// block into a fresh fp32 accumulator, and folds the block sums into its fp32 carry with the block's scales
// ("from_q8.rs", module doc: the lanes contracted over the int8 rows, then folded down each column with their scales,
// into an fp32 carry).  The MMA's K order is the relabeling of the register-fed kernel: MMA reduction index 2t, 2t+1,
// 2t+8, 2t+9 is weight row 4t, 4t+1, 4t+2, 4t+3, so a lane's activation fragment is 4 consecutive activations.
//
// Activations are read from L2 (ld.global.cg), two blocks ahead.  With programmatic dependent launch every thread
// waits for the previous kernel (griddepcontrol.wait) before it reads x or writes y; with Q8_FLAG_CONSTANT_WEIGHTS
// the first two stages' weights are already requested before that wait.
#include "q8_launch.h"

namespace q8 {

namespace {

constexpr int kWarpsS = 8;
constexpr int kThreadsS = 32 * kWarpsS;
constexpr int kUnit = kBlock * kTmaColumns;  // 4096 bytes of values per 32 x 128 unit
constexpr int kUnitScales = kTmaColumns;     // 128 fp32
constexpr int kStageS = kUnit + kUnitScales * 4;
// Ring stages per warp: three with two CTAs per SM (m <= 8), five with one (m > 8, twice the accumulators).
template <int NT> struct StreamShape {
    static constexpr int kDepth = NT == 1 ? 3 : 5;
    static constexpr int kSmem = kWarpsS * kDepth * kStageS;
};

__device__ __forceinline__ uint32_t smem_addr(const void *p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ void cp_async16(void *dst, const void *src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N> __device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ void mma_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                          uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// The same MMA into a fresh accumulator (C = 0): the first 16 rows of a block start the block's sums.
__device__ __forceinline__ void mma_16816_first(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                                uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%10, %10, %10, %10};"
        : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(0.0f));
}

__device__ __forceinline__ uint2 ld_cg_u2(const void *p) {
    uint2 v;
    asm volatile("ld.global.cg.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "l"(p));
    return v;
}

// Packed fp32 pairs (one 64-bit register pair) for the CUDA-core inner loop.
__device__ __forceinline__ unsigned long long pack_f32x2(float lo, float hi) {
    unsigned long long d;
    asm("mov.b64 %0, {%1, %2};" : "=l"(d) : "f"(lo), "f"(hi));
    return d;
}
__device__ __forceinline__ void unpack_f32x2(unsigned long long v, float &lo, float &hi) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ unsigned long long fma_f32x2(unsigned long long a, unsigned long long b,
                                                        unsigned long long c) {
    unsigned long long d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
// Bytes e and e + 1 of a sign-flipped int8 word (see q8_to_f32) as the exact fp32 pair {q_e, q_e+1}: two byte
// permutes into the mantissa of 2^23 and one packed subtract of 2^23 + 128.
template <int E> __device__ __forceinline__ unsigned long long q8x2_to_f32x2(uint32_t u, unsigned long long magic) {
    unsigned long long d;
    asm("{\n .reg .b32 a, b;\n .reg .b64 p;\n prmt.b32 a, %1, 0x4B000000, %2;\n prmt.b32 b, %1, 0x4B000000, %3;\n"
        " mov.b64 p, {a, b};\n sub.rn.f32x2 %0, p, %4;\n}"
        : "=l"(d)
        : "r"(u), "n"(0x7540 + E), "n"(0x7540 + E + 1), "l"(magic));
    return d;
}

// Copy unit `u` (values and scales) into `stage`: 8 + 1 cp.async of 16 bytes per lane.
__device__ __forceinline__ void issue_unit(unsigned char *stage, const int8_t *q, const float *s, size_t u, int lane) {
    const unsigned char *src = reinterpret_cast<const unsigned char *>(q) + u * kUnit + lane * 16;
#pragma unroll
    for (int seg = 0; seg < 8; ++seg) cp_async16(stage + seg * 512 + lane * 16, src + seg * 512);
    cp_async16(stage + kUnit + lane * 16, reinterpret_cast<const unsigned char *>(s + u * kUnitScales) + lane * 16);
}

template <int NT, bool ARGMAX>
__global__ void __launch_bounds__(kThreadsS, NT == 1 ? 2 : 1)
    stream_kernel(Args a, const __grid_constant__ Parts parts, const int prefetch_weights) {
    constexpr int MR = 8 * NT;
    constexpr int kDepth = StreamShape<NT>::kDepth;
    extern __shared__ __align__(16) unsigned char smem_s[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, t = lane & 3;
    const int tile = select_part(parts, blockIdx.x, a);
    const int rank = blockIdx.y;
    const int c0 = (int)((long long)a.nb * rank / a.ksplit);
    const int c1 = (int)((long long)a.nb * (rank + 1) / a.ksplit);
    const int b0 = c0 + (c1 - c0) * warp / kWarpsS;
    const int b1 = c0 + (c1 - c0) * (warp + 1) / kWarpsS;
    const int n = b1 - b0;
    unsigned char *ring = smem_s + warp * kDepth * kStageS;
    const size_t unit0 = (size_t)tile * a.nb + b0;

    float acc[NT][8][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int p = 0; p < 8; ++p)
#pragma unroll
            for (int i = 0; i < 4; ++i) acc[nt][p][i] = 0.0f;

    // Prologue: the first kDepth - 1 units (one commit group each, empty past the run).
    if (prefetch_weights) {
#pragma unroll
        for (int i = 0; i < kDepth - 1; ++i) {
            if (i < n) issue_unit(ring + i * kStageS, a.q, a.s, unit0 + i, lane);
            cp_async_commit();
        }
    }
    asm volatile("griddepcontrol.wait;" ::: "memory");
    if (!prefetch_weights) {
#pragma unroll
        for (int i = 0; i < kDepth - 1; ++i) {
            if (i < n) issue_unit(ring + i * kStageS, a.q, a.s, unit0 + i, lane);
            cp_async_commit();
        }
    }

    // Activation rows this lane feeds to the MMA (rows at or past m are zeros).
    const uint16_t *xrow[NT];
    bool xlive[NT];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
        const int r = 8 * nt + g;
        xlive[nt] = r < a.m;
        xrow[nt] = a.x + (size_t)(xlive[nt] ? r : 0) * a.K + 4 * t;
    }
    // Activation fragments two blocks ahead (L2 latency exceeds a block's work): xn1 for block i + 1, xn2 for i + 2.
    uint2 xn1[2][NT], xn2[2][NT];
    auto load_x = [&](uint2 (&dst)[2][NT], int b) {
#pragma unroll
        for (int step = 0; step < 2; ++step)
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
                dst[step][nt] = xlive[nt] ? ld_cg_u2(xrow[nt] + (size_t)b * kBlock + 16 * step) : make_uint2(0u, 0u);
    };
    if (n > 0) load_x(xn1, b0);
    if (n > 1) load_x(xn2, b0 + 1);

    for (int i = 0; i < n; ++i) {
        const int ahead = i + kDepth - 1;
        if (ahead < n) issue_unit(ring + (ahead % kDepth) * kStageS, a.q, a.s, unit0 + ahead, lane);
        cp_async_commit();
        cp_async_wait<kDepth - 1>();  // this lane's copies of unit i have landed
        __syncwarp();                 // ... and every other lane's (the scales are read across lanes)
        const unsigned char *st = ring + (i % kDepth) * kStageS;
        uint2 xc[2][NT];
#pragma unroll
        for (int step = 0; step < 2; ++step)
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                xc[step][nt] = xn1[step][nt];
                xn1[step][nt] = xn2[step][nt];
            }
        if (i + 2 < n) load_x(xn2, b0 + i + 2);

        float d[NT][8][4];  // the block's sums, started by the first step's MMAs
#pragma unroll
        for (int step = 0; step < 2; ++step) {
            uint4 w[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) w[j] = *reinterpret_cast<const uint4 *>(st + (step * 4 + j) * 512 + lane * 16);
#pragma unroll
            for (int wi = 0; wi < 4; ++wi) {
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
                for (int h = 0; h < 2; ++h) {
                    const int p = 2 * wi + h;
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt) {
                        if (step == 0)
                            mma_16816_first(d[nt][p], lo[2 * h], lo[2 * h + 1], hi[2 * h], hi[2 * h + 1],
                                            xc[step][nt].x, xc[step][nt].y);
                        else
                            mma_16816(d[nt][p], lo[2 * h], lo[2 * h + 1], hi[2 * h], hi[2 * h + 1], xc[step][nt].x,
                                      xc[step][nt].y);
                    }
                }
            }
        }
        const float *ss = reinterpret_cast<const float *>(st + kUnit) + 16 * g;
        float sc[16];
#pragma unroll
        for (int v4 = 0; v4 < 4; ++v4) {
            const float4 f = *reinterpret_cast<const float4 *>(ss + 4 * v4);
            sc[4 * v4 + 0] = f.x;
            sc[4 * v4 + 1] = f.y;
            sc[4 * v4 + 2] = f.z;
            sc[4 * v4 + 3] = f.w;
        }
        __syncwarp();  // every lane is done with this stage before it is refilled
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int p = 0; p < 8; ++p) {
                acc[nt][p][0] = fmaf(sc[2 * p], d[nt][p][0], acc[nt][p][0]);
                acc[nt][p][1] = fmaf(sc[2 * p], d[nt][p][1], acc[nt][p][1]);
                acc[nt][p][2] = fmaf(sc[2 * p + 1], d[nt][p][2], acc[nt][p][2]);
                acc[nt][p][3] = fmaf(sc[2 * p + 1], d[nt][p][3], acc[nt][p][3]);
            }
    }
    cp_async_wait<0>();
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    __syncthreads();  // every warp is done with its ring: the shared memory holds the epilogue now

    // D fragment: element 0/1 -> activation rows 2t, 2t+1 of MMA row g (column 16g + 2p); 2/3 -> the same rows of
    // MMA row g + 8 (column 16g + 2p + 1).
    float *red = reinterpret_cast<float *>(smem_s);  // [kWarpsS][MR][128]
    float *mine = red + warp * MR * kTmaColumns;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int p = 0; p < 8; ++p) {
            const int r = 8 * nt + 2 * t;
            const int c = 16 * g + 2 * p;
            *reinterpret_cast<float2 *>(mine + r * kTmaColumns + c) = make_float2(acc[nt][p][0], acc[nt][p][2]);
            *reinterpret_cast<float2 *>(mine + (r + 1) * kTmaColumns + c) = make_float2(acc[nt][p][1], acc[nt][p][3]);
        }
    __syncthreads();
    finish_n<kWarpsS, MR, kTmaColumns, kThreadsS, ARGMAX>(a, red, tile);
}


// The CUDA-core inner loop over the same stream, for m <= 2 (where the per-row FMAs are cheaper than packing bf16
// MMA operands).  In segment (s, j) lane L = 4g + u holds 16 columns 16g .. 16g + 15 of weight row 16s + 4u + j: it
// converts each pair of values to an exact fp32 pair and accumulates x[r, row] * q into the block's sums with packed
// fp32x2 FMAs, folds the sums into its carry with the block's scales, and at the end the four lanes u of a column
// group add their carries (rows 4u + j of every step) in a fixed order.
template <int M, bool ARGMAX>
__global__ void __launch_bounds__(kThreadsS, 2)
    stream_simt_kernel(Args a, const __grid_constant__ Parts parts, const int prefetch_weights) {
    constexpr int kDepth = StreamShape<1>::kDepth;
    extern __shared__ __align__(16) unsigned char smem_s[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, u = lane & 3;
    const int tile = select_part(parts, blockIdx.x, a);
    const int rank = blockIdx.y;
    const int c0 = (int)((long long)a.nb * rank / a.ksplit);
    const int c1 = (int)((long long)a.nb * (rank + 1) / a.ksplit);
    const int b0 = c0 + (c1 - c0) * warp / kWarpsS;
    const int b1 = c0 + (c1 - c0) * (warp + 1) / kWarpsS;
    const int n = b1 - b0;
    unsigned char *ring = smem_s + warp * kDepth * kStageS;
    const size_t unit0 = (size_t)tile * a.nb + b0;

    unsigned long long acc[M][8];  // fp32 pairs: columns 16g + 2p, 16g + 2p + 1
#pragma unroll
    for (int r = 0; r < M; ++r)
#pragma unroll
        for (int p = 0; p < 8; ++p) acc[r][p] = 0ull;

    if (prefetch_weights) {
#pragma unroll
        for (int i = 0; i < kDepth - 1; ++i) {
            if (i < n) issue_unit(ring + i * kStageS, a.q, a.s, unit0 + i, lane);
            cp_async_commit();
        }
    }
    asm volatile("griddepcontrol.wait;" ::: "memory");
    if (!prefetch_weights) {
#pragma unroll
        for (int i = 0; i < kDepth - 1; ++i) {
            if (i < n) issue_unit(ring + i * kStageS, a.q, a.s, unit0 + i, lane);
            cp_async_commit();
        }
    }

    // x[r][32b + 16s + 4u .. + 3]: the activations of this lane's rows, two 8-byte loads per row and block.
    uint2 xn1[M][2], xn2[M][2];  // blocks i + 1 and i + 2
    auto load_x = [&](uint2 (&dst)[M][2], int b) {
#pragma unroll
        for (int r = 0; r < M; ++r)
#pragma unroll
            for (int s = 0; s < 2; ++s) dst[r][s] = ld_cg_u2(a.x + (size_t)r * a.K + (size_t)b * kBlock + 16 * s + 4 * u);
    };
    if (n > 0) load_x(xn1, b0);
    if (n > 1) load_x(xn2, b0 + 1);

    for (int i = 0; i < n; ++i) {
        const int ahead = i + kDepth - 1;
        if (ahead < n) issue_unit(ring + (ahead % kDepth) * kStageS, a.q, a.s, unit0 + ahead, lane);
        cp_async_commit();
        cp_async_wait<kDepth - 1>();
        __syncwarp();
        const unsigned char *st = ring + (i % kDepth) * kStageS;
        uint2 xc[M][2];
#pragma unroll
        for (int r = 0; r < M; ++r)
#pragma unroll
            for (int s = 0; s < 2; ++s) {
                xc[r][s] = xn1[r][s];
                xn1[r][s] = xn2[r][s];
            }
        if (i + 2 < n) load_x(xn2, b0 + i + 2);

        unsigned long long part[M][8];
#pragma unroll
        for (int r = 0; r < M; ++r)
#pragma unroll
            for (int p = 0; p < 8; ++p) part[r][p] = 0ull;
#pragma unroll
        for (int s = 0; s < 2; ++s)
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const uint4 w = *reinterpret_cast<const uint4 *>(st + (s * 4 + j) * 512 + lane * 16);
                unsigned long long xx[M];
#pragma unroll
                for (int r = 0; r < M; ++r) {
                    const uint32_t pr = (j < 2) ? xc[r][s].x : xc[r][s].y;
                    const float xv = (j & 1) ? bf16_hi(pr) : bf16_lo(pr);
                    xx[r] = pack_f32x2(xv, xv);
                }
#pragma unroll
                for (int wi = 0; wi < 4; ++wi) {
                    const uint32_t uw = word_of(w, wi) ^ 0x80808080u;
                    const unsigned long long q01 = q8x2_to_f32x2<0>(uw, kMagicPair);
                    const unsigned long long q23 = q8x2_to_f32x2<2>(uw, kMagicPair);
#pragma unroll
                    for (int r = 0; r < M; ++r) {
                        part[r][2 * wi] = fma_f32x2(q01, xx[r], part[r][2 * wi]);
                        part[r][2 * wi + 1] = fma_f32x2(q23, xx[r], part[r][2 * wi + 1]);
                    }
                }
            }
        unsigned long long sc[8];
        const uint4 *ss = reinterpret_cast<const uint4 *>(st + kUnit) + 4 * g;
#pragma unroll
        for (int v4 = 0; v4 < 4; ++v4) {
            const uint4 f = ss[v4];
            sc[2 * v4] = ((unsigned long long)f.y << 32) | f.x;
            sc[2 * v4 + 1] = ((unsigned long long)f.w << 32) | f.z;
        }
        __syncwarp();  // every lane is done with this stage before it is refilled
#pragma unroll
        for (int r = 0; r < M; ++r)
#pragma unroll
            for (int p = 0; p < 8; ++p) acc[r][p] = fma_f32x2(sc[p], part[r][p], acc[r][p]);
    }
    cp_async_wait<0>();
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    __syncthreads();

    float *red = reinterpret_cast<float *>(smem_s);  // [kWarpsS][M][128]
    float *mine = red + warp * M * kTmaColumns;
#pragma unroll
    for (int r = 0; r < M; ++r)
#pragma unroll
        for (int p = 0; p < 8; ++p) {
            float lo, hi;
            unpack_f32x2(acc[r][p], lo, hi);
            lo += __shfl_xor_sync(0xffffffffu, lo, 1);
            hi += __shfl_xor_sync(0xffffffffu, hi, 1);
            lo += __shfl_xor_sync(0xffffffffu, lo, 2);
            hi += __shfl_xor_sync(0xffffffffu, hi, 2);
            if (u == 0) *reinterpret_cast<float2 *>(mine + r * kTmaColumns + 16 * g + 2 * p) = make_float2(lo, hi);
        }
    __syncthreads();
    finish_n<kWarpsS, M, kTmaColumns, kThreadsS, ARGMAX>(a, red, tile);
}


// m = 9..16: two tiles of 8 activation rows.  The accumulators of 16 rows x 128 columns would not fit one warp's
// registers at two CTAs per SM, so a block's columns are split between a warp pair: warp 2k + h streams and converts
// columns 64h .. 64h + 63 of every unit of its K range (each value is still converted once).  Each warp keeps its
// own ring of five half-units (2 KB of values and 256 B of scales each); lane (g, t) of warp h holds 8 columns
// 64h + 8g .. 64h + 8g + 7, the second half of chunk 4h + g/2 of its row group t.
constexpr int kHalfUnit = kUnit / 2;
constexpr int kHalfStage = kHalfUnit + kUnitScales * 2;
constexpr int kPairDepth = 5;
constexpr int kPairSmem = kWarpsS * kPairDepth * kHalfStage;

__device__ __forceinline__ void issue_half_unit(unsigned char *stage, const int8_t *q, const float *s, size_t u,
                                                int h, int lane) {
    const unsigned char *src = reinterpret_cast<const unsigned char *>(q) + u * kUnit + 256 * h + (lane & 15) * 16;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        const int seg = 2 * c + (lane >> 4);
        cp_async16(stage + seg * 256 + (lane & 15) * 16, src + seg * 512);
    }
    if (lane < 16)
        cp_async16(stage + kHalfUnit + lane * 16,
                   reinterpret_cast<const unsigned char *>(s + u * kUnitScales + 64 * h) + lane * 16);
}

template <bool ARGMAX>
__global__ void __launch_bounds__(kThreadsS, 2)
    stream_pair_kernel(Args a, const __grid_constant__ Parts parts, const int prefetch_weights) {
    constexpr int NT = 2, MR = 16, NP = 4, kDepth = kPairDepth, kRanges = kWarpsS / 2;
    extern __shared__ __align__(16) unsigned char smem_s[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, t = lane & 3;
    const int h = warp & 1, kr = warp >> 1;
    const int tile = select_part(parts, blockIdx.x, a);
    const int rank = blockIdx.y;
    const int c0 = (int)((long long)a.nb * rank / a.ksplit);
    const int c1 = (int)((long long)a.nb * (rank + 1) / a.ksplit);
    const int b0 = c0 + (c1 - c0) * kr / kRanges;
    const int b1 = c0 + (c1 - c0) * (kr + 1) / kRanges;
    const int n = b1 - b0;
    unsigned char *ring = smem_s + warp * kDepth * kHalfStage;
    const size_t unit0 = (size_t)tile * a.nb + b0;

    float acc[NT][NP][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int p = 0; p < NP; ++p)
#pragma unroll
            for (int i = 0; i < 4; ++i) acc[nt][p][i] = 0.0f;

    if (prefetch_weights) {
#pragma unroll
        for (int i = 0; i < kDepth - 1; ++i) {
            if (i < n) issue_half_unit(ring + i * kHalfStage, a.q, a.s, unit0 + i, h, lane);
            cp_async_commit();
        }
    }
    asm volatile("griddepcontrol.wait;" ::: "memory");
    if (!prefetch_weights) {
#pragma unroll
        for (int i = 0; i < kDepth - 1; ++i) {
            if (i < n) issue_half_unit(ring + i * kHalfStage, a.q, a.s, unit0 + i, h, lane);
            cp_async_commit();
        }
    }

    const uint16_t *xrow[NT];
    bool xlive[NT];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
        const int r = 8 * nt + g;
        xlive[nt] = r < a.m;
        xrow[nt] = a.x + (size_t)(xlive[nt] ? r : 0) * a.K + 4 * t;
    }
    uint2 xn1[2][NT], xn2[2][NT];
    auto load_x = [&](uint2 (&dst)[2][NT], int b) {
#pragma unroll
        for (int step = 0; step < 2; ++step)
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
                dst[step][nt] = xlive[nt] ? ld_cg_u2(xrow[nt] + (size_t)b * kBlock + 16 * step) : make_uint2(0u, 0u);
    };
    if (n > 0) load_x(xn1, b0);
    if (n > 1) load_x(xn2, b0 + 1);
    const int woff = (4 * (g >> 1) + t) * 16 + 8 * (g & 1);  // this lane's 8 bytes within a 256-byte half-segment

    for (int i = 0; i < n; ++i) {
        const int ahead = i + kDepth - 1;
        if (ahead < n) issue_half_unit(ring + (ahead % kDepth) * kHalfStage, a.q, a.s, unit0 + ahead, h, lane);
        cp_async_commit();
        cp_async_wait<kDepth - 1>();
        __syncwarp();
        const unsigned char *st = ring + (i % kDepth) * kHalfStage;
        uint2 xc[2][NT];
#pragma unroll
        for (int step = 0; step < 2; ++step)
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                xc[step][nt] = xn1[step][nt];
                xn1[step][nt] = xn2[step][nt];
            }
        if (i + 2 < n) load_x(xn2, b0 + i + 2);

        float d[NT][NP][4];  // the block's sums, started by the first step's MMAs
#pragma unroll
        for (int step = 0; step < 2; ++step) {
            uint2 w[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) w[j] = *reinterpret_cast<const uint2 *>(st + (step * 4 + j) * 256 + woff);
#pragma unroll
            for (int wi = 0; wi < 2; ++wi) {
                const uint32_t u0 = word_of(w[0], wi) ^ 0x80808080u;
                const uint32_t u1 = word_of(w[1], wi) ^ 0x80808080u;
                const uint32_t u2 = word_of(w[2], wi) ^ 0x80808080u;
                const uint32_t u3 = word_of(w[3], wi) ^ 0x80808080u;
                uint32_t lo[4], hi[4];
                lo[0] = q8x2_to_bf16x2<0>(u0, u1, kMagicPair);
                lo[1] = q8x2_to_bf16x2<1>(u0, u1, kMagicPair);
                lo[2] = q8x2_to_bf16x2<2>(u0, u1, kMagicPair);
                lo[3] = q8x2_to_bf16x2<3>(u0, u1, kMagicPair);
                hi[0] = q8x2_to_bf16x2<0>(u2, u3, kMagicPair);
                hi[1] = q8x2_to_bf16x2<1>(u2, u3, kMagicPair);
                hi[2] = q8x2_to_bf16x2<2>(u2, u3, kMagicPair);
                hi[3] = q8x2_to_bf16x2<3>(u2, u3, kMagicPair);
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    const int p = 2 * wi + hh;
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt) {
                        if (step == 0)
                            mma_16816_first(d[nt][p], lo[2 * hh], lo[2 * hh + 1], hi[2 * hh], hi[2 * hh + 1],
                                            xc[step][nt].x, xc[step][nt].y);
                        else
                            mma_16816(d[nt][p], lo[2 * hh], lo[2 * hh + 1], hi[2 * hh], hi[2 * hh + 1],
                                      xc[step][nt].x, xc[step][nt].y);
                    }
                }
            }
        }
        const float *ss = reinterpret_cast<const float *>(st + kHalfUnit) + 8 * g;
        float sc[8];
#pragma unroll
        for (int v4 = 0; v4 < 2; ++v4) {
            const float4 f = *reinterpret_cast<const float4 *>(ss + 4 * v4);
            sc[4 * v4 + 0] = f.x;
            sc[4 * v4 + 1] = f.y;
            sc[4 * v4 + 2] = f.z;
            sc[4 * v4 + 3] = f.w;
        }
        __syncwarp();
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
    cp_async_wait<0>();
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    __syncthreads();

    float *red = reinterpret_cast<float *>(smem_s);  // [kRanges][MR][128]
    float *mine = red + kr * MR * kTmaColumns;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int p = 0; p < NP; ++p) {
            const int r = 8 * nt + 2 * t;
            const int c = 64 * h + 8 * g + 2 * p;
            *reinterpret_cast<float2 *>(mine + r * kTmaColumns + c) = make_float2(acc[nt][p][0], acc[nt][p][2]);
            *reinterpret_cast<float2 *>(mine + (r + 1) * kTmaColumns + c) = make_float2(acc[nt][p][1], acc[nt][p][3]);
        }
    __syncthreads();
    finish_n<kRanges, MR, kTmaColumns, kThreadsS, ARGMAX>(a, red, tile);
}

static_assert(finish_smem_n(kWarpsS / 2, 16, kTmaColumns) <= kPairSmem, "the epilogue fits in the rings");
static_assert(2 * kPairSmem <= 227 * 1024, "two CTAs per SM");

static_assert(finish_smem_n(kWarpsS, 8, kTmaColumns) <= StreamShape<1>::kSmem, "the epilogue fits in the rings");
static_assert(finish_smem_n(kWarpsS, 16, kTmaColumns) <= StreamShape<2>::kSmem, "the epilogue fits in the rings");
static_assert(2 * StreamShape<1>::kSmem <= 227 * 1024 && StreamShape<2>::kSmem <= 227 * 1024, "residency");

template <typename Kernel>
cudaError_t launch_stream_kernel(Kernel kernel, int kSmemS, const Args &a, const Parts &pt, cudaStream_t stream,
                                 bool pdl, bool prefetch) {
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemS);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)pt.tile_end[pt.count - 1], (unsigned)a.ksplit, 1);
    cfg.blockDim = dim3(kThreadsS, 1, 1);
    cfg.dynamicSmemBytes = kSmemS;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    int na = 0;
    if (a.ksplit > 1) {
        attr[na].id = cudaLaunchAttributeClusterDimension;
        attr[na].val.clusterDim.x = 1;
        attr[na].val.clusterDim.y = (unsigned)a.ksplit;
        attr[na].val.clusterDim.z = 1;
        ++na;
    }
    if (pdl) {
        attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[na].val.programmaticStreamSerializationAllowed = 1;
        ++na;
    }
    cfg.attrs = attr;
    cfg.numAttrs = na;
    return cudaLaunchKernelEx(&cfg, kernel, a, pt, prefetch ? 1 : 0);
}

}  // namespace

int stream_ctas_per_sm(int) { return 2; }

cudaError_t launch_stream(const Args &a, const Parts &pt, bool argmax, cudaStream_t stream, bool pdl,
                          bool prefetch_weights) {
    constexpr int s1 = StreamShape<1>::kSmem;
    const bool p = prefetch_weights;
    switch (a.m) {
        case 1:
            return argmax ? launch_stream_kernel(stream_simt_kernel<1, true>, s1, a, pt, stream, pdl, p)
                          : launch_stream_kernel(stream_simt_kernel<1, false>, s1, a, pt, stream, pdl, p);
        case 2:
            return argmax ? launch_stream_kernel(stream_simt_kernel<2, true>, s1, a, pt, stream, pdl, p)
                          : launch_stream_kernel(stream_simt_kernel<2, false>, s1, a, pt, stream, pdl, p);
        default:
            break;
    }
    if (a.m <= 8)
        return argmax ? launch_stream_kernel(stream_kernel<1, true>, s1, a, pt, stream, pdl, p)
                      : launch_stream_kernel(stream_kernel<1, false>, s1, a, pt, stream, pdl, p);
    return argmax ? launch_stream_kernel(stream_pair_kernel<true>, kPairSmem, a, pt, stream, pdl, p)
                  : launch_stream_kernel(stream_pair_kernel<false>, kPairSmem, a, pt, stream, pdl, p);
}

}  // namespace q8
