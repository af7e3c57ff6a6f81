// Device building blocks shared by the Q8_0 GEMV kernels (sm_103a).
//
// The product, from "logicaffeine_compile/spatial/passes/from_q8.rs" (module doc and `q8_fold`):
//     y[r, n] = sum_b s[b, n] * sum_{i<32} x[r, 32b + i] * q[32b + i, n]
// with bf16 activations, int8 values, one fp32 scale per 32-row block and column, and fp32 accumulation.
//
// Work decomposition used by every kernel here:
//   - a CTA owns one tile of TC output columns for all m rows and a contiguous range of the K/32 blocks;
//   - its warps (6, 8 or 12 by kernel) split that range again, each streaming whole 32-row blocks of its columns;
//   - per block, the 32 lane products are summed first and then multiplied by the block's scale, as the formula
//     groups them, and added into an fp32 carry that starts at zero;
//   - the warps' carries are summed in shared memory in warp order, then, when K is split across the CTAs of a
//     thread-block cluster (N too narrow to fill the SMs: "plan.rs", `split_counts`: K divided so that every SM
//     gets blocks), each CTA sums one slice of the columns over the cluster's ranks through distributed shared
//     memory, in rank order, four columns a thread.  Every sum has a fixed order, so results are bit-reproducible
//     and need no scratch memory.
#pragma once

#include <cooperative_groups.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace q8 {

constexpr int kBlock = 32;   // rows of a Q8_0 block
constexpr int kMaxClusterRanks = 16;  // the largest K split across a cluster (non-portable above 8 CTAs)
constexpr int kWarps = 8;    // warps per CTA of the kernels launched through launch_tiles (q8_simt.cu, q8_mma.cu)
constexpr int kThreads = 32 * kWarps;

struct Args {
    const uint16_t *x;         // bf16 bit patterns [m][K]
    const int8_t *q;           // [K][Np]
    const float *s;            // [K/32][Np]
    float *y;                  // [m][Np], or null (arg-max without logits; gated pair with only a bf16 output)
    unsigned long long *keys;  // [m] packed arg-max keys, or null
    int m, K, N, Np, nb;       // nb = K / 32
    int ksplit;                // CTAs of a cluster splitting K (grid.y)
    uint16_t *ybf;             // gated pair: bf16 [m][Np] copy of the output; norm: the normed bf16 [m][Np]
    const float *res;          // norm: residual fp32 [m][Np] (h = res + y is written to y; may be y itself)
    const float *gamma;        // norm: fp32 [Np]
    float eps;                 // norm: added to the mean square
    unsigned int *count;       // norm: the completion counters (0 on entry, reset to 0 by the last CTA of a group);
                               // null: write h only, a launch of its own runs the norm
    int count_slot;            // norm: row group g counts in at count[(count_slot + g) % kNormSlots]
    int groups;                // set on the device: the launch's row groups (ceil(m / 16))
    unsigned char *yq;         // gated pair / norm: the quantized form of the bf16 output, codes [m][Np] (or null)
    float *yd;                 //   and its scales [m][Np / 32]
    int tile0;                 // stream kernels: added to grid x (column tiles; the gated pair: its CTAs, two a
                               // tile, so even); nonzero only for the second launch of a launch split in two
};

constexpr int kGroupRows = 16;   // activation rows of one row group (m > 16 runs ceil(m / 16) groups in one grid)
constexpr int kNormSlots = 64;   // completion counters of the residual-norm launches (row groups in flight at once)

// Row groups: grid x holds `groups` = ceil(m / 16) consecutive CTAs per column tile (the row groups of a tile side
// by side, so that they read the tile's weight units at about the same time and the later ones find them in L2).
__device__ __forceinline__ int row_groups(const Args &a) { return (a.m + kGroupRows - 1) / kGroupRows; }

// The Args of row group `group`'s rows, applied just before the epilogue (so that the main loop keeps no extra
// pointers live): y, its bf16 copy, the residual and the arg-max keys move to the group's first row, m becomes the
// group's row count and the norm counter the group's own.
__device__ __forceinline__ void apply_group(Args &a, int group, int groups) {
    a.groups = groups;
    if (groups > 1) {
        const int row0 = group * kGroupRows;
        const size_t off = (size_t)row0 * a.Np;
        if (a.y) a.y += off;
        if (a.ybf) a.ybf += off;
        if (a.yq) a.yq += off;
        if (a.yd) a.yd += (size_t)row0 * (a.Np / kBlock);
        if (a.res) a.res += off;
        if (a.keys) a.keys += row0;
        a.count_slot += group;
        a.m = a.m - row0 < kGroupRows ? a.m - row0 : kGroupRows;
    }
}

// Several weights that multiply one activation in one launch ("plan.rs", `Launch::GemmParts`: the projections that
// share an activation run together, their outputs placed next to each other).  Part p owns the column tiles
// [tile_end[p-1], tile_end[p]) of the launch's grid; q, s and y are its own, as is N.
constexpr int kMaxParts = 8;
struct Parts {
    const int8_t *q[kMaxParts];
    const float *s[kMaxParts];
    float *y[kMaxParts];
    int N[kMaxParts];
    int tile_end[kMaxParts];
    int count;
};

// The part owning grid tile `tile` and the tile's index within it; `a` gets that part's q, s, y and N.
__device__ __forceinline__ int select_part(const Parts &pt, int tile, Args &a) {
    int p = 0, first = 0;
#pragma unroll 1
    while (p + 1 < pt.count && tile >= pt.tile_end[p]) {
        first = pt.tile_end[p];
        ++p;
    }
    a.q = pt.q[p];
    a.s = pt.s[p];
    a.y = pt.y[p];
    a.N = pt.N[p];
    a.Np = (pt.N[p] + kBlock - 1) / kBlock * kBlock;
    return tile - first;
}

// What a launch's epilogue does with the product.
constexpr int kEpiStore = 0;   // write y
constexpr int kEpiArgmax = 1;  // write y (if any) and fold the row arg-max keys
constexpr int kEpiGlu = 2;     // gated pair: part 0 is the gate, part 1 the up projection; write silu(g) * u
constexpr int kEpiNorm = 3;    // residual add into h; with counters (Args::count) the last CTA also runs the norm

// A gated-pair launch interleaves the two weights' CTAs: grid x = 2 * (tile * groups + group) + part, clusters of 2
// along x (the gate's and the up projection's CTAs of one tile, row group and K range side by side).

// The CTA's column tile within its part and its row group (GROUPS: the kernel takes m > 16), with its part's q, s,
// y, N and Np in `a`; the gated pair interleaves the parts (x = 2 * (tile * groups + group) + p).
template <int EPI, bool GROUPS>
__device__ __forceinline__ int select_cta(const Parts &pt, Args &a, int &group) {
    const int groups = GROUPS ? row_groups(a) : 1;
    int x = (int)blockIdx.x + a.tile0;
    if (EPI == kEpiGlu) {
        const int p = x & 1;
        a.q = pt.q[p];
        a.s = pt.s[p];
        x >>= 1;
    }
    group = GROUPS ? x % groups : 0;
    x = GROUPS ? x / groups : x;
    return EPI == kEpiGlu ? x : select_part(pt, x, a);
}

// apply_group for the CTA's own row group, found again from the grid index (m is still the launch's).
template <int EPI, bool GROUPS> __device__ __forceinline__ void apply_cta_group(Args &a) {
    if (!GROUPS) {
        a.groups = 1;
        return;
    }
    const int groups = row_groups(a);
    const int x = EPI == kEpiGlu ? (int)(blockIdx.x + a.tile0) >> 1 : (int)blockIdx.x + a.tile0;
    apply_group(a, x % groups, groups);
}

// ------------------------------------------------------------------------------------------------------------------
// loads
// ------------------------------------------------------------------------------------------------------------------

template <int BYTES> struct Vec;
template <> struct Vec<4> { using T = uint32_t; };
template <> struct Vec<8> { using T = uint2; };
template <> struct Vec<16> { using T = uint4; };

__device__ __forceinline__ uint32_t word_of(const uint32_t &v, int) { return v; }
__device__ __forceinline__ uint32_t word_of(const uint2 &v, int i) { return i == 0 ? v.x : v.y; }
__device__ __forceinline__ uint32_t word_of(const uint4 &v, int i) {
    return i == 0 ? v.x : (i == 1 ? v.y : (i == 2 ? v.z : v.w));
}

// The weight is read exactly once per call: bypass L1 (the data has no reuse inside an SM).
__device__ __forceinline__ void ld_stream(uint32_t &v, const void *p) {
    asm("ld.global.nc.L1::no_allocate.u32 %0, [%1];" : "=r"(v) : "l"(p));
}
__device__ __forceinline__ void ld_stream(uint2 &v, const void *p) {
    asm("ld.global.nc.L1::no_allocate.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "l"(p));
}
__device__ __forceinline__ void ld_stream(uint4 &v, const void *p) {
    asm("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
        : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
        : "l"(p));
}

// ------------------------------------------------------------------------------------------------------------------
// exact conversions
// ------------------------------------------------------------------------------------------------------------------

// int8 -> fp32, exactly.  `u` is four int8 values with their sign bits flipped (x ^ 0x80808080), so byte e holds
// q + 128 in 0..255.  Placing that byte in the low mantissa of 2^23 gives the float 2^23 + q + 128 (the mantissa's
// unit is 1 at this exponent); subtracting 2^23 + 128, an exact difference of two floats in [2^23, 2^24), gives q.
__device__ __forceinline__ float q8_to_f32(uint32_t u, int e) {
    return __uint_as_float(__byte_perm(u, 0x4B000000u, 0x7540u | (uint32_t)e)) - 8388736.0f;
}

// bf16 -> fp32 of the low or high half of a 32-bit pair: bf16 is the top half of an fp32.
__device__ __forceinline__ float bf16_lo(uint32_t pair) { return __uint_as_float(pair << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t pair) { return __uint_as_float(pair & 0xFFFF0000u); }

// The packed fp32 pair {2^23 + 128, 2^23 + 128}: subtracted from two magic floats it leaves two int8 values.
constexpr unsigned long long kMagicPair = 0x4B0000804B000080ull;

// Byte e of two sign-flipped int8 words (see q8_to_f32) as one exact bf16 pair, lo from `ua` in the low half: the two
// magic floats are made by byte permutes, reduced to the integers by one packed fp32x2 subtract, then packed to bf16
// (exact: |q| <= 127 needs 8 significant bits).  `magic` is kMagicPair, held in a register pair by the caller.
template <int E>
__device__ __forceinline__ uint32_t q8x2_to_bf16x2(uint32_t ua, uint32_t ub, unsigned long long magic) {
    uint32_t out;
    asm("{\n .reg .b32 a, b;\n .reg .b64 p, d;\n .reg .f32 lo, hi;\n prmt.b32 a, %1, 0x4B000000, %3;\n"
        " prmt.b32 b, %2, 0x4B000000, %3;\n mov.b64 p, {a, b};\n sub.rn.f32x2 d, p, %4;\n mov.b64 {lo, hi}, d;\n"
        " cvt.rn.bf16x2.f32 %0, hi, lo;\n}"
        : "=r"(out)
        : "r"(ua), "r"(ub), "n"(0x7540 + E), "l"(magic));
    return out;
}

// Two small integers (|v| <= 127, at most 8 significant bits) as a bf16 pair, exactly: lo in the low half.
__device__ __forceinline__ uint32_t bf16x2_exact(float lo, float hi) {
    __nv_bfloat162 p = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&p);
}

// ------------------------------------------------------------------------------------------------------------------
// arg-max keys
// ------------------------------------------------------------------------------------------------------------------

// A 64-bit key whose unsigned order is (logit, then lower index first): the logit's bits made order-preserving in
// the high word (-0.0 counted as +0.0), 0xFFFFFFFF - n in the low word.  Every real key is nonzero, so 0 is the
// identity of the max.
__device__ __forceinline__ unsigned long long argmax_key(float v, int n) {
    // -0.0 keys as +0.0; every NaN (either sign, any payload) as the positive quiet NaN, above +inf
    uint32_t b = (v == 0.0f) ? 0u : (v != v) ? 0x7FC00000u : __float_as_uint(v);
    const uint32_t ord = (b & 0x80000000u) ? ~b : (b | 0x80000000u);
    return ((unsigned long long)ord << 32) | (unsigned long long)(0xFFFFFFFFu - (uint32_t)n);
}

// ------------------------------------------------------------------------------------------------------------------
// work ranges
// ------------------------------------------------------------------------------------------------------------------

// Blocks [b0, b1) this warp streams: the CTA's share of the K/32 blocks (rank blockIdx.y of ksplit), then the warp's
// share of that.
__device__ __forceinline__ void warp_blocks(const Args &a, int warp, int &b0, int &b1) {
    const int rank = blockIdx.y;
    const int c0 = (int)((long long)a.nb * rank / a.ksplit);
    const int c1 = (int)((long long)a.nb * (rank + 1) / a.ksplit);
    b0 = c0 + (c1 - c0) * warp / kWarps;
    b1 = c0 + (c1 - c0) * (warp + 1) / kWarps;
}

// Shared-memory bytes of the epilogue: NRED partial slabs of MR rows of RS floats (TC columns used), the CTA's sum,
// the row keys.
__host__ __device__ constexpr int finish_smem_n(int NRED, int MR, int TC, int RS = 0) {
    return (NRED * MR * (RS ? RS : TC) + MR * TC) * 4 + MR * 8;
}
__host__ __device__ constexpr int finish_smem_bytes(int MR, int TC) { return finish_smem_n(kWarps, MR, TC); }

// The epilogue.  On entry the CTA's NRED partial carries sit in red[NRED][MR][RS] (rows < MR, columns < TC of this
// CTA's column tile `tile` of the output; RS >= TC is the slab row stride) and the CTA has synchronised.  Sums the
// slabs in order, then (ksplit > 1) the cluster's ranks in order, writes y (0 in the pad columns) and folds this
// CTA's columns into the per-row arg-max keys.
// The quantized form of an activation ("plan.rs", `QBLOCK`: 32 values share one scale), the rule of q8_quantize_act:
// from the bit pattern of the block's largest magnitude, d = amax / 127 (IEEE fp32 quotient), a value's code is
// value / d rounded half away from zero and clamped to 127; a block of zeros has d = 0, a block holding inf or NaN
// d = NaN, both with codes 0.
__device__ __forceinline__ float act_scale(uint32_t amax_bits) {
    if (amax_bits >= 0x7F800000u) return __uint_as_float(0x7FC00000u);
    if (amax_bits == 0u) return 0.0f;
    return __fdiv_rn(__uint_as_float(amax_bits), 127.0f);
}
// The code of v with the block's d.  The quotient is taken as v * (1 / d) (both IEEE products, at most about 2.5
// units in the last place from v / d for |v / d| < 128, i.e. below 2^-15) unless that product lies within 2^-14 of
// a half-integer, where the rounding could differ; there, and when 1 / d overflows, the IEEE quotient itself is
// used.  Both give the code of the correctly rounded quotient.
__device__ __forceinline__ float act_inv(float d) { return __frcp_rn(d); }
__device__ __forceinline__ uint32_t act_code(float v, float d, float inv, uint32_t amax_bits) {
    if (amax_bits >= 0x7F800000u || amax_bits == 0u) return 0u;
    float qv = v * inv;
    const float a = fabsf(qv);
    if (!(inv < 3.0e38f) || fabsf(a - floorf(a) - 0.5f) < 6.103515625e-05f) qv = __fdiv_rn(v, d);
    return (uint32_t)(int)fminf(fmaxf(roundf(qv), -127.0f), 127.0f) & 0xFFu;
}

// The cluster barrier after a rank's last read of the others' shared memory, which keeps every rank's shared memory
// alive until then.  Each rank's remote loads feed stores issued before it arrives (the loops below load a column only
// when they store it), so the arrival needs no release ordering: relaxed, it does not wait for the rank's global stores
// to be performed, which took the decode chain from 5,036 to 5,115 GB/s at one row and 4,069 to 4,173 at 16 (GB300,
// three runs each, one box).
__device__ __forceinline__ void cluster_sync_after_reads() {
    asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
    asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
}

// part[r][c] = the sum of the NRED slabs red[w][r][c] (row stride RS), in slab order from 0, four columns a thread
// (16-byte loads and stores: TC and RS are multiples of 4 and both buffers 16-byte aligned).
template <int NRED, int MR, int TC, int NTHREADS, int RS>
__device__ __forceinline__ void sum_slabs(const float *red, float *part, int rows) {
    static_assert(TC % 4 == 0 && RS % 4 == 0, "four columns a thread: 16-byte rows and slabs");
    constexpr int TC4 = TC / 4;
    for (int i = threadIdx.x; i < rows * TC4; i += NTHREADS) {
        const int r = i / TC4, c = 4 * (i - r * TC4);
        float4 v = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
#pragma unroll
        for (int w = 0; w < NRED; ++w) {
            const float4 p = *reinterpret_cast<const float4 *>(red + (w * MR + r) * RS + c);
            v.x += p.x;
            v.y += p.y;
            v.z += p.z;
            v.w += p.w;
        }
        *reinterpret_cast<float4 *>(part + r * TC + c) = v;
    }
}

// The sum of the four floats at buf + at in the shared memory of cluster ranks first, first + stride, ... (count of
// them), in that order from 0; eight ranks' loads are in flight before their adds.
__device__ __forceinline__ float4 cluster_sum4(cooperative_groups::cluster_group &cluster, float *buf, int at,
                                               int first, int stride, int count) {
    float4 v = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
#pragma unroll
    for (int h = 0; h < kMaxClusterRanks; h += 8) {
        if (h >= count) break;
        float4 pv[8];
#pragma unroll
        for (int j = 0; j < 8; ++j)
            if (h + j < count)
                pv[j] = *reinterpret_cast<const float4 *>(cluster.map_shared_rank(buf, first + stride * (h + j)) + at);
#pragma unroll
        for (int j = 0; j < 8; ++j)
            if (h + j < count) {
                v.x += pv[j].x;
                v.y += pv[j].y;
                v.z += pv[j].z;
                v.w += pv[j].w;
            }
    }
    return v;
}

template <int NRED, int MR, int TC, int NTHREADS, bool ARGMAX, int RS = TC>
__device__ __forceinline__ void finish_n(const Args &a, float *red, int tile) {
    namespace cg = cooperative_groups;
    constexpr int TC4 = TC / 4;
    float *part = red + NRED * MR * RS;  // [MR][TC]
    // Arg-max: up to 8 rows, the keys of this CTA's outputs (one a thread: the largest of its four columns),
    // [rows][width / 4], go over the slabs (free once `part` holds their sum) and one warp a row reduces them; 16 rows
    // fold each key into a row key in shared memory by atomicMax (measured on GB300: the warp reduction takes the tied
    // head at m = 8 from 119.4 to 114.9 us, but in the 16-row kernel its code made the main loop spill and the head
    // slower).
    constexpr bool kWarpReduce = MR <= 8;
    unsigned long long *keys = reinterpret_cast<unsigned long long *>(red);
    static_assert(NRED * RS >= 2 * TC, "the keys fit over the slabs");
    unsigned long long *rowkey = reinterpret_cast<unsigned long long *>(part + MR * TC);  // [MR]
    const int rows = a.m < MR ? a.m : MR;

    sum_slabs<NRED, MR, TC, NTHREADS, RS>(red, part, rows);
    if (ARGMAX && !kWarpReduce)
        for (int r = threadIdx.x; r < MR; r += NTHREADS) rowkey[r] = 0ull;

    const int ks = a.ksplit;
    if (ks > 1)
        cg::this_cluster().sync();
    else
        __syncthreads();

    // This rank's slice of the columns, cut at multiples of four; every rank's partial of a column is loaded before
    // any is added, and the sum is taken in rank order.
    const int rank = blockIdx.y;
    const int c0 = ks > 1 ? 4 * (TC4 * rank / ks) : 0;
    const int c1 = ks > 1 ? 4 * (TC4 * (rank + 1) / ks) : TC;
    const int width4 = (c1 - c0) / 4;
    for (int i = threadIdx.x; i < rows * width4; i += NTHREADS) {
        const int r = i / width4;
        const int c = c0 + 4 * (i - r * width4);
        const int n = tile * TC + c;  // Np is a multiple of 32: the four columns are all below it or all past it
        unsigned long long key = 0ull;
        if (n < a.Np) {
            float4 v;
            if (ks > 1) {
                cg::cluster_group cluster = cg::this_cluster();
                v = cluster_sum4(cluster, part, r * TC + c, 0, 1, ks);
            } else {
                v = *reinterpret_cast<const float4 *>(part + r * TC + c);
            }
            const float4 out = make_float4(n < a.N ? v.x : 0.0f, n + 1 < a.N ? v.y : 0.0f, n + 2 < a.N ? v.z : 0.0f,
                                           n + 3 < a.N ? v.w : 0.0f);
            if (a.y) *reinterpret_cast<float4 *>(a.y + (size_t)r * a.Np + n) = out;
            if (ARGMAX) {
                const float o4[4] = {out.x, out.y, out.z, out.w};
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    if (n + e < a.N) {
                        const unsigned long long k = argmax_key(o4[e], n + e);
                        key = key > k ? key : k;
                    }
            }
        }
        if (ARGMAX && !kWarpReduce && key) atomicMax(&rowkey[r], key);
        if (ARGMAX && kWarpReduce) keys[i] = key;
    }
    if (ARGMAX && !kWarpReduce) {
        __syncthreads();
        for (int r = threadIdx.x; r < rows; r += NTHREADS)
            if (rowkey[r]) atomicMax(&a.keys[r], rowkey[r]);
    }
    if (ARGMAX && kWarpReduce) {
        // each row's largest key by one warp (a lane's maximum over its entries, then a shuffle tree), and one
        // atomic a row into the call's keys: the maximum is the same in any order
        __syncthreads();
        constexpr int kWarpsE = NTHREADS / 32;
        const int lane = threadIdx.x & 31;
        for (int r = threadIdx.x >> 5; r < rows; r += kWarpsE) {
            unsigned long long k = 0ull;
            for (int c = lane; c < width4; c += 32) k = k > keys[r * width4 + c] ? k : keys[r * width4 + c];
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                const unsigned long long other = __shfl_xor_sync(0xffffffffu, k, o);
                k = k > other ? k : other;
            }
            if (lane == 0 && k) atomicMax(&a.keys[r], k);
        }
    }
    if (ks > 1) cluster_sync_after_reads();
}

// The gated pair's epilogue ("plan.rs", `Launch::GemvGlu`, SwiGLU: out = silu(x.wg) * (x.wu), silu(g) = g / (1 +
// exp(-g))).  The cluster is (2, ks): rank p + 2k holds part p's sums over K range k.  Each rank first sums its
// column slice over its part's K ranges (rank order), then the gate's rank of a slice reads the up projection's sums
// of the same slice and writes silu(g) * u (0 in the pad columns) to y and/or its bf16 copy.
template <int NRED, int MR, int TC, int NTHREADS, int RS = TC>
__device__ __forceinline__ void finish_glu(const Args &a, float *red, int tile) {
    namespace cg = cooperative_groups;
    cg::cluster_group cluster = cg::this_cluster();
    float *part = red + NRED * MR * RS;  // [MR][TC]: this CTA's sums over its K range
    float *mine = part + MR * TC;        // [MR][width]: this rank's slice summed over its part's K ranges
    const int rows = a.m < MR ? a.m : MR;
    sum_slabs<NRED, MR, TC, NTHREADS, RS>(red, part, rows);
    cluster.sync();
    const int ks = a.ksplit, p = blockIdx.x & 1, k = blockIdx.y;
    // slices of whole 32-column blocks (a warp then holds one block of one row for the quantized output)
    const int c0 = kBlock * ((TC / kBlock) * k / ks), c1 = kBlock * ((TC / kBlock) * (k + 1) / ks), width = c1 - c0;
    const int width4 = width / 4;
    for (int i = threadIdx.x; i < rows * width4; i += NTHREADS) {  // four columns a thread, ranks in order
        const int r = i / width4, c = c0 + 4 * (i - r * width4);
        *reinterpret_cast<float4 *>(mine + r * width + (c - c0)) = cluster_sum4(cluster, part, r * TC + c, p, 2, ks);
    }
    cluster.sync();
    if (p == 0) {
        const float *up = cluster.map_shared_rank(mine, 1 + 2 * k);
        for (int i = threadIdx.x; i < rows * width; i += NTHREADS) {
            const int r = i / width, c = c0 + (i - r * width);
            const int n = tile * TC + c;
            if (n < a.Np) {  // uniform across the warp: its 32 values are one 32-column block
                const float g = mine[i];
                const float o = n < a.N ? g / (1.0f + expf(-g)) * up[i] : 0.0f;
                const __nv_bfloat16 ob = __float2bfloat16_rn(o);
                if (a.y) a.y[(size_t)r * a.Np + n] = o;
                if (a.ybf) a.ybf[(size_t)r * a.Np + n] = __bfloat16_as_ushort(ob);
                if (a.yq) {  // the quantized form of the bf16 output
                    const float v = __bfloat162float(ob);
                    uint32_t mx = __float_as_uint(v) & 0x7FFFFFFFu;
#pragma unroll
                    for (int o2 = 16; o2 > 0; o2 >>= 1) mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o2));
                    const float d = act_scale(mx);
                    a.yq[(size_t)r * a.Np + n] = (unsigned char)act_code(v, d, act_inv(d), mx);
                    if ((n & (kBlock - 1)) == 0) a.yd[(size_t)r * (a.Np / kBlock) + n / kBlock] = d;
                }
            }
        }
    }
    cluster_sync_after_reads();  // the up projection's rank keeps its shared memory until the gate's rank has read it
}

// A projection followed by the residual add and the following RMS norm ("plan.rs", `Launch::Fold` of a projection
// with `Launch::Norm`, `gemv_norm_epilogue`: each block of the projection registers on a counter when done, and the
// block that registers last fetches every result again from L2 and normalises).  Every CTA finishes its columns as
// finish_n does, writing h = residual + y to y; then (with counters) it counts itself in.  The CTA that counts last
// reads the m rows of h back (through L2), forms each row's sum of squares in a fixed order (so the result does not
// depend on which CTA is last) and writes out = h / sqrt(mean + eps) * gamma as bf16 (0 in the pad columns).
// Nothing waits on another CTA.
template <int NRED, int MR, int TC, int NTHREADS, int RS = TC>
__device__ __forceinline__ void finish_norm(const Args &a, float *red, int tile) {
    namespace cg = cooperative_groups;
    constexpr int TC4 = TC / 4;
    float *part = red + NRED * MR * RS;  // [MR][TC]
    const int rows = a.m < MR ? a.m : MR;
    sum_slabs<NRED, MR, TC, NTHREADS, RS>(red, part, rows);
    const int ks = a.ksplit;
    if (ks > 1)
        cg::this_cluster().sync();
    else
        __syncthreads();
    // this rank's slice of the columns, cut at multiples of four, four columns a thread (the residual is read one
    // value at a time: it need only be 4-byte aligned)
    const int rank = blockIdx.y;
    const int c0 = ks > 1 ? 4 * (TC4 * rank / ks) : 0;
    const int c1 = ks > 1 ? 4 * (TC4 * (rank + 1) / ks) : TC;
    const int width4 = (c1 - c0) / 4;
    for (int i = threadIdx.x; i < rows * width4; i += NTHREADS) {
        const int r = i / width4;
        const int c = c0 + 4 * (i - r * width4);
        const int n = tile * TC + c;  // the four columns are all below Np or all past it
        if (n < a.Np) {
            float4 v;
            if (ks > 1) {
                cg::cluster_group cluster = cg::this_cluster();
                v = cluster_sum4(cluster, part, r * TC + c, 0, 1, ks);
            } else {
                v = *reinterpret_cast<const float4 *>(part + r * TC + c);
            }
            const size_t at = (size_t)r * a.Np + n;
            const float v4[4] = {v.x, v.y, v.z, v.w};
            float o4[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) o4[e] = n + e < a.N ? a.res[at + e] + v4[e] : 0.0f;
            *reinterpret_cast<float4 *>(a.y + at) = make_float4(o4[0], o4[1], o4[2], o4[3]);
        }
    }
    if (ks > 1) cluster_sync_after_reads();
    if (!a.count) return;  // the norm runs as a launch of its own (norm_rows_kernel)

    // Count in; the last CTA runs the norm.
    __shared__ unsigned int last;
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();  // this CTA's h is visible before its count
        const unsigned total = gridDim.x * gridDim.y / (unsigned)a.groups;  // this row group's CTAs
        last = atomicAdd(a.count + a.count_slot % kNormSlots, 1u) == total - 1 ? 1u : 0u;
    }
    __syncthreads();
    if (!last) return;
    __threadfence();  // every other CTA's h is visible to the reads below
    // Sums of squares: thread t takes the 16-byte column chunks t, t + NTHREADS, ... of every row at once (the
    // rows' loads are independent), then the threads' sums are added by a fixed shuffle tree and in warp order.
    constexpr int kWarpsN = NTHREADS / 32;
    const int chunks = a.Np / 4;  // Np is a multiple of 32; h is 16-byte aligned with a row pitch of Np floats
    float ss[MR];
#pragma unroll
    for (int r = 0; r < MR; ++r) ss[r] = 0.0f;
    // Rows past m read row m - 1 again (branch-free, so that every row's load is issued before the first add); their
    // sums are never used.
    for (int j = threadIdx.x; j < chunks; j += NTHREADS) {
        float4 v[MR];
#pragma unroll
        for (int r = 0; r < MR; ++r)
            v[r] = __ldcg(reinterpret_cast<const float4 *>(a.y + (size_t)(r < rows ? r : rows - 1) * a.Np) + j);
#pragma unroll
        for (int r = 0; r < MR; ++r) {
            ss[r] = fmaf(v[r].x, v[r].x, ss[r]);
            ss[r] = fmaf(v[r].y, v[r].y, ss[r]);
            ss[r] = fmaf(v[r].z, v[r].z, ss[r]);
            ss[r] = fmaf(v[r].w, v[r].w, ss[r]);
        }
    }
    float *wsum = red;              // [kWarpsN][MR]
    float *rstd = red + kWarpsN * MR;  // [MR]
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int r = 0; r < MR; ++r) {
        float v = ss[r];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
        if (lane == 0) wsum[warp * MR + r] = v;
    }
    __syncthreads();
    if (threadIdx.x < rows) {
        float v = 0.0f;
#pragma unroll
        for (int w = 0; w < kWarpsN; ++w) v += wsum[w * MR + threadIdx.x];
        rstd[threadIdx.x] = 1.0f / sqrtf(v / (float)a.N + a.eps);
    }
    __syncthreads();
    if (!a.yq) {
        // out = h * rstd * gamma as bf16, four columns a store; the pad columns get 0.
        for (int j = threadIdx.x; j < chunks; j += NTHREADS) {
            const int n = 4 * j;
            float g[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) g[e] = n + e < a.N ? a.gamma[n + e] : 0.0f;
            float4 hv[MR];
#pragma unroll
            for (int r = 0; r < MR; ++r)
                hv[r] = __ldcg(reinterpret_cast<const float4 *>(a.y + (size_t)(r < rows ? r : rows - 1) * a.Np) + j);
#pragma unroll
            for (int r = 0; r < MR; ++r)
                if (r < rows) {
                    const float4 v = hv[r];
                    const float rs = rstd[r];
                    const float o0 = n < a.N ? v.x * rs * g[0] : 0.0f;
                    const float o1 = n + 1 < a.N ? v.y * rs * g[1] : 0.0f;
                    const float o2 = n + 2 < a.N ? v.z * rs * g[2] : 0.0f;
                    const float o3 = n + 3 < a.N ? v.w * rs * g[3] : 0.0f;
                    const uint32_t lo = (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(o0)) |
                                        ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(o1)) << 16);
                    const uint32_t hi = (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(o2)) |
                                        ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(o3)) << 16);
                    *reinterpret_cast<uint2 *>(a.ybf + (size_t)r * a.Np + n) = make_uint2(lo, hi);
                }
        }
    } else {
        // With the quantized form: four columns a thread, the loop warp-uniform so that eight consecutive lanes
        // (one 32-column block; chunks is a multiple of 8) reduce the block's largest magnitude by shuffles; the
        // bf16 rows too when asked for.
        for (int j0 = threadIdx.x - lane; j0 < chunks; j0 += NTHREADS) {
            const int j = j0 + lane;
            const bool live = j < chunks;
            const int jc = live ? j : chunks - 1;
            const int n = 4 * jc;
            float g[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) g[e] = n + e < a.N ? a.gamma[n + e] : 0.0f;
            float4 hv[MR];
#pragma unroll
            for (int r = 0; r < MR; ++r)
                hv[r] = __ldcg(reinterpret_cast<const float4 *>(a.y + (size_t)(r < rows ? r : rows - 1) * a.Np) + jc);
#pragma unroll
            for (int r = 0; r < MR; ++r)
                if (r < rows) {
                    const float4 v = hv[r];
                    const float rs = rstd[r];
                    const __nv_bfloat16 b0 = __float2bfloat16_rn(n < a.N ? v.x * rs * g[0] : 0.0f);
                    const __nv_bfloat16 b1 = __float2bfloat16_rn(n + 1 < a.N ? v.y * rs * g[1] : 0.0f);
                    const __nv_bfloat16 b2 = __float2bfloat16_rn(n + 2 < a.N ? v.z * rs * g[2] : 0.0f);
                    const __nv_bfloat16 b3 = __float2bfloat16_rn(n + 3 < a.N ? v.w * rs * g[3] : 0.0f);
                    if (a.ybf && live) {
                        const uint32_t lo =
                            (uint32_t)__bfloat16_as_ushort(b0) | ((uint32_t)__bfloat16_as_ushort(b1) << 16);
                        const uint32_t hi =
                            (uint32_t)__bfloat16_as_ushort(b2) | ((uint32_t)__bfloat16_as_ushort(b3) << 16);
                        *reinterpret_cast<uint2 *>(a.ybf + (size_t)r * a.Np + n) = make_uint2(lo, hi);
                    }
                    const float v0 = __bfloat162float(b0), v1 = __bfloat162float(b1);
                    const float v2 = __bfloat162float(b2), v3 = __bfloat162float(b3);
                    uint32_t mx = max(max(__float_as_uint(v0) & 0x7FFFFFFFu, __float_as_uint(v1) & 0x7FFFFFFFu),
                                      max(__float_as_uint(v2) & 0x7FFFFFFFu, __float_as_uint(v3) & 0x7FFFFFFFu));
#pragma unroll
                    for (int o2 = 1; o2 < 8; o2 <<= 1) mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o2));
                    const float d = act_scale(mx), inv = act_inv(d);
                    const uint32_t codes = act_code(v0, d, inv, mx) | (act_code(v1, d, inv, mx) << 8) |
                                           (act_code(v2, d, inv, mx) << 16) | (act_code(v3, d, inv, mx) << 24);
                    if (live) {
                        *reinterpret_cast<uint32_t *>(a.yq + (size_t)r * a.Np + n) = codes;
                        if ((j & 7) == 0) a.yd[(size_t)r * (a.Np / kBlock) + j / 8] = d;
                    }
                }
        }
    }
    if (threadIdx.x == 0) a.count[a.count_slot % kNormSlots] = 0u;  // ready for the next launch that takes it
}

template <int MR, int TC, bool ARGMAX>
__device__ __forceinline__ void finish(const Args &a, float *smem) {
    finish_n<kWarps, MR, TC, kThreads, ARGMAX>(a, smem, blockIdx.x);
}

}  // namespace q8
