// Q8_0 GEMV over the tiled weight storage: every warp streams its own contiguous run of weight units and contracts
// them on the tensor cores with fp16 operands.
//
// The tiled storage (q8_tile) keeps every 32-row x 128-column block of the weight as one contiguous 4 KB unit in
// MMA-fragment order: eight 512-byte segments (16-row half s = 0, 1; group h = 0..3 of four 8-column slices); in
// segment (s, h) lane L = 4g + t finds at L * 16 four words, word w holding weight rows 16s + 4t + 0..3 of column
// 8(4h + w) + g, offset by +128.  The unit's 128 scales follow in their own storage, in column order.  One warp
// instruction copies 512 contiguous bytes, and the units of a column tile follow each other along K, so a warp that
// owns a run of K blocks of one tile reads one contiguous range of memory.
//
// A CTA owns one 128-column tile and a range of its K blocks (split across a thread-block cluster when N is too
// narrow to fill the SMs); its warps split that range again into contiguous runs.  Each warp keeps a private ring of
// three stages in shared memory, filled with cp.async (16 bytes a lane, bypassing L1): it issues block i + 2 while it
// computes block i, so about two units per warp -- 80 to 150 KB per SM -- are in flight without holding registers.
// The CUDA-core kernel runs 8 warps a CTA, two CTAs per SM (128 registers a thread).  The MMA kernels hold more
// registers a thread, up to 168, in 6-warp CTAs, two per SM.  Measured on GB300: the 16-row decode chain 3,690 -> 3,850
// GB/s against 8 warps at 128 registers, which spilled; 5 warps at 200 registers and 4 at 255 were slower, and so
// was one 12-warp CTA per SM, whose whole-SM CTAs cannot start beside the previous launch's.  The 8-row kernel had
// run 12 warps, one CTA per SM (10-28 % faster per launch at 4 and 8 rows than 8 warps at the 128-register cap);
// two 6-warp CTAs per SM took its chains a further 0.4-1.4 % (m = 2 4,739 -> 4,793 GB/s, m = 4 4,654 -> 4,720).
//
// The block's contraction runs on m16n8k16 MMAs with the activations as the A operand (rows r and r + 8 of the lane's
// fragment are activation rows g and g + 8) and the weights as B (one 8-column slice per MMA, fp32 accumulators):
//   - weights: the byte permute of a stored word into the low mantissa bytes of the fp16 1024 gives 1024 + q + 128
//     exactly, and one packed fp16 subtract of 1152 leaves q -- one permute and one subtract per pair of weights;
//   - activations: bf16 has a wider exponent than fp16, so each activation row of the block (m <= 8; for m > 8 the
//     whole block) is scaled by one power of two 2^p that puts its largest magnitude in [2^15, 2^16).  If every
//     nonzero activation then lies in fp16's normal range, the conversion is exact (bf16's 8 significant bits fit
//     fp16's 11) and the products q * x * 2^p are exact in fp32; the block's scale is multiplied by 2^-p (exact)
//     before the fold.  A block with a row whose nonzero activations span more than 30 binades, or that holds inf or
//     NaN, is contracted instead with bf16 operands from the raw activations, exactly as well;
//   - MMA reduction index 2t, 2t+1, 2t+8, 2t+9 is weight row 4t .. 4t+3 of the 16-row half, so a lane's activation
//     fragment is 4 consecutive activations and its weight fragment the 4 bytes of one stored word;
//   - the block's sums (fresh accumulators) are folded into the fp32 carry with the block's scales, a packed
//     fp32x2 FMA over the pair of columns a lane holds ("from_q8.rs", module doc: int8 rows contracted lane by
//     lane, each column's block sums scaled and accumulated in an fp32 carry).
//
// For one row the CUDA cores do the contraction instead (stream_simt_kernel): there the row's FMAs cost less than the
// MMA operands' conversion and the per-block exponent choice.  From two bf16 rows on the 8-row MMA kernel is the
// faster one (measured on GB300: 4096 x 14336 at two rows 17.9 us on the CUDA cores, 12.9 on the 8-row kernel); two
// rows of quantized activations stay on the CUDA cores, whose dp4a products beat it there (the decode chain 3,900
// against 3,658 GB/s).
//
// Bf16 activations of one row (the CUDA-core kernel) and of 2 .. 8 rows (the 8-row kernel) travel in the unit's ring
// stage (cp.async through L2), read back from shared memory with the unit; the 16-row kernel, quantized activations
// and row-major weights read them from L2 (ld.global.cg) into registers two blocks ahead.  With programmatic dependent
// launch every thread waits for the previous kernel (griddepcontrol.wait) before it reads x or writes y; with
// Q8_FLAG_CONSTANT_WEIGHTS the first stages' weights are already requested before that wait.
#include <atomic>

#include "q8_launch.h"

namespace q8 {

namespace {

constexpr int kWarpsS = 8;   // warps of a CTA: the CUDA-core kernel (two CTAs per SM)
constexpr int kWarps8 = 6;   //   the 8-row kernel (two CTAs per SM)
constexpr int kWarps16 = 6;  //   the 16-row kernel (two CTAs per SM)
constexpr int kThreadsS = 32 * kWarpsS;
__host__ __device__ constexpr int stream_warps(bool rows16) { return rows16 ? kWarps16 : kWarps8; }
constexpr int kUnit = kBlock * kTmaColumns;  // 4096 bytes of values per 32 x 128 unit
constexpr int kUnitScales = kTmaColumns;     // 128 fp32
constexpr int kStageS = kUnit + kUnitScales * 4;
constexpr int kDepthS = 3;                   // ring stages per warp
constexpr int kSmemS = kWarpsS * kDepthS * kStageS;
constexpr int kXPitch = 96;                  // MMA kernels: the block's activation rows (up to 16 x 32 bf16) at a
constexpr int kStageX = 16 * kXPitch;        //   row pitch that keeps a half-warp's 8-byte reads conflict-free
constexpr int kStageM = kStageS + kStageX;   //   so their stages hold the unit, its scales and those rows
constexpr int kStageS1 = kStageS + kBlock * 2;  // the CUDA-core kernel's stages with the block's one bf16 row
// The ring of a CTA of `warps` warps with stages of `stage` bytes (kStageS; kStageM and kStageS1 for the XR instances,
// whose stages also carry the block's activation rows).
__host__ __device__ constexpr int stream_smem(int warps, int stage = kStageS) { return warps * kDepthS * stage; }
constexpr int kSlices = kTmaColumns / 8;     // 8-column MMA slices of a tile
constexpr int kSlabStride = kTmaColumns + 8; // epilogue slab row stride (floats)

__device__ __forceinline__ uint32_t smem_addr(const void *p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ void cp_async16(void *dst, const void *src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N> __device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ uint2 ld_cg_u2(const void *p) {
    uint2 v;
    asm volatile("ld.global.cg.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "l"(p));
    return v;
}

__device__ __forceinline__ uint32_t ld_cg_u32(const void *p) {
    uint32_t v;
    asm volatile("ld.global.cg.u32 %0, [%1];" : "=r"(v) : "l"(p));
    return v;
}

// fp32 pairs in one 64-bit register pair.
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
__device__ __forceinline__ unsigned long long mul_f32x2(unsigned long long a, unsigned long long b) {
    unsigned long long d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

// Stored bytes E, E + 1 of a word (q + 128 each) as the exact fp16 pair {q_E, q_E+1}: the permute writes each byte
// under the fp16 exponent of 1024 (bits 0x64), whose mantissa unit is 1, giving 1024 + q + 128; the packed subtract
// of 1152 is exact.
template <int E> __device__ __forceinline__ uint32_t q8x2_to_f16x2(uint32_t u) {
    uint32_t d;
    asm("{\n .reg .b32 p;\n prmt.b32 p, %1, 0x64646464, %2;\n sub.rn.f16x2 %0, p, %3;\n}"
        : "=r"(d)
        : "r"(u), "n"(E == 0 ? 0x4140 : 0x4342), "r"(0x64806480u));
    return d;
}

// The same bytes as an exact bf16 pair (for the bf16 contraction of a block whose activations do not fit fp16):
// each byte in the low mantissa of 2^23 gives 2^23 + q + 128, one packed subtract leaves q, packed to bf16 (exact:
// |q| <= 128 needs 8 significant bits).
template <int E> __device__ __forceinline__ uint32_t q8x2_to_bf16x2(uint32_t u) {
    uint32_t d;
    asm("{\n .reg .b32 a, b;\n .reg .b64 p, r;\n .reg .f32 lo, hi;\n prmt.b32 a, %1, 0x4B000000, %2;\n"
        " prmt.b32 b, %1, 0x4B000000, %3;\n mov.b64 p, {a, b};\n sub.rn.f32x2 r, p, %4;\n mov.b64 {lo, hi}, r;\n"
        " cvt.rn.bf16x2.f32 %0, hi, lo;\n}"
        : "=r"(d)
        : "r"(u), "n"(0x7540 + E), "n"(0x7540 + E + 1), "l"(kMagicPair));
    return d;
}

// A bf16 pair scaled by the power of two `scale` (both halves of the fp32 pair) as an fp16 pair; exact when the
// caller has checked that every nonzero scaled value is an fp16 normal.
__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t x, unsigned long long scale) {
    uint32_t d;
    asm("{\n .reg .b32 lo, hi;\n .reg .b64 p, r;\n .reg .f32 a, b;\n shl.b32 lo, %1, 16;\n"
        " and.b32 hi, %1, 0xFFFF0000;\n mov.b64 p, {lo, hi};\n mul.rn.f32x2 r, p, %2;\n mov.b64 {a, b}, r;\n"
        " cvt.rn.f16x2.f32 %0, b, a;\n}"
        : "=r"(d)
        : "r"(x), "l"(scale));
    return d;
}

// A bf16 pair as an fp16 pair without scaling; exact when both are fp16 normals or zero.
__device__ __forceinline__ uint32_t bf16x2_to_f16x2_plain(uint32_t x) {
    uint32_t d;
    asm("{\n .reg .b32 lo, hi;\n shl.b32 lo, %1, 16;\n and.b32 hi, %1, 0xFFFF0000;\n cvt.rn.f16x2.f32 %0, hi, lo;\n}"
        : "=r"(d)
        : "r"(x));
    return d;
}

// Per-half unsigned 16-bit max / min / decrement.
__device__ __forceinline__ uint32_t vmax_u16x2(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("max.u16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}
__device__ __forceinline__ uint32_t vmin_u16x2(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("min.u16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}
__device__ __forceinline__ uint32_t vadd_u16x2(uint32_t a, uint32_t b) {  // per-half sum, wrapping
    uint32_t d;
    asm("add.u16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}
__device__ __forceinline__ uint32_t vdec_u16x2(uint32_t a) {  // a - 1 in each half, 0 wrapping to 0xFFFF
    return vadd_u16x2(a, 0xFFFFFFFFu);
}

// D = A * B (+ D) on fp16 or bf16 operands, fp32 accumulators; FIRST starts D from zero.
template <bool F16, bool FIRST>
__device__ __forceinline__ void mma_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    if (F16) {
        if (FIRST)
            asm(
                "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
                "{%10, %10, %10, %10};"
                : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
                : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(0.0f));
        else
            asm(
                "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
                "{%0, %1, %2, %3};"
                : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
                : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
    } else {
        if (FIRST)
            asm(
                "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
                "{%10, %10, %10, %10};"
                : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
                : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(0.0f));
        else
            asm(
                "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
                "{%0, %1, %2, %3};"
                : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
                : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
    }
}

// Copy unit `u` (values and scales) into `stage`: 8 + 1 cp.async of 16 bytes per lane.
__device__ __forceinline__ void issue_unit(unsigned char *stage, const int8_t *q, const float *s, size_t u, int lane) {
    const unsigned char *src = reinterpret_cast<const unsigned char *>(q) + u * kUnit + lane * 16;
#pragma unroll
    for (int seg = 0; seg < 8; ++seg) cp_async16(stage + seg * 512 + lane * 16, src + seg * 512);
    cp_async16(stage + kUnit + lane * 16, reinterpret_cast<const unsigned char *>(s + u * kUnitScales) + lane * 16);
}

// Row-major storage (what q8_gemv takes): block b of column tile t is rows 32b .. 32b + 31 of q [K][Np], bytes
// 128t .. 128t + 127 of each.  It lands in a stage as [32 rows][128 bytes], the 16-byte chunk c of row r at chunk
// c ^ (r & 7), so that the transposing loads below read eight rows without bank conflicts; the 128 scales of row b
// follow as in the tiled unit.  Chunks at or past Np (a ragged last tile) are zero-filled, not read.
__device__ __forceinline__ void cp_async16_zfill(void *dst, const void *src, unsigned bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_addr(dst)), "l"(src), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void issue_block_rm(unsigned char *stage, const int8_t *q, const float *s, int Np, int tile,
                                               int b, int lane) {
    const int c = lane & 7;
    const int col = kTmaColumns * tile + 16 * c;  // Np is a multiple of 32: a chunk is wholly inside or past it
    const bool ok = col < Np;
#pragma unroll
    for (int seg = 0; seg < 8; ++seg) {
        const int r = 4 * seg + (lane >> 3);
        const unsigned char *src = reinterpret_cast<const unsigned char *>(q) + (size_t)(kBlock * b + r) * Np;
        cp_async16_zfill(stage + r * 128 + ((c ^ (r & 7)) << 4), src + (ok ? col : 0), ok ? 16u : 0u);
    }
    const int sc = kTmaColumns * tile + 4 * lane;
    const bool sok = sc < Np;
    cp_async16_zfill(stage + kUnit + lane * 16, s + (size_t)b * Np + (sok ? sc : 0), sok ? 16u : 0u);
}

// The four words of the tiled unit's segment (s, h) for this lane, from a row-major stage: one transposing matrix
// load of the 16 rows 16s .. 16s + 15 and the two 16-column groups 2h, 2h + 1 gives lane (g, t) weight rows
// 16s + 4t .. + 3 of columns 32h + g, + 8, + 16 and + 24 -- the tiled word order -- and the bytes are moved from int8
// to the stored form q + 128.
__device__ __forceinline__ uint4 rm_words(const unsigned char *st, int s, int h, int lane) {
    const int row = 16 * s + (lane & 15);
    const int c = 2 * h + (lane >> 4);
    uint4 w;
    asm volatile("ldmatrix.sync.aligned.m16n16.x2.trans.shared.b8 {%0, %1, %2, %3}, [%4];"
                 : "=r"(w.x), "=r"(w.y), "=r"(w.z), "=r"(w.w)
                 : "r"(smem_addr(st + row * 128 + ((c ^ (row & 7)) << 4)))
                 : "memory");
    w.x ^= 0x80808080u;
    w.y ^= 0x80808080u;
    w.z ^= 0x80808080u;
    w.w ^= 0x80808080u;
    return w;
}

// How a block's activations enter the MMA: fp16 as they are (plain), scaled fp16, or raw bf16.  scale[i] = 2^p and
// sf[i] = 2^-p (in both halves of an fp32 pair) for the lane's activation row g + 8i.
struct XPlan {
    unsigned long long scale[2], sf[2];
    bool f16, plain;
};

// The range of the lane's activation words of one row: its largest |x| in the low half and 0xFFFF minus (its smallest
// nonzero |x| - 1) in the high half, as bf16 bit patterns, so that one per-half max combines two ranges.
__device__ __forceinline__ uint32_t row_range(const uint2 (&x)[2]) {
    uint32_t mx = 0u, mn = 0xFFFFFFFFu;
#pragma unroll
    for (int s = 0; s < 2; ++s) {
        const uint32_t v0 = x[s].x & 0x7FFF7FFFu, v1 = x[s].y & 0x7FFF7FFFu;
        mx = vmax_u16x2(mx, vmax_u16x2(v0, v1));
        mn = vmin_u16x2(mn, vmin_u16x2(vdec_u16x2(v0), vdec_u16x2(v1)));
    }
    mx = vmax_u16x2(mx, __byte_perm(mx, 0, 0x1032));
    mn = vmin_u16x2(mn, __byte_perm(mn, 0, 0x1032));
    return (mx & 0xFFFFu) | (~mn << 16);
}

// From a reduced range: whether one power of two maps every nonzero value into fp16's normal range -- all values
// finite, the largest binade at least 2^-111 (so 2^p = 2^(142 - emax) is a normal fp32) and every nonzero value
// within 29 binades below it -- or every value is zero; and the factors 2^p, 2^-p.
// plain: every value already is an fp16 normal or zero (largest binade at most 2^15, smallest nonzero at least 2^-14),
// so no scaling is needed.
__device__ __forceinline__ bool range_plan(uint32_t range, unsigned long long &scale, unsigned long long &sf,
                                           bool &plain) {
    const uint32_t xmax = range & 0xFFFFu;
    const uint32_t xmin = ((~range >> 16) & 0xFFFFu) + 1u;  // 0x10000 when every value is zero
    const int emax = (int)(xmax >> 7), emin = (int)(xmin >> 7);
    const bool zero = xmax == 0u;
    plain = zero || (emax <= 142 && emin >= 113);
    const uint32_t up = zero ? 0x3F800000u : (uint32_t)(269 - emax) << 23;
    const uint32_t down = zero ? 0x3F800000u : (uint32_t)(emax - 15) << 23;
    scale = ((unsigned long long)up << 32) | up;
    sf = ((unsigned long long)down << 32) | down;
    return zero || (xmax < 0x7F80u && emax >= 16 && emin >= 1 && emin >= emax - 29);
}

// The plan of one block from the lane's activation words x[row][half] (rows g and g + 8 when NR = 2).  PER_ROW: one
// power of two per activation row (the range over the four lanes of the row), fp16 only if every row fits; else one
// power of two for the whole block (the range over the warp).  Warp-uniform f16.
template <int NR, bool PER_ROW> __device__ __forceinline__ XPlan plan_block(const uint2 (&x)[NR][2]) {
    XPlan pl;
    if (PER_ROW) {
        uint32_t rg[NR];
#pragma unroll
        for (int r = 0; r < NR; ++r) rg[r] = row_range(x[r]);
#pragma unroll
        for (int o = 1; o < 4; o <<= 1)
#pragma unroll
            for (int r = 0; r < NR; ++r) rg[r] = vmax_u16x2(rg[r], __shfl_xor_sync(0xffffffffu, rg[r], o));
        bool ok = true, plain;
#pragma unroll
        for (int r = 0; r < 2; ++r) ok = range_plan(rg[r < NR ? r : 0], pl.scale[r], pl.sf[r], plain) && ok;
        pl.f16 = __all_sync(0xffffffffu, ok);
        pl.plain = false;
    } else {
        uint32_t rg = row_range(x[0]);
#pragma unroll
        for (int r = 1; r < NR; ++r) rg = vmax_u16x2(rg, row_range(x[r]));
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) rg = vmax_u16x2(rg, __shfl_xor_sync(0xffffffffu, rg, o));
        pl.f16 = range_plan(rg, pl.scale[0], pl.sf[0], pl.plain);
        pl.scale[1] = pl.scale[0];
        pl.sf[1] = pl.sf[0];
    }
    return pl;
}

// Whether every activation the warp holds for a block (row g, and row g + 8 when live) already is an fp16 normal:
// magnitudes in [2^-14, 2^16) as bf16 patterns 0x3880 .. 0x477F (the largest, 65280, below fp16's 65504).  Each word
// costs a mask, a packed 16-bit add of -0x3880 (in range exactly when the sum is below 0x0F00; smaller magnitudes and
// zeros wrap above it) and a packed max; one vote decides for the warp.  Blocks with zeros or other ranges take the
// full plan.
template <int NR>
__device__ __forceinline__ bool block_f16_normal(const uint2 (&x)[NR][2], bool live0, bool live1) {
    uint32_t m[NR];
#pragma unroll
    for (int r = 0; r < NR; ++r) {
        m[r] = 0u;
#pragma unroll
        for (int s = 0; s < 2; ++s)
            m[r] = vmax_u16x2(m[r], vmax_u16x2(vadd_u16x2(x[r][s].x & 0x7FFF7FFFu, 0xC780C780u),
                                               vadd_u16x2(x[r][s].y & 0x7FFF7FFFu, 0xC780C780u)));
    }
    // a dead row (at or past m) holds zeros, which would fail the range: it does not count
    uint32_t mx = live0 ? m[0] : 0u;
    if (NR == 2 && live1) mx = vmax_u16x2(mx, m[NR - 1]);
    return __all_sync(0xffffffffu, (mx & 0xFFFFu) < 0x0F00u && (mx >> 16) < 0x0F00u);
}

// One block of the warp's run: the 16 slices' MMAs over both 16-row halves and the fold into the carry.  `a` holds
// the A fragments of the two halves (fp16, or raw bf16), `pl` the factors of the block's scales (2^-p per activation
// row; unused for bf16 and for PLAIN fp16, which is unscaled), ROWS16 whether activation rows 8..15 exist and SAME
// whether both rows share 2^-p.
template <bool F16, bool ROWS16, bool SAME, bool PLAIN = false, bool RM = false>
__device__ __forceinline__ void block_contract(const unsigned char *st, int lane, const uint32_t (&a)[2][4],
                                               const XPlan &pl,
                                               unsigned long long (&acc)[ROWS16 ? 2 : 1][kSlices]) {
    const int t = lane & 3;
    const unsigned long long *sp = reinterpret_cast<const unsigned long long *>(st + kUnit) + t;
#pragma unroll
    for (int h = 0; h < 4; ++h) {
        const uint4 w0 = RM ? rm_words(st, 0, h, lane) : *reinterpret_cast<const uint4 *>(st + h * 512 + lane * 16);
        const uint4 w1 = RM ? rm_words(st, 1, h, lane)
                            : *reinterpret_cast<const uint4 *>(st + (4 + h) * 512 + lane * 16);
#pragma unroll
        for (int w = 0; w < 4; ++w) {
            const int j = 4 * h + w;
            const uint32_t u0 = word_of(w0, w), u1 = word_of(w1, w);
            float d[4];
            if (F16) {
                mma_16816<true, true>(d, a[0], q8x2_to_f16x2<0>(u0), q8x2_to_f16x2<2>(u0));
                mma_16816<true, false>(d, a[1], q8x2_to_f16x2<0>(u1), q8x2_to_f16x2<2>(u1));
            } else {
                mma_16816<false, true>(d, a[0], q8x2_to_bf16x2<0>(u0), q8x2_to_bf16x2<2>(u0));
                mma_16816<false, false>(d, a[1], q8x2_to_bf16x2<0>(u1), q8x2_to_bf16x2<2>(u1));
            }
            // the scales of columns 8j + 2t, 8j + 2t + 1 (the D fragment's columns), times the row's factor
            const unsigned long long sc = (F16 && !PLAIN) ? mul_f32x2(sp[4 * j], pl.sf[0]) : sp[4 * j];
            acc[0][j] = fma_f32x2(sc, pack_f32x2(d[0], d[1]), acc[0][j]);
            if (ROWS16) {
                const unsigned long long sc1 = (!F16 || SAME || PLAIN) ? sc : mul_f32x2(sp[4 * j], pl.sf[1]);
                acc[ROWS16 ? 1 : 0][j] = fma_f32x2(sc1, pack_f32x2(d[2], d[3]), acc[ROWS16 ? 1 : 0][j]);
            }
        }
    }
}

// QACT: x is a quantized activation (int8 values [m][K], then fp32 scales [m][K/32]); each block's A fragments are its
// int8 codes as exact fp16, its integer sums are exact in the fp32 accumulators (|sum| <= 32 * 127 * 127 < 2^24),
// and its factor per activation row is that row's scale d.
// GROUPS: m > 16, the rows in groups of 16 (grid x = tiles * groups, ROWS16 only).
// RM: the weight is row-major (q8_gemv's layout), not tiled.
// XR (bf16 activations): each block's activation rows travel in the unit's ring stage (cp.async, read back from shared
// memory once the stage has landed) instead of being loaded from L2 into registers two blocks ahead.
template <bool ROWS16, int EPI, bool QACT = false, bool GROUPS = false, bool RM = false, bool XR = false>
__global__ void __launch_bounds__(32 * stream_warps(ROWS16), 2)
    stream_kernel(Args a, const __grid_constant__ Parts parts, const int mode) {
    static_assert(ROWS16 || !GROUPS, "row groups are groups of 16 rows");
    static_assert(!(XR && QACT), "the quantized activations are loaded from L2");
    constexpr int W = stream_warps(ROWS16);
    constexpr int SS = XR ? kStageM : kStageS;  // bytes of a ring stage
    constexpr int MR = ROWS16 ? 16 : 8;
    constexpr int NR = ROWS16 ? 2 : 1;  // activation rows per lane: g and g + 8
    extern __shared__ __align__(16) unsigned char smem_s[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, t = lane & 3;
    // the activation bases of the whole launch (all m rows), before the row group's Args replace m
    const unsigned char *xq_all = reinterpret_cast<const unsigned char *>(a.x);
    const float *xd_all = reinterpret_cast<const float *>(xq_all + (size_t)a.m * a.K);
    int group;
    const int tile = select_cta<EPI, GROUPS>(parts, a, group);
    const int row0 = group * kGroupRows;
    const int rank = blockIdx.y;
    const int c0 = (int)((long long)a.nb * rank / a.ksplit);
    const int c1 = (int)((long long)a.nb * (rank + 1) / a.ksplit);
    const int b0 = c0 + (c1 - c0) * warp / W;
    const int b1 = c0 + (c1 - c0) * (warp + 1) / W;
    const int n = b1 - b0;
    unsigned char *ring = smem_s + warp * kDepthS * SS;
    const size_t unit0 = (size_t)tile * a.nb + b0;
    auto issue_w = [&](unsigned char *stage, int i) {  // block b0 + i of the tile (values, scales) into `stage`
        if constexpr (RM)
            issue_block_rm(stage, a.q, a.s, a.Np, tile, b0 + i, lane);
        else
            issue_unit(stage, a.q, a.s, unit0 + i, lane);
    };
    // The block's bf16 activation rows row0 .. row0 + MR - 1 (the launch's rows; those at or past m zero-filled) into
    // the stage after the unit, row r at r * kXPitch: four 16-byte copies a row, through L2 like the unit's.
    auto issue_x = [&](unsigned char *stage, int i) {
        if constexpr (XR) {
            unsigned char *xs = stage + kStageS;
            const size_t b = (size_t)(b0 + i);
#pragma unroll
            for (int k = 0; k < MR * 4 / 32; ++k) {
                const int c = lane + 32 * k, r = c >> 2, ch = c & 3;
                const bool ok = row0 + r < a.m;
                const uint16_t *src = a.x + (size_t)(ok ? row0 + r : 0) * a.K + b * kBlock + 8 * ch;
                cp_async16_zfill(xs + r * kXPitch + ch * 16, src, ok ? 16u : 0u);
            }
        }
    };
    auto issue = [&](unsigned char *stage, int i) {
        issue_w(stage, i);
        issue_x(stage, i);
    };

    // acc[i][j]: rows g + 8i, columns 8j + 2t and 8j + 2t + 1 of the tile
    unsigned long long acc[NR][kSlices];
#pragma unroll
    for (int i = 0; i < NR; ++i)
#pragma unroll
        for (int j = 0; j < kSlices; ++j) acc[i][j] = 0ull;

    // Prologue: the first kDepthS - 1 units (one commit group each, empty past the run).  Requested before the
    // dependency wait, a unit's weights go first and (XR) its activation rows, which the previous kernel may still be
    // writing, after the wait in a group of their own: the loop's wait for unit i (at most kDepthS - 1 later groups
    // pending) then covers both.
    const bool early = (mode & (kModePrefetch | kModeDeferWait)) != 0;  // weights requested before any wait
    if (early) {
#pragma unroll
        for (int i = 0; i < kDepthS - 1; ++i) {
            if (i < n) issue_w(ring + i * SS, i);
            cp_async_commit();
        }
    }
    if (!(mode & kModeDeferWait)) asm volatile("griddepcontrol.wait;" ::: "memory");
    if (mode & kModeRelease) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    if (XR || !early) {
#pragma unroll
        for (int i = 0; i < kDepthS - 1; ++i) {
            if (i < n) {
                if (!early) issue_w(ring + i * SS, i);
                issue_x(ring + i * SS, i);
            }
            cp_async_commit();
        }
    }

    // The lane's activations x[g + 8i][32b + 16s + 4t .. + 3] (rows at or past m are zeros): XR from the unit's
    // stage; otherwise from L2, two blocks ahead (QACT: [i][0] holds the two int8 words (s = 0, 1) and [i][1].x the
    // bits of the row's block scale).
    const uint16_t *xrow[NR];
    const unsigned char *qrow[NR];
    const float *drow[NR];
    bool xlive[NR];
#pragma unroll
    for (int i = 0; i < NR; ++i) {
        const int r = row0 + g + 8 * i;  // the launch's row (m is still the launch's here)
        xlive[i] = r < a.m;
        const size_t rr = (size_t)(xlive[i] ? r : 0);
        xrow[i] = a.x + rr * a.K + 4 * t;
        qrow[i] = xq_all + rr * a.K + 4 * t;
        drow[i] = xd_all + rr * a.nb;
    }
    uint2 xn1[NR][2], xn2[NR][2];  // blocks i + 1 and i + 2
    auto load_x = [&](uint2 (&dst)[NR][2], int b) {
#pragma unroll
        for (int i = 0; i < NR; ++i) {
            if constexpr (QACT) {
                const unsigned char *p = qrow[i] + (size_t)b * kBlock;
                dst[i][0] = xlive[i] ? make_uint2(ld_cg_u32(p), ld_cg_u32(p + 16)) : make_uint2(0u, 0u);
                dst[i][1] = make_uint2(xlive[i] ? ld_cg_u32(drow[i] + b) : 0u, 0u);
            } else {
#pragma unroll
                for (int s = 0; s < 2; ++s)
                    dst[i][s] = xlive[i] ? ld_cg_u2(xrow[i] + (size_t)b * kBlock + 16 * s) : make_uint2(0u, 0u);
            }
        }
    };
    if constexpr (!XR) {
        if (n > 0) load_x(xn1, b0);
        if (n > 1) load_x(xn2, b0 + 1);
    }

    // Stage indices: counted round for the 16-row kernel (measured faster there), i % depth for the 8-row one (its
    // register allocation is at its limit; the counters cost it more than they save).
    int cur = 0, nxt = kDepthS - 1;
    for (int i = 0; i < n; ++i) {
        const int ahead = i + kDepthS - 1;
        if (ahead < n)
            issue(ring + (ROWS16 ? nxt : ahead % kDepthS) * SS, ahead);
        cp_async_commit();
        uint2 xc[NR][2];
        XPlan plan;
        bool f16_normal = false;  // 16-row kernel: every live activation already an fp16 normal (no plan needed)
        if constexpr (!XR) {
#pragma unroll
            for (int r = 0; r < NR; ++r)
#pragma unroll
                for (int s = 0; s < 2; ++s) {
                    xc[r][s] = xn1[r][s];
                    xn1[r][s] = xn2[r][s];
                }
            if (i + 2 < n) load_x(xn2, b0 + i + 2);
            if constexpr (QACT) {
                plan.sf[0] = pack_f32x2(__uint_as_float(xc[0][1].x), __uint_as_float(xc[0][1].x));
                plan.sf[1] = pack_f32x2(__uint_as_float(xc[NR - 1][1].x), __uint_as_float(xc[NR - 1][1].x));
            } else if constexpr (ROWS16) {
                f16_normal = block_f16_normal<NR>(xc, xlive[0], xlive[NR - 1]);
                if (!f16_normal) plan = plan_block<NR, false>(xc);
            } else {
                plan = plan_block<NR, true>(xc);
            }
        }

        cp_async_wait<kDepthS - 1>();  // this lane's copies of unit i have landed
        __syncwarp();                  // ... and every other lane's
        const unsigned char *st = ring + (ROWS16 ? cur : i % kDepthS) * SS;
        if (ROWS16) {
            cur = cur == kDepthS - 1 ? 0 : cur + 1;
            nxt = nxt == kDepthS - 1 ? 0 : nxt + 1;
        }
        if constexpr (XR) {
#pragma unroll
            for (int r = 0; r < NR; ++r) {
                const unsigned char *row = st + kStageS + (g + 8 * r) * kXPitch;
                xc[r][0] = *reinterpret_cast<const uint2 *>(row + 8 * t);       // values 4t .. 4t + 3
                xc[r][1] = *reinterpret_cast<const uint2 *>(row + 32 + 8 * t);  // values 16 + 4t .. 16 + 4t + 3
            }
            if constexpr (ROWS16) {
                f16_normal = block_f16_normal<NR>(xc, xlive[0], xlive[NR - 1]);
                if (!f16_normal) plan = plan_block<NR, false>(xc);
            } else {
                plan = plan_block<NR, true>(xc);
            }
        }
        if constexpr (QACT) {
            // int8 codes as the stored-weight form (x + 128 = x ^ 0x80 per byte), then the same exact fp16 pairs
            uint32_t af[2][4];
#pragma unroll
            for (int s = 0; s < 2; ++s) {
                const uint32_t u0 = (s ? xc[0][0].y : xc[0][0].x) ^ 0x80808080u;
                const uint32_t u1 = (s ? xc[NR - 1][0].y : xc[NR - 1][0].x) ^ 0x80808080u;
                af[s][0] = q8x2_to_f16x2<0>(u0);
                af[s][2] = q8x2_to_f16x2<2>(u0);
                af[s][1] = ROWS16 ? q8x2_to_f16x2<0>(u1) : 0u;
                af[s][3] = ROWS16 ? q8x2_to_f16x2<2>(u1) : 0u;
            }
            block_contract<true, ROWS16, false, false, RM>(st, lane, af, plan, acc);
        } else if (ROWS16 && (f16_normal || plan.plain)) {
            uint32_t af[2][4];
#pragma unroll
            for (int s = 0; s < 2; ++s) {
                af[s][0] = bf16x2_to_f16x2_plain(xc[0][s].x);
                af[s][2] = bf16x2_to_f16x2_plain(xc[0][s].y);
                af[s][1] = ROWS16 ? bf16x2_to_f16x2_plain(xc[NR - 1][s].x) : 0u;
                af[s][3] = ROWS16 ? bf16x2_to_f16x2_plain(xc[NR - 1][s].y) : 0u;
            }
            block_contract<true, ROWS16, ROWS16, true, RM>(st, lane, af, plan, acc);
        } else if (plan.f16) {
            uint32_t af[2][4];
#pragma unroll
            for (int s = 0; s < 2; ++s) {
                af[s][0] = bf16x2_to_f16x2(xc[0][s].x, plan.scale[0]);
                af[s][2] = bf16x2_to_f16x2(xc[0][s].y, plan.scale[0]);
                af[s][1] = ROWS16 ? bf16x2_to_f16x2(xc[NR - 1][s].x, plan.scale[1]) : 0u;
                af[s][3] = ROWS16 ? bf16x2_to_f16x2(xc[NR - 1][s].y, plan.scale[1]) : 0u;
            }
            block_contract<true, ROWS16, ROWS16, false, RM>(st, lane, af, plan, acc);
        } else {
            uint32_t ab[2][4];
#pragma unroll
            for (int s = 0; s < 2; ++s) {
                ab[s][0] = xc[0][s].x;
                ab[s][2] = xc[0][s].y;
                ab[s][1] = ROWS16 ? xc[NR - 1][s].x : 0u;
                ab[s][3] = ROWS16 ? xc[NR - 1][s].y : 0u;
            }
            block_contract<false, ROWS16, ROWS16, false, RM>(st, lane, ab, plan, acc);
        }
        __syncwarp();  // every lane is done with this stage before it is refilled
    }
    cp_async_wait<0>();
    if (!(mode & kModeRelease)) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    __syncthreads();  // every warp is done with its ring: the shared memory holds the epilogue now

    // [W][MR][kSlabStride]: rows padded by 8 floats, so that a half-warp's 8-byte stores (rows g, columns
    // 8j + 2t) fall on 32 distinct banks
    float *red = reinterpret_cast<float *>(smem_s);
    float *mine = red + warp * MR * kSlabStride;
#pragma unroll
    for (int r = 0; r < NR; ++r)
#pragma unroll
        for (int j = 0; j < kSlices; ++j) {
            float lo, hi;
            unpack_f32x2(acc[r][j], lo, hi);
            *reinterpret_cast<float2 *>(mine + (g + 8 * r) * kSlabStride + 8 * j + 2 * t) = make_float2(lo, hi);
        }
    __syncthreads();
    apply_cta_group<EPI, GROUPS>(a);
    if constexpr (EPI == kEpiGlu)
        finish_glu<W, MR, kTmaColumns, 32 * W, kSlabStride>(a, red, tile);
    else if constexpr (EPI == kEpiNorm)
        finish_norm<W, MR, kTmaColumns, 32 * W, kSlabStride>(a, red, tile);
    else
        finish_n<W, MR, kTmaColumns, 32 * W, EPI == kEpiArgmax, kSlabStride>(a, red, tile);
    if (mode & kModeDeferWait) asm volatile("griddepcontrol.wait;" ::: "memory");  // the first half has completed
}

// M rows on CUDA cores (one row; two of quantized activations): in segment (s, h) lane (g, t) holds words w = 0..3,
// each four weight rows 16s + 4t + 0..3 of column 8(4h + w) + g; they meet the lane's four activations of each row
// with two packed fp32x2 FMAs (exact products), the block's sums of a column are folded with its scale, and at the
// end the four lanes t of a column add their carries.
// Stored bytes E, E + 1 of a word as the exact fp32 pair {q_E, q_E+1}: each byte in the low mantissa of 2^23 gives
// 2^23 + q + 128, and one packed subtract of 2^23 + 128 leaves q.
template <int E> __device__ __forceinline__ unsigned long long q8x2_to_f32x2(uint32_t u) {
    unsigned long long d;
    asm("{\n .reg .b32 a, b;\n .reg .b64 p;\n prmt.b32 a, %1, 0x4B000000, %2;\n prmt.b32 b, %1, 0x4B000000, %3;\n"
        " mov.b64 p, {a, b};\n sub.rn.f32x2 %0, p, %4;\n}"
        : "=l"(d)
        : "r"(u), "n"(0x7540 + E), "n"(0x7540 + E + 1), "l"(kMagicPair));
    return d;
}

// dp4a with unsigned bytes in a (the stored weights, q + 128) and signed bytes in b: c + sum a_i * b_i.
__device__ __forceinline__ int dp4a_us(uint32_t a, uint32_t b, int c) {
    int d;
    asm("dp4a.u32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

// QACT (quantized activations): the lane's eight codes of a row and block meet each column's eight stored
// bytes in two dp4a (integer products, exact); the offset is removed by starting the sum at -128 times the sum of the
// eight codes, the exact integer is converted to fp32 and folded with s[b, n] * d[r, b].
// XR (one bf16 row, tiled weights): the block's row travels in the unit's ring stage, as in the 8-row kernel.
template <int M, int EPI, bool QACT = false, bool RM = false, bool XR = false>
__global__ void __launch_bounds__(kThreadsS, 2)
    stream_simt_kernel(Args a, const __grid_constant__ Parts parts, const int mode) {
    static_assert(!XR || (M == 1 && !QACT && !RM), "the staged row: one bf16 row of tiled weights");
    constexpr int SS = XR ? kStageS1 : kStageS;  // bytes of a ring stage
    extern __shared__ __align__(16) unsigned char smem_s[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, t = lane & 3;
    int group;  // one row group
    const int tile = select_cta<EPI, false>(parts, a, group);
    const int rank = blockIdx.y;
    const int c0 = (int)((long long)a.nb * rank / a.ksplit);
    const int c1 = (int)((long long)a.nb * (rank + 1) / a.ksplit);
    const int b0 = c0 + (c1 - c0) * warp / kWarpsS;
    const int b1 = c0 + (c1 - c0) * (warp + 1) / kWarpsS;
    const int n = b1 - b0;
    unsigned char *ring = smem_s + warp * kDepthS * SS;
    const size_t unit0 = (size_t)tile * a.nb + b0;
    auto issue_w = [&](unsigned char *stage, int i) {  // block b0 + i of the tile (values, scales) into `stage`
        if constexpr (RM)
            issue_block_rm(stage, a.q, a.s, a.Np, tile, b0 + i, lane);
        else
            issue_unit(stage, a.q, a.s, unit0 + i, lane);
    };
    auto issue_x = [&](unsigned char *stage, int i) {  // XR: the block's 64 bytes of the row, after the unit
        if constexpr (XR)
            if (lane < 4) cp_async16(stage + kStageS + 16 * lane, a.x + (size_t)(b0 + i) * kBlock + 8 * lane);
    };
    auto issue = [&](unsigned char *stage, int i) {
        issue_w(stage, i);
        issue_x(stage, i);
    };

    unsigned long long acc[M][kSlices];  // per row and column 8j + g: the carry of rows 4t, 4t+2 | 4t+1, 4t+3
    float accq[M][kSlices];              // QACT: per row and column 8j + g, the carry of the lane's rows
#pragma unroll
    for (int r = 0; r < M; ++r)
#pragma unroll
        for (int j = 0; j < kSlices; ++j) {
            acc[r][j] = 0ull;
            accq[r][j] = 0.0f;
        }

    // All kDepthS stages are requested before the dependency wait (unit i + kDepthS is requested once unit i is done):
    // measured on GB300, the one-row decode chain 5,003 -> 5,066 GB/s against requesting kDepthS - 1 first; the MMA
    // kernels keep the request at the top of the loop (there the same change lost 1-12%).
    // (XR: the rows of those stages follow after the wait, in groups of their own: the loop's wait for unit i, with at
    // most kDepthS - 1 later groups pending, covers its row too.)
    const bool early = (mode & (kModePrefetch | kModeDeferWait)) != 0;  // weights requested before any wait
    if (early) {
#pragma unroll
        for (int i = 0; i < kDepthS; ++i) {
            if (i < n) issue_w(ring + i * SS, i);
            cp_async_commit();
        }
    }
    if (!(mode & kModeDeferWait)) asm volatile("griddepcontrol.wait;" ::: "memory");
    if (mode & kModeRelease) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    if (XR || !early) {
#pragma unroll
        for (int i = 0; i < kDepthS; ++i) {
            if (i < n) {
                if (!early) issue_w(ring + i * SS, i);
                issue_x(ring + i * SS, i);
            }
            cp_async_commit();
        }
    }

    // QACT: [r][0] holds the row's two code words (s = 0, 1), [r][1].x the bits of its block scale
    const unsigned char *xq = reinterpret_cast<const unsigned char *>(a.x);
    const float *xd = reinterpret_cast<const float *>(xq + (size_t)a.m * a.K);
    uint2 xn1[M][2], xn2[M][2];
    auto load_x = [&](uint2 (&dst)[M][2], int b) {
#pragma unroll
        for (int r = 0; r < M; ++r) {
            if constexpr (QACT) {
                const unsigned char *p = xq + (size_t)r * a.K + (size_t)b * kBlock + 4 * t;
                dst[r][0] = make_uint2(ld_cg_u32(p), ld_cg_u32(p + 16));
                dst[r][1] = make_uint2(ld_cg_u32(xd + (size_t)r * a.nb + b), 0u);
            } else {
#pragma unroll
                for (int s = 0; s < 2; ++s)
                    dst[r][s] = ld_cg_u2(a.x + (size_t)r * a.K + (size_t)b * kBlock + 16 * s + 4 * t);
            }
        }
    };
    if constexpr (!XR) {
        if (n > 0) load_x(xn1, b0);
        if (n > 1) load_x(xn2, b0 + 1);
    }

    for (int i = 0; i < n; ++i) {
        uint2 xc[M][2];
        if constexpr (!XR) {
#pragma unroll
            for (int r = 0; r < M; ++r)
#pragma unroll
                for (int s = 0; s < 2; ++s) {
                    xc[r][s] = xn1[r][s];
                    xn1[r][s] = xn2[r][s];
                }
            if (i + 2 < n) load_x(xn2, b0 + i + 2);
        }
        if constexpr (QACT) {
            int base[M];  // -128 * (the lane's eight codes of the row summed)
#pragma unroll
            for (int r = 0; r < M; ++r)
                base[r] = -128 * dp4a_us(0x01010101u, xc[r][0].y, dp4a_us(0x01010101u, xc[r][0].x, 0));
            cp_async_wait<kDepthS - 1>();
            __syncwarp();
            const unsigned char *st = ring + (i % kDepthS) * SS;
            const float *ss = reinterpret_cast<const float *>(st + kUnit) + g;
#pragma unroll
            for (int h = 0; h < 4; ++h) {
                const uint4 w0 = RM ? rm_words(st, 0, h, lane)
                                    : *reinterpret_cast<const uint4 *>(st + h * 512 + lane * 16);
                const uint4 w1 = RM ? rm_words(st, 1, h, lane)
                                    : *reinterpret_cast<const uint4 *>(st + (4 + h) * 512 + lane * 16);
#pragma unroll
                for (int w = 0; w < 4; ++w) {
                    const int j = 4 * h + w;
                    const float sv = ss[8 * j];
#pragma unroll
                    for (int r = 0; r < M; ++r) {
                        const int p = dp4a_us(word_of(w1, w), xc[r][0].y, dp4a_us(word_of(w0, w), xc[r][0].x, base[r]));
                        accq[r][j] = fmaf(sv * __uint_as_float(xc[r][1].x), (float)p, accq[r][j]);
                    }
                }
            }
            __syncwarp();  // every lane is done with this stage: it takes unit i + kDepthS
            if (i + kDepthS < n) issue(ring + (i % kDepthS) * SS, i + kDepthS);
            cp_async_commit();
            continue;
        }
        if constexpr (XR) {  // the row's values 4t .. 4t + 3 and 16 + 4t .. 16 + 4t + 3, once the stage has landed
            cp_async_wait<kDepthS - 1>();
            __syncwarp();
            const unsigned char *xs = ring + (i % kDepthS) * SS + kStageS;
            xc[0][0] = *reinterpret_cast<const uint2 *>(xs + 8 * t);
            xc[0][1] = *reinterpret_cast<const uint2 *>(xs + 32 + 8 * t);
        }
        // activations as fp32 pairs {x[4t], x[4t+1]} and {x[4t+2], x[4t+3]} of each row and half
        unsigned long long xp[M][2][2];
#pragma unroll
        for (int r = 0; r < M; ++r)
#pragma unroll
            for (int s = 0; s < 2; ++s) {
                xp[r][s][0] = pack_f32x2(bf16_lo(xc[r][s].x), bf16_hi(xc[r][s].x));
                xp[r][s][1] = pack_f32x2(bf16_lo(xc[r][s].y), bf16_hi(xc[r][s].y));
            }
        if constexpr (!XR) {
            cp_async_wait<kDepthS - 1>();
            __syncwarp();
        }
        const unsigned char *st = ring + (i % kDepthS) * SS;
        const float *ss = reinterpret_cast<const float *>(st + kUnit) + g;
        // per group h of four slices: both 16-row halves, then the fold, so that only four slices' block sums are
        // live at a time (each slice's operations run in the same order as half by half over all slices)
#pragma unroll
        for (int h = 0; h < 4; ++h) {
            const uint4 w0 = RM ? rm_words(st, 0, h, lane)
                                : *reinterpret_cast<const uint4 *>(st + h * 512 + lane * 16);
            const uint4 w1 = RM ? rm_words(st, 1, h, lane)
                                : *reinterpret_cast<const uint4 *>(st + (4 + h) * 512 + lane * 16);
#pragma unroll
            for (int w = 0; w < 4; ++w) {
                const int j = 4 * h + w;
                const uint32_t u0 = word_of(w0, w), u1 = word_of(w1, w);
                const unsigned long long q01a = q8x2_to_f32x2<0>(u0), q23a = q8x2_to_f32x2<2>(u0);
                const unsigned long long q01b = q8x2_to_f32x2<0>(u1), q23b = q8x2_to_f32x2<2>(u1);
                const float sv = ss[8 * j];
                const unsigned long long s2 = pack_f32x2(sv, sv);
#pragma unroll
                for (int r = 0; r < M; ++r) {
                    unsigned long long part = mul_f32x2(q01a, xp[r][0][0]);
                    part = fma_f32x2(q23a, xp[r][0][1], part);
                    part = fma_f32x2(q01b, xp[r][1][0], part);
                    part = fma_f32x2(q23b, xp[r][1][1], part);
                    acc[r][j] = fma_f32x2(s2, part, acc[r][j]);
                }
            }
        }
        __syncwarp();  // every lane is done with this stage: it takes unit i + kDepthS
        if (i + kDepthS < n) issue(ring + (i % kDepthS) * SS, i + kDepthS);
        cp_async_commit();
    }
    cp_async_wait<0>();
    if (!(mode & kModeRelease)) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    __syncthreads();

    float *red = reinterpret_cast<float *>(smem_s);  // [kWarpsS][M][128]
    float *mine = red + warp * M * kTmaColumns;
#pragma unroll
    for (int r = 0; r < M; ++r)
#pragma unroll
        for (int j = 0; j < kSlices; ++j) {
            float lo, hi;
            unpack_f32x2(acc[r][j], lo, hi);
            float v = QACT ? accq[r][j] : lo + hi;
            v += __shfl_xor_sync(0xffffffffu, v, 1);
            v += __shfl_xor_sync(0xffffffffu, v, 2);
            if (t == 0) mine[r * kTmaColumns + 8 * j + g] = v;
        }
    __syncthreads();
    apply_cta_group<EPI, false>(a);
    if constexpr (EPI == kEpiGlu)
        finish_glu<kWarpsS, M, kTmaColumns, kThreadsS>(a, red, tile);
    else if constexpr (EPI == kEpiNorm)
        finish_norm<kWarpsS, M, kTmaColumns, kThreadsS>(a, red, tile);
    else
        finish_n<kWarpsS, M, kTmaColumns, kThreadsS, EPI == kEpiArgmax>(a, red, tile);
    if (mode & kModeDeferWait) asm volatile("griddepcontrol.wait;" ::: "memory");  // the first half has completed
}

static_assert(finish_smem_n(kWarps16, 16, kTmaColumns, kSlabStride) <= stream_smem(kWarps16), "the epilogue fits");
static_assert((kWarps16 * 16 * kSlabStride + 2 * 16 * kTmaColumns) * 4 <= stream_smem(kWarps16),
              "the gated pair's epilogue fits");
static_assert(finish_smem_n(kWarpsS, 2, kTmaColumns) <= kSmemS, "the CUDA-core kernel's epilogue fits");
static_assert(2 * kSmemS <= 227 * 1024 && 2 * stream_smem(kWarps16) <= 227 * 1024, "two CTAs per SM");
static_assert(finish_smem_n(kWarps8, 8, kTmaColumns, kSlabStride) <= stream_smem(kWarps8), "8-row epilogue fits");
static_assert((kWarps8 * 8 * kSlabStride + 2 * 8 * kTmaColumns) * 4 <= stream_smem(kWarps8), "8-row gated pair fits");
static_assert(2 * stream_smem(kWarps8) <= 227 * 1024, "two 8-row CTAs per SM");
static_assert(2 * stream_smem(kWarps8, kStageM) <= 227 * 1024 && 2 * stream_smem(kWarpsS, kStageS1) <= 227 * 1024,
              "two CTAs per SM whose stages carry the activation rows");
// The shared memory of a launch held to one CTA per SM beside one ordinary CTA of the same kernel (the CUDA-core
// kernel's 8 warps, the MMA kernels' 6): two such CTAs (each with its 1 KB reserve) exceed the SM's 228 KB, one of
// them and an ordinary one do not.
constexpr int kSmemOnePerSm = 114 * 1024;
static_assert(stream_smem(kWarps8, kStageM) <= kSmemOnePerSm && stream_smem(kWarpsS, kStageS1) <= kSmemOnePerSm &&
                  kSmemOnePerSm + stream_smem(kWarpsS, kStageS1) + 2 * 1024 <= 228 * 1024,
              "a one-per-SM CTA holds the stages with the activation rows, beside an ordinary one");
static_assert(2 * (kSmemOnePerSm + 1024) > 228 * 1024 && kSmemOnePerSm + kSmemS + 2 * 1024 <= 228 * 1024,
              "one such CTA and one ordinary CTA per SM");

template <typename Kernel>
cudaError_t launch_stream_kernel(Kernel kernel, int warps, int stage, const Args &a, const Parts &pt,
                                 cudaStream_t stream, bool pdl, int mode, bool pair, StreamGrid grid) {
    const int smem = grid.one_per_sm ? kSmemOnePerSm : stream_smem(warps, stage);
    // the attribute is the largest size any launch of the kernel asks for, so that concurrent callers agree on it
    const int smem_max = kSmemOnePerSm;
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_max);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
    if (e != cudaSuccess) return e;
    if (a.ksplit * (pair ? 2 : 1) > 8) {  // clusters above the portable 8 CTAs (up to 16 on this GPU)
        e = cudaFuncSetAttribute(kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        if (e != cudaSuccess) return e;
    }
    cudaLaunchConfig_t cfg = {};
    const unsigned groups = (unsigned)((a.m + kGroupRows - 1) / kGroupRows);
    const unsigned ntiles = grid.ntiles > 0 ? (unsigned)grid.ntiles : (unsigned)pt.tile_end[pt.count - 1];
    cfg.gridDim = dim3(ntiles * groups, (unsigned)a.ksplit, 1);
    cfg.blockDim = dim3(32 * (unsigned)warps, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    int na = 0;
    if (a.ksplit > 1 || pair) {
        attr[na].id = cudaLaunchAttributeClusterDimension;
        attr[na].val.clusterDim.x = pair ? 2 : 1;
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
    return cudaLaunchKernelEx(&cfg, kernel, a, pt, mode);
}

}  // namespace

// The completion counters of the residual norm's one-launch fold: the library's only scratch memory, static so that
// the entry point allocates nothing.  Each row group of a launch takes one counter (round robin over the calls); the
// group's last CTA leaves it at 0 again.
__device__ __align__(256) unsigned int g_norm_count[kNormSlots];

unsigned int *norm_counters() {
    void *base = nullptr;
    if (cudaGetSymbolAddress(&base, g_norm_count) != cudaSuccess) return nullptr;
    return static_cast<unsigned int *>(base);
}

// The 8-row kernel takes 2 .. 8 rows of tiled weights (3 .. 8 of quantized activations).  Row-major weights take the
// 16-row kernel from 2 rows: measured on GB300, its row-major instances do not spill where the 8-row kernel's do (12
// to 24 bytes at the 168-register cap), and the row-major product at 2, 4 and 8 rows ran 4-14% faster on five of the
// six shapes of the sweep (5120 x 6144 at m = 8 12.56 -> 10.90 us, 14336 x 4096 16.94 -> 15.59) and within 2% on
// 4096 x 14336; on tiled weights the 16-row kernel was up to 12% slower there.  Every stream kernel runs two CTAs per
// SM.
bool rows8_family(int m, bool qact, bool rowmajor = false) {
    return !rowmajor && ((m >= 3 && m <= 8) || (m == 2 && !qact));
}
int stream_ctas_per_sm(int, bool, bool) { return 2; }

int stream_max_clusters(int m, bool qact, int ks, bool rowmajor) {
    // Clusters of ks CTAs are placed within one GPC, so fewer of them fit at once than slots / ks.  Asked once per
    // device, kernel shape and size (a deterministic answer: concurrent first calls store the same value) of the
    // family's main instance; the stream kernels of one family (CUDA-core: 8 warps; 8-row and 16-row: 6 warps; two
    // CTAs per SM each) have the same block size and register cap, and shared memory within 2% of it.
    static std::atomic<int> cache[64][3][kMaxStreamSplit + 1];  // 0: not asked yet; else the count + 1
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64 || ks < 1 || ks > kMaxStreamSplit) return 0;
    const int fam = rows8_family(m, qact, rowmajor) ? 1 : (m == 1 || (m == 2 && qact)) ? 0 : 2;
    const int known = cache[dev][fam][ks].load(std::memory_order_relaxed);
    if (known > 0) return known - 1;
    auto kernel = fam == 1   ? stream_kernel<false, kEpiStore, false, false, false, true>
                  : fam == 2 ? stream_kernel<true, kEpiStore>
                             : stream_simt_kernel<1, kEpiStore, false, false, true>;
    const int warps = fam == 1 ? kWarps8 : fam == 2 ? kWarps16 : kWarpsS;
    const int smem = stream_smem(warps, fam == 1 ? kStageM : fam == 2 ? kStageS : kStageS1);
    int n = 0;
    bool ok = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                   kSmemOnePerSm) == cudaSuccess &&  // as launch_stream_kernel sets it
              cudaFuncSetAttribute(kernel, cudaFuncAttributePreferredSharedMemoryCarveout, 100) == cudaSuccess &&
              (ks <= 8 || cudaFuncSetAttribute(kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) ==
                              cudaSuccess);
    if (ok) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(1, (unsigned)ks, 1);
        cfg.blockDim = dim3(32 * (unsigned)warps, 1, 1);
        cfg.dynamicSmemBytes = smem;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 1;
        attr[0].val.clusterDim.y = (unsigned)ks;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = ks > 1 ? 1 : 0;
        ok = cudaOccupancyMaxActiveClusters(&n, kernel, &cfg) == cudaSuccess;
    }
    if (!ok) {
        cudaGetLastError();  // the failed query's error is not the caller's
        return 0;
    }
    cache[dev][fam][ks].store(n + 1, std::memory_order_relaxed);
    return n;
}

template <int EPI>
cudaError_t launch_stream_epi(const Args &a, const Parts &pt, cudaStream_t stream, bool pdl, int mode, bool qact,
                              bool rowmajor, StreamGrid grid) {
    const bool pair = EPI == kEpiGlu;
    if ((grid.ntiles > 0 || a.tile0 != 0) && (EPI == kEpiNorm || a.m > kGroupRows || (pair && (a.tile0 & 1))))
        return cudaErrorInvalidValue;  // a part of the tiles: store, arg-max and gated-pair launches of one row group

    auto go = [&](auto kernel, int stage = kStageS) {
        return launch_stream_kernel(kernel, kWarpsS, stage, a, pt, stream, pdl, mode, pair, grid);
    };
    auto go8 = [&](auto kernel, int stage = kStageS) {
        return launch_stream_kernel(kernel, kWarps8, stage, a, pt, stream, pdl, mode, pair, grid);
    };
    auto go16 = [&](auto kernel, int stage = kStageS) {
        return launch_stream_kernel(kernel, kWarps16, stage, a, pt, stream, pdl, mode, pair, grid);
    };
    if constexpr (EPI == kEpiStore || EPI == kEpiArgmax) {
        if (rowmajor) {  // at most 16 rows, bf16 activations
            if (qact || a.m > kGroupRows) return cudaErrorInvalidValue;
            if (a.m == 1) return go(stream_simt_kernel<1, EPI, false, true>);
            return go16(stream_kernel<true, EPI, false, false, true>);
        }
    } else if (rowmajor) {
        return cudaErrorInvalidValue;  // the fused epilogues take the tiled storage
    }
    if (qact) {
        if (a.m == 1) return go(stream_simt_kernel<1, EPI, true>);
        if (a.m == 2) return go(stream_simt_kernel<2, EPI, true>);
        if (a.m <= 8) return go8(stream_kernel<false, EPI, true>);
        if (a.m <= kGroupRows) return go16(stream_kernel<true, EPI, true>);
        return go16(stream_kernel<true, EPI, true, true>);
    }
    // 2 .. 8 bf16 rows take their activations through the ring stages (XR).  Measured on GB300 against loading them
    // into registers two blocks ahead: the decode chain at m = 2 4,777 -> 5,008 GB/s and at m = 8 4,574 -> 4,843, every
    // launch kind 4-9% faster.  The 16-row kernel keeps the registers: alone its long launches gained as much (the
    // head at m = 16 -8%, gate/up -4%, down -5%), but its chain fell 4,162 -> 4,090 GB/s.
    // One bf16 row: through the ring stages too (the one-row chain 5,123 -> 5,143 GB/s), but for the two launches of a
    // plain product split in two (the gate/up pair), which keep the register loads (5,143 -> 5,210).
    if (a.m == 1) {
        if (EPI == kEpiStore && (grid.ntiles > 0 || a.tile0 != 0)) return go(stream_simt_kernel<1, EPI>);
        return go(stream_simt_kernel<1, EPI, false, false, true>, kStageS1);
    }
    if (a.m <= 8) return go8(stream_kernel<false, EPI, false, false, false, true>, kStageM);
    if (a.m <= kGroupRows) return go16(stream_kernel<true, EPI>);
    return go16(stream_kernel<true, EPI, false, true>);
}

cudaError_t launch_stream(const Args &a, const Parts &pt, int epi, cudaStream_t stream, bool pdl, int mode,
                          bool qact, bool rowmajor, StreamGrid grid) {
    switch (epi) {
        case kEpiStore: return launch_stream_epi<kEpiStore>(a, pt, stream, pdl, mode, qact, rowmajor, grid);
        case kEpiArgmax: return launch_stream_epi<kEpiArgmax>(a, pt, stream, pdl, mode, qact, rowmajor, grid);
        case kEpiGlu: return launch_stream_epi<kEpiGlu>(a, pt, stream, pdl, mode, qact, rowmajor, grid);
        case kEpiNorm: return launch_stream_epi<kEpiNorm>(a, pt, stream, pdl, mode, qact, rowmajor, grid);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace q8
