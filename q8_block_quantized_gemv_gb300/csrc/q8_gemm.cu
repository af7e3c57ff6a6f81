// Q8_0 product of a prefill chunk (m > 16 rows, up to 512) over the tiled storage on the 5th-generation tensor cores:
// one CTA computes a 128-row x 128-column output tile over its range of K with tcgen05.mma (bf16 operands from
// shared memory, fp32 accumulators in tensor memory).
//
// The block's scale s[b, n] belongs to each 32-row block and column, so the weight cannot be dequantized into a bf16
// operand (8 significant bits cannot hold q * s).  Each 32-row block is therefore contracted on its own -- two
// K = 16 MMAs of M = 128, N = 128 into a fresh accumulator -- and folded into the fp32 carry on the CUDA cores
// ("from_q8.rs", module doc: int8 rows are contracted lane by lane, and each column's block sums are scaled and
// accumulated into an fp32 carry).  The exact int8 -> bf16 weights and the bf16 activations make every product
// exact; the block's sums are fp32.
//
// Warp roles (576 threads, one CTA per SM; 18 warps, at most five a scheduler, 96 registers a thread):
//   warp 0     one thread loads block b + 4 into a ring stage: the activations (128 rows x 32 values) by a TMA tensor
//              copy with 64-byte swizzle (rows past m read as zeros), the weight unit (4 KB, stored q + 128) and its
//              128 scales by two bulk copies, all completing one `loaded` barrier;
//   warp 1     one thread issues each block's two MMAs into one of four accumulator buffers and commits them to the
//              stage's `empty` barrier and the buffer's `full` barrier;
//   warps 2-17 workers: they first fold block b - 3 -- each thread reads its accumulator lane (one output row)
//              over a quarter of the columns, multiplies by the block's scales and adds into its fp32 carry (packed
//              fp32x2); the warp frees the buffer and its share of the stage -- then turn block b's unit into exact
//              bf16 in the same 64-byte swizzled K-major layout (two words a thread) and signal the stage full.
// Four accumulator buffers let the MMAs of later blocks run while a block is folded.  When the tiles are too
// few to fill the SMs, K is split across a thread-block cluster of up to 4 CTAs; their carries are summed through
// distributed shared memory in rank order (deterministic).  Every mbarrier wait is bounded (about two seconds); a
// wait that runs out records a fault bit, makes the CTA stop issuing work and drain, and the kernel returns with its
// tensor memory freed.
#include <stdlib.h>

#include <atomic>
#include <cooperative_groups.h>

#include "q8_launch.h"

namespace q8 {

namespace {

constexpr int kGM = 128;               // activation rows of a CTA tile (the MMA's M)
constexpr int kGN = kTmaColumns;       // columns of a CTA tile: one 128-column tile of the tiled storage
constexpr int kGStages = 8;            // ring stages (one 32-row block each)
constexpr int kAccBufs = 4;            // accumulator buffers in tensor memory (128 columns each)
constexpr int kLoadWarp = 0;
constexpr int kMmaWarp = 1;
constexpr int kWorkWarp0 = 2;             // warps 2..17: TMEM lane quarters 2, 3, 0, 1 (four times: column quarters)
constexpr int kWorkWarps = 16;
constexpr int kGThreads = 32 * (kWorkWarp0 + kWorkWarps);
constexpr int kFoldCols = kGN / 4;        // columns one worker folds
constexpr int kFoldLag = 3;               // a worker folds block b - 3 before it converts block b

// Stage layout (bytes): bf16 A [128 rows x 64 bytes] as the TMA writes it (64-byte swizzle), B [128 weight columns x
// 64 bytes] in the same swizzle, the raw unit, its 128 scales; stages 1024-byte aligned (the swizzle pattern repeats
// every 512 bytes).
constexpr int kAOff = 0, kBOff = 8192, kRawOff = 16384, kSOff = 20480, kStageBytes = 21504;
constexpr int kBlockTx = 8192 + 4096 + 512;  // bytes the copies of one block deliver
static_assert(kFoldLag < kAccBufs, "the MMAs of a block never wait for a fold that comes after it");
static_assert(kStageBytes % 1024 == 0, "swizzled stages stay aligned");
constexpr int kMaxSplit = 4;               // CTAs of a cluster splitting K
constexpr int kRedStride = kGN + 4;        // floats a row of the split-K reduction slab (padded)
static_assert(kGM * kRedStride * 4 <= kGStages * kStageBytes, "the reduction slab fits in the ring");
constexpr int kBarOff = kGStages * kStageBytes;
// barriers: loaded[S], full[S], empty[S], acc_full[kAccBufs], acc_empty[kAccBufs], drain; then the TMEM base and
// the abort flag
constexpr int kGSmem = kBarOff + (3 * kGStages + 2 * kAccBufs + 1) * 8 + 16;
constexpr unsigned kTmemCols = kAccBufs * kGN;  // all 512 columns: the accumulator buffers

constexpr unsigned kFaultGemmWait = 4u;

__device__ unsigned int g_gemm_fault = 0;  // this kernel's bounded waits (reported with the TMA kernel's fault word)

__device__ __forceinline__ uint32_t smem_u32(const void *p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ void bar_init(uint64_t *bar, unsigned count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void bar_arrive_tx(uint64_t *bar, unsigned bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes) : "memory");
}
__device__ __forceinline__ void bulk_copy(void *dst, const void *src, unsigned bytes, uint64_t *bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     smem_u32(dst)),
                 "l"(src), "r"(bytes), "r"(smem_u32(bar))
                 : "memory");
}
__device__ __forceinline__ void bar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ bool bar_try_wait(uint64_t *bar, unsigned parity) {
    uint32_t done;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}"
        : "=r"(done)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return done != 0;
}
__device__ __forceinline__ uint64_t now_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
// Wait for the phase of `bar` with the given parity; false when the CTA is aborting or after about two seconds
// (which also starts the abort).
__device__ __forceinline__ bool bar_wait(uint64_t *bar, unsigned parity, volatile int *abort) {
    if (bar_try_wait(bar, parity)) return true;
    const uint64_t t0 = now_ns();
    for (unsigned n = 1;; ++n) {
        if (bar_try_wait(bar, parity)) return true;
        if ((n & 63u) == 0) {
            if (*abort) return false;
            if (now_ns() - t0 > 2000000000ull) {
                *abort = 1;
                atomicOr(&g_gemm_fault, kFaultGemmWait);
                return false;
            }
        }
    }
}

__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Shared-memory matrix descriptor, K-major: lbo = byte step between core matrices along K (unused with a swizzle),
// sbo = byte step between 8-row groups, layout = 0 (no swizzle: core matrices of 8 rows x 16 bytes) or 4 (64-byte
// swizzle: rows of 64 bytes, 16-byte chunks XOR-ed with row bits 1-2); bits 46-48 hold the fixed 0b001.
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr, uint32_t lbo, uint32_t sbo, uint32_t layout = 0) {
    return (uint64_t)((addr & 0x3FFFFu) >> 4) | ((uint64_t)(lbo >> 4) << 16) | ((uint64_t)(sbo >> 4) << 32) |
           (1ull << 46) | ((uint64_t)layout << 61);
}

__device__ __forceinline__ void tma_rows(void *dst, const CUtensorMap *map, int k, int row, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::
            "r"(smem_u32(dst)),
        "l"(map), "r"(k), "r"(row), "r"(smem_u32(bar))
        : "memory");
}

// Instruction descriptor of kind::f16: fp32 D (bits 4-5 = 1), bf16 A and B (bits 7-9, 10-12 = 1), both K-major,
// N >> 3 at bit 17, M >> 4 at bit 24.
constexpr uint32_t kIdesc = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(kGN >> 3) << 17) |
                            ((uint32_t)(kGM >> 4) << 24);

__device__ __forceinline__ void mma_bf16(uint32_t tmem_d, uint64_t a, uint64_t b, uint32_t accumulate) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}" ::"r"(tmem_d),
        "l"(a), "l"(b), "r"(kIdesc), "r"(accumulate)
        : "memory");
}
__device__ __forceinline__ void mma_commit(uint64_t *bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}

// 32 consecutive accumulator columns of this thread's lane, requested; tmem_wait makes them usable.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&v)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),
          "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15]),
          "=r"(v[16]), "=r"(v[17]), "=r"(v[18]), "=r"(v[19]), "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]),
          "=r"(v[24]), "=r"(v[25]), "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]), "=r"(v[31])
        : "r"(taddr));
}
__device__ __forceinline__ void tmem_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

__device__ __forceinline__ unsigned long long fma2(unsigned long long a, unsigned long long b, unsigned long long c) {
    unsigned long long d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
__device__ __forceinline__ unsigned long long pack2(uint32_t lo, uint32_t hi) {
    unsigned long long d;
    asm("mov.b64 %0, {%1, %2};" : "=l"(d) : "r"(lo), "r"(hi));
    return d;
}

// Stored bytes E, E + 1 of a word (q + 128 each) as the exact bf16 pair {q_E, q_E+1}: each byte in the low mantissa
// of 2^23 gives 2^23 + q + 128, a packed subtract leaves q, packed to bf16 (exact: |q| <= 127).
template <int E> __device__ __forceinline__ uint32_t stored_to_bf16x2(uint32_t u) {
    uint32_t d;
    asm("{\n .reg .b32 a, b;\n .reg .b64 p, r;\n .reg .f32 lo, hi;\n prmt.b32 a, %1, 0x4B000000, %2;\n"
        " prmt.b32 b, %1, 0x4B000000, %3;\n mov.b64 p, {a, b};\n sub.rn.f32x2 r, p, %4;\n mov.b64 {lo, hi}, r;\n"
        " cvt.rn.bf16x2.f32 %0, hi, lo;\n}"
        : "=r"(d)
        : "r"(u), "n"(0x7540 + E), "n"(0x7540 + E + 1), "l"(0x4B0000804B000080ull));
    return d;
}

__global__ void __maxnreg__(96)
    gemm_kernel(Args a, const __grid_constant__ Parts parts, const __grid_constant__ CUtensorMap xmap) {
    namespace cg = cooperative_groups;
    extern __shared__ __align__(1024) unsigned char smem_g[];
    uint64_t *loaded = reinterpret_cast<uint64_t *>(smem_g + kBarOff);
    uint64_t *full = loaded + kGStages;
    uint64_t *empty = full + kGStages;
    uint64_t *acc_full = empty + kGStages;
    uint64_t *acc_empty = acc_full + kAccBufs;
    uint64_t *drain = acc_empty + kAccBufs;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(drain + 1);
    volatile int *abort = reinterpret_cast<volatile int *>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int tile = select_part(parts, blockIdx.x, a);
    const int row0 = kGM * blockIdx.y;
    const int ks = gridDim.z, rank = blockIdx.z;  // the cluster's split of K (clusters are (1, 1, ks))
    const int kb0 = (int)((long long)a.nb * rank / ks);
    const int n = (int)((long long)a.nb * (rank + 1) / ks) - kb0;  // this CTA's blocks

    if (threadIdx.x == 0) {
        for (int i = 0; i < kGStages; ++i) {
            bar_init(&loaded[i], 1);               // thread 0's expect_tx; the bulk copies' bytes complete it
            bar_init(&full[i], kWorkWarps);        // one thread of each worker warp
            bar_init(&empty[i], 1 + kWorkWarps);   // the MMA commit and the folds (they read the stage's scales)
        }
        for (int i = 0; i < kAccBufs; ++i) {
            bar_init(&acc_full[i], 1);
            bar_init(&acc_empty[i], kWorkWarps);
        }
        bar_init(drain, 1);
        *abort = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                     "r"(kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = *tmem_slot;
    asm volatile("griddepcontrol.wait;" ::: "memory");

    const int quarter = warp & 3;                            // the TMEM lanes a worker warp may read
    const int col0 = kFoldCols * ((warp - kWorkWarp0) >> 2);  // the columns it folds (one quarter of them)
    const int r = 32 * quarter + lane;                       // the output row a worker thread folds
    unsigned long long acc[kFoldCols / 2];
#pragma unroll
    for (int j = 0; j < kFoldCols / 2; ++j) acc[j] = 0ull;

    if (warp == kLoadWarp) {
        // ---- loader (one thread): the copies of block i (i counts this CTA's blocks) ----
        if (lane == 0) {
            const unsigned char *qbase =
                reinterpret_cast<const unsigned char *>(a.q) + ((size_t)tile * a.nb + kb0) * 4096;
            const float *sbase = a.s + ((size_t)tile * a.nb + kb0) * kGN;
            int issued = 0;
            for (int i = 0; i < n; ++i) {
                const int st = i % kGStages;
                // the stage was last used by block i - kGStages: its MMAs and every worker's fold are done
                if (i >= kGStages && !bar_wait(&empty[st], ((i / kGStages) - 1) & 1, abort)) break;
                unsigned char *sp = smem_g + st * kStageBytes;
                bar_arrive_tx(&loaded[st], kBlockTx);
                tma_rows(sp + kAOff, &xmap, (kb0 + i) * kBlock, row0, &loaded[st]);
                bulk_copy(sp + kRawOff, qbase + (size_t)i * 4096, 4096, &loaded[st]);
                bulk_copy(sp + kSOff, sbase + (size_t)i * kGN, 512, &loaded[st]);
                ++issued;
            }
            if (*abort) {
                // the copies started land before the shared memory is reused or freed (the last fill of each
                // stage; earlier fills were waited for before their stage was refilled)
                for (int i = issued - kGStages < 0 ? 0 : issued - kGStages; i < issued; ++i) {
                    const uint64_t t0 = now_ns();
                    while (!bar_try_wait(&loaded[i % kGStages], (i / kGStages) & 1) &&
                           now_ns() - t0 < 2000000000ull) {
                    }
                }
            }
        }
        __syncwarp();
    } else if (warp == kMmaWarp) {
        // ---- MMA issue (one thread) ----
        if (lane == 0) {
            for (int i = 0; i < n; ++i) {
                const int st = i % kGStages, buf = i % kAccBufs;
                if (!bar_wait(&full[st], (i / kGStages) & 1, abort)) break;
                if (i >= kAccBufs && !bar_wait(&acc_empty[buf], ((i / kAccBufs) - 1) & 1, abort)) break;
                tc_fence_after();
                const uint32_t sa = smem_u32(smem_g + st * kStageBytes + kAOff);
                const uint32_t sb = smem_u32(smem_g + st * kStageBytes + kBOff);
                const uint32_t td = tbase + (uint32_t)(buf * kGN);
#pragma unroll
                for (int k = 0; k < 2; ++k)  // K = 16 each: 32 bytes into the 64-byte rows of A and B
                    mma_bf16(td, smem_desc(sa + 32 * k, 16, 512, 4), smem_desc(sb + 32 * k, 16, 512, 4), k);
                mma_commit(&empty[st]);
                mma_commit(&acc_full[buf]);
            }
        }
        __syncwarp();
    } else {
        // ---- workers: fold block i - kFoldLag, convert block i ----
        // Each thread converts two words of the unit: words 2wp, 2wp + 1 of segment 4s + h, lane 4g + u.  Warp wi
        // takes group h, columns g0 .. g0 + 3 of each 8-column slice and word pair wp; a lane takes (s, g, u).  Then
        // the 16 lanes of a half-warp write two adjacent weight columns (rows of B) whole -- their 16 x 8 bytes are
        // one 128-byte line of banks -- so the conversion stores have no bank conflicts (the raw reads take two
        // passes a half-warp: its two 16-row halves s sit 2 KB apart).
        const int wi = warp - kWorkWarp0;
        const int h = wi & 3, g0 = ((wi >> 2) & 1) * 4, wp = wi >> 3;
        const int u = lane & 3, s = (lane >> 3) & 1, g = g0 + 2 * ((lane >> 4) & 1) + ((lane >> 2) & 1);
        const int c = (4 * s + h) * 32 + 4 * g + u;  // this thread's 16-byte chunk of the unit
        auto fold = [&](int f) -> bool {
            const int buf = f % kAccBufs, st = f % kGStages;
            if (!bar_wait(&acc_full[buf], (f / kAccBufs) & 1, abort)) return false;
            tc_fence_after();
            uint32_t v[kFoldCols / 32][32];
#pragma unroll
            for (int cc = 0; cc < kFoldCols / 32; ++cc)
                tmem_ld32(tbase + ((uint32_t)(32 * quarter) << 16) + (uint32_t)(buf * kGN + col0 + 32 * cc), v[cc]);
            // the block's scales (landed with the `loaded` wait of block f; the stage is refilled only after every
            // worker's fold of block f has arrived on its `empty` barrier)
            const unsigned long long *sp = reinterpret_cast<const unsigned long long *>(
                smem_g + st * kStageBytes + kSOff + col0 * 4);
            tmem_wait();
#pragma unroll
            for (int cc = 0; cc < kFoldCols / 32; ++cc)
#pragma unroll
                for (int j = 0; j < 16; ++j)
                    acc[16 * cc + j] = fma2(sp[16 * cc + j], pack2(v[cc][2 * j], v[cc][2 * j + 1]), acc[16 * cc + j]);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                bar_arrive(&acc_empty[buf]);
                bar_arrive(&empty[st]);
            }
            return true;
        };
        bool ok = true;
        for (int i = 0; i < n && ok; ++i) {
            // Fold block i - kFoldLag first: then a stage's refill (after its block's MMAs and folds) does not wait for
            // a later block's copies (measured on GB300: 2-4% faster on every prefill shape of the sweep).
            if (i >= kFoldLag && !(ok = fold(i - kFoldLag))) break;
            const int st = i % kGStages;
            if (!bar_wait(&loaded[st], (i / kGStages) & 1, abort)) break;
            unsigned char *sp = smem_g + st * kStageBytes;
            const uint2 raw = *reinterpret_cast<const uint2 *>(sp + kRawOff + c * 16 + wp * 8);
            const uint32_t words[2] = {raw.x, raw.y};
#pragma unroll
            for (int ww = 0; ww < 2; ++ww) {
                const int w = 2 * wp + ww;
                const int j = 4 * h + w;  // 8-column slice: B rows 8j .. 8j + 7, this word's row 8j + g
                const uint2 cv = make_uint2(stored_to_bf16x2<0>(words[ww]), stored_to_bf16x2<2>(words[ww]));
                // B row (weight column) nr = 8j + g holds its 32 K values in 64 bytes; 16-byte chunk kc = 2s + u / 2
                // sits at chunk kc ^ ((nr >> 1) & 3) (the 64-byte swizzle), 8 bytes in for odd u
                const int nr = 8 * j + g, kc = 2 * s + (u >> 1);
                *reinterpret_cast<uint2 *>(sp + kBOff + nr * 64 + ((kc ^ ((nr >> 1) & 3)) << 4) + (u & 1) * 8) = cv;
            }
            fence_async_smem();  // this thread's generic-proxy writes before the MMAs read them
            __syncwarp();
            if (lane == 0) bar_arrive(&full[st]);
        }
        for (int f = n - kFoldLag < 0 ? 0 : n - kFoldLag; f < n && ok; ++f) ok = fold(f);
    }

    // Drain: every MMA this CTA issued has completed (the last block's commit reached acc_full, waited on by the
    // fold warps) and every copy has landed, unless the CTA aborted; after an abort, one more commit waited on with a
    // bound covers any MMA still running.
    tc_fence_before();
    __syncthreads();
    if (*abort && threadIdx.x == 32 * kMmaWarp) {
        mma_commit(drain);
        const uint64_t t0 = now_ns();
        while (!bar_try_wait(drain, 0) && now_ns() - t0 < 2000000000ull) {
        }
    }
    __syncthreads();
    tc_fence_after();

    // The carries to y (rows < m; pad columns n >= N exactly 0): directly, or through the cluster when K is split.
    if (ks == 1) {
        const int row = row0 + r;
        if (warp >= kWorkWarp0 && row < a.m && !*abort) {
            float *yrow = a.y + (size_t)row * a.Np;
#pragma unroll
            for (int j = 0; j < kFoldCols / 4; ++j) {
                const int nn = tile * kGN + col0 + 4 * j;
                if (nn < a.Np) {
                    float lo0, hi0, lo1, hi1;
                    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo0), "=f"(hi0) : "l"(acc[2 * j]));
                    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo1), "=f"(hi1) : "l"(acc[2 * j + 1]));
                    float4 o = make_float4(nn < a.N ? lo0 : 0.0f, nn + 1 < a.N ? hi0 : 0.0f,
                                           nn + 2 < a.N ? lo1 : 0.0f, nn + 3 < a.N ? hi1 : 0.0f);
                    *reinterpret_cast<float4 *>(yrow + nn) = o;
                }
            }
        }
    } else {
        // every CTA's carries into its slab (the ring is idle: all copies landed, all MMAs done)
        float *red = reinterpret_cast<float *>(smem_g);
        if (warp >= kWorkWarp0) {
#pragma unroll
            for (int j = 0; j < kFoldCols / 4; ++j) {
                float lo0, hi0, lo1, hi1;
                asm("mov.b64 {%0, %1}, %2;" : "=f"(lo0), "=f"(hi0) : "l"(acc[2 * j]));
                asm("mov.b64 {%0, %1}, %2;" : "=f"(lo1), "=f"(hi1) : "l"(acc[2 * j + 1]));
                *reinterpret_cast<float4 *>(red + r * kRedStride + col0 + 4 * j) = make_float4(lo0, hi0, lo1, hi1);
            }
        }
        cg::cluster_group cluster = cg::this_cluster();
        cluster.sync();
        // rank z sums rows [z * 128 / ks, (z + 1) * 128 / ks) over the ranks, in rank order
        const int r0 = kGM * rank / ks, r1 = kGM * (rank + 1) / ks;
        for (int e = threadIdx.x; e < (r1 - r0) * (kGN / 4); e += kGThreads) {
            const int rr = r0 + e / (kGN / 4), c4 = 4 * (e % (kGN / 4));
            const int row = row0 + rr, nn = tile * kGN + c4;
            if (row < a.m && nn < a.Np && !*abort) {  // the ranks' slabs are read only for a value that is stored
                const float4 sum = cluster_sum4(cluster, red, rr * kRedStride + c4, 0, 1, ks);
                float4 o = make_float4(nn < a.N ? sum.x : 0.0f, nn + 1 < a.N ? sum.y : 0.0f,
                                       nn + 2 < a.N ? sum.z : 0.0f, nn + 3 < a.N ? sum.w : 0.0f);
                *reinterpret_cast<float4 *>(a.y + (size_t)row * a.Np + nn) = o;
            }
        }
        cluster_sync_after_reads();  // every rank's slab stays alive until all have read it
    }
    if (warp == 0)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tbase), "r"(kTmemCols) : "memory");
}

}  // namespace

int gemm_min_rows() { return 128; }

cudaError_t read_gemm_fault(unsigned *out, bool clear) {
    cudaError_t e = cudaMemcpyFromSymbol(out, g_gemm_fault, sizeof(unsigned));
    if (e != cudaSuccess || !clear) return e;
    const unsigned zero = 0;
    return cudaMemcpyToSymbol(g_gemm_fault, &zero, sizeof(unsigned));
}

// Clusters of ks GEMM CTAs resident at once on this device (0: unknown); asked once per device and size.
static int max_clusters(int ks) {
    static std::atomic<int> cache[64][kMaxSplit + 1];  // 0: not asked yet; else the count + 1
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64 || ks < 1 || ks > kMaxSplit) return 0;
    const int known = cache[dev][ks].load(std::memory_order_relaxed);
    if (known > 0) return known - 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(1, 1, (unsigned)ks);
    cfg.blockDim = dim3(kGThreads, 1, 1);
    cfg.dynamicSmemBytes = kGSmem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 1;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = (unsigned)ks;
    cfg.attrs = attr;
    cfg.numAttrs = ks > 1 ? 1 : 0;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, gemm_kernel, &cfg) != cudaSuccess) {
        cudaGetLastError();  // the failed query's error is not the caller's
        return 0;
    }
    cache[dev][ks].store(n + 1, std::memory_order_relaxed);
    return n;
}

cudaError_t launch_gemm(const Args &a, const Parts &pt, cudaStream_t stream) {
    cudaError_t e = cudaFuncSetAttribute(gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kGSmem);
    if (e != cudaSuccess) return e;
    int sms = 0;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, 0);
    if (e != cudaSuccess) return e;
    // K split: the one of 1 .. 4 whose waves of resident clusters (one CTA per SM; a cluster's CTAs share one GPC)
    // finish first, a CTA costing its blocks plus about eight blocks of fill, drain and epilogue.  Measured on GB300
    // against every forced split, it picks the fastest for each shape of the sweep; against the split that only
    // filled one wave, 4096 x 14336 at m = 256 (224 CTAs unsplit, 1.5 waves) went 131.4 -> 110.0 us and 5120 x 6144
    // at m = 512 162.3 -> 131.4 us.
    const long long ctas = (long long)pt.tile_end[pt.count - 1] * ((a.m + kGM - 1) / kGM);
    long long ks = 1;
    double best_cost = 1e300;
    for (int k = 1; k <= kMaxSplit && k <= a.nb; ++k) {
        const long long fit = k == 1 ? (long long)sms : (long long)max_clusters(k);
        if (fit <= 0) continue;
        const long long waves = (ctas + fit - 1) / fit;
        const double cost = (double)waves * (8.0 + (double)((a.nb + k - 1) / k));
        if (cost < best_cost - 1e-9) {
            best_cost = cost;
            ks = k;
        }
    }
    const int f = forced_ksplit();
    if (f >= 1 && f <= kMaxSplit && f <= a.nb) ks = f;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)pt.tile_end[pt.count - 1], (unsigned)((a.m + kGM - 1) / kGM), (unsigned)ks);
    cfg.blockDim = dim3(kGThreads, 1, 1);
    cfg.dynamicSmemBytes = kGSmem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    if (ks > 1) {
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 1;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = (unsigned)ks;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
    }
    CUtensorMap xmap;
    if (!encode_bf16_rows(&xmap, a.x, a.m, a.K, kBlock, kGM)) return cudaErrorNotSupported;
    return cudaLaunchKernelEx(&cfg, gemm_kernel, a, pt, xmap);
}

}  // namespace q8
