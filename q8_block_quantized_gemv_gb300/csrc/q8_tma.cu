// Q8_0 GEMV with a TMA-fed shared-memory pipeline (sm_103a).
//
// One CTA owns a tile of 128 output columns for all m rows and a contiguous range of the K/32 Q8_0 blocks (the
// range is split across a thread-block cluster when N is too narrow to fill the SMs).  Its warps are specialised:
//   - one producer warp: a single lane streams the CTA's blocks through a ring of 14 (m <= 8) or 15 stages guarded
//     by mbarriers
//     (full: bytes landed; empty: consumers done).  A stage is one 32-row Q8_0 block: its 32 x 128 int8 values (a
//     2-D TMA box with the 128-byte swizzle), its 128 fp32 scales and the matching 32 activations of every row
//     (a box of 8 or 16 rows; rows at or past m arrive as zeros from the box's out-of-range fill);
//   - seven consumer warps (six for m > 8, in pairs that split a block's columns): each converts the int8 values
//     exactly to bf16, multiplies them with the activations on the tensor cores (m16n8k16, fp32 accumulation into a
//     fresh accumulator per block), then folds the block sums into an fp32 carry with the block's scales
//     ("from_q8.rs", module doc: int8 rows contracted lane by lane, each column's block sums scaled and
//     accumulated in an fp32 carry).
// The MMA's K order is a relabeling of the block's rows chosen so that a warp's shared-memory reads of the swizzled
// weight box are bank-conflict-free: lane quad t reads rows 2t, 2t+8, 2t+1, 2t+9 of each 16-row step (MMA reduction
// index 2t, 2t+1, 2t+8, 2t+9), and its activation fragment pairs x[2t] with x[2t+8] and x[2t+1] with x[2t+9].  MMA
// row g is weight column c + 2p and row g+8 is column c + 2p + 1.
//
// Two CTAs are resident per SM (eight warps each at 128 registers; 72-85 KB of shared memory each), so up to 30
// stages -- about 140 KB -- are in flight per SM.
//
// Programmatic dependent launch: the kernel's CTAs may start before the previous kernel on the stream has finished.
// Every thread waits for it (griddepcontrol.wait) before touching memory that kernel may write -- the activations,
// y and the arg-max keys.  Only when the caller declares the weights constant (Q8_FLAG_CONSTANT_WEIGHTS) does the
// producer start streaming the first stages' weights and scales before that wait.  A CTA lets its own dependents
// launch once its blocks are consumed.
//
// Every wait on an mbarrier is bounded (about two seconds of %globaltimer); a wait that runs out records a fault
// bit in the library's device fault word (q8_device_fault), the CTA waits (bounded again) for the copies it issued
// and finishes without hanging.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "q8_launch.h"

namespace q8 {

__device__ unsigned int g_fault_word = 0;

constexpr int kMaxStages = 16;                      // pipeline depth bound (one 32-row Q8_0 block a stage)
constexpr int kWeightStage = kBlock * kTmaColumns;  // 4 KB of int8 values
constexpr int kScaleStage = kTmaColumns * 4;        // 512 B of fp32 scales

constexpr unsigned kFaultFullWait = 1u;
constexpr unsigned kFaultEmptyWait = 2u;

template <int NT> struct TmaShape {
    static constexpr int kConsumers = NT == 1 ? 7 : 6;
    static constexpr int kClasses = kConsumers / NT;  // blocks in flight across the consumers
    // Stages: a multiple of the classes, so that every block of a stage is consumed by the same class, in order.
    // An mbarrier parity wait is defined only for the barrier's current or preceding phase; with a stage shared by
    // two classes a class that ran ahead could wait two phases ahead and see the older phase of its parity as
    // complete.  With one class a stage, a class waits for the next fill of its stage only after consuming the last.
    static constexpr int kStages = (kMaxStages / kClasses) * kClasses;
    static constexpr int kThreads = 32 * (kConsumers + 1);
    static constexpr int MR = 8 * NT;                 // activation rows held (zeros past m)
    static constexpr int kXStage = MR * kBlock * 2;   // bf16 activations of one block
    static constexpr int kScaleOff = kStages * kWeightStage;  // (kStages of this shape)
    static constexpr int kXOff = kScaleOff + kStages * kScaleStage;
    static constexpr int kBarOff = kXOff + kStages * kXStage;
    static constexpr int kSmem = 1024 /* alignment slack */ + kBarOff + 2 * kStages * 8;
};

__device__ __forceinline__ uint32_t smem_u32(const void *p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ void mbar_init(uint64_t *bar, unsigned count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, unsigned bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, unsigned parity) {
    uint32_t done;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}"
        : "=r"(done)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return done != 0;
}
__device__ __forceinline__ uint64_t global_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
// Wait for the phase of `bar` with the given parity to complete; false after about two seconds.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *bar, unsigned parity) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_ns();
    for (unsigned n = 1;; ++n) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((n & 255u) == 0 && global_ns() - t0 > 2000000000ull) return false;
    }
}

__device__ __forceinline__ void tma_load_2d(void *dst, const CUtensorMap *map, uint64_t *bar, int c0, int c1) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::
            "r"(smem_u32(dst)),
        "l"(map), "r"(c0), "r"(c1), "r"(smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                               uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

template <int V> struct SmemVec;
template <> struct SmemVec<16> {
    using T = uint4;
    static __device__ __forceinline__ T load(const unsigned char *p) { return *reinterpret_cast<const uint4 *>(p); }
};
template <> struct SmemVec<8> {
    using T = uint2;
    static __device__ __forceinline__ T load(const unsigned char *p) { return *reinterpret_cast<const uint2 *>(p); }
};

// NT row tiles of 8 activation rows (m <= 8 * NT).  For NT = 2 each block is shared by a pair of warps, one per
// half of the columns, so that the per-lane accumulators stay in registers.
template <int NT, bool ARGMAX>
__global__ void __maxnreg__(128)
    tma_mma_kernel(const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap smap,
                   const __grid_constant__ CUtensorMap xmap, const Args a, const int prefetch_weights) {
    using S = TmaShape<NT>;
    constexpr int kStages = S::kStages;
    constexpr int V = 16 / NT;  // columns per lane
    constexpr int NP = V / 2;   // MMAs per 16-row step and row tile
    constexpr int MR = S::MR;
    constexpr int NCLS = S::kClasses;
    constexpr unsigned kStageTx = kWeightStage + kScaleStage + S::kXStage;
    extern __shared__ unsigned char smem_raw[];
    unsigned char *smem = reinterpret_cast<unsigned char *>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    unsigned char *wring = smem;                                    // [kStages][32][128] int8, swizzled
    float *sring = reinterpret_cast<float *>(smem + S::kScaleOff);  // [kStages][128] fp32
    unsigned char *xring = smem + S::kXOff;                         // [kStages][MR][32] bf16
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + S::kBarOff);
    uint64_t *empty = full + kStages;
    __shared__ int bail;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int tile = blockIdx.x;
    const int rank = blockIdx.y;
    const int cb0 = (int)((long long)a.nb * rank / a.ksplit);
    const int cb1 = (int)((long long)a.nb * (rank + 1) / a.ksplit);
    const int nblk = cb1 - cb0;

    if (threadIdx.x == 0) {
        for (int i = 0; i < kStages; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], NT);
        }
        bail = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();

    float acc[NT][NP][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int p = 0; p < NP; ++p)
#pragma unroll
            for (int i = 0; i < 4; ++i) acc[nt][p][i] = 0.0f;

    const int g = lane >> 2, t = lane & 3;
    const int hc = warp % NT, cls = warp / NT;
    const int ccol = hc * 64 * (NT - 1) + g * V;  // first column of this lane within the tile
    int issued = 0;                                // stages the producer issued (producer lane only)

    // The weight and scale bytes of block cb0 + i into stage `slot` (2-D TMA boxes of the row-major tensors).
    auto load_weights = [&](int slot, int i) {
        tma_load_2d(wring + slot * kWeightStage, &qmap, &full[slot], tile * kTmaColumns, (cb0 + i) * kBlock);
        tma_load_2d(sring + slot * kTmaColumns, &smap, &full[slot], tile * kTmaColumns, cb0 + i);
    };

    if (warp == S::kConsumers) {
        // ---------------- producer ----------------
        if (lane == 0) {
            asm volatile("prefetch.tensormap [%0];" ::"l"(&qmap) : "memory");
            asm volatile("prefetch.tensormap [%0];" ::"l"(&smap) : "memory");
            asm volatile("prefetch.tensormap [%0];" ::"l"(&xmap) : "memory");
            // Constant weights: the first stages' weights and scales may stream before the previous kernel ends.
            const int early = prefetch_weights ? (nblk < kStages ? nblk : kStages) : 0;
            for (int i = 0; i < early; ++i) {
                mbar_arrive_expect_tx(&full[i], kStageTx);
                load_weights(i, i);
            }
            asm volatile("griddepcontrol.wait;" ::: "memory");
            for (int i = 0; i < nblk; ++i) {
                const int slot = i % kStages;
                if (i >= early) {
                    if (i >= kStages && !mbar_wait_bounded(&empty[slot], ((i / kStages) - 1) & 1)) {
                        atomicOr(&g_fault_word, kFaultEmptyWait);
                        bail = 1;
                        break;
                    }
                    mbar_arrive_expect_tx(&full[slot], kStageTx);
                    load_weights(slot, i);
                }
                tma_load_2d(xring + slot * S::kXStage, &xmap, &full[slot], (cb0 + i) * kBlock, 0);
                issued = i + 1;
            }
        }
    } else {
        // ---------------- consumers ----------------
        asm volatile("griddepcontrol.wait;" ::: "memory");
        const int chunk = ccol >> 4, within = ccol & 15;
        int roff[4];  // byte offset of this lane's rows 2t, 2t+8, 2t+1, 2t+9 (+ swizzle) within a 16-row step
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int row = 2 * t + 8 * (j & 1) + (j >> 1);
            roff[j] = row * kTmaColumns + ((chunk ^ (row & 7)) << 4) + within;
        }
        for (int i = cls; i < nblk; i += NCLS) {
            const int slot = i % kStages;
            // Every lane waits (each needs the barrier's acquire of the stage's bytes); the warp then agrees on the
            // outcome so that a timeout never splits it before an MMA.
            const bool landed = __all_sync(0xffffffffu, mbar_wait_bounded(&full[slot], (i / kStages) & 1));
            if (!landed) {
                if (lane == 0) {
                    atomicOr(&g_fault_word, kFaultFullWait);
                    bail = 1;
                }
                break;
            }
            const unsigned char *ws = wring + slot * kWeightStage;
            const unsigned char *xs = xring + slot * S::kXStage;
            float d[NT][NP][4];
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int p = 0; p < NP; ++p)
#pragma unroll
                    for (int e = 0; e < 4; ++e) d[nt][p][e] = 0.0f;
#pragma unroll
            for (int step = 0; step < 2; ++step) {
                uint32_t b0[NT], b1[NT];
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    const unsigned char *xr = xs + (8 * nt + g) * (kBlock * 2) + (16 * step + 2 * t) * 2;
                    const uint32_t lo = *reinterpret_cast<const uint32_t *>(xr);       // x[2t], x[2t+1]
                    const uint32_t hi = *reinterpret_cast<const uint32_t *>(xr + 16);  // x[2t+8], x[2t+9]
                    b0[nt] = __byte_perm(lo, hi, 0x5410);  // x[2t],   x[2t+8]
                    b1[nt] = __byte_perm(lo, hi, 0x7632);  // x[2t+1], x[2t+9]
                }
                typename SmemVec<V>::T w[4];
#pragma unroll
                for (int j = 0; j < 4; ++j) w[j] = SmemVec<V>::load(ws + step * 16 * kTmaColumns + roff[j]);
#pragma unroll
                for (int wi = 0; wi < V / 4; ++wi) {
                    const uint32_t u0 = word_of(w[0], wi) ^ 0x80808080u;
                    const uint32_t u1 = word_of(w[1], wi) ^ 0x80808080u;
                    const uint32_t u2 = word_of(w[2], wi) ^ 0x80808080u;
                    const uint32_t u3 = word_of(w[3], wi) ^ 0x80808080u;
                    uint32_t lo[4], hi[4];
                    // rows 2t, 2t+8 (lo) and 2t+1, 2t+9 (hi) of each of the word's four columns
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
                        for (int nt = 0; nt < NT; ++nt)
                            mma_bf16_16816(d[nt][p], lo[2 * h], lo[2 * h + 1], hi[2 * h], hi[2 * h + 1], b0[nt],
                                           b1[nt]);
                    }
                }
            }
            float sc[V];
            const float *ss = sring + slot * kTmaColumns + ccol;
#pragma unroll
            for (int v4 = 0; v4 < V / 4; ++v4) {
                const float4 f = *reinterpret_cast<const float4 *>(ss + 4 * v4);
                sc[4 * v4 + 0] = f.x;
                sc[4 * v4 + 1] = f.y;
                sc[4 * v4 + 2] = f.z;
                sc[4 * v4 + 3] = f.w;
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[slot]);
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
    }

    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    __syncthreads();
    if (bail) {
        // A wait ran out: before the ring is reused, wait (bounded) for every copy the producer issued.
        if (warp == S::kConsumers && lane == 0) {
            for (int s = 0; s < kStages && s < issued; ++s) {
                const int last = s + ((issued - 1 - s) / kStages) * kStages;
                if (!mbar_wait_bounded(&full[s], (last / kStages) & 1)) break;
            }
        }
        __syncthreads();
    }
    // Every issued stage has landed and been read: the ring is free for the epilogue.
    float *red = reinterpret_cast<float *>(smem);  // [NCLS][MR][128]
    if (warp < S::kConsumers) {
        float *mine = red + cls * MR * kTmaColumns;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int p = 0; p < NP; ++p) {
                const int r = 8 * nt + 2 * t;
                const int c = ccol + 2 * p;
                *reinterpret_cast<float2 *>(mine + r * kTmaColumns + c) = make_float2(acc[nt][p][0], acc[nt][p][2]);
                *reinterpret_cast<float2 *>(mine + (r + 1) * kTmaColumns + c) =
                    make_float2(acc[nt][p][1], acc[nt][p][3]);
            }
    }
    __syncthreads();
    finish_n<NCLS, MR, kTmaColumns, S::kThreads, ARGMAX>(a, red, blockIdx.x);
}

static_assert(finish_smem_n(TmaShape<1>::kClasses, 8, kTmaColumns) <= TmaShape<1>::kStages * kWeightStage,
              "epilogue fits");
static_assert(finish_smem_n(TmaShape<2>::kClasses, 16, kTmaColumns) <= TmaShape<2>::kStages * kWeightStage,
              "epilogue fits");
static_assert(TmaShape<1>::kStages % TmaShape<1>::kClasses == 0 && TmaShape<2>::kStages % TmaShape<2>::kClasses == 0,
              "one consumer class a stage");
static_assert(TmaShape<1>::kSmem * 2 <= 227 * 1024 && TmaShape<2>::kSmem * 2 <= 227 * 1024, "two CTAs per SM");

// ---------------------------------------------------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------------------------------------------------

static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static bool tried = false;
    if (!tried) {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
        tried = true;
    }
    return fn;
}

static bool encode_2d(PFN_cuTensorMapEncodeTiled_v12000 encode, CUtensorMap *map, CUtensorMapDataType type,
                      const void *base, cuuint64_t inner, cuuint64_t outer, cuuint64_t pitch_bytes, cuuint32_t box_in,
                      cuuint32_t box_out, CUtensorMapSwizzle swizzle) {
    cuuint64_t dims[2] = {inner, outer};
    cuuint64_t strides[1] = {pitch_bytes};
    cuuint32_t box[2] = {box_in, box_out};
    cuuint32_t estr[2] = {1, 1};
    return encode(map, type, 2, const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode_bf16_rows(CUtensorMap *map, const void *base, int rows, int K, int box_k, int box_rows) {
    PFN_cuTensorMapEncodeTiled_v12000 encode = encode_fn();
    return encode && encode_2d(encode, map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, base, (cuuint64_t)K, (cuuint64_t)rows,
                               (cuuint64_t)K * 2, (cuuint32_t)box_k, (cuuint32_t)box_rows, CU_TENSOR_MAP_SWIZZLE_64B);
}

template <int NT, bool ARGMAX>
static cudaError_t launch_tma_nt(const Args &a, const CUtensorMap &qmap, const CUtensorMap &smap,
                                 const CUtensorMap &xmap, cudaStream_t stream, bool pdl, bool prefetch) {
    using S = TmaShape<NT>;
    auto kernel = tma_mma_kernel<NT, ARGMAX>;
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, S::kSmem);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((a.Np + kTmaColumns - 1) / kTmaColumns), (unsigned)a.ksplit, 1);
    cfg.blockDim = dim3(S::kThreads, 1, 1);
    cfg.dynamicSmemBytes = S::kSmem;
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
    return cudaLaunchKernelEx(&cfg, kernel, qmap, smap, xmap, a, prefetch ? 1 : 0);
}

bool tma_supported(const Args &a) { return a.Np >= kTmaColumns; }

cudaError_t launch_tma(const Args &a, bool argmax, cudaStream_t stream, bool pdl, bool prefetch_weights) {
    PFN_cuTensorMapEncodeTiled_v12000 encode = encode_fn();
    if (!encode) return cudaErrorNotSupported;
    const int MR = a.m <= 8 ? 8 : 16;
    CUtensorMap qmap, smap, xmap;
    if (!encode_2d(encode, &qmap, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.q, a.Np, a.K, a.Np, kTmaColumns, kBlock,
                   CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_2d(encode, &smap, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, a.s, a.Np, a.nb, (cuuint64_t)a.Np * 4, kTmaColumns,
                   1, CU_TENSOR_MAP_SWIZZLE_NONE))
        return cudaErrorInvalidValue;
    if (!encode_2d(encode, &xmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a.x, a.K, a.m, (cuuint64_t)a.K * 2, kBlock, MR,
                   CU_TENSOR_MAP_SWIZZLE_NONE))
        return cudaErrorInvalidValue;
    if (MR == 8)
        return argmax ? launch_tma_nt<1, true>(a, qmap, smap, xmap, stream, pdl, prefetch_weights)
                      : launch_tma_nt<1, false>(a, qmap, smap, xmap, stream, pdl, prefetch_weights);
    return argmax ? launch_tma_nt<2, true>(a, qmap, smap, xmap, stream, pdl, prefetch_weights)
                  : launch_tma_nt<2, false>(a, qmap, smap, xmap, stream, pdl, prefetch_weights);
}

cudaError_t read_fault_word(unsigned *out, bool clear) {
    cudaError_t e = cudaMemcpyFromSymbol(out, g_fault_word, sizeof(unsigned));
    if (e != cudaSuccess || !clear) return e;
    const unsigned zero = 0;
    return cudaMemcpyToSymbol(g_fault_word, &zero, sizeof(unsigned));
}

}  // namespace q8
