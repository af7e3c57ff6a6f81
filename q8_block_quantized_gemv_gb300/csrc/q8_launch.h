// Host-side launch helpers shared by the kernel translation units of libq8gemv.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include "q8_device.cuh"

namespace q8 {

// Launch `kernel` over the column tiles of width TC (grid.x) and the K split (grid.y, one thread-block cluster of
// ksplit CTAs per tile when ksplit > 1).
template <typename Kernel>
inline cudaError_t launch_tiles(Kernel kernel, const Args &a, int TC, int smem_bytes, cudaStream_t stream) {
    if (smem_bytes > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes);
        if (e != cudaSuccess) return e;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((a.Np + TC - 1) / TC), (unsigned)a.ksplit, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = (size_t)smem_bytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    cfg.numAttrs = 0;
    if (a.ksplit > 1) {
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 1;
        attr[0].val.clusterDim.y = (unsigned)a.ksplit;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
    }
    return cudaLaunchKernelEx(&cfg, kernel, a);
}

// Column tile width of each kernel family for a given per-thread width V.
__host__ __device__ constexpr int simt_tile(int V) { return 32 * V; }
__host__ __device__ constexpr int mma_tile(int V) { return 8 * V; }

// Defined in q8_simt.cu / q8_mma.cu.  Return cudaErrorInvalidValue for a combination that is not built.
cudaError_t launch_simt(const Args &a, int V, bool argmax, cudaStream_t stream);
cudaError_t launch_mma(const Args &a, int V, bool argmax, cudaStream_t stream);

// Defined in q8_tma.cu.
bool tma_supported(const Args &a);
// A tensor map of bf16 rows [rows][K] (row pitch K), boxes of box_k x box_rows values, 64-byte swizzle, zero fill
// past the last row; false when the driver entry point or the encoding fails.
bool encode_bf16_rows(CUtensorMap *map, const void *base, int rows, int K, int box_k, int box_rows);
cudaError_t launch_tma(const Args &a, bool argmax, cudaStream_t stream, bool pdl, bool prefetch_weights);

// Defined in q8_stream.cu (the tiled layout).
// The largest K split of a stream-kernel launch: a cluster of up to 16 CTAs (above 8 the non-portable size, which the
// launch and the residency query ask for).
constexpr int kMaxStreamSplit = kMaxClusterRanks;
// Resident CTAs per SM of the stream kernel that takes m rows (qact: of quantized activations; rowmajor: of row-major
// weights), and how many clusters of ks such CTAs are resident at once on this device (0: unknown).
int stream_ctas_per_sm(int m, bool qact, bool rowmajor = false);
int stream_max_clusters(int m, bool qact, int ks, bool rowmajor = false);
// How a stream launch takes part in programmatic dependent launch (bits of `mode`):
constexpr int kModePrefetch = 1;   // request the first ring stages' weights before the dependency wait
constexpr int kModeRelease = 2;    // release the next launch right after the dependency wait, not after the main loop
constexpr int kModeDeferWait = 4;  // no dependency wait before the main loop (the launch before released this one
                                   // only after its own wait); wait just before exiting instead
// A stream launch's grid: every column tile of the parts (ntiles = 0), or ntiles grid columns from Args::tile0 (m <= 16,
// one row group; the gated pair has two columns a tile); one_per_sm asks for enough shared memory that an SM holds one
// CTA of the launch and still one ordinary CTA of the same kernel (the kernels that run two CTAs per SM).
struct StreamGrid {
    int ntiles = 0;
    bool one_per_sm = false;
};
// epi: kEpiStore, kEpiArgmax, kEpiGlu (parts 0 and 1 the gate and up weights, grid x = 2 * tiles) or kEpiNorm.
// qact: a.x is a quantized activation (int8 values [m][K], then fp32 scales [m][K/32]) instead of bf16 values.
// rowmajor: the parts' weights are row-major ([K][Np] int8, [K/32][Np] fp32), not tiled (kEpiStore and kEpiArgmax,
// bf16 activations, m <= 16).
cudaError_t launch_stream(const Args &a, const Parts &parts, int epi, cudaStream_t stream, bool pdl, int mode,
                          bool qact, bool rowmajor = false, StreamGrid grid = StreamGrid());
cudaError_t read_fault_word(unsigned *out, bool clear);

// Defined in q8_gemm.cu: the tcgen05 GEMM for prefill chunks (tiled storage, bf16 activations, plain store).
int gemm_min_rows();  // the row count from which the planner takes it
cudaError_t launch_gemm(const Args &a, const Parts &parts, cudaStream_t stream);
cudaError_t read_gemm_fault(unsigned *out, bool clear);
unsigned int *norm_counters();  // device address of the kNormSlots completion counters (null on a CUDA error)

// Defined in q8_api.cu: the K split a test or benchmark forces through q8_set_tuning (0: the planner's).
int forced_ksplit();

// Defined in q8_norm.cu: the residual norm's RMS norm as a launch of its own, one CTA per row of h, after a product
// launch whose epilogue wrote h and stopped there (Args::count null).
struct NormRows {
    const float *h;      // [m][Np], pad columns 0
    const float *gamma;  // [N]
    float eps;
    uint16_t *ybf;       // bf16 [m][Np], or null
    unsigned char *yq;   // quantized form: int8 codes [m][Np], or null
    float *yd;           // its fp32 scales [m][Np / 32] (with yq)
    int N, Np;
};
cudaError_t launch_norm_rows(const NormRows &a, int m, cudaStream_t stream, bool pdl);
constexpr int kTmaColumns = 128;

// Widths built for each family (descending), used by the planner.
bool simt_has(int m, int V);
bool mma_has(int m, int V);

}  // namespace q8
