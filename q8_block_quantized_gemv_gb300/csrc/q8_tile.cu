// The tiled storage of a Q8_0 weight: the row-major values [K][Np] and scales [K/32][Np] rearranged so that every
// 32-row x 128-column block is one contiguous 4 KB unit in MMA-fragment order (and its 128 scales one 512-byte unit),
// the units of a 128-column tile following each other along K.  A warp that owns a run of a tile's K blocks then
// reads one contiguous range of memory, 512 contiguous bytes per instruction, and finds each lane's operand bytes
// where that lane loads them.
//
// Layout (Nt = N rounded up to a multiple of 128, T = Nt / 128 tiles, nb = K / 32 blocks):
//   values  uint8 unit (t, b) at byte (t * nb + b) * 4096: eight 512-byte segments, segment 4s + h (s = 0, 1: the
//                 16-row half of the block; h = 0..3: a group of four 8-column slices).  In segment (s, h) the 16 bytes
//                 at 16 * L, L = 4g + u (g = 0..7, u = 0..3), are four words; word w holds the values of weight rows
//                 32b + 16s + 4u + k (k = 0..3, byte k) in column 128t + 8(4h + w) + g, each stored as q + 128
//   scales  fp32  unit (t, b) at element (t * nb + b) * 128; element c = s[b][128t + c]
//   columns >= N hold q = 0 (byte 128) and scale 0.
#include <string.h>

#include "../../include/q8_gemv.h"
#include "q8_launch.h"

namespace q8 {
void set_last_cuda_error(int e);  // q8_host.cpp
}

namespace {

constexpr int kTileCols = 128;

// One thread per 16-byte chunk of the tiled values (four rows of four columns); the first 8 threads of a unit also
// write its scales.
__global__ void tile_values_kernel(const int8_t *__restrict__ q, const float *__restrict__ s, int K, int N, int Np,
                                   int8_t *__restrict__ qt, float *__restrict__ st, long long chunks) {
    const long long id = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (id >= chunks) return;
    const int nb = K / Q8_BLOCK;
    const long long unit = id / 256;  // 4096 B = 256 chunks per unit
    const int within = (int)(id % 256);
    const int seg = within / 32, L = within % 32;
    const int step = seg / 4, h = seg % 4, g = L / 4, u = L % 4;
    const int t = (int)(unit / nb), b = (int)(unit % nb);
    const long long krow = (long long)Q8_BLOCK * b + 16 * step + 4 * u;  // first of the chunk's four weight rows
    unsigned char tmp[16];
    for (int w = 0; w < 4; ++w) {
        const int c = kTileCols * t + 8 * (4 * h + w) + g;
        for (int k = 0; k < 4; ++k)
            tmp[4 * w + k] = (unsigned char)((c < N ? (int)q[(krow + k) * Np + c] : 0) + 128);
    }
    uint4 v;
    memcpy(&v, tmp, 16);
    *reinterpret_cast<uint4 *>(qt + id * 16) = v;
    if (within < 8) {  // the unit's scales: 8 threads x 16 fp32
        for (int i = 0; i < 16; ++i) {
            const int c = 16 * within + i;
            const int n = kTileCols * t + c;
            st[unit * kTileCols + c] = n < N ? s[(long long)b * Np + n] : 0.0f;
        }
    }
}

q8_status check_tile_args(const void *q, const void *s, int K, int N, const void *qt, const void *st) {
    if (!q || !s || !qt || !st) return Q8_ERR_ARG;
    if (K <= 0 || K % Q8_BLOCK != 0 || N <= 0 || q8_tiled_n(N) < 0) return Q8_ERR_SHAPE;
    return Q8_OK;
}

}  // namespace

extern "C" int q8_tiled_n(int N) {
    if (N <= 0) return -1;
    const long long p = ((long long)N + kTileCols - 1) / kTileCols * kTileCols;
    return p > 0x7FFFFFFFLL ? -1 : (int)p;
}

extern "C" q8_status q8_tile(const int8_t *q, const float *s, int K, int N, int8_t *qt, float *st) {
    q8_status stt = check_tile_args(q, s, K, N, qt, st);
    if (stt != Q8_OK) return stt;
    const int Np = q8_padded_n(N), Nt = q8_tiled_n(N), nb = K / Q8_BLOCK, T = Nt / kTileCols;
    for (int t = 0; t < T; ++t) {
        for (int b = 0; b < nb; ++b) {
            const size_t unit = (size_t)t * nb + b;
            int8_t *dst = qt + unit * (Q8_BLOCK * kTileCols);
            for (int r = 0; r < Q8_BLOCK; ++r) {
                const int step = r / 16, u = (r % 16) / 4, k = r % 4;
                for (int c = 0; c < kTileCols; ++c) {
                    const int n = kTileCols * t + c;
                    const int j = c / 8, g = c % 8;
                    const size_t at = (size_t)(4 * step + j / 4) * 512 + 16 * (4 * g + u) + 4 * (j % 4) + k;
                    const int v = n < N ? (int)q[((size_t)Q8_BLOCK * b + r) * Np + n] : 0;
                    dst[at] = (int8_t)(unsigned char)(v + 128);
                }
            }
            for (int c = 0; c < kTileCols; ++c) {
                const int n = kTileCols * t + c;
                st[unit * kTileCols + c] = n < N ? s[(size_t)b * Np + n] : 0.0f;
            }
        }
    }
    return Q8_OK;
}

extern "C" q8_status q8_tile_device(const int8_t *q, const float *s, int K, int N, int8_t *qt, float *st,
                                    q8_stream_t stream) {
    q8_status stt = check_tile_args(q, s, K, N, qt, st);
    if (stt != Q8_OK) return stt;
    if (((uintptr_t)q & 15) || ((uintptr_t)qt & 15) || ((uintptr_t)s & 3) || ((uintptr_t)st & 3))
        return Q8_ERR_ALIGN;
    const int Np = q8_padded_n(N), Nt = q8_tiled_n(N);
    const long long chunks = (long long)K * Nt / 16;
    const int threads = 256;
    const long long blocks = (chunks + threads - 1) / threads;
    if (blocks > 0x7FFFFFFFLL) return Q8_ERR_SHAPE;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)blocks, 1, 1);
    cfg.blockDim = dim3(threads, 1, 1);
    cfg.stream = (cudaStream_t)stream;
    cudaError_t e = cudaLaunchKernelEx(&cfg, tile_values_kernel, q, s, K, N, Np, qt, st, chunks);
    if (e != cudaSuccess) {
        q8::set_last_cuda_error((int)e);
        return Q8_ERR_CUDA;
    }
    return Q8_OK;
}
