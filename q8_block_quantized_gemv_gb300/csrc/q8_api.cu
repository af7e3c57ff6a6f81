// Device entry points of libq8gemv: argument checks, the launch plan, and the arg-max finish.
#include <stdint.h>

#include <stdlib.h>

#include <atomic>

#include "../../include/q8_gemv.h"
#include "q8_launch.h"

namespace q8 {
void set_last_cuda_error(int e);  // q8_host.cpp
}

using q8::Args;

namespace {

q8_status cuda_fail(cudaError_t e) {
    q8::set_last_cuda_error((int)e);
    return Q8_ERR_CUDA;
}

bool aligned(const void *p, uintptr_t a) { return ((uintptr_t)p & (a - 1)) == 0; }

bool overlaps(const void *a, size_t na, const void *b, size_t nb) {
    const uintptr_t a0 = (uintptr_t)a, b0 = (uintptr_t)b;
    return a0 < b0 + nb && b0 < a0 + na;
}

// SM count of the current device, cached per device (a read-only property).
int sm_count(int *out) {
    static std::atomic<int> cache[64];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return (int)e;
    if (dev >= 0 && dev < 64) {
        const int c = cache[dev].load(std::memory_order_relaxed);
        if (c > 0) {
            *out = c;
            return 0;
        }
    }
    int n = 0;
    e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return (int)e;
    if (dev >= 0 && dev < 64) cache[dev].store(n, std::memory_order_relaxed);
    *out = n;
    return 0;
}

// The test and benchmark overrides of the planner (q8_set_tuning): a forced K split, the prefill GEMM forced on or
// off, the residual norm's route and the two-launch split.  Each starts from its environment variable (Q8_KSPLIT,
// Q8_GEMM, Q8_NORM_LAUNCH, Q8_SPLIT), read once per process at the first call that needs it; a call then reads one
// relaxed atomic.
constexpr int kTuneOptions = 4;

struct Tuning {
    std::atomic<int> value[kTuneOptions];
    Tuning() {
        const char *k = getenv("Q8_KSPLIT");
        const char *g = getenv("Q8_GEMM");
        const char *r = getenv("Q8_NORM_LAUNCH");
        const char *sp = getenv("Q8_SPLIT");
        const int ks = k ? atoi(k) : 0;
        value[Q8_TUNE_KSPLIT].store(ks >= 1 && ks <= 8 ? ks : 0, std::memory_order_relaxed);
        value[Q8_TUNE_GEMM].store(g && g[0] == '0' ? 0 : g && g[0] == '1' ? 1 : -1, std::memory_order_relaxed);
        value[Q8_TUNE_NORM_FOLD].store(r && r[0] == '0' ? 1 : 0, std::memory_order_relaxed);
        value[Q8_TUNE_SPLIT].store(sp && sp[0] == '0' ? 0 : 1, std::memory_order_relaxed);
    }
};

Tuning &tuning_table() {
    static Tuning t;  // initialised once, thread-safely, at the first use
    return t;
}

int tuning(int option) { return tuning_table().value[option].load(std::memory_order_relaxed); }

constexpr int kVariantStream = 100;  // internal: the tiled-layout kernel

struct Plan {
    int variant;  // Q8_VARIANT_SIMT or Q8_VARIANT_MMA
    int V;        // columns per lane
    int ksplit;   // CTAs of a cluster splitting K
};

// Kernel family, per-lane width and K split for a shape.  The widest tile that still gives every SM a CTA is
// preferred; K is split across a cluster (at most 8 CTAs, the portable size) until the grid holds about as many CTAs
// as are resident at once (two per SM; one for the 8-row stream kernel).
Plan make_plan(int m, int K, int Np, int variant, bool tiled, int sms, long long tiled_tiles = 0, bool qact = false,
               bool rowmajor = false) {
    const int nb = K / Q8_BLOCK;
    if (tiled) {
        // The tiled layout: per-warp cp.async streams, 128-column tiles.  Measured on GB300, the best K split is
        // the largest one whose CTAs still fit in one wave of resident CTAs (a second, partial wave and the cluster
        // reduction both cost more than the idle SMs of a short wave): ks = resident slots / tiles, at least 1,
        // lowered while the tiles' clusters of ks CTAs would not all be resident at once (a cluster's CTAs share
        // one GPC, so fewer clusters fit than slots / ks).
        const long long groups = (m + q8::kGroupRows - 1) / q8::kGroupRows;
        const long long tiles = groups * (tiled_tiles > 0 ? tiled_tiles : (Np + q8::kTmaColumns - 1) / q8::kTmaColumns);
        const long long slots = (long long)q8::stream_ctas_per_sm(m, qact, rowmajor) * sms;
        // Clusters above the portable 8 CTAs only where 8 would leave more than half of the SMs idle (measured:
        // 5120 x 40 at m = 1 3.66 -> 2.83 us with 16; 5120 x 3000 at m = 16 8.90 -> 9.27 us with 12).
        const long long cap = tiles * 8 * 2 < sms ? q8::kMaxStreamSplit : 8;
        long long ks = slots / tiles;
        if (ks > cap) ks = cap;
        if (ks > nb) ks = nb;
        if (ks < 1) ks = 1;
        while (ks > 1) {
            const int fit = q8::stream_max_clusters(m, qact, (int)ks, rowmajor);
            if (fit <= 0 || tiles <= fit) break;
            --ks;
        }
        int best = (int)ks;
        const int f = tuning(Q8_TUNE_KSPLIT);
        if (f >= 1 && f <= nb) best = f;
        return Plan{kVariantStream, 16, best};
    }
    if (variant == Q8_VARIANT_AUTO) variant = Q8_VARIANT_TMA;
    if (variant == Q8_VARIANT_TMA && Np < q8::kTmaColumns) variant = Q8_VARIANT_MMA;
    if (variant == Q8_VARIANT_TMA) {
        // 128-column tiles, two resident CTAs per SM.  A CTA costs its blocks plus a fixed overhead (pipeline fill,
        // epilogue, cluster reduction) of about eight blocks; the K split is the one whose waves of CTAs finish first.
        const long long tiles = (Np + q8::kTmaColumns - 1) / q8::kTmaColumns;
        const long long slots = 2LL * sms;
        int best = 1;
        double best_cost = 1e300;
        for (int ks = 1; ks <= 8 && ks <= nb; ++ks) {
            const long long waves = (tiles * ks + slots - 1) / slots;
            const double cost = (double)waves * (8.0 + (double)((nb + ks - 1) / ks));
            if (cost < best_cost) {
                best_cost = cost;
                best = ks;
            }
        }
        const int f = tuning(Q8_TUNE_KSPLIT);
        if (f >= 1 && f <= nb) best = f;
        return Plan{Q8_VARIANT_TMA, 16, best};
    }
    if (variant == Q8_VARIANT_SIMT && !q8::simt_has(m, 4)) variant = Q8_VARIANT_MMA;
    static const int widths[3] = {16, 8, 4};
    Plan best = {variant, 0, 1};
    for (int i = 0; i < 3; ++i) {
        const int V = widths[i];
        const bool has = variant == Q8_VARIANT_SIMT ? q8::simt_has(m, V) : q8::mma_has(m, V);
        if (!has) continue;
        const int TC = variant == Q8_VARIANT_SIMT ? q8::simt_tile(V) : q8::mma_tile(V);
        const long long tiles = (Np + TC - 1) / TC;
        long long ks = (2LL * sms + tiles - 1) / tiles;
        if (ks > 8) ks = 8;
        if (ks > nb) ks = nb;
        if (ks < 1) ks = 1;
        best.V = V;
        best.ksplit = (int)ks;
        if (tiles * ks >= sms) break;
    }
    return best;
}

// m may be 1 .. 16, or 1 .. 512 over the tiled storage (row groups of 16 in one launch).
q8_status check_gemv_args(const void *x, const int8_t *q, const float *s, int m, int K, int N, unsigned flags) {
    if (!x || !q || !s) return Q8_ERR_ARG;
    const int max_rows = (flags & Q8_FLAG_TILED) ? Q8_MAX_CHUNK : Q8_MAX_ROWS;
    if (m < 1 || m > max_rows || K <= 0 || K % Q8_BLOCK != 0 || N <= 0) return Q8_ERR_SHAPE;
    if (q8_padded_n(N) < 0) return Q8_ERR_SHAPE;
    if (!aligned(x, 16) || !aligned(q, 16) || !aligned(s, 16)) return Q8_ERR_ALIGN;
    return Q8_OK;
}

int tiles_of(int N) { return (N + q8::kTmaColumns - 1) / q8::kTmaColumns; }

constexpr unsigned kKnownFlags = Q8_FLAG_CONSTANT_WEIGHTS | Q8_FLAG_TILED | Q8_FLAG_Q8_ACT;

// Flags a product entry point takes: the known ones, the quantized activation only over the tiled storage.
bool flags_ok(unsigned flags) {
    return (flags & ~kKnownFlags) == 0 && (!(flags & Q8_FLAG_Q8_ACT) || (flags & Q8_FLAG_TILED));
}

// Bytes of the activation operand: bf16 [m][K], or the quantized form (int8 [m][K] and fp32 [m][K/32]).
size_t x_bytes(unsigned flags, int m, int K) {
    return (flags & Q8_FLAG_Q8_ACT) ? (size_t)q8_act_bytes(m, K) : (size_t)m * K * 2;
}

// Whether a tiled call runs on the tcgen05 GEMM (prefill chunks of bf16 activations with a plain store) rather than
// the row groups of the streaming kernel: from gemm_min_rows() rows, when its 128 x 128 tiles (times the largest K
// split, 4) give at least 64 CTAs; a narrow weight keeps the row groups, whose grid is 8 times finer.  Q8_GEMM=0 in
// the tuning (Q8_TUNE_GEMM) keeps the row groups, 1 takes the GEMM for every such call whatever its width (both for
// comparison and tests).
bool use_gemm(int m, int epi, bool qact, long long col_tiles) {
    if (m < q8::gemm_min_rows() || epi != q8::kEpiStore || qact) return false;
    const int force = tuning(Q8_TUNE_GEMM);
    if (force == 0) return false;
    if (force == 1) return true;
    return col_tiles * ((m + 127) / 128) * 4 >= 64;
}

// A plain product (store or arg-max) or a gated pair of at most 16 rows whose one-launch plan has no K split but whose
// column tiles do not fill the resident slots evenly runs as two launches on the stream (a balance of the "plan.rs"
// `split_counts` kind: every SM gets about the same share of the blocks):
//   - tiles > SMs but below the slots (two CTAs per SM): the first launch takes one tile per SM, its CTAs held to one
//     per SM by their shared-memory size; the second takes the other tiles with K split over clusters of ks CTAs,
//     sized to the free half of every SM.  The gate/up pair (224 tiles on 152 SMs) then gives every SM 128 + 64 K
//     blocks instead of 256 on 72 SMs and 128 on the other 80;
//   - tiles above the slots: the first launch takes the whole waves, the second the last partial wave's tiles with K
//     split so that they fill one wave (the tied head's 1002 tiles: 3 waves of 304, then 90 tiles x 3).
// The first launch releases the second right after its own dependency wait, so the second's CTAs take the slots the
// first leaves free; the second waits for the first only before it exits, so whatever follows on the stream still
// sees both complete.  A K split below 2 would gain nothing, so it plans no split.
struct Split {
    int tiles_a = 0;  // tiles of the first launch (0: one launch)
    int ks_b = 1;     // the second launch's K split
    bool one_per_sm = false;
};
// pair: the gated pair, whose tiles are two CTAs each (the gate's and the up projection's, a cluster of 2 x ks, ks at
// most 4); else one CTA a tile (ks at most 8).
Split plan_split(long long tiles, int nb, int m, bool qact, int sms, int ks, bool pair = false, bool rowmajor = false) {
    Split none;
    // (a forced K split keeps one launch, so that it applies to every tile)
    if (tuning(Q8_TUNE_SPLIT) == 0 || tuning(Q8_TUNE_KSPLIT) != 0 || ks != 1 || m > q8::kGroupRows || sms <= 0)
        return none;
    const long long per = pair ? 2 : 1;  // CTAs a tile
    const long long slots = (long long)q8::stream_ctas_per_sm(m, qact, rowmajor) * sms;
    const long long ctas = per * tiles;
    long long ta;
    bool co;
    if (slots > sms && ctas > sms && ctas < slots) {
        ta = sms / per;
        co = true;
    } else if (ctas > slots && ctas % slots != 0) {
        ta = ctas / slots * slots / per;
        co = false;
    } else {
        return none;
    }
    const long long tb = tiles - ta;
    long long kb = (co ? sms : slots) / (per * tb);
    if (kb > 8 / per) kb = 8 / per;
    if (kb > nb) kb = nb;
    while (kb > 1) {  // clusters that are all resident at once (beside the first launch's CTAs: about half as many)
        const int fit = q8::stream_max_clusters(m, qact, (int)(per * kb), rowmajor);
        if (fit > 0 && tb <= (co ? fit / 2 : fit)) break;
        --kb;
    }
    if (kb < 2) return none;
    Split sp;
    sp.tiles_a = (int)ta;
    sp.ks_b = (int)kb;
    sp.one_per_sm = co;
    return sp;
}

q8_status run(const Args &a, int variant, unsigned flags, bool argmax, cudaStream_t stream,
              const q8::Parts *parts = nullptr) {
    const int epi = argmax ? q8::kEpiArgmax : q8::kEpiStore;
    int sms = 0;
    int e = sm_count(&sms);
    if (e != 0) return cuda_fail((cudaError_t)e);
    const bool tiled = (flags & Q8_FLAG_TILED) != 0;
    // the streaming kernels: tiled weights, and row-major ones when the caller leaves the kernel family to the library
    const bool streaming = tiled || variant == Q8_VARIANT_AUTO;
    q8::Parts one = {};
    if (streaming && !parts) {
        one.q[0] = a.q;
        one.s[0] = a.s;
        one.y[0] = a.y;
        one.N[0] = a.N;
        one.tile_end[0] = tiles_of(a.N);
        one.count = 1;
        parts = &one;
    }
    const bool qact = (flags & Q8_FLAG_Q8_ACT) != 0;
    const Plan p = make_plan(a.m, a.K, a.Np, variant, streaming, sms, parts ? parts->tile_end[parts->count - 1] : 0,
                             qact, !tiled);
    Args b = a;
    b.ksplit = p.ksplit;
    const bool prefetch = (flags & Q8_FLAG_CONSTANT_WEIGHTS) != 0;
    if (p.variant == kVariantStream && use_gemm(a.m, epi, qact, parts->tile_end[parts->count - 1])) {
        cudaError_t ce = q8::launch_gemm(b, *parts, stream);
        if (ce != cudaSuccess) return cuda_fail(ce);
        return Q8_OK;
    }
    const int mode = prefetch ? q8::kModePrefetch : 0;
    if (p.variant == kVariantStream) {
        const int tiles = parts->tile_end[parts->count - 1];
        const Split sp = plan_split(tiles, a.nb, a.m, qact, sms, b.ksplit, false, !tiled);
        if (sp.tiles_a > 0) {
            q8::StreamGrid ga;
            ga.ntiles = sp.tiles_a;
            ga.one_per_sm = sp.one_per_sm;
            cudaError_t ce = q8::launch_stream(b, *parts, epi, stream, true, mode | q8::kModeRelease, qact, !tiled, ga);
            if (ce != cudaSuccess) return cuda_fail(ce);
            Args c = b;
            c.tile0 = sp.tiles_a;
            c.ksplit = sp.ks_b;
            q8::StreamGrid gb;
            gb.ntiles = tiles - sp.tiles_a;
            ce = q8::launch_stream(c, *parts, epi, stream, true, mode | q8::kModeDeferWait, qact, !tiled, gb);
            if (ce != cudaSuccess) return cuda_fail(ce);
            return Q8_OK;
        }
    }
    cudaError_t ce = p.variant == kVariantStream    ? q8::launch_stream(b, *parts, epi, stream, true, mode, qact,
                                                                        !tiled)
                     : p.variant == Q8_VARIANT_TMA  ? q8::launch_tma(b, argmax, stream, true, prefetch)
                     : p.variant == Q8_VARIANT_SIMT ? q8::launch_simt(b, p.V, argmax, stream)
                                                    : q8::launch_mma(b, p.V, argmax, stream);
    if (ce != cudaSuccess) return cuda_fail(ce);
    return Q8_OK;
}

}  // namespace

extern "C" int q8_plan_launches(int m, int K, const int *Ns, int nparts, unsigned int flags) {
    if (!Ns || nparts < 1 || nparts > Q8_MAX_PARTS || !flags_ok(flags)) return -Q8_ERR_ARG;
    const bool tiled = (flags & Q8_FLAG_TILED) != 0;
    const int max_rows = tiled ? Q8_MAX_CHUNK : Q8_MAX_ROWS;
    if (m < 1 || m > max_rows || K <= 0 || K % Q8_BLOCK != 0) return -Q8_ERR_SHAPE;
    long long tiles = 0;
    for (int i = 0; i < nparts; ++i) {
        if (Ns[i] <= 0 || q8_padded_n(Ns[i]) < 0 || (tiled && q8_tiled_n(Ns[i]) < 0)) return -Q8_ERR_SHAPE;
        tiles += tiles_of(Ns[i]);
    }
    int sms = 0;
    if (sm_count(&sms) != 0) return -Q8_ERR_CUDA;
    const bool qact = (flags & Q8_FLAG_Q8_ACT) != 0;
    const Plan p = make_plan(m, K, q8_padded_n(Ns[0]), Q8_VARIANT_AUTO, true, sms, tiles, qact, !tiled);
    return plan_split(tiles, K / Q8_BLOCK, m, qact, sms, p.ksplit, false, !tiled).tiles_a > 0 ? 2 : 1;
}

namespace {

// keys[r] (the packed maximum written by the GEMV) -> the 0-based index it encodes, in place.
__global__ void argmax_decode(int64_t *idx, int m) {
    for (int r = threadIdx.x; r < m; r += blockDim.x) {
        const unsigned long long key = (unsigned long long)idx[r];
        idx[r] = (int64_t)(0xFFFFFFFFull - (key & 0xFFFFFFFFull));
    }
}

}  // namespace

extern "C" q8_status q8_gemv_ex(const void *x, const int8_t *q, const float *s, float *y, int m, int K, int N,
                                int variant, unsigned int flags, q8_stream_t stream) {
    q8_status st = check_gemv_args(x, q, s, m, K, N, flags);
    if (st != Q8_OK) return st;
    if (!y) return Q8_ERR_ARG;
    if (variant < Q8_VARIANT_AUTO || variant > Q8_VARIANT_TMA) return Q8_ERR_ARG;
    if (!flags_ok(flags)) return Q8_ERR_ARG;
    if ((flags & Q8_FLAG_TILED) && variant != Q8_VARIANT_AUTO) return Q8_ERR_ARG;
    if ((flags & Q8_FLAG_TILED) && q8_tiled_n(N) < 0) return Q8_ERR_SHAPE;
    if (!aligned(y, 16)) return Q8_ERR_ALIGN;
    const int Np = q8_padded_n(N);
    const size_t wcols = (flags & Q8_FLAG_TILED) ? (size_t)q8_tiled_n(N) : (size_t)Np;
    const size_t ybytes = (size_t)m * Np * 4;
    if (overlaps(y, ybytes, x, x_bytes(flags, m, K)) || overlaps(y, ybytes, q, (size_t)K * wcols) ||
        overlaps(y, ybytes, s, (size_t)(K / Q8_BLOCK) * wcols * 4))
        return Q8_ERR_ARG;
    Args a = {static_cast<const uint16_t *>(x), q, s, y, nullptr, m, K, N, Np, K / Q8_BLOCK, 1};
    return run(a, variant, flags, false, (cudaStream_t)stream);
}

extern "C" q8_status q8_gemv(const void *x, const int8_t *q, const float *s, float *y, int m, int K, int N,
                             q8_stream_t stream) {
    return q8_gemv_ex(x, q, s, y, m, K, N, Q8_VARIANT_AUTO, 0u, stream);
}

extern "C" q8_status q8_gemv_argmax_ex(const void *x, const int8_t *q, const float *s, int64_t *idx, float *logits,
                                       int m, int K, int N, unsigned int flags, q8_stream_t stream) {
    q8_status st = check_gemv_args(x, q, s, m, K, N, flags);
    if (st != Q8_OK) return st;
    if (!idx) return Q8_ERR_ARG;
    if (!flags_ok(flags)) return Q8_ERR_ARG;
    if ((flags & Q8_FLAG_TILED) && q8_tiled_n(N) < 0) return Q8_ERR_SHAPE;
    if (!aligned(idx, 8) || (logits && !aligned(logits, 16))) return Q8_ERR_ALIGN;
    const int Np = q8_padded_n(N);
    const size_t wcols = (flags & Q8_FLAG_TILED) ? (size_t)q8_tiled_n(N) : (size_t)Np;
    if (logits) {
        const size_t ybytes = (size_t)m * Np * 4;
        if (overlaps(logits, ybytes, x, x_bytes(flags, m, K)) || overlaps(logits, ybytes, q, (size_t)K * wcols) ||
            overlaps(logits, ybytes, s, (size_t)(K / Q8_BLOCK) * wcols * 4) ||
            overlaps(logits, ybytes, idx, (size_t)m * 8))
            return Q8_ERR_ARG;
    }
    if (overlaps(idx, (size_t)m * 8, x, x_bytes(flags, m, K))) return Q8_ERR_ARG;
    cudaStream_t cs = (cudaStream_t)stream;
    cudaError_t ce = cudaMemsetAsync(idx, 0, (size_t)m * sizeof(int64_t), cs);
    if (ce != cudaSuccess) return cuda_fail(ce);
    Args a = {static_cast<const uint16_t *>(x), q, s, logits, reinterpret_cast<unsigned long long *>(idx),
              m, K, N, Np, K / Q8_BLOCK, 1};
    st = run(a, Q8_VARIANT_AUTO, flags, true, cs);
    if (st != Q8_OK) return st;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(1, 1, 1);
    cfg.blockDim = dim3(m > 32 ? 128 : 32, 1, 1);
    cfg.stream = cs;
    ce = cudaLaunchKernelEx(&cfg, argmax_decode, idx, m);
    if (ce != cudaSuccess) return cuda_fail(ce);
    return Q8_OK;
}

extern "C" q8_status q8_gemv_argmax(const void *x, const int8_t *q, const float *s, int64_t *idx, float *logits,
                                    int m, int K, int N, q8_stream_t stream) {
    return q8_gemv_argmax_ex(x, q, s, idx, logits, m, K, N, 0u, stream);
}

extern "C" q8_status q8_gemv_parts(const void *x, const q8_part *parts, int nparts, int m, int K,
                                   unsigned int flags, q8_stream_t stream) {
    if (!x || !parts) return Q8_ERR_ARG;
    if (nparts < 1 || nparts > Q8_MAX_PARTS) return Q8_ERR_ARG;
    if (!flags_ok(flags)) return Q8_ERR_ARG;
    const bool tiled = (flags & Q8_FLAG_TILED) != 0;
    for (int i = 0; i < nparts; ++i) {
        const q8_part &p = parts[i];
        q8_status st = check_gemv_args(x, p.q, p.s, m, K, p.N, flags);
        if (st != Q8_OK) return st;
        if (!p.y) return Q8_ERR_ARG;
        if (!aligned(p.y, 16)) return Q8_ERR_ALIGN;
        if (tiled && q8_tiled_n(p.N) < 0) return Q8_ERR_SHAPE;
    }
    // No output may overlap the activation, any weight or any other output.
    for (int i = 0; i < nparts; ++i) {
        const size_t ybytes = (size_t)m * q8_padded_n(parts[i].N) * 4;
        if (overlaps(parts[i].y, ybytes, x, x_bytes(flags, m, K))) return Q8_ERR_ARG;
        for (int j = 0; j < nparts; ++j) {
            const size_t wcols = tiled ? (size_t)q8_tiled_n(parts[j].N) : (size_t)q8_padded_n(parts[j].N);
            if (overlaps(parts[i].y, ybytes, parts[j].q, (size_t)K * wcols) ||
                overlaps(parts[i].y, ybytes, parts[j].s, (size_t)(K / Q8_BLOCK) * wcols * 4))
                return Q8_ERR_ARG;
            if (j != i && overlaps(parts[i].y, ybytes, parts[j].y, (size_t)m * q8_padded_n(parts[j].N) * 4))
                return Q8_ERR_ARG;
        }
    }
    cudaStream_t cs = (cudaStream_t)stream;
    q8::Parts pt = {};
    int tiles = 0;
    for (int i = 0; i < nparts; ++i) {
        pt.q[i] = parts[i].q;
        pt.s[i] = parts[i].s;
        pt.y[i] = parts[i].y;
        pt.N[i] = parts[i].N;
        tiles += tiles_of(parts[i].N);
        pt.tile_end[i] = tiles;
    }
    pt.count = nparts;
    Args a = {static_cast<const uint16_t *>(x), parts[0].q, parts[0].s, parts[0].y, nullptr, m, K, parts[0].N,
              q8_padded_n(parts[0].N), K / Q8_BLOCK, 1};
    return run(a, Q8_VARIANT_AUTO, flags, false, cs, &pt);
}

// The K split of a gated-pair launch: its clusters are (2, ks), a gate's and an up projection's CTA for each K range
// of one column tile, so the one-wave rule counts 2 * tiles * ks CTAs and clusters of 2 * ks (at most 8).
int plan_glu(long long tiles, int nb, int sms, int m, bool qact) {
    const long long slots = (long long)q8::stream_ctas_per_sm(m, qact) * sms;
    long long ks = slots / (2 * tiles);
    if (ks > 4) ks = 4;
    if (ks > nb) ks = nb;
    if (ks < 1) ks = 1;
    while (ks > 1) {
        const int fit = q8::stream_max_clusters(m, qact, (int)(2 * ks));
        if (fit <= 0 || tiles <= fit) break;
        --ks;
    }
    const int f = tuning(Q8_TUNE_KSPLIT);
    if (f >= 1 && f <= 4 && f <= nb) ks = f;
    return (int)ks;
}

extern "C" int q8_plan_glu_launches(int m, int K, int N, unsigned int flags) {
    if (!flags_ok(flags) || !(flags & Q8_FLAG_TILED)) return -Q8_ERR_ARG;
    if (m < 1 || m > Q8_MAX_CHUNK || K <= 0 || K % Q8_BLOCK != 0 || N <= 0 || q8_tiled_n(N) < 0) return -Q8_ERR_SHAPE;
    int sms = 0;
    if (sm_count(&sms) != 0) return -Q8_ERR_CUDA;
    const bool qact = (flags & Q8_FLAG_Q8_ACT) != 0;
    const int groups = (m + q8::kGroupRows - 1) / q8::kGroupRows;
    const long long tiles = (long long)tiles_of(N) * groups;
    const int ks = plan_glu(tiles, K / Q8_BLOCK, sms, m, qact);
    return plan_split(tiles, K / Q8_BLOCK, m, qact, sms, ks, true).tiles_a > 0 ? 2 : 1;
}

extern "C" q8_status q8_gemv_glu_ex(const void *x, const int8_t *qg, const float *sg, const int8_t *qu,
                                    const float *su, float *out, void *out_bf16, void *out_q8, int m, int K, int N,
                                    unsigned int flags, q8_stream_t stream) {
    q8_status st = check_gemv_args(x, qg, sg, m, K, N, flags);
    if (st != Q8_OK) return st;
    st = check_gemv_args(x, qu, su, m, K, N, flags);
    if (st != Q8_OK) return st;
    if (!out && !out_bf16 && !out_q8) return Q8_ERR_ARG;
    if (!flags_ok(flags)) return Q8_ERR_ARG;
    if (!(flags & Q8_FLAG_TILED)) return Q8_ERR_ARG;  // the gated pair runs on the tiled storage only
    if (q8_tiled_n(N) < 0) return Q8_ERR_SHAPE;
    if ((out && !aligned(out, 16)) || (out_bf16 && !aligned(out_bf16, 16)) || (out_q8 && !aligned(out_q8, 16)))
        return Q8_ERR_ALIGN;
    const int Np = q8_padded_n(N);
    const size_t wcols = (size_t)q8_tiled_n(N);
    const size_t obytes[3] = {(size_t)m * Np * 4, (size_t)m * Np * 2, (size_t)q8_act_bytes(m, Np)};
    const void *outs[3] = {out, out_bf16, out_q8};
    for (int o = 0; o < 3; ++o) {
        if (!outs[o]) continue;
        if (overlaps(outs[o], obytes[o], x, x_bytes(flags, m, K)) ||
            overlaps(outs[o], obytes[o], qg, (size_t)K * wcols) || overlaps(outs[o], obytes[o], qu, (size_t)K * wcols) ||
            overlaps(outs[o], obytes[o], sg, (size_t)(K / Q8_BLOCK) * wcols * 4) ||
            overlaps(outs[o], obytes[o], su, (size_t)(K / Q8_BLOCK) * wcols * 4))
            return Q8_ERR_ARG;
        for (int p = 0; p < o; ++p)
            if (outs[p] && overlaps(outs[o], obytes[o], outs[p], obytes[p])) return Q8_ERR_ARG;
    }
    int sms = 0;
    int e = sm_count(&sms);
    if (e != 0) return cuda_fail((cudaError_t)e);
    const int tiles = tiles_of(N);
    const int groups = (m + q8::kGroupRows - 1) / q8::kGroupRows;
    q8::Parts pt = {};
    pt.q[0] = qg;
    pt.s[0] = sg;
    pt.q[1] = qu;
    pt.s[1] = su;
    pt.N[0] = pt.N[1] = N;
    pt.tile_end[0] = tiles;
    pt.tile_end[1] = 2 * tiles;  // grid x: the two parts' CTAs of each tile side by side
    pt.count = 2;
    Args a = {static_cast<const uint16_t *>(x), qg, sg, out, nullptr, m, K, N, Np, K / Q8_BLOCK, 1,
              static_cast<uint16_t *>(out_bf16)};
    if (out_q8) {
        a.yq = static_cast<unsigned char *>(out_q8);
        a.yd = reinterpret_cast<float *>(a.yq + (size_t)m * Np);
    }
    const bool qact = (flags & Q8_FLAG_Q8_ACT) != 0;
    const int mode = (flags & Q8_FLAG_CONSTANT_WEIGHTS) ? q8::kModePrefetch : 0;
    a.ksplit = plan_glu((long long)tiles * groups, K / Q8_BLOCK, sms, m, qact);
    const Split sp = plan_split((long long)tiles * groups, K / Q8_BLOCK, m, qact, sms, a.ksplit, true);
    cudaError_t ce;
    if (sp.tiles_a > 0) {
        q8::StreamGrid ga;
        ga.ntiles = 2 * sp.tiles_a;  // grid columns: two CTAs a tile
        ga.one_per_sm = sp.one_per_sm;
        ce = q8::launch_stream(a, pt, q8::kEpiGlu, (cudaStream_t)stream, true, mode | q8::kModeRelease, qact, false,
                               ga);
        if (ce != cudaSuccess) return cuda_fail(ce);
        Args c = a;
        c.tile0 = 2 * sp.tiles_a;
        c.ksplit = sp.ks_b;
        q8::StreamGrid gb;
        gb.ntiles = 2 * (tiles - sp.tiles_a);
        ce = q8::launch_stream(c, pt, q8::kEpiGlu, (cudaStream_t)stream, true, mode | q8::kModeDeferWait, qact, false,
                               gb);
    } else {
        ce = q8::launch_stream(a, pt, q8::kEpiGlu, (cudaStream_t)stream, true, mode, qact);
    }
    if (ce != cudaSuccess) return cuda_fail(ce);
    return Q8_OK;
}

extern "C" q8_status q8_gemv_glu(const void *x, const int8_t *qg, const float *sg, const int8_t *qu,
                                 const float *su, float *out, void *out_bf16, int m, int K, int N, unsigned int flags,
                                 q8_stream_t stream) {
    return q8_gemv_glu_ex(x, qg, sg, qu, su, out, out_bf16, nullptr, m, K, N, flags, stream);
}

// Whether a residual-norm call runs its RMS norm as a launch of its own (one CTA per row, chained by programmatic
// dependent launch) rather than in the product's last CTA.  Measured on GB300 (4096 x 4096, bf16 output), the own
// launch is faster at every row count: 8.4 against 10.0 us a call at m = 1, 12.8 against 21.9 at m = 16, since the
// last CTA's pass over every row is the fold's tail.  The tuning Q8_TUNE_NORM_FOLD = 1 keeps the norm in the
// product's last CTA (for comparison and tests).
bool norm_own_launch() { return tuning(Q8_TUNE_NORM_FOLD) == 0; }

extern "C" q8_status q8_gemv_residual_norm_ex(const void *x, const int8_t *q, const float *s, const float *residual,
                                              const float *gamma, float eps, float *h, void *out_bf16, void *out_q8,
                                              int m, int K, int N, unsigned int flags, q8_stream_t stream) {
    q8_status st = check_gemv_args(x, q, s, m, K, N, flags);
    if (st != Q8_OK) return st;
    if (!residual || !gamma || !h || (!out_bf16 && !out_q8)) return Q8_ERR_ARG;
    if (!flags_ok(flags)) return Q8_ERR_ARG;
    if (!(flags & Q8_FLAG_TILED)) return Q8_ERR_ARG;  // the tiled storage only
    if (!(eps >= 0.0f) || !(eps < INFINITY)) return Q8_ERR_ARG;
    if (q8_tiled_n(N) < 0) return Q8_ERR_SHAPE;
    if (!aligned(h, 16) || (out_bf16 && !aligned(out_bf16, 16)) || (out_q8 && !aligned(out_q8, 16)) ||
        !aligned(residual, 4) || !aligned(gamma, 4))
        return Q8_ERR_ALIGN;
    const int Np = q8_padded_n(N);
    const size_t wcols = (size_t)q8_tiled_n(N);
    const size_t hbytes = (size_t)m * Np * 4, obytes = (size_t)m * Np * 2, qbytes = (size_t)q8_act_bytes(m, Np);
    // h may be the residual itself (in place) but may not overlap it otherwise, nor any other operand.
    if (h != residual && overlaps(h, hbytes, residual, hbytes)) return Q8_ERR_ARG;
    const void *ins[4] = {x, q, s, gamma};
    const size_t inb[4] = {x_bytes(flags, m, K), (size_t)K * wcols, (size_t)(K / Q8_BLOCK) * wcols * 4, (size_t)Np * 4};
    const void *outs[2] = {out_bf16, out_q8};
    const size_t outb[2] = {obytes, qbytes};
    for (int o = 0; o < 2; ++o) {
        if (!outs[o]) continue;
        for (int i = 0; i < 4; ++i)
            if (overlaps(outs[o], outb[o], ins[i], inb[i])) return Q8_ERR_ARG;
        if (overlaps(outs[o], outb[o], h, hbytes) || overlaps(outs[o], outb[o], residual, hbytes)) return Q8_ERR_ARG;
    }
    for (int i = 0; i < 4; ++i)
        if (overlaps(h, hbytes, ins[i], inb[i])) return Q8_ERR_ARG;
    if (out_bf16 && out_q8 && overlaps(out_bf16, obytes, out_q8, qbytes)) return Q8_ERR_ARG;
    q8::NormRows nr = {h, gamma, eps, static_cast<uint16_t *>(out_bf16), static_cast<unsigned char *>(out_q8),
                       out_q8 ? reinterpret_cast<float *>(static_cast<unsigned char *>(out_q8) + (size_t)m * Np)
                              : nullptr,
                       N, Np};
    const bool own_launch = norm_own_launch();
    Args a = {static_cast<const uint16_t *>(x), q, s, h, nullptr, m, K, N, Np, K / Q8_BLOCK, 1, nullptr, residual,
              gamma, eps, nullptr, 0};
    if (!own_launch) {
        // one completion counter per row group, taken round robin
        static std::atomic<unsigned> next_counter{0};
        const unsigned groups = (unsigned)((m + q8::kGroupRows - 1) / q8::kGroupRows);
        a.count_slot = (int)(next_counter.fetch_add(groups, std::memory_order_relaxed) % q8::kNormSlots);
        a.count = q8::norm_counters();
        if (!a.count) return cuda_fail(cudaGetLastError());
        a.ybf = nr.ybf;
        a.yq = nr.yq;
        a.yd = nr.yd;
    }
    int sms = 0;
    int e = sm_count(&sms);
    if (e != 0) return cuda_fail((cudaError_t)e);
    q8::Parts pt = {};
    pt.q[0] = q;
    pt.s[0] = s;
    pt.y[0] = h;
    pt.N[0] = N;
    pt.tile_end[0] = tiles_of(N);
    pt.count = 1;
    const Plan p = make_plan(m, K, Np, Q8_VARIANT_AUTO, true, sms, pt.tile_end[0], (flags & Q8_FLAG_Q8_ACT) != 0);
    a.ksplit = p.ksplit;
    cudaError_t ce = q8::launch_stream(a, pt, q8::kEpiNorm, (cudaStream_t)stream, true,
                                       (flags & Q8_FLAG_CONSTANT_WEIGHTS) ? q8::kModePrefetch : 0,
                                       (flags & Q8_FLAG_Q8_ACT) != 0);
    if (ce != cudaSuccess) return cuda_fail(ce);
    if (own_launch) {
        ce = q8::launch_norm_rows(nr, m, (cudaStream_t)stream, true);
        if (ce != cudaSuccess) return cuda_fail(ce);
    }
    return Q8_OK;
}

extern "C" q8_status q8_gemv_residual_norm(const void *x, const int8_t *q, const float *s, const float *residual,
                                           const float *gamma, float eps, float *h, void *out_bf16, int m, int K,
                                           int N, unsigned int flags, q8_stream_t stream) {
    if (!out_bf16) return Q8_ERR_ARG;
    return q8_gemv_residual_norm_ex(x, q, s, residual, gamma, eps, h, out_bf16, nullptr, m, K, N, flags, stream);
}

extern "C" q8_status q8_device_fault(unsigned int *fault, int clear) {
    if (!fault) return Q8_ERR_ARG;
    unsigned gemm = 0;
    cudaError_t e = q8::read_fault_word(fault, clear != 0);
    if (e == cudaSuccess) e = q8::read_gemm_fault(&gemm, clear != 0);
    if (e != cudaSuccess) return cuda_fail(e);
    *fault |= gemm;
    return Q8_OK;
}

namespace q8 {
int forced_ksplit() { return tuning(Q8_TUNE_KSPLIT); }
}  // namespace q8

extern "C" q8_status q8_set_tuning(int option, int value) {
    if (option < 0 || option >= kTuneOptions) return Q8_ERR_ARG;
    const bool ok = option == Q8_TUNE_KSPLIT ? (value >= 0 && value <= 8)
                    : option == Q8_TUNE_GEMM ? (value >= -1 && value <= 1)
                                             : (value == 0 || value == 1);
    if (!ok) return Q8_ERR_ARG;
    tuning_table().value[option].store(value, std::memory_order_relaxed);
    return Q8_OK;
}

extern "C" int q8_get_tuning(int option) {
    if (option < 0 || option >= kTuneOptions) return -2;
    return tuning(option);
}

// ---------------------------------------------------------------------------------------------------------------------
// The residual norm's one-launch fold for callers that cannot allocate device memory
// ---------------------------------------------------------------------------------------------------------------------

namespace {

// The fold's only scratch: one completion counter per group of 16 rows, in this file's own static device array
// (every GPU that loads the library holds these 128 bytes until the process exits).  Every call uses counters
// 0 .. groups-1 and clears them first, so calls whose kernels overlap on a GPU race on them.
constexpr int kFoldStaticGroups = Q8_FOLD_STATIC_MAX_ROWS / q8::kGroupRows;
static __device__ __align__(256) unsigned int g_fold_static_counters[kFoldStaticGroups];
static_assert(kFoldStaticGroups <= q8::kNormSlots, "the kernel takes counter (slot + group) % kNormSlots");

// The device address of g_fold_static_counters on the current device.  In host code the array's name stands for a
// host-side shadow, not for device memory, so the address is asked of the runtime -- once per device, with that
// device current, on the first call there -- and kept.
cudaError_t fold_static_counters(unsigned int **out) {
    static std::atomic<unsigned int *> cache[64];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) {
        unsigned int *p = cache[dev].load(std::memory_order_acquire);
        if (p) {
            *out = p;
            return cudaSuccess;
        }
    }
    void *base = nullptr;
    e = cudaGetSymbolAddress(&base, g_fold_static_counters);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) cache[dev].store(static_cast<unsigned int *>(base), std::memory_order_release);
    *out = static_cast<unsigned int *>(base);
    return cudaSuccess;
}

}  // namespace

extern "C" q8_status q8_gemv_residual_norm_noalloc(const void *x, const int8_t *q, const float *s,
                                                   const float *residual, const float *gamma, float eps, float *h,
                                                   void *out_bf16, int m, int K, int N, unsigned int flags,
                                                   q8_stream_t stream) {
    if (m > Q8_FOLD_STATIC_MAX_ROWS) return Q8_ERR_SHAPE;  // more row groups than the static counters
    q8_status st = check_gemv_args(x, q, s, m, K, N, flags);
    if (st != Q8_OK) return st;
    if (!residual || !gamma || !h || !out_bf16) return Q8_ERR_ARG;
    if (!flags_ok(flags) || !(flags & Q8_FLAG_TILED)) return Q8_ERR_ARG;
    if (!(eps >= 0.0f) || !(eps < INFINITY)) return Q8_ERR_ARG;
    if (q8_tiled_n(N) < 0) return Q8_ERR_SHAPE;
    if (!aligned(h, 16) || !aligned(out_bf16, 16) || !aligned(residual, 4) || !aligned(gamma, 4)) return Q8_ERR_ALIGN;
    const int Np = q8_padded_n(N);
    const size_t wcols = (size_t)q8_tiled_n(N);
    const size_t hbytes = (size_t)m * Np * 4, obytes = (size_t)m * Np * 2;
    if (h != residual && overlaps(h, hbytes, residual, hbytes)) return Q8_ERR_ARG;
    const void *ins[4] = {x, q, s, gamma};
    const size_t inb[4] = {x_bytes(flags, m, K), (size_t)K * wcols, (size_t)(K / Q8_BLOCK) * wcols * 4, (size_t)Np * 4};
    for (int i = 0; i < 4; ++i)
        if (overlaps(out_bf16, obytes, ins[i], inb[i]) || overlaps(h, hbytes, ins[i], inb[i])) return Q8_ERR_ARG;
    if (overlaps(out_bf16, obytes, h, hbytes) || overlaps(out_bf16, obytes, residual, hbytes)) return Q8_ERR_ARG;

    unsigned int *counters = nullptr;
    cudaError_t ce = fold_static_counters(&counters);
    if (ce != cudaSuccess) return cuda_fail(ce);
    int sms = 0;
    int e = sm_count(&sms);
    if (e != 0) return cuda_fail((cudaError_t)e);
    cudaStream_t cs = (cudaStream_t)stream;
    const int groups = (m + q8::kGroupRows - 1) / q8::kGroupRows;
    // the counters must start at zero: a memset node, which allocates nothing
    ce = cudaMemsetAsync(counters, 0, (size_t)groups * sizeof(unsigned int), cs);
    if (ce != cudaSuccess) return cuda_fail(ce);
    q8::Parts pt = {};
    pt.q[0] = q;
    pt.s[0] = s;
    pt.y[0] = h;
    pt.N[0] = N;
    pt.tile_end[0] = tiles_of(N);
    pt.count = 1;
    Args a = {static_cast<const uint16_t *>(x), q, s, h, nullptr, m, K, N, Np, K / Q8_BLOCK, 1,
              static_cast<uint16_t *>(out_bf16), residual, gamma, eps, counters, 0};
    a.ksplit = make_plan(m, K, Np, Q8_VARIANT_AUTO, true, sms, pt.tile_end[0], (flags & Q8_FLAG_Q8_ACT) != 0).ksplit;
    // a plain stream-ordered launch after the memset (no programmatic dependent launch)
    ce = q8::launch_stream(a, pt, q8::kEpiNorm, cs, false, 0, (flags & Q8_FLAG_Q8_ACT) != 0);
    if (ce != cudaSuccess) return cuda_fail(ce);
    return Q8_OK;
}
