/*
 * q8_gemv.h -- C ABI of the GB300 Q8_0 block-quantized GEMV library (libq8gemv.so).
 *
 * The product (source: "logicaffeine_compile/spatial/passes/from_q8.rs", module doc):
 *
 *     y[r, n] = sum_b s[b, n] * sum_{i<32} x[r, 32b + i] * q[32b + i, n]        r < m, n < N
 *
 * over a weight stored Q8_0: int8 values q (`W__q8`, K x N) and one fp32 scale per 32-row block of each column
 * (`W__q8_scale`, K/32 x N), about 1.125 bytes a weight against 2 for bf16.  Activations x are bf16, accumulation is
 * fp32, and a batch of m <= 16 rows reads the weight once for all its rows.
 *
 * Layouts (all row-major, no strides):
 *   x  bf16    [m][K]        row pitch K elements
 *   q  int8    [K][Np]       row pitch Np bytes; Np = q8_padded_n(N) = N rounded up to a multiple of 32
 *   s  fp32    [K/32][Np]    row pitch Np elements
 *   y  fp32    [m][Np]       row pitch Np elements
 * Columns N .. Np-1 are the zero-padded last 32-column tile ("from_q8.rs", `q8_gemv_applies`): their q and s should
 * be 0 (q8_repack and q8_quantize write them so); the GEMV writes exactly 0.0f into y's pad columns regardless.
 *
 * Conventions shared by every entry point:
 *   - The caller owns every buffer and the library allocates no memory.  Its only state is read-only caches (per
 *     device: SM count, resident clusters), the device fault words (q8_device_fault), the planner overrides of
 *     q8_set_tuning, the residual norm's 64 static completion counters (used only by its one-launch fold; see
 *     q8_gemv_residual_norm for the limit this puts on overlapping calls) and the 32 static counters of
 *     q8_gemv_residual_norm_noalloc (see there).
 *   - Device entry points take device pointers and enqueue work on `stream` (a cudaStream_t; NULL is the legacy
 *     default stream).  They are asynchronous: Q8_OK means the work was enqueued.  An argument error is returned
 *     before anything is enqueued.  A CUDA error at launch returns Q8_ERR_CUDA; q8_last_cuda_error() then gives the
 *     cudaError_t value for the calling thread.
 *   - Host entry points take host pointers and run synchronously on the calling thread.
 *   - No entry point aborts, throws or prints.
 *   - Every call is thread-safe; calls on one stream run in order.  The exception is the residual norm's one-launch
 *     fold (q8_set_tuning Q8_TUNE_NORM_FOLD = 1): at most 64 of its row groups may be in flight at once over all
 *     streams and threads.
 */
#ifndef Q8_GEMV_H
#define Q8_GEMV_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ABI-identical to cudaStream_t; declared here so that the header needs no CUDA headers. */
struct CUstream_st;
typedef struct CUstream_st *q8_stream_t;

/* Rows of a Q8_0 block ("from_q8.rs", `Q8_BLOCK`). */
#define Q8_BLOCK 32
/* The most activation rows one call takes ("plan.rs", `GEMV_ROWS`: a GEMV launch multiplies at most 16 rows). */
#define Q8_MAX_ROWS 16

/* The most activation rows one call over the tiled storage takes ("plan.rs", `MAX_CHUNK`: the largest prefill chunk
 * a lane compiles, 512; its projections of more rows than the GEMV's 16 run on the tensor cores).  With
 * Q8_FLAG_TILED, m may be 1 .. 512: from 128 rows a plain product of bf16 activations runs as a tensor-core GEMM
 * (tcgen05, 128 x 128 output tiles, each 32-row block contracted exactly and folded with its scales); otherwise the
 * rows run as ceil(m / 16) groups of 16 in one launch, each group's CTAs of a column tile side by side so that the
 * weight is streamed from HBM about once. */
#define Q8_MAX_CHUNK 512

typedef enum {
    Q8_OK = 0,
    Q8_ERR_ARG = 1,      /* a required pointer is NULL, or an enum argument is out of range */
    Q8_ERR_SHAPE = 2,    /* m outside 1..16, K <= 0, K % 32 != 0, N <= 0, or a size that overflows */
    Q8_ERR_ALIGN = 3,    /* a device pointer is not 16-byte aligned */
    Q8_ERR_NOT_Q8_0 = 4, /* a weight or block that is not Q8_0 (see q8_quantize, q8_repack) */
    Q8_ERR_CUDA = 5      /* the CUDA runtime reported an error; see q8_last_cuda_error() */
} q8_status;

/* Kernel family selector for q8_gemv_ex (benchmarking and testing).  AUTO, what q8_gemv takes, runs the streaming
 * kernels: each warp copies its 32-row x 128-column blocks of the row-major weight into a shared-memory ring with
 * cp.async and reads them back transposed (ldmatrix .trans .b8) in the tiled storage's word order, so the row-major
 * weight streams through the same kernels as the tiled one.  The others are earlier designs kept for comparison. */
typedef enum {
    Q8_VARIANT_AUTO = 0,
    Q8_VARIANT_SIMT = 1, /* CUDA-core fp32 FMA, m-row accumulators per thread, weights loaded straight to registers */
    Q8_VARIANT_MMA = 2,  /* int8 -> bf16 exact dequant in registers, bf16 tensor-core MMA, fp32 per-block scale fold */
    Q8_VARIANT_TMA = 3   /* as MMA, the weight streamed by TMA through a 16-stage shared-memory pipeline by a producer
                            warp; launched with programmatic dependent launch.  Needs N > 96 (Np >= 128); smaller N
                            falls back to MMA. */
} q8_variant;

/* N rounded up to whole 32-column tiles ("from_q8.rs", `q8_gemv_applies`: the last tile is zero-padded).
 * Returns -1 when N <= 0 or the result would overflow an int. */
int q8_padded_n(int N);

/* y = x . W over the Q8_0 weight (q, s), m rows (source: "from_q8.rs", module doc and `q8_fold`).
 *   x  device, bf16 [m][K], 16-byte aligned        q  device, int8 [K][Np], 16-byte aligned
 *   s  device, fp32 [K/32][Np], 16-byte aligned    y  device, fp32 [m][Np] (written), 16-byte aligned
 *   1 <= m <= 16 (1 <= m <= 512 over the tiled storage, Q8_MAX_CHUNK), K > 0, K % 32 == 0 ("from_q8.rs",
 *   `q8_gemv_applies`), N > 0.
 * y must not overlap x, q or s.  Every output n < Np is written; outputs n >= N are 0.0f.
 * Each y[r, n] equals the real-number product within 1e-5 * sum_b |s[b,n]| sum_i |x[r,32b+i] q[32b+i,n]|; the
 * summation order is fixed for a given (m, K, N) and device, so repeated calls give identical bits. */
q8_status q8_gemv(const void *x, const int8_t *q, const float *s, float *y, int m, int K, int N, q8_stream_t stream);

/* Flags of q8_gemv_ex. */
#define Q8_FLAG_CONSTANT_WEIGHTS 1u /* no work enqueued before this call on `stream` writes q or s: the pipelined
                                       kernel may start streaming them before the previous kernel on the stream has
                                       finished (programmatic dependent launch); x and y are still ordered */

#define Q8_FLAG_TILED 2u            /* q and s are in the tiled layout of q8_tile (below), not row-major; read by the
                                       per-warp cp.async streaming kernel (variant must be AUTO) */

#define Q8_FLAG_Q8_ACT 4u           /* x is the quantized form of the activation written by q8_quantize_act (below),
                                       not bf16 values, and the product is the quantized numerics'
                                           y[r, n] = sum_b s[b, n] * d[r, b] * sum_i xq[r, 32b+i] * q[32b+i, n]
                                       (its integer inner sums exact); requires Q8_FLAG_TILED.  Every product entry
                                       point takes it; the bound is as before with xq * d in place of x */

/* q8_gemv with an explicit kernel family (q8_variant) and flags (Q8_FLAG_*; 0 for none).  Same arguments and
 * bound; Q8_ERR_ARG for an unknown variant or flag, for Q8_FLAG_TILED with a variant other than AUTO, or for
 * Q8_FLAG_Q8_ACT without Q8_FLAG_TILED. */
q8_status q8_gemv_ex(const void *x, const int8_t *q, const float *s, float *y, int m, int K, int N, int variant,
                     unsigned int flags, q8_stream_t stream);

/* The product followed by the arg-max that ends a decode step (source: "plan.rs", `Launch::ArgMax`, and
 * "int8_model.rs", `decode_step_lg`: the lowest index among the largest logits; its CUDA arg-max sends equal values to
 * the lower index).
 *   idx     device, int64 [m] (written), 8-byte aligned: idx[r] = the smallest n < N with y[r, n] equal to the
 *           largest y[r, n'] over n' < N, 0-based.  Pad columns never take part.  +0.0 and -0.0 count as equal.
 *           The buffer also serves as the call's cross-block scratch: its contents before the call do not matter.
 *   logits  device, fp32 [m][Np] (written, as q8_gemv's y) or NULL to skip storing the logits.
 * Other arguments as q8_gemv.  Logits that are NaN order above +inf (not reached for finite inputs). */
q8_status q8_gemv_argmax(const void *x, const int8_t *q, const float *s, int64_t *idx, float *logits, int m, int K,
                         int N, q8_stream_t stream);

/* q8_gemv_argmax with flags (Q8_FLAG_CONSTANT_WEIGHTS, Q8_FLAG_TILED). */
q8_status q8_gemv_argmax_ex(const void *x, const int8_t *q, const float *s, int64_t *idx, float *logits, int m,
                            int K, int N, unsigned int flags, q8_stream_t stream);

/* The tiled storage of a Q8_0 weight, for Q8_FLAG_TILED (no counterpart on the pages: a GPU storage order of the
 * same two tensors, made once when the weight is loaded, as the host repack of "from_q8.rs" `Q8Part` is).  Every
 * 32-row x 128-column block becomes one contiguous 4 KB unit laid out in the order the kernel's lanes load it, so a
 * warp streaming one column tile along K reads contiguous memory.  With Nt = q8_tiled_n(N), T = Nt / 128 tiles and
 * nb = K / 32 blocks:
 *   values  uint8 [T][nb][4096]: in unit (t, b), segment 4s + h (s = 0, 1; h = 0..3; 512 bytes each) holds at byte
 *           16 * (4g + u) (g = 0..7, u = 0..3) four words; word w holds weight rows 32b + 16s + 4u + k (byte k,
 *           k = 0..3) of column 128t + 8(4h + w) + g, each value stored as q + 128 (offset binary)
 *   scales  fp32 [T][nb][128]: element c of unit (t, b) is s[b][128t + c]
 * Columns >= N hold q = 0 (byte 128) and scale 0.  Sizes: K * Nt bytes of values, (K / 32) * Nt * 4 bytes of
 * scales. */
int q8_tiled_n(int N); /* N rounded up to a multiple of 128; -1 when N <= 0 or on overflow */

/* Host: row-major q [K][Np], s [K/32][Np] (as q8_gemv takes them) -> tiled qt, st (host buffers, written). */
q8_status q8_tile(const int8_t *q, const float *s, int K, int N, int8_t *qt, float *st);

/* Device: the same transform on device buffers, enqueued on `stream` (q, qt 16-byte aligned; s, st 4-byte aligned;
 * the input and output must not overlap). */
q8_status q8_tile_device(const int8_t *q, const float *s, int K, int N, int8_t *qt, float *st, q8_stream_t stream);

/* The gated pair ("plan.rs", `Launch::GemvGlu`: two projections of one activation through a gate,
 * out = act(x.wg + bg) * (x.wu + bu), silu gating (SwiGLU) by default; here without biases):
 *     out[r, n] = silu(g[r, n]) * u[r, n],   g = x . Wg,  u = x . Wu,   silu(g) = g / (1 + exp(-g)),
 * g and u each the Q8_0 product of q8_gemv (fp32 accumulation), silu and the product in fp32 (CUDA's expf, IEEE
 * division).  One launch (two when the planner splits it, Q8_TUNE_SPLIT, q8_plan_glu_launches): the gate's and the
 * up projection's CTAs of a column tile run side by side in a cluster.
 *   x         device, bf16 [m][K], 16-byte aligned
 *   qg, sg    device, the gate's weight in the tiled storage (q8_tile), 16-byte aligned
 *   qu, su    device, the up projection's weight, tiled, 16-byte aligned
 *   out       device, fp32 [m][Np] (written; pad columns 0), 16-byte aligned, or NULL
 *   out_bf16  device, bf16 [m][Np] (written: out rounded to nearest even; pads 0), 16-byte aligned, or NULL
 *             -- a down projection's activation as q8_gemv takes it (row pitch Np)
 *   flags     Q8_FLAG_TILED (required) | Q8_FLAG_CONSTANT_WEIGHTS
 * Errors: Q8_ERR_ARG (null inputs, both outputs null, flags without Q8_FLAG_TILED or with unknown bits, an output
 * overlapping an input or the other output), Q8_ERR_SHAPE, Q8_ERR_ALIGN, Q8_ERR_CUDA; nothing is launched on an
 * error.  inf and NaN propagate as IEEE arithmetic does (silu(-inf) = -inf / inf = NaN). */
q8_status q8_gemv_glu(const void *x, const int8_t *qg, const float *sg, const int8_t *qu, const float *su, float *out,
                      void *out_bf16, int m, int K, int N, unsigned int flags, q8_stream_t stream);

/* q8_gemv_glu with a third, optional output: out_q8 (device, q8_act_bytes(m, Np) bytes, 16-byte aligned, or NULL)
 * receives the quantized form of the bf16 output -- exactly what q8_quantize_act of out_bf16 (as [m][Np]) writes --
 * from the same launch ("plan.rs": an op may emit fp32, the quantized form, or the two together; `GluActMulQuant`),
 * ready for a Q8_FLAG_Q8_ACT product with K = Np.  At least one of out, out_bf16, out_q8; no two may overlap. */
q8_status q8_gemv_glu_ex(const void *x, const int8_t *qg, const float *sg, const int8_t *qu, const float *su,
                         float *out, void *out_bf16, void *out_q8, int m, int K, int N, unsigned int flags,
                         q8_stream_t stream);

/* A projection followed by the residual add and the following RMS norm ("plan.rs", `Launch::Fold` of a projection
 * with `Launch::Norm`, `gemv_norm_epilogue`: each block of the projection registers on a counter when done, and the
 * block that registers last fetches every result again from L2 and normalises; the norm launch is the lane's
 * "rmsnorm"):
 *     y = x . W (the Q8_0 product of q8_gemv),   h = residual + y,
 *     out[r, n] = h[r, n] / sqrt(mean_{n' < N} h[r, n']^2 + eps) * gamma[n]
 * Every CTA of the product writes its columns of h.  A second launch on the same stream, chained by programmatic
 * dependent launch (it waits for all of h), then runs the norm with one CTA per row: the row's mean square in a fixed
 * order, then out.  The one-launch fold of the source, where the product's last CTA to finish (a completion counter
 * from a fixed set of 64 in static device memory: the library allocates nothing) reads the rows of h back and runs
 * the norm, is kept for comparison (q8_set_tuning Q8_TUNE_NORM_FOLD = 1); measured on GB300 it is slower at every m.
 * Either way the result depends only on the inputs, never on which CTA finishes last.
 *   x, q, s   as q8_gemv, the weight in the tiled storage (q8_tile)
 *   residual  device, fp32 [m][Np], 4-byte aligned (read)
 *   gamma     device, fp32 [N] (at least N values), 4-byte aligned
 *   eps       >= 0 and finite
 *   h         device, fp32 [m][Np] (written: residual + y, pads 0), 16-byte aligned; may be residual itself
 *   out_bf16  device, bf16 [m][Np] (written: out rounded to nearest even, pads 0), 16-byte aligned -- the next
 *             projection's activation as q8_gemv takes it (row pitch Np)
 *   flags     Q8_FLAG_TILED (required) | Q8_FLAG_CONSTANT_WEIGHTS
 * Under the one-launch fold each group of 16 rows takes the next of 64 static completion counters in turn (a counter
 * is back to 0 when its launch ends), so at most 64 row groups may be in flight at once.
 * Errors: Q8_ERR_ARG (null pointers, flags without Q8_FLAG_TILED or unknown bits, eps < 0 or not finite, outputs
 * overlapping an input or each other other than h == residual), Q8_ERR_SHAPE, Q8_ERR_ALIGN, Q8_ERR_CUDA; nothing is
 * launched on an argument error (a Q8_ERR_CUDA from the norm's own launch leaves h written and out unspecified). */
q8_status q8_gemv_residual_norm(const void *x, const int8_t *q, const float *s, const float *residual,
                                const float *gamma, float eps, float *h, void *out_bf16, int m, int K, int N,
                                unsigned int flags, q8_stream_t stream);

/* q8_gemv_residual_norm with the normed output as bf16 (out_bf16) and/or its quantized form (out_q8, q8_act_bytes(m,
 * Np) bytes, 16-byte aligned: what q8_quantize_act of the bf16 rows writes; "plan.rs" `AddNormQuant`); at least one of
 * them, neither overlapping an input, h or the other. */
q8_status q8_gemv_residual_norm_ex(const void *x, const int8_t *q, const float *s, const float *residual,
                                   const float *gamma, float eps, float *h, void *out_bf16, void *out_q8, int m,
                                   int K, int N, unsigned int flags, q8_stream_t stream);

/* The rows one q8_gemv_residual_norm_noalloc call takes at most: its static scratch holds one completion counter per
 * group of 16 rows. */
#define Q8_FOLD_STATIC_MAX_ROWS 512

/* q8_gemv_residual_norm as one kernel launch that needs no device memory beyond its arguments and allocates none.
 * No counterpart on the pages: it serves callers that cannot call cudaMalloc or take memory from an allocator --
 * code running where device allocation is forbidden or would stall the pipeline (a real-time loop, a host
 * framework that owns all device memory and gives its plugins none, a step that must not synchronise the device).
 * It runs the source's one-launch fold (the product's last CTA per group of 16 rows reads h back and normalises),
 * whose completion counters live in a fixed array of this library (Q8_FOLD_STATIC_MAX_ROWS / 16 = 32 counters,
 * 128 bytes held by every GPU that loads the library until the process exits).
 *   Arguments, layouts, the result and its bound as q8_gemv_residual_norm (tiled storage; Q8_FLAG_TILED required,
 *   Q8_FLAG_CONSTANT_WEIGHTS and Q8_FLAG_Q8_ACT accepted), with 1 <= m <= Q8_FOLD_STATIC_MAX_ROWS.
 *   The call enqueues a memset that clears the counters it uses, then the product.
 * The first call on a device looks up the array's device address (cudaGetSymbolAddress) with that device current;
 * make that first call before any stream capture on the device.  Every call shares the one array: calls whose work
 * overlaps on a GPU (other streams, other threads) race on the counters and give wrong results; calls on one stream
 * are ordered and safe.
 * Errors: Q8_ERR_SHAPE for m > Q8_FOLD_STATIC_MAX_ROWS (and as q8_gemv_residual_norm); Q8_ERR_ARG, Q8_ERR_ALIGN,
 * Q8_ERR_CUDA as q8_gemv_residual_norm.  Nothing is enqueued on an argument error. */
q8_status q8_gemv_residual_norm_noalloc(const void *x, const int8_t *q, const float *s, const float *residual,
                                        const float *gamma, float eps, float *h, void *out_bf16, int m, int K, int N,
                                        unsigned int flags, q8_stream_t stream);

/* One weight of a multi-projection call: its Q8_0 values and scales (row-major, or tiled with Q8_FLAG_TILED), its
 * output y [m][q8_padded_n(N)] (written) and its N. */
typedef struct q8_part {
    const int8_t *q;
    const float *s;
    float *y;
    int N;
} q8_part;

#define Q8_MAX_PARTS 8

/* Several Q8_0 products of one activation: y_p = x . W_p for every part p (source: "plan.rs", `Launch::GemmParts`:
 * the projections that share an activation -- q/k/v, or gate/up -- run together, their outputs placed next to each
 * other).
 *   x      device bf16 [m][K], read once for all parts       parts  host array of nparts q8_part (read during the call)
 *   1 <= nparts <= Q8_MAX_PARTS; every part has the same K; N may differ.  Each y_p is as q8_gemv writes it.
 * The parts run as one kernel launch (two when the planner splits it, Q8_TUNE_SPLIT, q8_plan_launches), row-major
 * or (Q8_FLAG_TILED) in the q8_tile layout.  Flags and errors as
 * q8_gemv_ex; an output overlapping x, a weight or another output is Q8_ERR_ARG. */
q8_status q8_gemv_parts(const void *x, const q8_part *parts, int nparts, int m, int K, unsigned int flags,
                        q8_stream_t stream);

/* How many product kernels a q8_gemv_ex (Q8_VARIANT_AUTO), q8_gemv_argmax_ex or q8_gemv_parts call of these sizes
 * launches on the calling thread's current device under the current tuning: 1, or 2 when the planner splits it
 * (Q8_TUNE_SPLIT; plain products of at most 16 rows whose column tiles do not fill the SMs evenly).  The arg-max's
 * memset and index decode are not counted.  No counterpart on the pages: for callers that account for the kernels of
 * a captured graph, and for tests.
 *   Ns  host array of the nparts output widths N (one for q8_gemv_ex and q8_gemv_argmax_ex); 1 <= nparts <= 8
 * Returns the count, or a negative status: -Q8_ERR_ARG (null Ns, nparts out of range, unknown flags), -Q8_ERR_SHAPE
 * (sizes the call would reject), -Q8_ERR_CUDA (the device cannot be queried). */
int q8_plan_launches(int m, int K, const int *Ns, int nparts, unsigned int flags);

/* q8_plan_launches for a q8_gemv_glu(_ex) call of these sizes (flags as that call takes them, Q8_FLAG_TILED among
 * them): 1, or 2 when the planner splits the gated pair in two.  Returns the count or a negative status as
 * q8_plan_launches. */
int q8_plan_glu_launches(int m, int K, int N, unsigned int flags);

/* The quantized form of an activation (source: "plan.rs", `QBLOCK`: 32 consecutive values of the form share one
 * scale; `Buffer::quantized`: int8 codes plus one scale for every 32; `Launch::projected_input`: a product over
 * checkpoint rows takes its activation in this form unless the numerics are the exact ones).  One buffer of
 * q8_act_bytes(m, K) bytes:
 *   values  int8 [m][K]      at byte 0
 *   scales  fp32 [m][K/32]   at byte m * K (16-byte aligned when the buffer is, since K % 32 == 0)
 * The pages fix the form but not its rounding; the rule here is the weight rule of "from_q8.rs" `quantize`
 * (d = amax / 127, q = round(x / d)) in fp32: for each row and block of 32 values, amax = max |x|,
 * d = amax / 127 and q = x / d rounded half away from zero, both quotients IEEE fp32 (round to nearest even,
 * subnormals kept), q clamped to [-127, 127] (a guard: for bf16 input |x / d| <= 127 * (1 + 2^-10)).  A block of
 * zeros gets d = 0 and q = 0; a block holding inf or NaN gets d = NaN and q = 0, so every product over it is NaN. */
int64_t q8_act_bytes(int m, int K); /* m * K + m * (K / 32) * 4; -1 when m < 1, K <= 0 or K % 32 != 0 */

/* Device: quantize x into xa, enqueued on `stream` (asynchronous; errors as q8_gemv).
 *   x   device, bf16 [m][K] row-major, 16-byte aligned
 *   xa  device, q8_act_bytes(m, K) bytes (written), 16-byte aligned, not overlapping x
 * Any m >= 1 (not limited to 16). */
q8_status q8_quantize_act(const void *x, void *xa, int m, int K, q8_stream_t stream);

/* Host repack of checkpoint blocks into the two stored tensors (source: "from_q8.rs", `Q8Part`: the host repacks the
 * checkpoint's blocks into the int8 values `q8_0.values` and the fp32 scales `q8_0.scales`).
 *   blocks  host, N * (K/32) blocks of 36 bytes, column-major by block: column n's blocks b = 0 .. K/32-1 in order;
 *           each block is a little-endian fp32 scale d followed by 32 int8 values (rows 32b .. 32b+31).
 *   q       host, int8 [K][Np] (written, pad columns 0)     s  host, fp32 [K/32][Np] (written, pad columns 0)
 * Returns Q8_ERR_NOT_Q8_0 when a value is -128 (outside the Q8_0 range |q| <= 127) or a scale is not finite; q and s
 * are then left partly written. */
q8_status q8_repack(const void *blocks, int K, int N, int8_t *q, float *s);

/* q8_repack for GGML-style checkpoint blocks ("plan.rs" names the checkpoint format `GgmlType::Q8_0`): each block is
 * 34 bytes, a little-endian IEEE binary16 scale d followed by 32 int8 values, in the same column-major block order.
 * The scale is widened to fp32 exactly (subnormals kept).  Errors as q8_repack (a non-finite scale or a value of
 * -128 is Q8_ERR_NOT_Q8_0). */
q8_status q8_repack_f16(const void *blocks, int K, int N, int8_t *q, float *s);

/* Host Q8_0 quantization of a declared weight (source: "from_q8.rs", `quantize`).
 *   w  host, fp64 [K][N] row-major (the declared values, as the pages' rule takes them)
 *   q  host, int8 [K][Np] (written, pad columns 0)     s  host, fp32 [K/32][Np] (written, pad columns 0)
 * For every 32-row block and column: amax = max |w|; an all-zero block gets q = 0 and s = 0; otherwise
 * d = amax / 127 (in fp64) must be exactly an fp32 value, and every w / d must lie within 1e-9 of an integer r with
 * |r| <= 127 and r * d == w exactly.  Any failure returns Q8_ERR_NOT_Q8_0 (q and s then hold no meaning). */
q8_status q8_quantize(const double *w, int K, int N, int8_t *q, float *s);

/* Reads the device fault word of the current device: nonzero when a kernel's bounded wait on a pipeline barrier ran
 * out (bit 0: a consumer waited about two seconds for a stage's data; bit 1: the producer waited as long for a free
 * stage; bit 2: a wait of the prefill GEMM ran out) and the kernel finished early -- that call's outputs are then
 * wrong.  Synchronous with respect to the
 * device.  `clear` != 0 resets the word to 0.  Returns Q8_ERR_ARG for a NULL `fault`, Q8_ERR_CUDA on a CUDA error. */
q8_status q8_device_fault(unsigned int *fault, int clear);

/* Planner overrides for tests and benchmarks (no counterpart on the pages).  Process-wide: every later call on every
 * thread and device sees the value, so set them only while no other thread is enqueuing work.  Each option starts
 * from an environment variable, read once, at the first call that plans a launch.
 *   Q8_TUNE_KSPLIT     0: the planner's K split (default); 1..8: every K-split cluster takes this many CTAs (capped
 *                      at the number of K blocks; the gated pair and the prefill GEMM take at most 4).
 *                      Environment: Q8_KSPLIT.
 *   Q8_TUNE_GEMM       -1: the planner's choice (default); 0: calls of 128 rows or more keep the row groups; 1: they
 *                      run on the tcgen05 GEMM whatever the weight's width.  Environment: Q8_GEMM (0 or 1).
 *   Q8_TUNE_NORM_FOLD  0: the residual norm as a launch of its own (default); 1: the one-launch fold, where the
 *                      product's last CTA runs the norm.  Environment: Q8_NORM_LAUNCH=0 selects 1.
 *   Q8_TUNE_SPLIT      1: the planner may run a plain product (q8_gemv, q8_gemv_argmax, q8_gemv_parts) or a gated
 *                      pair (q8_gemv_glu) of m <= 16 rows as two launches, the column tiles that do not fill the
 *                      SMs evenly given their own K split (default); 0: always one launch.  Environment: Q8_SPLIT=0
 *                      selects 0. */
#define Q8_TUNE_KSPLIT 0
#define Q8_TUNE_GEMM 1
#define Q8_TUNE_NORM_FOLD 2
#define Q8_TUNE_SPLIT 3

/* Sets an override.  Returns Q8_ERR_ARG for an unknown option or a value outside its range. */
q8_status q8_set_tuning(int option, int value);

/* The current value of an override (its environment default until set); -2 for an unknown option. */
int q8_get_tuning(int option);

/* A static, human-readable name for a status code. */
const char *q8_status_string(q8_status status);

/* The cudaError_t of the last CUDA failure on the calling thread (0 when none). */
int q8_last_cuda_error(void);

/* Library version, major * 10000 + minor * 100 + patch. */
int q8_version(void);

#ifdef __cplusplus
}
#endif

#endif /* Q8_GEMV_H */
