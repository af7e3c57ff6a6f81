// Host entry points of libq8gemv: padding, the Q8_0 quantize rule, the checkpoint-block repack, status strings.
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <string.h>

#include "../../include/q8_gemv.h"

namespace q8 {
static thread_local int g_last_cuda_error = 0;
void set_last_cuda_error(int e) { g_last_cuda_error = e; }
}  // namespace q8

extern "C" int q8_padded_n(int N) {
    if (N <= 0) return -1;
    const long long p = ((long long)N + Q8_BLOCK - 1) / Q8_BLOCK * Q8_BLOCK;
    return p > 0x7FFFFFFFLL ? -1 : (int)p;
}

extern "C" int q8_last_cuda_error(void) { return q8::g_last_cuda_error; }

extern "C" int q8_version(void) { return 1 * 10000 + 0 * 100 + 0; }

extern "C" const char *q8_status_string(q8_status status) {
    switch (status) {
        case Q8_OK: return "ok";
        case Q8_ERR_ARG: return "invalid argument (null pointer, overlapping buffers or unknown variant)";
        case Q8_ERR_SHAPE: return "invalid shape (m outside 1..16, K not a positive multiple of 32, or N <= 0)";
        case Q8_ERR_ALIGN: return "misaligned pointer (16 bytes for x, q, s, y and logits; 8 for idx)";
        case Q8_ERR_NOT_Q8_0: return "weight is not Q8_0";
        case Q8_ERR_CUDA: return "CUDA runtime error (see q8_last_cuda_error)";
    }
    return "unknown status";
}

// "from_q8.rs", `quantize`: per 32-row block and column, amax = max |w|; a zero block is skipped (q = 0, d = 0);
// d = amax / 127 must round-trip through fp32, and every w / d must be within 1e-9 of an integer r, |r| <= 127, with
// r * d == w exactly.  The rounding of w / d is half away from zero (C `round`), as Rust's `f64::round`.
extern "C" q8_status q8_quantize(const double *w, int K, int N, int8_t *q, float *s) {
    if (!w || !q || !s) return Q8_ERR_ARG;
    if (K <= 0 || K % Q8_BLOCK != 0 || N <= 0) return Q8_ERR_SHAPE;
    const int Np = q8_padded_n(N);
    if (Np < 0) return Q8_ERR_SHAPE;
    const int nb = K / Q8_BLOCK;
    memset(q, 0, (size_t)K * Np);
    memset(s, 0, (size_t)nb * Np * sizeof(float));
    for (int b = 0; b < nb; ++b) {
        for (int n = 0; n < N; ++n) {
            double amax = 0.0;
            for (int i = 0; i < Q8_BLOCK; ++i) {
                const double a = fabs(w[(size_t)(Q8_BLOCK * b + i) * N + n]);
                if (a != a) return Q8_ERR_NOT_Q8_0;  // a NaN is no multiple of any scale
                if (a > amax) amax = a;
            }
            if (amax == 0.0) continue;
            const double d = amax / 127.0;
            if ((double)(float)d != d) return Q8_ERR_NOT_Q8_0;
            for (int i = 0; i < Q8_BLOCK; ++i) {
                const double wv = w[(size_t)(Q8_BLOCK * b + i) * N + n];
                const double v = wv / d;
                const double r = round(v);
                if (!(fabs(v - r) <= 1e-9) || fabs(r) > 127.0 || r * d != wv) return Q8_ERR_NOT_Q8_0;
                q[(size_t)(Q8_BLOCK * b + i) * Np + n] = (int8_t)r;
            }
            s[(size_t)b * Np + n] = (float)d;
        }
    }
    return Q8_OK;
}

namespace {

// An IEEE binary16 bit pattern widened to binary32 (exact: every binary16 value is a binary32 value), from the
// format's definition: sign, 5-bit exponent (bias 15), 10-bit fraction; exponent 0 holds zeros and subnormals
// (f * 2^-24), exponent 31 infinities and NaNs.
float half_to_float(uint16_t h) {
    const uint32_t sign = (uint32_t)(h & 0x8000u) << 16;
    const uint32_t e = (h >> 10) & 0x1Fu;
    uint32_t f = h & 0x3FFu;
    uint32_t bits;
    if (e == 31u) {
        bits = sign | 0x7F800000u | (f << 13);  // inf or NaN
    } else if (e != 0u) {
        bits = sign | ((e + 112u) << 23) | (f << 13);  // normal: exponent re-biased from 15 to 127
    } else if (f == 0u) {
        bits = sign;  // signed zero
    } else {
        // subnormal f * 2^-24: normalise so that the leading 1 of f sits at bit 10
        uint32_t shift = 0;
        while ((f & 0x400u) == 0u) {
            f <<= 1;
            ++shift;
        }
        bits = sign | ((113u - shift) << 23) | ((f & 0x3FFu) << 13);
    }
    float v;
    memcpy(&v, &bits, sizeof v);
    return v;
}

// Both block forms: `scale_bytes` (4: fp32, 2: binary16) little-endian scale, then 32 int8 values.
q8_status repack_blocks(const void *blocks, int K, int N, int8_t *q, float *s, int scale_bytes) {
    if (!blocks || !q || !s) return Q8_ERR_ARG;
    if (K <= 0 || K % Q8_BLOCK != 0 || N <= 0) return Q8_ERR_SHAPE;
    const int Np = q8_padded_n(N);
    if (Np < 0) return Q8_ERR_SHAPE;
    const int nb = K / Q8_BLOCK;
    const size_t block_bytes = (size_t)scale_bytes + Q8_BLOCK;
    const unsigned char *src = static_cast<const unsigned char *>(blocks);
    memset(q, 0, (size_t)K * Np);
    memset(s, 0, (size_t)nb * Np * sizeof(float));
    for (int n = 0; n < N; ++n) {
        for (int b = 0; b < nb; ++b) {
            const unsigned char *blk = src + ((size_t)n * nb + b) * block_bytes;
            float d;
            if (scale_bytes == 4) {
                const uint32_t bits = (uint32_t)blk[0] | ((uint32_t)blk[1] << 8) | ((uint32_t)blk[2] << 16) |
                                      ((uint32_t)blk[3] << 24);
                memcpy(&d, &bits, sizeof d);
            } else {
                d = half_to_float((uint16_t)(blk[0] | (blk[1] << 8)));
            }
            if (!isfinite(d)) return Q8_ERR_NOT_Q8_0;
            for (int i = 0; i < Q8_BLOCK; ++i) {
                const int8_t v = (int8_t)blk[scale_bytes + i];
                if (v == -128) return Q8_ERR_NOT_Q8_0;
                q[(size_t)(Q8_BLOCK * b + i) * Np + n] = v;
            }
            s[(size_t)b * Np + n] = d;
        }
    }
    return Q8_OK;
}

}  // namespace

// "from_q8.rs", `Q8Part`: the checkpoint's blocks repacked into the int8 values [K][Np] and the fp32 scales
// [K/32][Np], column-major by block; q8_repack takes 36-byte blocks (fp32 scale), q8_repack_f16 the GGML-style
// 34-byte blocks of "plan.rs" `GgmlType::Q8_0` (binary16 scale).
extern "C" q8_status q8_repack_f16(const void *blocks, int K, int N, int8_t *q, float *s) {
    return repack_blocks(blocks, K, N, q, s, 2);
}

extern "C" q8_status q8_repack(const void *blocks, int K, int N, int8_t *q, float *s) {
    return repack_blocks(blocks, K, N, q, s, 4);
}

