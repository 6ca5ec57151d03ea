// Host-only parts of the C ABI: status strings, scale-array sizes and the
// per-layer factor preparation helpers.  No CUDA calls.
//
// Built with -ffp-contract=off so that every fp64 operation below is one
// separately rounded IEEE operation on every host architecture.
#include <cmath>
#include <cstdint>

#include "kq.h"
#include "kq_records.h"

extern "C" {

const char *kq_status_string(kq_status status)
{
    switch (status) {
    case KQ_OK: return "ok";
    case KQ_ERR_NULL: return "a required pointer is NULL";
    case KQ_ERR_SHAPE: return "invalid shape (m < 0, d <= 0, d % 32 != 0, lda < d, ldq < d/2, ...)";
    case KQ_ERR_ALIGN: return "misaligned pointer or leading dimension (16-byte rules)";
    case KQ_ERR_LAYOUT: return "unknown layout, format, variant or sign value";
    case KQ_ERR_CUDA: return "CUDA runtime or driver error";
    case KQ_ERR_UNSUPPORTED: return "current device is not compute capability 10.3 (GB300)";
    }
    return "unknown status";
}

size_t kq_sf_bytes(int64_t m, int64_t d, kq_sf_layout sf_layout)
{
    if (m < 0 || d <= 0 || d % 32 != 0) return 0;
    const int64_t nb = d / 32;
    if (sf_layout == KQ_SF_ROWMAJOR) return static_cast<size_t>(m * nb);
    if (sf_layout == KQ_SF_BLOCKED_128x4)
        return static_cast<size_t>(((m + 127) / 128) * 128 * ((nb + 3) / 4) * 4);
    return 0;
}

size_t kq_expanded_bytes(int64_t nb, kq_kfmt fmt)
{
    if (nb <= 0) return 0;
    if (fmt == KQ_K_FP32) return static_cast<size_t>(nb) * 32 * 32 * 4;
    if (fmt == KQ_K_BF16X3) return static_cast<size_t>(nb) * kq::kUmmaRecordBytes;
    return 0;
}

// eq. (6) of "KroQuant: Kronecker-Structured Block Transforms for Efficient
// Post-Training Quantization of Diffusion Transformers":
// G = [[1, 0], [c, 1]] . [[a, b], [0, u22]], u22 = det_sign / a.
kq_status kq_lu_to_factors(const float *lu, int64_t nb, int det_sign, float *factors)
{
    if (lu == nullptr || factors == nullptr) return KQ_ERR_NULL;
    if (nb <= 0) return KQ_ERR_SHAPE;
    if (det_sign != 1 && det_sign != -1) return KQ_ERR_LAYOUT;
    for (int64_t k = 0; k < nb * 5; ++k) {
        const double a = lu[3 * k];
        if (a == 0.0 || !std::isfinite(a)) return KQ_ERR_SHAPE;
    }
    for (int64_t k = 0; k < nb * 5; ++k) {
        const double a = lu[3 * k], b = lu[3 * k + 1], c = lu[3 * k + 2];
        const double u22 = (det_sign < 0 ? -1.0 : 1.0) / a;
        factors[4 * k + 0] = static_cast<float>(a);
        factors[4 * k + 1] = static_cast<float>(b);
        factors[4 * k + 2] = static_cast<float>(c * a);
        factors[4 * k + 3] = static_cast<float>(c * b + u22);
    }
    return KQ_OK;
}

// G^{-T} = [[g11, -g10], [-g01, g00]] / det G  (Sec. 3.2: the inverse of a
// Kronecker product is the product of the inverses; eq. (1): W T^{-T}).
kq_status kq_invert_transpose_factors(const float *factors, int64_t nb, float *out)
{
    if (factors == nullptr || out == nullptr) return KQ_ERR_NULL;
    if (nb <= 0) return KQ_ERR_SHAPE;
    for (int64_t k = 0; k < nb * 5; ++k) {
        const double g00 = factors[4 * k], g01 = factors[4 * k + 1];
        const double g10 = factors[4 * k + 2], g11 = factors[4 * k + 3];
        const double det = g00 * g11 - g01 * g10;
        if (det == 0.0 || !std::isfinite(det)) return KQ_ERR_SHAPE;
    }
    for (int64_t k = 0; k < nb * 5; ++k) {
        const double g00 = factors[4 * k], g01 = factors[4 * k + 1];
        const double g10 = factors[4 * k + 2], g11 = factors[4 * k + 3];
        const double det = g00 * g11 - g01 * g10;
        out[4 * k + 0] = static_cast<float>(g11 / det);
        out[4 * k + 1] = static_cast<float>(-g10 / det);
        out[4 * k + 2] = static_cast<float>(-g01 / det);
        out[4 * k + 3] = static_cast<float>(g00 / det);
    }
    return KQ_OK;
}

}  // extern "C"
