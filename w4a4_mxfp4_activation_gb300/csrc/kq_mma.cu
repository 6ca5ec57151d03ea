// Tensor-core variant of the KroQuant block transform (placeholder until
// the mma.sync kernel lands).
#include "kq_internal.h"

namespace kq {

kq_status launch_quant_mma(const uint16_t *, int64_t, const void *, const QuantParams &,
                           cudaStream_t)
{
    return KQ_ERR_UNSUPPORTED;
}

}  // namespace kq
