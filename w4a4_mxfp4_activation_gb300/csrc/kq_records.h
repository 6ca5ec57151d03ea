// Sizes of the operand records that kq_expand_blocks writes in KQ_K_BF16X3
// (host and device code; no CUDA headers).
#pragma once

#include <cstdint>

namespace kq {

// Bytes of one block's operand record of the tcgen05 kernel: the dense K_j
// as three bf16 terms (hi, mid, lo), laid out as the B operands of the
// block's two K = 16 MMA steps.  K_expanded in KQ_K_BF16X3 holds nb records.
constexpr int64_t kUmmaRecordBytes = 6144;

}  // namespace kq
