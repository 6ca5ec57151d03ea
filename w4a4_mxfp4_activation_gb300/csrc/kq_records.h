// Sizes of the operand records that kq_expand_blocks writes in KQ_K_BF16X3
// (host and device code; no CUDA headers).
#pragma once

#include <cstdint>

namespace kq {

// Bytes of one block's operand record for the two tensor-core variants:
// tcgen05 (dense K_j, three bf16 terms) and mma.sync (K'_j terms + G1).
// K_expanded in KQ_K_BF16X3 holds nb tcgen05 records, then nb mma.sync ones.
constexpr int64_t kUmmaRecordBytes = 6144;
constexpr int64_t kMmaRecordBytes = 1552;

}  // namespace kq
