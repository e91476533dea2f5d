// The kernels and launch sequences for bf16 target logits and bf16 draft logits
// (bf16 logits are held as their uint16_t bit patterns).
#include "launch.cuh"

namespace sv {
const PairOps ops_bf16_bf16 = make_ops<uint16_t, uint16_t>();
}  // namespace sv
