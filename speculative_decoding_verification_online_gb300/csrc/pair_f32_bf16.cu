// The kernels and launch sequences for f32 target logits and bf16 draft logits
// (bf16 logits are held as their uint16_t bit patterns).
#include "launch.cuh"

namespace sv {
const PairOps ops_f32_bf16 = make_ops<float, uint16_t>();
}  // namespace sv
