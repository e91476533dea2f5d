// The kernels and launch sequences for f32 target logits and f32 draft logits
// (bf16 logits are held as their uint16_t bit patterns).
#include "launch.cuh"

namespace sv {
const PairOps ops_f32_f32 = make_ops<float, float>();
}  // namespace sv
