// Paged decode attention kernels for block size 8 (all GQA groups, with and
// without the fused cache write).
#include "attention_kernel.cuh"

namespace pkv {
namespace attn {

PKV_DEFINE_LAUNCH_SPLIT(8)

}  // namespace attn
}  // namespace pkv
