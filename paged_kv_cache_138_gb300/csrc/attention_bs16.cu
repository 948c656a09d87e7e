// Paged decode attention kernels for block size 16 (all GQA groups, with and
// without the fused cache write).
#include "attention_kernel.cuh"

namespace pkv {
namespace attn {

PKV_DEFINE_LAUNCH_SPLIT(16)

}  // namespace attn
}  // namespace pkv
