// tc_inst_split_vbias.cu -- instantiates the key-split kernel's packed-sequence
// variants with a post-scale bias (bf16 / fp16 inputs, 16-bit / fp32 bias).
#include "tc_split.cuh"

namespace triattn {
namespace tc {

TRIATTN_SPLIT_VARLEN_BIAS_VARIANTS(TRIATTN_SPLIT_INSTANTIATE)

}  // namespace tc
}  // namespace triattn
