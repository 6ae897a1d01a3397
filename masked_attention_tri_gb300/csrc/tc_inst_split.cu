// tc_inst_split.cu -- instantiates the key-split kernel's triangle-form variants
// (bf16 / fp16 inputs, 16-bit / fp32 bias).
#include "tc_split.cuh"

namespace triattn {
namespace tc {

TRIATTN_SPLIT_TRI_VARIANTS(TRIATTN_SPLIT_INSTANTIATE)

}  // namespace tc
}  // namespace triattn
