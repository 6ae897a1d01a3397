// tc_inst_split.cu -- instantiates the key-split triangle-form kernel (D <= 64)
// for bf16 / fp16 inputs and 16-bit / fp32 bias.
#include "tc_split.cuh"

namespace triattn {
namespace tc {

TRIATTN_SPLIT_VARIANTS(TRIATTN_SPLIT_INSTANTIATE)

}  // namespace tc
}  // namespace triattn
