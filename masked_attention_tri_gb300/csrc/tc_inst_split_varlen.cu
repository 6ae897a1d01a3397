// tc_inst_split_varlen.cu -- instantiates the key-split kernel's packed-sequence
// variants (bf16 / fp16 inputs, scale folded into the exponent or not).
#include "tc_split.cuh"

namespace triattn {
namespace tc {

TRIATTN_SPLIT_VARLEN_VARIANTS(TRIATTN_SPLIT_INSTANTIATE)

}  // namespace tc
}  // namespace triattn
