// tc_inst_varlen.cu -- instantiates the packed-sequence (bf16 and fp16) variants of the tcgen05 forward
// kernel (split across files so they compile in parallel).
#include "tc_kernel.cuh"

namespace triattn {
namespace tc {

TRIATTN_TC_INSTANTIATE(2, true, true, false, false)
TRIATTN_TC_INSTANTIATE(2, true, true, false, true)
TRIATTN_TC_INSTANTIATE(2, true, false, false, false)
TRIATTN_TC_INSTANTIATE(2, true, false, false, true)

}  // namespace tc
}  // namespace triattn
