// tc_inst_bf16_tri.cu -- instantiates the bf16 triangle-form variants of the tcgen05 forward
// kernel (split across files so they compile in parallel).
#include "tc_kernel.cuh"

namespace triattn {
namespace tc {

TRIATTN_TC_INSTANTIATE(1, false, true, false, false)
TRIATTN_TC_INSTANTIATE(1, false, true, true, false)
TRIATTN_TC_INSTANTIATE(2, false, true, false, false)
TRIATTN_TC_INSTANTIATE(2, false, true, true, false)

}  // namespace tc
}  // namespace triattn
