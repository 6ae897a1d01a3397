// tc_inst_f16_tri.cu -- instantiates the fp16 triangle-form variants of the tcgen05 forward
// kernel (split across files so they compile in parallel).
#include "tc_kernel.cuh"

namespace triattn {
namespace tc {

TRIATTN_TC_INSTANTIATE(1, false, false, false, false)
TRIATTN_TC_INSTANTIATE(1, false, false, true, false)
TRIATTN_TC_INSTANTIATE(2, false, false, false, false)
TRIATTN_TC_INSTANTIATE(2, false, false, true, false)

}  // namespace tc
}  // namespace triattn
