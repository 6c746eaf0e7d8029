// Tensor-core implicit GEMM (tcgen05): not built yet; the configuration check
// rejects the fp16x3 precision until it is.
#include "tc_gemm.h"

namespace codec {

bool tc_eligible(int, int) { return false; }
bool tc_pack_weights(const float*, int, int, int, TcWeights*, std::vector<void*>&) { return false; }
bool tc_scratch_alloc(TcScratch*, size_t, std::vector<void*>&) { return false; }
cudaError_t launch_gemm_tc(const GemmArgs&, const TcWeights&, PlanView, int, TcScratch*, cudaStream_t, int*)
{
    return cudaErrorNotSupported;
}

}  // namespace codec
