// tcgen05 tensor-core kernels (sm_103a).
#include "tc.h"

namespace qg {

bool tc_gemm_supported(const GemmArgs&) { return false; }
mm_status launch_tc_gemm(const GemmArgs&, unsigned*, cudaStream_t) { return MM_ERR_UNSUPPORTED; }
bool tc_qlinear_supported(const QLinearArgs&) { return false; }
size_t tc_qlinear_workspace_bytes(int64_t, int64_t, int64_t, int64_t) { return 0; }
mm_status launch_tc_qlinear(const QLinearArgs&, void*, unsigned*, cudaStream_t) { return MM_ERR_UNSUPPORTED; }
bool tc_grouped_supported(const GroupedArgs&) { return false; }
size_t tc_grouped_workspace_bytes(int64_t, int64_t, int64_t) { return 0; }
mm_status launch_tc_grouped(const GroupedArgs&, void*, unsigned*, cudaStream_t) { return MM_ERR_UNSUPPORTED; }

}  // namespace qg
