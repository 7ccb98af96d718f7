// Tensor-core (tcgen05 / TMEM / TMA) paths for sm_103a.  Each *_supported()
// says whether the operands' types and layouts fit the kernels; the launchers
// enqueue the work on `stream`.
#pragma once

#include "kernels.h"

namespace qg {

// Limit of each pipeline wait in the tensor-core kernels (0 = the 2 s default).
void tc_set_wait_limit_ns(unsigned long long ns);

bool tc_gemm_supported(const GemmArgs& g);
mm_status launch_tc_gemm(const GemmArgs& g, unsigned* status, cudaStream_t stream);

bool tc_qlinear_supported(const QLinearArgs& q);
size_t tc_qlinear_workspace_bytes(int64_t M, int64_t N, int64_t K, int64_t a_count, int64_t b_count);
mm_status launch_tc_qlinear(const QLinearArgs& q, void* workspace, unsigned* status, cudaStream_t stream);

bool tc_grouped_supported(const GroupedArgs& g);
size_t tc_grouped_workspace_bytes(const GroupedArgs& g);
// GroupedArgs with wq != 0 take the fused-dequantisation kernel (CTA pairs):
// the weights stay int8/uint8 in memory and are dequantised in shared memory.
mm_status launch_tc_grouped(const GroupedArgs& g, void* workspace, unsigned* status, cudaStream_t stream);

}  // namespace qg
