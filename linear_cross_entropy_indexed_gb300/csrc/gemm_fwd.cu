// Forward tensor-core kernel: H W^T tiles -> per-group running (max, sum) of the row
// softmax denominator (Liger-CCE blog, §三 "CCE" linear-LSE; ai-infra-kb M011, §05).
// A = H [N, Hd] K-major, B = W [V, Hd] K-major.
#include "tc_gemm.cuh"

namespace flce {

cudaError_t launch_linear_lse(const CUtensorMap& tmH, const CUtensorMap& tmW, const Sched& s,
                              const EpiLseParams& p, unsigned long long* err, int grid,
                              cudaStream_t st) {
  return launch_gemm<EpiLse, false, false>(tmH, tmH, tmW, s, p, err, grid, st);
}

cudaError_t set_gemm_smem_attributes_fwd() { return set_smem_attr<EpiLse, false, false>(); }

}  // namespace flce
