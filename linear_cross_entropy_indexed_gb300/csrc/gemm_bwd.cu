// Backward tensor-core kernels (ai-infra-kb M011, §06: recompute the logit tile from
// the saved LSE, dH summed over vocabulary tiles, dW summed over tokens).
//   dZ chunk : A = H [N, Hd] K-major,        B = W rows of the chunk, K-major
//   dW chunk : A = dZ^T (dZ [N, Vc], MN-major), B = H (MN-major)
//   dH       : A = dZ [N, Vc] K-major,        B = W rows of the chunk, MN-major
#include "tc_gemm.cuh"

namespace flce {

cudaError_t launch_dz(const CUtensorMap& tmH, const CUtensorMap& tmW, const Sched& s,
                      const EpiDzParams& p, unsigned long long* err, int grid, cudaStream_t st) {
  return launch_gemm<EpiDz, false, false>(tmH, tmH, tmW, s, p, err, grid, st);
}

cudaError_t launch_dw(const CUtensorMap& tmDz, const CUtensorMap& tmDz2, const CUtensorMap& tmH, const Sched& s,
                      const EpiDwParams& p, unsigned long long* err, int grid, cudaStream_t st) {
  return launch_gemm<EpiDw, true, true>(tmDz, tmDz2, tmH, s, p, err, grid, st);
}

cudaError_t launch_dh(const CUtensorMap& tmDz, const CUtensorMap& tmDz2, const CUtensorMap& tmW, const Sched& s,
                      const EpiDhParams& p, unsigned long long* err, int grid, cudaStream_t st) {
  return launch_gemm<EpiDh, false, true>(tmDz, tmDz2, tmW, s, p, err, grid, st);
}

cudaError_t set_gemm_smem_attributes_bwd() {
  cudaError_t e = set_smem_attr<EpiDz, false, false>();
  if (e != cudaSuccess) return e;
  e = set_smem_attr<EpiDw, true, true>();
  if (e != cudaSuccess) return e;
  return set_smem_attr<EpiDh, false, true>();
}

}  // namespace flce
