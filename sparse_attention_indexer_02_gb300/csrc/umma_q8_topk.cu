// tcgen05 scorer with the fused per-row selection, fp8 keys with fp8 q (see umma_kernel.cuh).
#include "umma_kernel.cuh"

namespace qsa {
namespace umma {

cudaError_t launch_q8_topk(int heads, const CUtensorMap& kv, const CUtensorMap& qm, const UmmaParams& up,
                           const Layout& L, int grid, cudaStream_t s) {
  return launch_any<kKindFp8Q, true>(heads, kv, qm, up, L, grid, s);
}

}  // namespace umma
}  // namespace qsa
