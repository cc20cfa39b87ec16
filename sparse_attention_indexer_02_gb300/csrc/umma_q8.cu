// tcgen05 scorer instantiations for fp8 q with fp8 keys (see umma_kernel.cuh).
#include "umma_kernel.cuh"

namespace qsa {
namespace umma {

cudaError_t launch_q8(int heads, const CUtensorMap& kv, const CUtensorMap& qm, const UmmaParams& up,
                      const Layout& L, int grid, cudaStream_t s) {
  return launch_any<kKindFp8Q>(heads, kv, qm, up, L, grid, s);
}

}  // namespace umma
}  // namespace qsa
