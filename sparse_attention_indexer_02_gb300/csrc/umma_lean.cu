// tcgen05 scorer instantiations of the lean form (see umma_kernel.cuh): bf16
// keys, and fp8 keys with fp8 q, for groups of at most 64 rows x heads.
#include "umma_kernel.cuh"

namespace qsa {
namespace umma {

cudaError_t launch_lean(int heads, int kind, const CUtensorMap& kv, const CUtensorMap& qm, const UmmaParams& up,
                        const Layout& L, int grid, cudaStream_t s) {
  if (kind == kKindFp8Q) return launch_any<kKindFp8Q, false, true>(heads, kv, qm, up, L, grid, s);
  return launch_any<kKindBf16, false, true>(heads, kv, qm, up, L, grid, s);
}

}  // namespace umma
}  // namespace qsa
