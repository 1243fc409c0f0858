// fa_bwd_strided.cu -- the backward main pass of head dims 64 and 128 for calls whose q-side
// or kv-side tensors are [batch, rows, heads, dim] in memory (sm_103a). The kernel is the one
// of fa_bwd_main.cuh with its STRIDED flag set; compiled apart from fa_bwd.cu, which
// instantiates the default layout.
#include "fa_bwd_main.cuh"

namespace fa {

cudaError_t launch_main_strided(const BwdArgs& a, const BwdMaps& m, cudaStream_t s) {
  if (a.d == 64 && a.dval == 64) return launch_main_layout<64, 64, true>(a, m, s);
  if (a.d == 128 && a.dval == 128) return launch_main_layout<128, 128, true>(a, m, s);
  if (a.d == 128 && a.dval == 64) return launch_main_layout<128, 64, true>(a, m, s);
  return cudaErrorInvalidValue;
}

}  // namespace fa
