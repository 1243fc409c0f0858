// fa_band.cuh -- which kv tiles a block of query rows must visit under the visibility band.
//
// Key j is visible to query row i iff q_abs + lo_off <= j <= q_abs + hi_off (and j < kl), with
// q_abs = kl - ql + i: the bottom-right causal diagonal of the mlx-native training forward
// (page "mlx-native tests/test_flash_attn_train.rs", `sdpa_reference_with_logsumexp`) when
// hi_off = 0, widened or narrowed by a local window.
#pragma once

#include "fa_launch.h"

namespace fa {

// Kv tiles [first, last) of BN keys that rows r0 .. r1 (inclusive, r1 < ql) must visit.
// Without a window every range starts at tile 0 (an empty range is [0, 0)). With one, a row
// block whose band misses every key gets first = last = -1.
template <int BN, int BAND>
__device__ __forceinline__ void band_kv_tiles(int r0, int r1, int ql, int kl, int lo_off,
                                              int hi_off, int& first, int& last) {
  const int off = kl - ql;
  if (BAND != kBandWindow) {
    int kend = kl;
    if (BAND == kBandCausal) kend = min(kend, off + r1 + 1);  // exclusive key bound
    first = 0;
    last = kend <= 0 ? 0 : (kend + BN - 1) / BN;
    return;
  }
  const long long klo = max(0LL, (long long)off + r0 + lo_off);
  const long long khi = min((long long)kl, (long long)off + r1 + hi_off + 1);  // exclusive
  if (khi <= klo) {
    first = last = -1;
    return;
  }
  first = (int)(klo / BN);
  last = (int)((khi + BN - 1) / BN);
}

}  // namespace fa
