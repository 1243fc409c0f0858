// fa_once.h -- run a setup step once per key (a CUDA device ordinal), thread-safely.
//
// Kernel attributes such as the dynamic shared-memory limit belong to a device context: a
// process that drives two GPUs must set them on each one. OncePerKey keeps one bit per key
// and runs the step under a lock the first time a key is seen; a step that fails leaves the
// bit clear, so the next call tries again. The fast path (already done) is one atomic load.
// Plain C++: no CUDA header, so the logic is tested on its own with a host compiler.
#pragma once

#include <atomic>
#include <mutex>
#include <stdint.h>

namespace fa {

template <int N = 64>
class OncePerKey {
 public:
  // Calls fn() unless it already succeeded for `key`; fn returns a status whose value-initialised
  // form R{} means success (cudaSuccess, 0). Keys outside [0, N) are not remembered: fn runs
  // every time.
  template <class F>
  auto run(int key, F&& fn) -> decltype(fn()) {
    using R = decltype(fn());
    if (key < 0 || key >= N) return fn();
    const uint64_t bit = uint64_t(1) << (key % 64);
    std::atomic<uint64_t>& word = done_[key / 64];
    if (word.load(std::memory_order_acquire) & bit) return R{};
    std::lock_guard<std::mutex> lk(mu_);
    if (word.load(std::memory_order_relaxed) & bit) return R{};
    R r = fn();
    if (r == R{}) word.fetch_or(bit, std::memory_order_release);
    return r;
  }

  bool done(int key) const {
    if (key < 0 || key >= N) return false;
    return (done_[key / 64].load(std::memory_order_acquire) >> (key % 64)) & 1u;
  }

 private:
  static constexpr int kWords = (N + 63) / 64;
  std::atomic<uint64_t> done_[kWords] = {};
  std::mutex mu_;
};

}  // namespace fa
