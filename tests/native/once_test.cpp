// Host test of fa::OncePerKey (the per-device kernel-attribute cache): many threads and keys,
// each key's step must succeed exactly once; a failing step must be retried; keys outside the
// range run every time. Prints "ok" and exits 0 on success.
#include <stdio.h>

#include <atomic>
#include <thread>
#include <vector>

#include "../../flash_attention_gb300/csrc/fa_once.h"

int main() {
  constexpr int kKeys = 70;  // spans two words of the bit set (N = 128)
  static fa::OncePerKey<128> once;
  std::atomic<int> calls[kKeys];
  for (auto& c : calls) c = 0;
  std::atomic<int> fail_left{5};  // key 3 fails its first five attempts
  std::vector<std::thread> th;
  for (int t = 0; t < 16; ++t) {
    th.emplace_back([&, t] {
      for (int rep = 0; rep < 2000; ++rep) {
        const int key = (t * 7 + rep) % kKeys;
        int r = once.run(key, [&] {
          calls[key]++;
          if (key == 3 && fail_left.fetch_sub(1) > 0) return 1;  // a failed step
          return 0;
        });
        (void)r;
      }
    });
  }
  for (auto& x : th) x.join();
  int bad = 0;
  for (int k = 0; k < kKeys; ++k) {
    const int want = k == 3 ? 6 : 1;
    if (calls[k] != want || !once.done(k)) {
      printf("key %d: %d calls (want %d), done %d\n", k, calls[k].load(), want, (int)once.done(k));
      ++bad;
    }
  }
  int outside = 0;
  for (int i = 0; i < 3; ++i) once.run(-1, [&] { ++outside; return 0; });
  for (int i = 0; i < 3; ++i) once.run(128, [&] { ++outside; return 0; });
  if (outside != 6) {
    printf("out-of-range keys ran %d times (want 6)\n", outside);
    ++bad;
  }
  if (bad) return 1;
  printf("ok\n");
  return 0;
}
