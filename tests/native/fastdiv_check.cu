// Host check of fa::FastDiv (the unit decode's division by a multiply-high): against plain
// unsigned division, for edge numerators of many divisors and for random pairs. Prints the
// number of mismatches and exits non-zero on any.
#include <cstdint>
#include <cstdio>
#include <random>

#include "fa_fwd_kernel.cuh"

int main() {
  std::mt19937_64 gen(12345);
  long long checked = 0, bad = 0;
  auto check = [&](uint32_t n, uint32_t d) {
    const fa::FastDiv f = fa::FastDiv::make(d);
    ++checked;
    if (f.div(n) != n / d) {
      if (bad < 5) std::printf("mismatch: %u / %u: %u vs %u\n", n, d, f.div(n), n / d);
      ++bad;
    }
  };
  const uint32_t ds[] = {1u, 2u, 3u, 5u, 7u, 12u, 48u, 96u, 127u, 128u, 152u, 641u, 65535u, 65536u,
                         1000003u, 0x7fffffffu, 0x80000000u, 0xfffffffeu, 0xffffffffu};
  for (uint32_t d : ds) {
    const uint32_t edge[] = {0u, 1u, d - 1u, d, d + 1u, 2u * d - 1u, 2u * d, 0x7fffffffu,
                             0x80000000u, 0xfffffffeu, 0xffffffffu};
    for (uint32_t n : edge) check(n, d);
    for (int i = 0; i < 200000; ++i) check(static_cast<uint32_t>(gen()), d);
  }
  for (int i = 0; i < 1000000; ++i) {
    uint32_t d = static_cast<uint32_t>(gen()) >> (gen() % 32);
    if (d == 0u) d = 1u;
    check(static_cast<uint32_t>(gen()) >> (gen() % 32), d);
  }
  std::printf("checked %lld, mismatches %lld\n", checked, bad);
  return bad == 0 ? 0 : 1;
}
