// Shared device/host helpers: status codes, the per-device error word, bounded
// mbarrier waits, element-type traits.
#pragma once
#include <cstdint>
#include <cuda_runtime.h>

#include "../../include/ssdnn.h"
#include "ptx.cuh"

namespace ssdnn {

// Error bits recorded by kernels in the per-device error word.
enum : uint32_t { kErrTimeout = 1u, kErrInternal = 2u };

// Kernels receive the device address of the per-device error word (a
// file-scope __device__ variable of the C-ABI translation unit).
__device__ __forceinline__ void record_error(uint32_t* err, uint32_t bits) {
  if (err) atomicOr(err, bits);
}

// Upper bound on any single mbarrier wait inside a kernel (wall clock).
constexpr uint64_t kWaitLimitNs = 2000ull * 1000ull * 1000ull;

// Waits for the given phase parity of `bar`. Gives up after limit_ns, records a
// timeout and returns false; the caller then stops issuing work.
__device__ __forceinline__ bool wait_bounded(uint64_t* bar, uint32_t parity, uint32_t* err,
                                             uint64_t limit_ns = kWaitLimitNs) {
  if (ptx::mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = ptx::globaltimer_ns();
  uint32_t n = 0;
  while (true) {
    if (ptx::mbar_try_wait(bar, parity)) return true;
    if ((++n & 63u) == 0) {
      if (ptx::globaltimer_ns() - t0 > limit_ns) {
        record_error(err, kErrTimeout);
        return false;
      }
    }
  }
}

// 2:4 selection of one group of four magnitudes m0..m3 (stored bits, sign
// cleared): the two largest are kept, equal magnitudes going to the lower
// position. Each magnitude is tagged with (3 - position) in its two low bits, so
// the keys are distinct and a larger key is the preferred element; the top two
// keys of four come out of a five-comparison min/max network. Returns the
// metadata nibble j0 | j1 << 2 with j0 < j1.
__device__ __forceinline__ uint32_t top2_nibble(uint32_t m0, uint32_t m1, uint32_t m2, uint32_t m3) {
  const uint32_t k0 = (m0 << 2) | 3u, k1 = (m1 << 2) | 2u, k2 = (m2 << 2) | 1u, k3 = m3 << 2;
  const uint32_t a = max(k0, k1), b = min(k0, k1), c = max(k2, k3), d = min(k2, k3);
  const uint32_t t1 = max(a, c), t2 = max(min(a, c), max(b, d));
  const uint32_t i1 = 3u - (t1 & 3u), i2 = 3u - (t2 & 3u);
  return min(i1, i2) | (max(i1, i2) << 2);
}

template <int DT>
struct Elem;  // DT: 0 = f16, 1 = bf16, 2 = e4m3
template <>
struct Elem<0> {
  static constexpr int bytes = 2;
  static constexpr uint32_t mag_mask = 0x7FFFu;
  static constexpr uint32_t mma_fmt = 0;  // kind::f16, F16
  static constexpr bool f8 = false;
};
template <>
struct Elem<1> {
  static constexpr int bytes = 2;
  static constexpr uint32_t mag_mask = 0x7FFFu;
  static constexpr uint32_t mma_fmt = 1;  // kind::f16, BF16
  static constexpr bool f8 = false;
};
template <>
struct Elem<2> {
  static constexpr int bytes = 1;
  static constexpr uint32_t mag_mask = 0x7Fu;
  static constexpr uint32_t mma_fmt = 0;  // kind::f8f6f4, E4M3
  static constexpr bool f8 = true;
};

inline int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }
inline int64_t round_up(int64_t a, int64_t b) { return ceil_div(a, b) * b; }

}  // namespace ssdnn
