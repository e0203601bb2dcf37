// 2:4 magnitude prune + compress.
//
// The 2:4 pattern: in each contiguous group of four values along K two are zero,
// and the matrix is kept as its nonzero values plus small position metadata
// ("NVIDIA A100 benchmarks" blog page, 2:4 paragraph and Figure 1 caption).
// Criterion (reading): keep the two largest |w| of each group, ties to the lower
// position, comparing the stored bits with the sign cleared as integers.
//
// One thread owns 32 consecutive elements of a row (8 groups): 64 B of fp16/bf16
// or 32 B of e4m3 read with 16-byte loads, 32 B / 16 B of values and 4 B of
// canonical metadata written, plus the word of the tensor-core operand layout of
// the metadata. The grid also covers the 128-row and K-block padding of that
// layout, which it fills with the (0,1) pattern.
#include "common.cuh"
#include "kernels.h"

namespace ssdnn {
namespace {

template <int EB>
__device__ __forceinline__ uint32_t elem(const uint32_t (&w)[16], int j) {
  if constexpr (EB == 2) {
    return (w[j >> 1] >> ((j & 1) * 16)) & 0xFFFFu;
  } else {
    return (w[j >> 2] >> ((j & 3) * 8)) & 0xFFu;
  }
}

// Block = 16 rows x 16 chunks (a warp reads 1 KB / 512 B contiguous of each of
// two rows); grid.y walks 16-row groups of the 128-row-padded matrix.
template <int EB>
__global__ void __launch_bounds__(256) k_sp24_compress(const uint8_t* __restrict__ W, int64_t M, int64_t K,
                                                       int64_t ldw_b, uint8_t* __restrict__ values,
                                                       int64_t ldv_b, uint8_t* __restrict__ meta, int64_t ldm,
                                                       uint8_t* __restrict__ meta_hw, int64_t KBhw,
                                                       int64_t chunks_pad, bool vec_ok) {
  constexpr uint32_t kMask = (EB == 2) ? 0x7FFFu : 0x7Fu;
  __shared__ uint32_t s_nib[16][17];
  const int tr = threadIdx.x >> 4, tc = threadIdx.x & 15;
  const int64_t i = static_cast<int64_t>(blockIdx.y) * 16 + tr;
  const int64_t c = static_cast<int64_t>(blockIdx.x) * 16 + tc;
  const int64_t k0 = c * 32;
  const int64_t Kp = (K + 31) / 32 * 32;

  uint32_t nib = 0x44444444u;
  uint32_t outv[8] = {0, 0, 0, 0, 0, 0, 0, 0};  // 16 values packed (EB bytes each)
  if (i < M && k0 < K) {
    uint32_t w[16];
    const uint8_t* src = W + i * ldw_b + k0 * EB;
    if (vec_ok && k0 + 32 <= K) {
#pragma unroll
      for (int q = 0; q < 2 * EB; ++q) {  // 32 elements = 2 * EB 16-byte loads
        const uint4 v = __ldg(reinterpret_cast<const uint4*>(src) + q);
        w[4 * q + 0] = v.x;
        w[4 * q + 1] = v.y;
        w[4 * q + 2] = v.z;
        w[4 * q + 3] = v.w;
      }
      if constexpr (EB == 1) {
#pragma unroll
        for (int q = 8; q < 16; ++q) w[q] = 0;
      }
    } else {
#pragma unroll
      for (int q = 0; q < 16; ++q) w[q] = 0;
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        if (k0 + j >= K) break;
        uint32_t e = (EB == 2) ? static_cast<uint32_t>(reinterpret_cast<const uint16_t*>(src)[j])
                               : static_cast<uint32_t>(src[j]);
        if constexpr (EB == 2)
          w[j >> 1] |= e << ((j & 1) * 16);
        else
          w[j >> 2] |= e << ((j & 3) * 8);
      }
    }
#pragma unroll
    for (int g = 0; g < 8; ++g) {
      if (k0 + 4 * g + 4 > K) break;  // K % 4 == 0: a group is entirely in or out
      const uint32_t e0 = elem<EB>(w, 4 * g + 0), e1 = elem<EB>(w, 4 * g + 1);
      const uint32_t e2 = elem<EB>(w, 4 * g + 2), e3 = elem<EB>(w, 4 * g + 3);
      const uint32_t sel = top2_nibble(e0 & kMask, e1 & kMask, e2 & kMask, e3 & kMask);
      const uint32_t j0 = sel & 3u, j1 = sel >> 2;
      nib = (nib & ~(0xFu << (4 * g))) | (sel << (4 * g));
      // gather the two kept values with one byte permute of the group's bytes
      if constexpr (EB == 2) {
        outv[g] = __byte_perm(w[2 * g], w[2 * g + 1],
                              (2 * j0) | ((2 * j0 + 1) << 4) | ((2 * j1) << 8) | ((2 * j1 + 1) << 12));
      } else {
        outv[g >> 1] |= __byte_perm(w[g], 0u, j0 | (j1 << 4) | 0x4400u) << ((g & 1) * 16);
      }
    }
  }
  if (i < M && k0 < Kp) {
    uint8_t* dv = values + i * ldv_b + c * 16 * EB;
    reinterpret_cast<uint4*>(dv)[0] = make_uint4(outv[0], outv[1], outv[2], outv[3]);
    if constexpr (EB == 2) reinterpret_cast<uint4*>(dv)[1] = make_uint4(outv[4], outv[5], outv[6], outv[7]);
    if (meta) *reinterpret_cast<uint32_t*>(meta + i * ldm + c * 4) = nib;
  }
  const int64_t mb = i >> 7, r = i & 127;
  if constexpr (EB == 1) {
    // e4m3 operand order = canonical nibbles, 16 bytes per row per 128 columns of K
    if (c < chunks_pad)
      *reinterpret_cast<uint32_t*>(meta_hw + ((mb * KBhw + (c >> 2)) * 128 + r) * 16 + (c & 3) * 4) = nib;
  } else {
    // 16-bit operand order: rows r and r ^ 8 share one 32-bit word per 32-column
    // span (lower row: groups 0..3 of both rows; upper row: groups 4..7 of both),
    // each span in its own even TMEM column (odd words zero).
    s_nib[tr][tc] = nib;
    __syncthreads();
    const uint32_t partner = s_nib[tr ^ 8][tc];
    const uint32_t hw = (tr & 8) ? ((partner >> 16) | (nib & 0xFFFF0000u)) : ((nib & 0xFFFFu) | (partner << 16));
    if (c < chunks_pad)
      *reinterpret_cast<uint2*>(meta_hw + ((mb * KBhw + (c >> 1)) * 128 + r) * 16 + (c & 1) * 8) =
          make_uint2(hw, 0u);
  }
}

}  // namespace

cudaError_t launch_sp24_compress(int dt, const void* W, int64_t M, int64_t K, int64_t ldw, void* values,
                                 uint8_t* meta, uint8_t* meta_hw, cudaStream_t s, uint32_t* err) {
  (void)err;
  const int EB = (dt == SSDNN_E4M3) ? 1 : 2;
  const int64_t span = (EB == 1) ? 128 : 64;          // K columns per operand metadata block
  const int64_t MB = ceil_div(M, 128), KBhw = ceil_div(K, span);
  const int64_t chunks_pad = KBhw * (span / 32);
  if (MB == 0 || KBhw == 0) return cudaSuccess;
  const int64_t Kp = round_up(K, 32);
  const bool vec_ok = (reinterpret_cast<uintptr_t>(W) % 16 == 0) && ((ldw * EB) % 16 == 0);
  const dim3 grid(static_cast<unsigned>(ceil_div(chunks_pad, 16)), static_cast<unsigned>(MB * 8));
  if (EB == 2)
    k_sp24_compress<2><<<grid, 256, 0, s>>>(static_cast<const uint8_t*>(W), M, K, ldw * 2,
                                            static_cast<uint8_t*>(values), Kp / 2 * 2, meta, Kp / 8, meta_hw, KBhw,
                                            chunks_pad, vec_ok);
  else
    k_sp24_compress<1><<<grid, 256, 0, s>>>(static_cast<const uint8_t*>(W), M, K, ldw,
                                            static_cast<uint8_t*>(values), Kp / 2, meta, Kp / 8, meta_hw, KBhw,
                                            chunks_pad, vec_ok);
  return cudaGetLastError();
}

}  // namespace ssdnn
