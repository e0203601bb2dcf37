// Tile-wise (TW) prune and the tile-vector-wise (TVW) hybrid.
//
// "Accelerating Sparse DNNs Based on Tiled GEMM" (TL;DR, Abstract, Figure 3):
// each GEMM tile keeps its own subset of K rows of the activation operand, so the
// pattern is regular inside a tile and irregular across tiles; TVW additionally
// applies 2:4 inside the kept rows. Readings (the page gives no formulas): a tile
// is 128 rows of W; score s_t[k] = fp32 sum over the tile's rows, in ascending
// row order, of |w_ik|; the tile keeps the first L_t of (score descending, k
// ascending), listed ascending; TVW groups are four consecutive kept columns.
//
// Three kernels:
//   k_tw_score   one thread per (tile, 8 consecutive k): walks the tile's rows
//                with 16-byte loads (coalesced across threads), fp32 sums in row
//                order, writes scores to the caller's workspace.
//   k_tw_select  one CTA per tile: exact top-L by a 4-pass 8-bit radix select on
//                the score bits (non-negative floats order like their bits), then
//                an ascending-k compaction with block prefix sums that takes ties
//                at the threshold from the lowest k.
//   k_tw_pack    one warp per (tile, 64-column chunk, row), 16 rows per CTA:
//                gathers the kept columns of the row into the chunk-blocked packed
//                operand; TVW selects 2 of every 4 and writes values plus metadata
//                in the canonical and the tensor-core operand order (which pairs
//                rows r and r ^ 8, exchanged through shared memory).
#include <cuda_fp16.h>

#include "common.cuh"
#include "kernels.h"

namespace ssdnn {
namespace {

template <int DT>
__device__ __forceinline__ float mag16(uint32_t h) {
  h &= 0x7FFFu;
  if constexpr (DT == 1) {
    return __uint_as_float(h << 16);
  } else {
    return __half2float(__ushort_as_half(static_cast<unsigned short>(h)));
  }
}

template <int DT>
__global__ void __launch_bounds__(256) k_tw_score(const uint8_t* __restrict__ W, int64_t M, int64_t K,
                                                  int64_t ldw_b, float* __restrict__ scores, bool vec_ok) {
  const int64_t t = blockIdx.y;
  const int64_t k0 = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) * 8;
  if (k0 >= K) return;
  const int64_t r0 = t * 128;
  const int64_t r1 = min(M, r0 + 128);
  float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  if (vec_ok && k0 + 8 <= K) {
    const uint8_t* p = W + r0 * ldw_b + k0 * 2;
#pragma unroll 8
    for (int64_t i = r0; i < r1; ++i, p += ldw_b) {
      const uint4 v = __ldg(reinterpret_cast<const uint4*>(p));
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        acc[2 * j] = acc[2 * j] + mag16<DT>(w[j] & 0xFFFFu);
        acc[2 * j + 1] = acc[2 * j + 1] + mag16<DT>(w[j] >> 16);
      }
    }
  } else {
    for (int64_t i = r0; i < r1; ++i) {
      const uint16_t* p = reinterpret_cast<const uint16_t*>(W + i * ldw_b) + k0;
#pragma unroll
      for (int j = 0; j < 8; ++j)
        if (k0 + j < K) acc[j] = acc[j] + mag16<DT>(p[j]);
    }
  }
#pragma unroll
  for (int j = 0; j < 8; ++j)
    if (k0 + j < K) scores[t * K + k0 + j] = acc[j];
}

// Exclusive prefix sum over a 1024-thread block; returns this thread's prefix and
// writes the block total to *total. `ws` holds 32 words of shared scratch.
__device__ __forceinline__ uint32_t block_excl_scan(uint32_t v, uint32_t* ws, uint32_t* total) {
  const uint32_t lane = threadIdx.x & 31u, warp = threadIdx.x >> 5;
  uint32_t x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= static_cast<uint32_t>(o)) x += y;
  }
  if (lane == 31) ws[warp] = x;
  __syncthreads();
  if (warp == 0) {
    uint32_t s = (lane < (blockDim.x >> 5)) ? ws[lane] : 0u;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_up_sync(0xffffffffu, s, o);
      if (lane >= static_cast<uint32_t>(o)) s += y;
    }
    ws[lane] = s;  // inclusive scan of warp totals
  }
  __syncthreads();
  const uint32_t warp_prefix = (warp == 0) ? 0u : ws[warp - 1];
  *total = ws[(blockDim.x >> 5) - 1];
  __syncthreads();
  return warp_prefix + x - v;
}

__global__ void __launch_bounds__(1024) k_tw_select(const float* __restrict__ scores, int64_t K,
                                                    const int32_t* __restrict__ offsets,
                                                    int32_t* __restrict__ indices) {
  __shared__ uint32_t hist[256];
  __shared__ uint32_t ws[32];
  __shared__ uint32_t s_prefix, s_remaining;
  const int64_t t = blockIdx.x;
  const int32_t L = offsets[t + 1] - offsets[t];
  if (L <= 0) return;
  int32_t* out = indices + offsets[t];
  const uint32_t* key = reinterpret_cast<const uint32_t*>(scores + t * K);

  uint32_t prefix = 0, mask = 0, remaining = static_cast<uint32_t>(L);
  for (int pass = 0; pass < 4; ++pass) {
    const int shift = 24 - 8 * pass;
    for (int i = threadIdx.x; i < 256; i += blockDim.x) hist[i] = 0;
    __syncthreads();
    for (int64_t k = threadIdx.x; k < K; k += blockDim.x) {
      const uint32_t x = key[k];
      if ((x & mask) == prefix) atomicAdd(&hist[(x >> shift) & 255u], 1u);
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      uint32_t cum = 0;
      for (int d = 255; d >= 0; --d) {
        const uint32_t h = hist[d];
        if (cum + h >= remaining) {
          s_prefix = prefix | (static_cast<uint32_t>(d) << shift);
          s_remaining = remaining - cum;
          break;
        }
        cum += h;
      }
    }
    __syncthreads();
    prefix = s_prefix;
    remaining = s_remaining;
    mask |= 255u << shift;
    __syncthreads();
  }
  // prefix = the L-th largest key; take every key above it and the `remaining`
  // lowest-k keys equal to it.
  const uint32_t thr = prefix, take_eq = remaining;
  uint32_t base = 0, eq_base = 0;
  for (int64_t k0 = 0; k0 < K; k0 += blockDim.x) {
    const int64_t k = k0 + threadIdx.x;
    const uint32_t x = (k < K) ? key[k] : 0u;
    const uint32_t gt = (k < K && x > thr) ? 1u : 0u;
    const uint32_t eq = (k < K && x == thr) ? 1u : 0u;
    uint32_t eq_total, take_total;
    const uint32_t eq_rank = eq_base + block_excl_scan(eq, ws, &eq_total);
    const uint32_t take = gt | ((eq && eq_rank < take_eq) ? 1u : 0u);
    const uint32_t pos = base + block_excl_scan(take, ws, &take_total);
    if (take) out[pos] = static_cast<int32_t>(k);
    base += take_total;
    eq_base += eq_total;
  }
}

// 512 threads = 16 warps = 16 consecutive rows of one 64-column chunk of a tile:
// blockIdx.x = chunk * 8 + row group, blockIdx.y = schedule entry (t, L, P, Q).
template <int DT, bool TVW>
__global__ void __launch_bounds__(512) k_tw_pack(const uint8_t* __restrict__ W, int64_t M, int64_t ldw_b,
                                                 const int32_t* __restrict__ offsets,
                                                 const int32_t* __restrict__ indices,
                                                 const int32_t* __restrict__ schedule, uint16_t* __restrict__ packed,
                                                 uint8_t* __restrict__ meta, uint8_t* __restrict__ meta_hw) {
  __shared__ uint32_t s_words[16][2];
  const int32_t* e = schedule + 4 * blockIdx.y;
  const int64_t t = e[0], L = e[1], P = e[2], Q = e[3];
  const int64_t R = (L + 63) / 64 * 64;
  const int64_t c = blockIdx.x >> 3;
  if (c * 64 >= R) return;  // uniform over the block
  const uint32_t warp = threadIdx.x >> 5, lane = threadIdx.x & 31u;
  const int64_t r = 16 * (blockIdx.x & 7) + warp;
  const int64_t row = t * 128 + r;
  const int32_t* idx = indices + offsets[t];
  const uint16_t* wrow = reinterpret_cast<const uint16_t*>(W + (row < M ? row : 0) * ldw_b);
  if constexpr (!TVW) {
    uint32_t v = 0;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int64_t j = c * 64 + 2 * lane + h;
      if (j < L && row < M) v |= static_cast<uint32_t>(wrow[idx[j]]) << (16 * h);
    }
    *reinterpret_cast<uint32_t*>(packed + 128 * P + 8192 * c + 64 * r + 2 * lane) = v;
  } else {
    uint32_t nib = 0;
    if (lane < 16) {
      const int64_t j = c * 64 + 4 * lane;
      uint32_t v01 = 0;
      nib = 0x4u;
      if (j < L && row < M) {  // L % 4 == 0: the group is entirely kept
        const uint32_t e0 = wrow[idx[j]], e1 = wrow[idx[j + 1]], e2 = wrow[idx[j + 2]], e3 = wrow[idx[j + 3]];
        nib = top2_nibble(e0 & 0x7FFFu, e1 & 0x7FFFu, e2 & 0x7FFFu, e3 & 0x7FFFu);
        const uint32_t j0 = nib & 3u, j1 = nib >> 2;
        v01 = __byte_perm(e0 | (e1 << 16), e2 | (e3 << 16),
                          (2 * j0) | ((2 * j0 + 1) << 4) | ((2 * j1) << 8) | ((2 * j1 + 1) << 12));
      }
      *reinterpret_cast<uint32_t*>(packed + 64 * P + 4096 * c + 32 * r + 2 * lane) = v01;
    }
    // the 16 nibbles of this row and chunk: lanes 0-7 form word 0, lanes 8-15 word 1
    uint32_t word = (lane < 16) ? (nib << (4 * (lane & 7))) : 0u;
#pragma unroll
    for (int o = 1; o < 8; o <<= 1) word |= __shfl_xor_sync(0xffffffffu, word, o);
    const uint32_t word1 = __shfl_sync(0xffffffffu, word, 8);
    if (lane == 0) {
      *reinterpret_cast<uint2*>(meta + 16 * P + r * (R / 8) + 8 * c) = make_uint2(word, word1);
      s_words[warp][0] = word;
      s_words[warp][1] = word1;
    }
    __syncthreads();
    if (lane == 0) {
      // tensor-core operand order: rows r and r ^ 8 share a word per 32-column span
      uint32_t hw[2];
#pragma unroll
      for (int jj = 0; jj < 2; ++jj) {
        const uint32_t own = s_words[warp][jj], partner = s_words[warp ^ 8][jj];
        hw[jj] = (warp & 8) ? ((partner >> 16) | (own & 0xFFFF0000u)) : ((own & 0xFFFFu) | (partner << 16));
      }
      *reinterpret_cast<uint4*>(meta_hw + 2048 * (Q + c) + 16 * r) = make_uint4(hw[0], 0u, hw[1], 0u);
    }
  }
}

// Block-wise: bs[t, b] = fp32 sum over the block's 64 column scores, ascending.
__global__ void __launch_bounds__(256) k_bw_block_scores(const float* __restrict__ scores, int64_t K, int64_t nt,
                                                         float* __restrict__ bs) {
  const int64_t KB = K / 64;
  const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= nt * KB) return;
  const int64_t t = i / KB, b = i - t * KB;
  const float* src = scores + t * K + 64 * b;
  float acc = 0.f;
#pragma unroll 8
  for (int j = 0; j < 64; ++j) acc = acc + src[j];
  bs[i] = acc;
}

// Block-wise: the kept blocks' column lists, in the blocks' order (64 per block).
__global__ void __launch_bounds__(256) k_bw_expand(const int32_t* __restrict__ blocks, int64_t n_blocks,
                                                   int32_t* __restrict__ cols) {
  const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= 64 * n_blocks) return;
  cols[i] = 64 * blocks[i >> 6] + static_cast<int32_t>(i & 63);
}

}  // namespace

cudaError_t launch_bw_prune(int dt, const void* W, int64_t M, int64_t K, int64_t ldw, const TwTables& tabs,
                            const int32_t* blk_offsets, int32_t* blk_indices, int64_t n_blocks,
                            const int32_t* col_offsets, int32_t* col_indices, const int32_t* schedule, void* packed,
                            float* scores, float* block_scores, cudaStream_t s) {
  if (tabs.nt == 0 || K == 0) return cudaSuccess;
  const auto* w8 = static_cast<const uint8_t*>(W);
  const bool vec_ok = (reinterpret_cast<uintptr_t>(W) % 16 == 0) && ((ldw * 2) % 16 == 0);
  cudaError_t e;
  dim3 g(static_cast<unsigned>(ceil_div(ceil_div(K, 8), 256)), static_cast<unsigned>(tabs.nt));
  if (dt == SSDNN_BF16)
    k_tw_score<1><<<g, 256, 0, s>>>(w8, M, K, ldw * 2, scores, vec_ok);
  else
    k_tw_score<0><<<g, 256, 0, s>>>(w8, M, K, ldw * 2, scores, vec_ok);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  const int64_t nb_all = tabs.nt * (K / 64);
  k_bw_block_scores<<<static_cast<unsigned>(ceil_div(nb_all, 256)), 256, 0, s>>>(scores, K, tabs.nt, block_scores);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  // the tile-wise top-L selection, over blocks: (score descending, index ascending)
  k_tw_select<<<static_cast<unsigned>(tabs.nt), 1024, 0, s>>>(block_scores, K / 64, blk_offsets, blk_indices);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  if (n_blocks == 0) return cudaSuccess;
  k_bw_expand<<<static_cast<unsigned>(ceil_div(64 * n_blocks, 256)), 256, 0, s>>>(blk_indices, n_blocks, col_indices);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  // the kept columns packed exactly as a tile-wise operand
  dim3 gp(static_cast<unsigned>((tabs.max_R / 64) * 8), static_cast<unsigned>(tabs.nt));
  auto* pk = static_cast<uint16_t*>(packed);
  if (dt == SSDNN_BF16)
    k_tw_pack<1, false><<<gp, 512, 0, s>>>(w8, M, ldw * 2, col_offsets, col_indices, schedule, pk, nullptr, nullptr);
  else
    k_tw_pack<0, false><<<gp, 512, 0, s>>>(w8, M, ldw * 2, col_offsets, col_indices, schedule, pk, nullptr, nullptr);
  return cudaGetLastError();
}

cudaError_t launch_row_select(const float* scores, int64_t rows, int64_t K, const int32_t* offsets, int32_t* indices,
                              cudaStream_t s) {
  if (rows == 0) return cudaSuccess;
  k_tw_select<<<static_cast<unsigned>(rows), 1024, 0, s>>>(scores, K, offsets, indices);
  return cudaGetLastError();
}

cudaError_t launch_tw_prune(int dt, int tvw, const void* W, int64_t M, int64_t K, int64_t ldw,
                            const TwTables& tabs, const int32_t* offsets, int32_t* indices,
                            const int32_t* schedule, void* packed, uint8_t* meta, uint8_t* meta_hw,
                            float* scores, cudaStream_t s, uint32_t* err) {
  (void)err;
  if (tabs.nt == 0) return cudaSuccess;
  const auto* w8 = static_cast<const uint8_t*>(W);
  const bool vec_ok = (reinterpret_cast<uintptr_t>(W) % 16 == 0) && ((ldw * 2) % 16 == 0);
  cudaError_t e;
  if (K > 0) {
    dim3 g(static_cast<unsigned>(ceil_div(ceil_div(K, 8), 256)), static_cast<unsigned>(tabs.nt));
    if (dt == SSDNN_BF16)
      k_tw_score<1><<<g, 256, 0, s>>>(w8, M, K, ldw * 2, scores, vec_ok);
    else
      k_tw_score<0><<<g, 256, 0, s>>>(w8, M, K, ldw * 2, scores, vec_ok);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    k_tw_select<<<static_cast<unsigned>(tabs.nt), 1024, 0, s>>>(scores, K, offsets, indices);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  if (tabs.max_R > 0) {
    dim3 g(static_cast<unsigned>((tabs.max_R / 64) * 8), static_cast<unsigned>(tabs.nt));
    auto* pk = static_cast<uint16_t*>(packed);
    if (dt == SSDNN_BF16) {
      if (tvw)
        k_tw_pack<1, true><<<g, 512, 0, s>>>(w8, M, ldw * 2, offsets, indices, schedule, pk, meta, meta_hw);
      else
        k_tw_pack<1, false><<<g, 512, 0, s>>>(w8, M, ldw * 2, offsets, indices, schedule, pk, meta, meta_hw);
    } else {
      if (tvw)
        k_tw_pack<0, true><<<g, 512, 0, s>>>(w8, M, ldw * 2, offsets, indices, schedule, pk, meta, meta_hw);
      else
        k_tw_pack<0, false><<<g, 512, 0, s>>>(w8, M, ldw * 2, offsets, indices, schedule, pk, meta, meta_hw);
    }
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace ssdnn
