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
//   k_tw_score   one CTA per (tile, 128 consecutive k): stages the tile's 128 x
//                128 block in shared memory (one TMA box, k_tw_score_tma, when W's
//                base and pitch are 16-byte aligned; else 16-byte or element loads),
//                then one thread per k sums the rows in order (fp32), into the
//                caller's workspace.
//   k_tw_select  one CTA per tile: exact top-L by a 4-pass 8-bit radix select on
//                the score bits (non-negative floats order like their bits; each
//                pass's digit found by one warp's scan of the histogram), then an
//                ascending-k compaction with one block prefix sum per 1024 keys
//                that takes ties at the threshold from the lowest k.
//   k_tw_pack    one warp per (row or TVW row pair, four 64-column chunks of a
//                tile): gathers the kept columns of the row into the chunk-blocked
//                packed operand; TVW selects 2 of every 4 and writes values plus
//                metadata in the canonical and the tensor-core operand order (which
//                pairs rows r and r ^ 8, the two halves of one warp).
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

// One CTA per (tile, 128 consecutive k): the tile's 128 rows x 128 columns (32 KB)
// are loaded with coalesced 16-byte loads into shared memory, then thread j sums
// column j over the rows in ascending order.
template <int DT>
__global__ void __launch_bounds__(128) k_tw_score(const uint8_t* __restrict__ W, int64_t M, int64_t K,
                                                  int64_t ldw_b, float* __restrict__ scores, bool vec_ok) {
  __shared__ __align__(16) uint16_t s_w[128][128];
  const int64_t t = blockIdx.y;
  const int64_t kb = static_cast<int64_t>(blockIdx.x) * 128;
  const int64_t r0 = t * 128;
  const int rows = static_cast<int>(M - r0 < 128 ? M - r0 : 128);
  // 16-byte segment `seg` of rows rsub, rsub + 8, ...: 16 threads cover a row's 256 bytes
  const int seg = static_cast<int>(threadIdx.x & 15u), rsub = static_cast<int>(threadIdx.x >> 4);
  const int64_t kseg = kb + 8 * seg;
#pragma unroll 1
  for (int half = 0; half < 2; ++half) {
    uint4 v[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int r = rsub + 8 * (8 * half + i);
      v[i] = make_uint4(0u, 0u, 0u, 0u);
      if (r < rows) {
        const uint8_t* p = W + (r0 + r) * ldw_b + kseg * 2;
        if (vec_ok && kseg + 8 <= K) {
          v[i] = __ldg(reinterpret_cast<const uint4*>(p));
        } else {
          uint32_t e[4] = {0u, 0u, 0u, 0u};
          for (int j = 0; j < 8; ++j)
            if (kseg + j < K) e[j >> 1] |= static_cast<uint32_t>(reinterpret_cast<const uint16_t*>(p)[j]) << (16 * (j & 1));
          v[i] = make_uint4(e[0], e[1], e[2], e[3]);
        }
      }
    }
#pragma unroll
    for (int i = 0; i < 8; ++i)
      *reinterpret_cast<uint4*>(&s_w[rsub + 8 * (8 * half + i)][8 * seg]) = v[i];
  }
  __syncthreads();
  const int64_t k = kb + threadIdx.x;
  if (k >= K) return;
  float acc = 0.f;
#pragma unroll 8
  for (int r = 0; r < rows; ++r) acc = acc + mag16<DT>(s_w[r][threadIdx.x]);
  scores[t * K + k] = acc;
}

// The same with the tile's 128 x 128 block brought in by one 2-D TMA box (rows past
// M and columns past K arrive as zeros): the copy engine fetches the 32 KB without
// the per-SM limit on 16-byte loads in flight that bounds the loop above.
template <int DT>
__global__ void __launch_bounds__(128) k_tw_score_tma(const __grid_constant__ CUtensorMap tmW, int64_t M, int64_t K,
                                                      float* __restrict__ scores, uint32_t* err) {
  __shared__ __align__(128) uint16_t s_w[128][128];
  __shared__ __align__(8) uint64_t bar;
  const int64_t t = blockIdx.y;
  const int64_t kb = static_cast<int64_t>(blockIdx.x) * 128;
  const int64_t r0 = t * 128;
  const int rows = static_cast<int>(M - r0 < 128 ? M - r0 : 128);
  if (threadIdx.x == 0) {
    ptx::mbar_init(&bar, 1);
    ptx::fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    ptx::mbar_arrive_expect_tx(&bar, 128u * 128u * 2u);
    ptx::tma_load_2d(&s_w[0][0], &tmW, &bar, static_cast<int32_t>(kb), static_cast<int32_t>(r0),
                     ptx::policy_evict_normal());
  }
  if (!wait_bounded(&bar, 0, err)) {
    wait_bounded(&bar, 0, nullptr);  // the copy may still be writing shared memory
    return;
  }
  const int64_t k = kb + threadIdx.x;
  if (k >= K) return;
  float acc = 0.f;
#pragma unroll 8
  for (int r = 0; r < rows; ++r) acc = acc + mag16<DT>(s_w[r][threadIdx.x]);
  scores[t * K + k] = acc;
}

// The score pass: by TMA where W's base and pitch allow it (16-byte aligned), else by
// 16-byte or element loads.
cudaError_t launch_score(int dt, const uint8_t* w8, int64_t M, int64_t K, int64_t ldw_b, float* scores, int64_t nt,
                         bool vec_ok, cudaStream_t s, uint32_t* err) {
  const dim3 g(static_cast<unsigned>(ceil_div(K, 128)), static_cast<unsigned>(nt));
  CUtensorMap m;
  if (vec_ok && make_map(&m, w8, 2, static_cast<uint64_t>(K), static_cast<uint64_t>(M), static_cast<uint64_t>(ldw_b),
                         128, 128, CU_TENSOR_MAP_SWIZZLE_NONE)) {
    if (dt == SSDNN_BF16)
      k_tw_score_tma<1><<<g, 128, 0, s>>>(m, M, K, scores, err);
    else
      k_tw_score_tma<0><<<g, 128, 0, s>>>(m, M, K, scores, err);
  } else if (dt == SSDNN_BF16) {
    k_tw_score<1><<<g, 128, 0, s>>>(w8, M, K, ldw_b, scores, vec_ok);
  } else {
    k_tw_score<0><<<g, 128, 0, s>>>(w8, M, K, ldw_b, scores, vec_ok);
  }
  return cudaGetLastError();
}

// Exclusive prefix sum over the block (whole warps, at most 1024 threads); returns
// this thread's prefix and writes the block total to *total. `ws` holds 32 words of
// shared scratch.
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

// NT threads per CTA: 1024 for the few tiles of a tile-wise weight (the CTA's latency
// is the kernel's), 256 for the many rows of the element-wise prune (more CTAs per SM).
template <int NT>
__global__ void __launch_bounds__(NT, NT >= 1024 ? 1 : 4) k_tw_select(const float* __restrict__ scores, int64_t K,
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

  // up to 4096 keys stay in registers (KPT a thread) for the four passes and the
  // compaction; longer rows are read from global memory on each pass
  constexpr int KPT = 4096 / NT;
  const bool cached = K <= static_cast<int64_t>(KPT) * NT;
  uint32_t kreg[KPT];
  if (cached) {
#pragma unroll
    for (int c = 0; c < KPT; ++c) {
      const int64_t k = static_cast<int64_t>(c) * NT + threadIdx.x;
      kreg[c] = k < K ? key[k] : 0u;
    }
  }

  uint32_t prefix = 0, mask = 0, remaining = static_cast<uint32_t>(L);
  for (int pass = 0; pass < 4; ++pass) {
    const int shift = 24 - 8 * pass;
    for (int i = threadIdx.x; i < 256; i += NT) hist[i] = 0;
    __syncthreads();
    if (cached) {
#pragma unroll
      for (int c = 0; c < KPT; ++c) {
        const uint32_t x = kreg[c];
        if (static_cast<int64_t>(c) * NT + threadIdx.x < K && (x & mask) == prefix)
          atomicAdd(&hist[(x >> shift) & 255u], 1u);
      }
    } else {
      for (int64_t k = threadIdx.x; k < K; k += NT) {
        const uint32_t x = key[k];
        if ((x & mask) == prefix) atomicAdd(&hist[(x >> shift) & 255u], 1u);
      }
    }
    __syncthreads();
    if (threadIdx.x < 32) {
      // the digit whose keys, counted from the largest digit down, reach `remaining`:
      // lane l sums bins 255 - 8 l .. 248 - 8 l, a warp scan orders the lanes, and
      // the first lane whose running count reaches `remaining` walks its eight bins
      const uint32_t lane = threadIdx.x;
      uint32_t h[8], sum = 0;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        h[i] = hist[255u - 8u * lane - static_cast<uint32_t>(i)];
        sum += h[i];
      }
      uint32_t inc = sum;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(0xffffffffu, inc, o);
        if (lane >= static_cast<uint32_t>(o)) inc += y;
      }
      const uint32_t found = __ballot_sync(0xffffffffu, inc >= remaining);
      if (found == 0u) {  // L > K (refused by the host): take every key
        if (lane == 0) {
          s_prefix = 0u;
          s_remaining = 0u;
        }
      } else if (lane == static_cast<uint32_t>(__ffs(found) - 1)) {
        uint32_t cum = inc - sum;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          if (cum + h[i] >= remaining) {
            s_prefix = prefix | ((255u - 8u * lane - static_cast<uint32_t>(i)) << shift);
            s_remaining = remaining - cum;
            break;
          }
          cum += h[i];
        }
      }
    }
    __syncthreads();
    prefix = s_prefix;
    remaining = s_remaining;
    mask |= 255u << shift;
  }
  // prefix = the L-th largest key; take every key above it and the `remaining`
  // lowest-k keys equal to it. A taken key's place is the number of larger keys
  // before it plus the number of equal keys before it (at most `remaining`): one
  // block scan of both counts (16 bits each) per 1024 keys.
  const uint32_t thr = prefix, take_eq = remaining;
  uint32_t gt_base = 0, eq_base = 0;
  auto compact = [&](uint32_t x, int64_t k) {  // every thread, once per NT keys
    const uint32_t gt = (k < K && x > thr) ? 1u : 0u;
    const uint32_t eq = (k < K && x == thr) ? 1u : 0u;
    uint32_t total;
    const uint32_t ex = block_excl_scan(gt | (eq << 16), ws, &total);
    const uint32_t gt_before = gt_base + (ex & 0xFFFFu), eq_before = eq_base + (ex >> 16);
    const bool take = gt != 0u || (eq != 0u && eq_before < take_eq);
    const uint32_t pos = gt_before + (eq_before < take_eq ? eq_before : take_eq);
    if (take && pos < static_cast<uint32_t>(L)) out[pos] = static_cast<int32_t>(k);
    gt_base += total & 0xFFFFu;
    eq_base += total >> 16;
  };
  if (cached) {
#pragma unroll
    for (int c = 0; c < KPT; ++c) {
      if (static_cast<int64_t>(c) * NT >= K) break;  // uniform over the block
      compact(kreg[c], static_cast<int64_t>(c) * NT + threadIdx.x);
    }
  } else {
    for (int64_t k0 = 0; k0 < K; k0 += NT) {
      const int64_t k = k0 + threadIdx.x;
      compact(k < K ? key[k] : 0u, k);
    }
  }
}

// 512 threads = 16 warps; blockIdx.y = schedule entry (t, L, P, Q), blockIdx.x = chunk
// group * row groups + row group. Each warp packs kPackChunks consecutive 64-column
// chunks, all index and weight loads of which are independent and issued together.
// TW: warp w packs row 16 g + w. TVW: warp w packs rows r and r + 8 (lanes 0-15 and
// 16-31, r = 32 g + 16 (w >> 3) + (w & 7)), so the pair of rows that share the
// tensor-core metadata words meets inside one warp.
constexpr int kPackChunks = 4;
template <int DT, bool TVW>
__global__ void __launch_bounds__(512) k_tw_pack(const uint8_t* __restrict__ W, int64_t M, int64_t ldw_b,
                                                 const int32_t* __restrict__ offsets,
                                                 const int32_t* __restrict__ indices,
                                                 const int32_t* __restrict__ schedule, uint16_t* __restrict__ packed,
                                                 uint8_t* __restrict__ meta, uint8_t* __restrict__ meta_hw) {
  constexpr int GROUPS = TVW ? 4 : 8;  // row groups per tile (32 or 16 rows each)
  const int32_t* e = schedule + 4 * blockIdx.y;
  const int64_t t = e[0], L = e[1], P = e[2], Q = e[3];
  const int64_t nch = (L + 63) / 64;  // chunks of the tile
  const int64_t c0 = static_cast<int64_t>(blockIdx.x / GROUPS) * kPackChunks;
  if (c0 >= nch) return;  // uniform over the block
  const int g = static_cast<int>(blockIdx.x % GROUPS);
  const uint32_t warp = threadIdx.x >> 5, lane = threadIdx.x & 31u;
  const int32_t* idx = indices + offsets[t];
  if constexpr (!TVW) {
    const int64_t r = 16 * g + warp;
    const int64_t row = t * 128 + r;
    const uint16_t* wrow = reinterpret_cast<const uint16_t*>(W + (row < M ? row : 0) * ldw_b);
    int32_t k[kPackChunks][2];
#pragma unroll
    for (int cc = 0; cc < kPackChunks; ++cc)
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int64_t j = (c0 + cc) * 64 + 2 * lane + h;
        k[cc][h] = (j < L && row < M) ? __ldg(idx + j) : -1;
      }
    uint32_t v[kPackChunks];
#pragma unroll
    for (int cc = 0; cc < kPackChunks; ++cc) {
      v[cc] = 0u;
#pragma unroll
      for (int h = 0; h < 2; ++h)
        if (k[cc][h] >= 0) v[cc] |= static_cast<uint32_t>(__ldg(wrow + k[cc][h])) << (16 * h);
    }
#pragma unroll
    for (int cc = 0; cc < kPackChunks; ++cc)
      if (c0 + cc < nch)
        *reinterpret_cast<uint32_t*>(packed + 128 * P + 8192 * (c0 + cc) + 64 * r + 2 * lane) = v[cc];
  } else {
    const uint32_t half = lane >> 4, hl = lane & 15u;
    const int64_t r = 32 * g + 16 * (warp >> 3) + (warp & 7u) + 8 * half;
    const int64_t row = t * 128 + r;
    const uint16_t* wrow = reinterpret_cast<const uint16_t*>(W + (row < M ? row : 0) * ldw_b);
    int32_t k[kPackChunks][4];
#pragma unroll
    for (int cc = 0; cc < kPackChunks; ++cc) {
      const int64_t j = (c0 + cc) * 64 + 4 * hl;  // L % 4 == 0: a group is entirely kept or not
      const bool ok = j < L && row < M;
#pragma unroll
      for (int q = 0; q < 4; ++q) k[cc][q] = ok ? __ldg(idx + j + q) : -1;
    }
    uint32_t ev[kPackChunks][4];
#pragma unroll
    for (int cc = 0; cc < kPackChunks; ++cc)
#pragma unroll
      for (int q = 0; q < 4; ++q) ev[cc][q] = k[cc][q] >= 0 ? static_cast<uint32_t>(__ldg(wrow + k[cc][q])) : 0u;
#pragma unroll
    for (int cc = 0; cc < kPackChunks; ++cc) {
      const int64_t c = c0 + cc;
      if (c >= nch) break;  // uniform over the warp
      uint32_t nib = 0x4u, v01 = 0u;
      if (k[cc][0] >= 0) {
        nib = top2_nibble(ev[cc][0] & 0x7FFFu, ev[cc][1] & 0x7FFFu, ev[cc][2] & 0x7FFFu, ev[cc][3] & 0x7FFFu);
        const uint32_t j0 = nib & 3u, j1 = nib >> 2;
        v01 = __byte_perm(ev[cc][0] | (ev[cc][1] << 16), ev[cc][2] | (ev[cc][3] << 16),
                          (2 * j0) | ((2 * j0 + 1) << 4) | ((2 * j1) << 8) | ((2 * j1 + 1) << 12));
      }
      *reinterpret_cast<uint32_t*>(packed + 64 * P + 4096 * c + 32 * r + 2 * hl) = v01;
      // the 16 nibbles of this row and chunk: lanes 0-7 of the half form word 0,
      // lanes 8-15 word 1
      uint32_t word = nib << (4 * (hl & 7u));
#pragma unroll
      for (int o = 1; o < 8; o <<= 1) word |= __shfl_xor_sync(0xffffffffu, word, o);
      const uint32_t w0 = __shfl_sync(0xffffffffu, word, 16 * half);
      const uint32_t w1 = __shfl_sync(0xffffffffu, word, 16 * half + 8);
      // tensor-core operand order: rows r and r + 8 share a word per 32-column span
      const uint32_t p0 = __shfl_xor_sync(0xffffffffu, w0, 16), p1 = __shfl_xor_sync(0xffffffffu, w1, 16);
      if (hl == 0) {
        *reinterpret_cast<uint2*>(meta + 16 * P + r * (nch * 8) + 8 * c) = make_uint2(w0, w1);
        const uint32_t h0 = half ? ((p0 >> 16) | (w0 & 0xFFFF0000u)) : ((w0 & 0xFFFFu) | (p0 << 16));
        const uint32_t h1 = half ? ((p1 >> 16) | (w1 & 0xFFFF0000u)) : ((w1 & 0xFFFFu) | (p1 << 16));
        *reinterpret_cast<uint4*>(meta_hw + 2048 * (Q + c) + 16 * r) = make_uint4(h0, 0u, h1, 0u);
      }
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
  if ((e = launch_score(dt, w8, M, K, ldw * 2, scores, tabs.nt, vec_ok, s, nullptr)) != cudaSuccess) return e;
  const int64_t nb_all = tabs.nt * (K / 64);
  k_bw_block_scores<<<static_cast<unsigned>(ceil_div(nb_all, 256)), 256, 0, s>>>(scores, K, tabs.nt, block_scores);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  // the tile-wise top-L selection, over blocks: (score descending, index ascending)
  k_tw_select<1024><<<static_cast<unsigned>(tabs.nt), 1024, 0, s>>>(block_scores, K / 64, blk_offsets, blk_indices);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  if (n_blocks == 0) return cudaSuccess;
  k_bw_expand<<<static_cast<unsigned>(ceil_div(64 * n_blocks, 256)), 256, 0, s>>>(blk_indices, n_blocks, col_indices);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  // the kept columns packed exactly as a tile-wise operand
  dim3 gp(static_cast<unsigned>(ceil_div(tabs.max_R / 64, kPackChunks) * 8), static_cast<unsigned>(tabs.nt));
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
  k_tw_select<256><<<static_cast<unsigned>(rows), 256, 0, s>>>(scores, K, offsets, indices);
  return cudaGetLastError();
}

cudaError_t launch_tw_prune(int dt, int tvw, const void* W, int64_t M, int64_t K, int64_t ldw,
                            const TwTables& tabs, const int32_t* offsets, int32_t* indices,
                            const int32_t* schedule, void* packed, uint8_t* meta, uint8_t* meta_hw,
                            float* scores, cudaStream_t s, uint32_t* err) {
  if (tabs.nt == 0) return cudaSuccess;
  const auto* w8 = static_cast<const uint8_t*>(W);
  const bool vec_ok = (reinterpret_cast<uintptr_t>(W) % 16 == 0) && ((ldw * 2) % 16 == 0);
  cudaError_t e;
  if (K > 0) {
    if ((e = launch_score(dt, w8, M, K, ldw * 2, scores, tabs.nt, vec_ok, s, err)) != cudaSuccess) return e;
    k_tw_select<1024><<<static_cast<unsigned>(tabs.nt), 1024, 0, s>>>(scores, K, offsets, indices);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  if (tabs.max_R > 0) {
    // 16 rows (TW) or 32 rows (TVW) and kPackChunks chunks per CTA
    const unsigned cg = static_cast<unsigned>(ceil_div(tabs.max_R / 64, kPackChunks));
    dim3 g(cg * (tvw ? 4u : 8u), static_cast<unsigned>(tabs.nt));
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
