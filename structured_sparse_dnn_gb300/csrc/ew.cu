// Element-wise (unstructured) sparsity: magnitude pruning to CSR and the
// sparse x dense product on the CUDA cores.
//
// "SparseRT: Accelerating Unstructured Sparsity on GPUs for Deep Learning
// Inference" (Abstract): individually pruned weights at 90-95 % sparsity, fully
// connected layers and 1x1 convolutions as sparse-weight x dense-activation
// products. "Accelerating Sparse DNNs Based on Tiled GEMM" (Figure 5 caption) uses
// the same EW pattern as its unstructured comparison point. Readings: every row
// keeps the same count k of its largest |w| (stored bits with the sign cleared,
// ties to the lower column), listed in ascending column order; CSR holds them.
//
// Kernels:
//   k_ew_mag     |w| as fp32 (exact for fp16/bf16), one row of keys per row of W;
//   k_tw_select  (shared with tile-wise) one CTA per row: exact top-k by radix
//                select, ascending compaction, ties to the lower column;
//   k_ew_values  the kept values' stored bits (k_ew_row_ptr: the row pointers);
//   k_ew_spmm    one CTA of 16 warps per (64 rows, 256 columns), one per SM: the X
//                panel streams through shared memory in 224-row chunks (two 112 KB
//                buffers filled by cp.async; long chunks, because the handling of each
//                (row, chunk) pair costs far more than an entry); each warp owns 4
//                rows and, for every kept entry of a row that falls in the chunk,
//                adds w times the chunk's X row into 8 fp32 accumulators per lane,
//                held and updated as packed pairs (the entries of a row are held 32
//                at a time in registers, one per lane, and broadcast by one shuffle
//                of the entry's chunk row and value bits).
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "common.cuh"
#include "kernels.h"

namespace ssdnn {

// The tile-wise top-L selection (csrc/tw.cu): one CTA per key row.
cudaError_t launch_row_select(const float* scores, int64_t rows, int64_t K, const int32_t* offsets, int32_t* indices,
                              cudaStream_t s);

namespace {

constexpr int kRowsW = 4;                          // output rows per warp
constexpr int kThreads = 512;
constexpr int kRows = (kThreads / 32) * kRowsW;    // output rows per CTA
constexpr int kCols = 256;                         // output columns per CTA (8 per lane)
constexpr int kChunk = 224;                        // X rows per shared-memory chunk (112 KB)

template <int DT>
__global__ void __launch_bounds__(256) k_ew_mag(const uint8_t* __restrict__ W, int64_t M, int64_t K, int64_t ldw_b,
                                                float* __restrict__ mag) {
  const int64_t i = blockIdx.y;
  for (int64_t k = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; k < K;
       k += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const uint32_t h = reinterpret_cast<const uint16_t*>(W + i * ldw_b)[k] & 0x7FFFu;
    float v;
    if constexpr (DT == 1)
      v = __uint_as_float(h << 16);
    else
      v = __half2float(__ushort_as_half(static_cast<unsigned short>(h)));
    mag[i * K + k] = v;
  }
}

__global__ void __launch_bounds__(256) k_ew_values(const uint8_t* __restrict__ W, int64_t M, int64_t ldw_b,
                                                   int64_t k, const int32_t* __restrict__ cols,
                                                   uint16_t* __restrict__ vals) {
  const int64_t j = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (j < M * k) {
    const int64_t i = j / k;
    vals[j] = reinterpret_cast<const uint16_t*>(W + i * ldw_b)[cols[j]];
  }
}

__global__ void __launch_bounds__(256) k_ew_row_ptr(int64_t M, int64_t k, int32_t* __restrict__ offsets) {
  const int64_t j = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (j <= M) offsets[j] = static_cast<int32_t>(j * k);
}

template <int DT>
__device__ __forceinline__ float to_f32(uint32_t h) {
  if constexpr (DT == 1) return __uint_as_float(h << 16);
  return __half2float(__ushort_as_half(static_cast<unsigned short>(h)));
}

template <int DT>
__global__ void __launch_bounds__(kThreads, 1) k_ew_spmm(int64_t M, int64_t N, int64_t K,
                                                         const int32_t* __restrict__ row_ptr,
                                                         const int32_t* __restrict__ col_idx,
                                                         const uint16_t* __restrict__ vals,
                                                         const uint16_t* __restrict__ X, int64_t ldx,
                                                         uint16_t* __restrict__ Y, int64_t ldy) {
  extern __shared__ __align__(16) uint8_t smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t row0 = static_cast<int64_t>(blockIdx.y) * kRows + warp * kRowsW;
  const int64_t n0 = static_cast<int64_t>(blockIdx.x) * kCols;
  const int64_t nchunks = (K + kChunk - 1) / kChunk;

  // this warp's kRowsW rows: next entry and end, and a register batch of the next 32
  // entries (lane l holds entry pos + l), refilled only when used up
  int32_t pos[kRowsW], end[kRowsW], bcol[kRowsW];
  uint32_t bval[kRowsW];
#pragma unroll
  for (int r = 0; r < kRowsW; ++r) {
    const int64_t i = row0 + r;
    pos[r] = i < M ? row_ptr[i] : 0;
    end[r] = i < M ? row_ptr[i + 1] : 0;
    const int32_t p = pos[r] + lane;
    bcol[r] = p < end[r] ? __ldg(col_idx + p) : INT32_MAX;
    bval[r] = p < end[r] ? __ldg(vals + p) : 0u;
  }
  int32_t used[kRowsW];  // entries of the current batch already consumed
#pragma unroll
  for (int r = 0; r < kRowsW; ++r) used[r] = 0;
  // fp32 accumulators as packed pairs: acc[r][h] holds columns 2h (low word) and 2h + 1
  uint64_t acc[kRowsW][4];
#pragma unroll
  for (int r = 0; r < kRowsW; ++r)
#pragma unroll
    for (int h = 0; h < 4; ++h) acc[r][h] = 0ull;

  // chunk loader: kChunk rows x 256 columns by 16-byte cp.async, zero past K / N
  auto load_chunk = [&](int64_t c, int buf) {
    uint8_t* dst = smem + buf * (kChunk * kCols * 2);
    for (int q = threadIdx.x; q < kChunk * (kCols / 8); q += kThreads) {
      const int rr = q / (kCols / 8), cc = q % (kCols / 8);
      const int64_t xr = c * kChunk + rr, xc = n0 + 8 * cc;
      uint32_t bytes = 0;
      const uint16_t* src = X;
      if (xr < K && xc < N) {
        bytes = static_cast<uint32_t>((N - xc < 8 ? N - xc : 8) * 2);
        src = X + xr * ldx + xc;
      }
      ptx::cp_async_16(dst + (rr * kCols + 8 * cc) * 2, src, bytes);
    }
    ptx::cp_async_commit();
  };

  load_chunk(0, 0);
  for (int64_t c = 0; c < nchunks; ++c) {
    if (c + 1 < nchunks) {
      load_chunk(c + 1, (c + 1) & 1);
      ptx::cp_async_wait<1>();
    } else {
      ptx::cp_async_wait<0>();
    }
    __syncthreads();
    const uint8_t* xs = smem + (c & 1) * (kChunk * kCols * 2) + lane * 16;
    const int32_t kend = static_cast<int32_t>(K < (c + 1) * kChunk ? K : (c + 1) * kChunk);
    const int32_t kbase = static_cast<int32_t>(c * kChunk);
#pragma unroll
    for (int r = 0; r < kRowsW; ++r) {
      // entries of row r inside this chunk: the batch is ascending, so those are the
      // lanes from `used` up to the first column at or past the chunk's end
      while (true) {
        const uint32_t in_chunk = __ballot_sync(0xffffffffu, bcol[r] < kend);
        const int n = __popc(in_chunk);
        // each lane's entry as one word: the row of the chunk and the value's bits. The
        // row is clamped to the chunk: under the contract (ascending columns) every
        // entry taken here lies in it, and an entry of a CSR that breaks the contract
        // reads a wrong row of the chunk rather than memory outside it.
        const uint32_t off = min(static_cast<uint32_t>(bcol[r] - kbase), static_cast<uint32_t>(kChunk - 1));
        const uint32_t ent = (off << 16) | (bval[r] & 0xFFFFu);
        // w times the X row of entry en
        auto add_entry = [&](uint32_t en) {
          const float w = to_f32<DT>(en & 0xFFFFu);
          const uint64_t w2 = ptx::f2_pack(w, w);
          const uint4 xv = *reinterpret_cast<const uint4*>(xs + (en >> 16) * (kCols * 2));
          const uint32_t xw[4] = {xv.x, xv.y, xv.z, xv.w};
#pragma unroll
          for (int h = 0; h < 4; ++h) {
            // the pair of X values as fp32 (bf16: the upper halves of two words)
            const uint64_t x2 =
                DT == 1 ? ptx::f2_pack(__uint_as_float(xw[h] << 16), __uint_as_float(xw[h] & 0xFFFF0000u))
                        : ptx::f2_pack(to_f32<DT>(xw[h] & 0xFFFFu), to_f32<DT>(xw[h] >> 16));
            acc[r][h] = ptx::f2_fma(w2, x2, acc[r][h]);
          }
        };
        // two entries a turn, so that their shuffles and shared-memory reads overlap
        int e = used[r];
        for (; e + 1 < n; e += 2) {
          const uint32_t en0 = __shfl_sync(0xffffffffu, ent, e), en1 = __shfl_sync(0xffffffffu, ent, e + 1);
          add_entry(en0);
          add_entry(en1);
        }
        if (e < n) add_entry(__shfl_sync(0xffffffffu, ent, e));
        used[r] = n;
        if (n < 32 || pos[r] + 32 >= end[r]) break;  // the batch reaches past this chunk, or the row ends
        // the whole batch was inside the chunk: fetch the next 32 entries
        pos[r] += 32;
        used[r] = 0;
        const int32_t p = pos[r] + lane;
        bcol[r] = p < end[r] ? __ldg(col_idx + p) : INT32_MAX;
        bval[r] = p < end[r] ? __ldg(vals + p) : 0u;
      }
    }
    __syncthreads();  // the buffer of chunk c is refilled by the next iteration's load
  }

  // kRowsW rows x 8 columns per lane, rounded once and stored 16 bytes at a time
  const int64_t col = n0 + 8 * lane;
#pragma unroll
  for (int r = 0; r < kRowsW; ++r) {
    const int64_t i = row0 + r;
    if (i >= M || col >= N) continue;
    uint32_t w[4];
#pragma unroll
    for (int h = 0; h < 4; ++h) {
      if constexpr (DT == 1) {
        const __nv_bfloat162 b = __floats2bfloat162_rn(ptx::f2_lo(acc[r][h]), ptx::f2_hi(acc[r][h]));
        w[h] = *reinterpret_cast<const uint32_t*>(&b);
      } else {
        const __half2 b = __floats2half2_rn(ptx::f2_lo(acc[r][h]), ptx::f2_hi(acc[r][h]));
        w[h] = *reinterpret_cast<const uint32_t*>(&b);
      }
    }
    uint16_t* dst = Y + i * ldy + col;
    if (col + 8 <= N) {
      *reinterpret_cast<uint4*>(dst) = make_uint4(w[0], w[1], w[2], w[3]);
    } else {
      for (int q = 0; q < 8; ++q)
        if (col + q < N) dst[q] = static_cast<uint16_t>(w[q >> 1] >> (16 * (q & 1)));
    }
  }
}

}  // namespace

cudaError_t launch_ew_prune(int dt, const void* W, int64_t M, int64_t K, int64_t ldw, int64_t k, int32_t* row_ptr,
                            int32_t* col_idx, void* vals, float* mag, cudaStream_t s) {
  cudaError_t e;
  k_ew_row_ptr<<<static_cast<unsigned>(ceil_div(M + 1, 256)), 256, 0, s>>>(M, k, row_ptr);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  if (M == 0 || k == 0) return cudaSuccess;
  const auto* w8 = static_cast<const uint8_t*>(W);
  const dim3 g(static_cast<unsigned>(std::min<int64_t>(ceil_div(K, 256), 64)), static_cast<unsigned>(M));
  if (dt == SSDNN_BF16)
    k_ew_mag<1><<<g, 256, 0, s>>>(w8, M, K, ldw * 2, mag);
  else
    k_ew_mag<0><<<g, 256, 0, s>>>(w8, M, K, ldw * 2, mag);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  if ((e = launch_row_select(mag, M, K, row_ptr, col_idx, s)) != cudaSuccess) return e;
  k_ew_values<<<static_cast<unsigned>(ceil_div(M * k, 256)), 256, 0, s>>>(w8, M, ldw * 2, k, col_idx,
                                                                          static_cast<uint16_t*>(vals));
  return cudaGetLastError();
}

cudaError_t launch_ew_spmm(int dt, int64_t M, int64_t N, int64_t K, const int32_t* row_ptr, const int32_t* col_idx,
                           const void* vals, const void* X, int64_t ldx, void* Y, int64_t ldy, cudaStream_t s) {
  if (M == 0 || N == 0) return cudaSuccess;
  constexpr int kSmem = 2 * kChunk * kCols * 2;
  const dim3 g(static_cast<unsigned>(ceil_div(N, kCols)), static_cast<unsigned>(ceil_div(M, kRows)));
  cudaError_t e;
  if (dt == SSDNN_BF16) {
    if ((e = cudaFuncSetAttribute(k_ew_spmm<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem)) != cudaSuccess)
      return e;
    k_ew_spmm<1><<<g, kThreads, kSmem, s>>>(M, N, K, row_ptr, col_idx, static_cast<const uint16_t*>(vals),
                                            static_cast<const uint16_t*>(X), ldx, static_cast<uint16_t*>(Y), ldy);
  } else {
    if ((e = cudaFuncSetAttribute(k_ew_spmm<0>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem)) != cudaSuccess)
      return e;
    k_ew_spmm<0><<<g, kThreads, kSmem, s>>>(M, N, K, row_ptr, col_idx, static_cast<const uint16_t*>(vals),
                                            static_cast<const uint16_t*>(X), ldx, static_cast<uint16_t*>(Y), ldy);
  }
  return cudaGetLastError();
}

}  // namespace ssdnn
