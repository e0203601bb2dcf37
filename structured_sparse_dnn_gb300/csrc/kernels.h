// Host-side launchers of the kernels; called by the C ABI after validation.
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace ssdnn {

// 2-D tensor map over a row-major matrix (rows x cols elements of eb bytes, pitch in
// bytes, boxes of box_cols x box_rows); false if the driver refuses the encoding.
bool make_map(CUtensorMap* m, const void* base, int eb, uint64_t cols, uint64_t rows, uint64_t pitch_bytes,
              uint32_t box_cols, uint32_t box_rows, CUtensorMapSwizzle swz);

// 2:4 magnitude prune + compress (one streaming pass over W).
cudaError_t launch_sp24_compress(int dt, const void* W, int64_t M, int64_t K, int64_t ldw, void* values,
                                 uint8_t* meta, uint8_t* meta_hw, cudaStream_t s, uint32_t* err);

struct GemmArgs {
  int dt, out_dt;
  int64_t M, N, K;
  const void* A;         // dense W, 2:4 values, or TW/TVW packed operand
  int64_t lda;           // elements (dense W pitch or values pitch)
  const uint8_t* meta_hw;
  const void* X;
  int64_t ldx;
  void* Y;
  int64_t ldy;
  float alpha;
  // tile-wise only
  int64_t nt;            // number of 128-row tiles
  int64_t packed_rows;   // rows of the packed operand seen as a (rows x 64 or 32) matrix
  const int32_t* offsets;
  const int32_t* indices;
  const int32_t* schedule;
  // 3x3 convolution (implicit GEMM): NHWC activations, K = 9 C_in ordered (tap, channel)
  int64_t conv_cin = 0, conv_h = 0, conv_w = 0, conv_nb = 0;
  // fused layer epilogue (out = round(y_scale * act(alpha * acc + bias[row])))
  const float* bias = nullptr;
  int act = 0;          // 0 none, 1 ReLU, 2 GELU
  float y_scale = 1.0f;
  // dense / 2:4 GEMM tile variant: 0 = chosen by shape; else one of kGemmVariants
  int variant = 0;
};

// Explicit tile variants of the dense and 2:4 GEMMs (tuning and tests):
// MT * 1000 + BN for single-CTA tiles of 128 MT rows x BN columns, 9256 for SM-pair
// 256 x 256 tiles with one 128-byte K step per stage, 19256 for SM-pair tiles with
// two K steps per stage (2:4 only).
bool gemm_variant_ok(int variant, bool sparse, int elem_bytes);

// mode: 0 dense, 1 sp24, 2 TW (dense packed + gather), 3 TVW (2:4 packed + gather),
// 4 block-wise (dense packed blocks, X panels by TMA), 5 / 6 3x3 convolution with a
// 2:4 / dense filter (activation taps by 4-D TMA boxes of NHWC X), 7 3x3 convolution
// with a tile-wise filter (the packed kept (tap, 64-channel) groups of each tile)
cudaError_t launch_gemm(int mode, const GemmArgs& a, cudaStream_t s, uint32_t* err);

// Y = round(y_scale * act(bias[row])) for every element (the fused epilogue of a
// product with no terms, K == 0); out_dt 0 f16, 1 bf16, 2 e4m3.
cudaError_t launch_fill_epilogue(void* Y, int64_t ldy, int64_t M, int64_t N, int out_dt, const float* bias, int act,
                                 float y_scale, cudaStream_t s);

// Tile-wise prune: scores -> per-tile top-L selection -> pack (TVW: + 2:4).
struct TwTables {
  int64_t nt;
  int64_t P_total;  // sum of round_up(L_t, 64)
  int64_t Q_total;  // metadata blocks: sum of R_t / 64
  int64_t max_R;    // max R_t
};
cudaError_t launch_tw_prune(int dt, int tvw, const void* W, int64_t M, int64_t K, int64_t ldw,
                            const TwTables& tabs, const int32_t* offsets, int32_t* indices,
                            const int32_t* schedule, void* packed, uint8_t* meta, uint8_t* meta_hw,
                            float* scores, cudaStream_t s, uint32_t* err);

// Block-wise prune: tile-wise column scores, 64-column block scores, per-tile top-B
// block selection, the kept blocks' column lists, and the tile-wise dense packing.
cudaError_t launch_bw_prune(int dt, const void* W, int64_t M, int64_t K, int64_t ldw, const TwTables& tabs,
                            const int32_t* blk_offsets, int32_t* blk_indices, int64_t n_blocks,
                            const int32_t* col_offsets, int32_t* col_indices, const int32_t* schedule, void* packed,
                            float* scores, float* block_scores, cudaStream_t s);

// Element-wise (unstructured) prune to CSR (k kept per row) and the CSR x dense product.
cudaError_t launch_ew_prune(int dt, const void* W, int64_t M, int64_t K, int64_t ldw, int64_t k, int32_t* row_ptr,
                            int32_t* col_idx, void* vals, float* mag, cudaStream_t s);
cudaError_t launch_ew_spmm(int dt, int64_t M, int64_t N, int64_t K, const int32_t* row_ptr, const int32_t* col_idx,
                           const void* vals, const void* X, int64_t ldx, void* Y, int64_t ldy, cudaStream_t s);

// Tensor-core issue-rate microbenchmark (operands resident on chip), one CTA per SM.
cudaError_t launch_mma_rate(int dt, int sparse, int n, int iters, cudaStream_t s, uint32_t* err);
cudaError_t launch_mma_rate_pair(int dt, int sparse, int iters, cudaStream_t s, uint32_t* err);

}  // namespace ssdnn
