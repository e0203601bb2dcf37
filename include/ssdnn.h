/*
 * ssdnn.h -- C ABI of the structured-sparse weight GEMM library for GB300 (sm_103a).
 *
 * The library computes Y = W_sparse . X for pruned fully connected layers and
 * 1x1 convolutions written as GEMMs, with two weight patterns:
 *
 *   2:4 fine-grained sparsity -- in every contiguous group of four weights along
 *   K two are zero; W is stored as its kept values plus 2-bit positions
 *   ("NVIDIA A100 benchmarks" blog page, paragraph on 2:4 structured sparsity
 *   and Figure 1 caption; "Accelerating Sparse Deep Neural Networks", Abstract).
 *
 *   Tile-wise (TW) sparsity and its tile-vector-wise (TVW) hybrid -- each tile of
 *   128 output rows keeps its own subset of K indices, applied where operands are
 *   fetched from global memory; TVW also applies 2:4 inside the kept indices
 *   ("Accelerating Sparse DNNs Based on Tiled GEMM", TL;DR, Abstract, Figure 3).
 *
 * Conventions (every function):
 *   - Returns an ssdnn_status; no exception or abort crosses the ABI.
 *   - Pointers are DEVICE pointers unless the parameter name ends in _host.
 *     The caller owns and allocates every buffer (the *_sizes functions give the
 *     sizes); the library allocates no memory.
 *   - Work is enqueued asynchronously on `stream` (a cudaStream_t, NULL = legacy
 *     default stream); outputs are valid once the stream has reached that point.
 *   - Matrices are row-major with explicit leading dimensions in ELEMENTS:
 *       W  M x K   (K contiguous),  X  K x N  (N contiguous),  Y  M x N.
 *     Base pointers must be 16-byte aligned and leading dimension x element size
 *     a multiple of 16 bytes; otherwise SSDNN_ERR_UNSUPPORTED.
 *   - Inputs must be finite. Element types: ssdnn_dtype.
 *   - A kernel whose internal wait exceeds its bound records it in a per-device
 *     error word and returns; ssdnn_check_device_error() reports it.
 *
 * Readings of the method where the pages are silent (magnitude criterion, tie
 * rules, layouts, tile height 128) are stated beside each call.
 */
#ifndef SSDNN_H
#define SSDNN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum { SSDNN_F16 = 0, SSDNN_BF16 = 1, SSDNN_E4M3 = 2 } ssdnn_dtype;

typedef enum {
  SSDNN_OK = 0,
  SSDNN_ERR_INVALID_ARG = 1, /* null pointer, negative size, bad enum, inconsistent counts */
  SSDNN_ERR_UNSUPPORTED = 2, /* shape / alignment / dtype combination not implemented */
  SSDNN_ERR_CUDA = 3,        /* a CUDA runtime or driver call failed */
  SSDNN_ERR_TIMEOUT = 4,     /* a bounded device-side wait expired */
  SSDNN_ERR_DEVICE = 5       /* a kernel recorded an internal error */
} ssdnn_status;

/* Constant string for a status code. */
const char* ssdnn_status_str(int status);

/* Library ABI version (major * 100 + minor). */
int ssdnn_version(void);

/* Synchronizes `stream`, then reads and clears this device's error word.
 * Returns SSDNN_OK, SSDNN_ERR_TIMEOUT or SSDNN_ERR_DEVICE. */
int ssdnn_check_device_error(void* stream);

/* Failure-detection self-test. Launches one thread on `stream` that waits,
 * through the same bounded wait the GEMM pipeline uses, on an mbarrier that
 * nothing arrives on. After `limit_us` microseconds (1 .. 1000000) the wait
 * gives up, sets the timeout bit of this device's error word and the kernel
 * returns normally, so the context stays usable; the following
 * ssdnn_check_device_error() then returns SSDNN_ERR_TIMEOUT. Returns
 * SSDNN_ERR_INVALID_ARG for a limit outside the range, else the launch status.
 * No passage of the pages defines this call: it tests the library's own
 * recovery path (kernels give up on a stalled pipeline instead of hanging). */
int ssdnn_selftest_wait_timeout(uint32_t limit_us, void* stream);

/* Tensor-core rate microbenchmark (measurement only; no output buffer).
 * Launches one CTA per SM on `stream`; each issues `iters` (1 .. 262144) steps
 * of tcgen05.mma with operands resident in shared memory and the fp32
 * accumulator in TMEM: M = 128 rows, N = `n` columns (128, 192 or 256), and
 * 128 bytes of K per step (64 elements for f16/bf16, 128 for e4m3), in the dense
 * (`sparse` = 0) or the 2:4-sparse (`sparse` = 1) form, where K counts the dense
 * width the sparse instruction covers. A step is 2 * 128 * n * (128 / elem
 * bytes) dense-equivalent flops per SM; the caller times the launch. The pages
 * state that the sparse tensor core doubles the dense math rate ("Accelerating
 * Sparse Deep Neural Networks", Abstract; "NVIDIA A100 benchmarks" page, 2:4
 * paragraph); this call measures both rates on the device at hand.
 * Returns SSDNN_ERR_INVALID_ARG / SSDNN_ERR_UNSUPPORTED for a bad dtype, flag,
 * step count or n, else the launch status. */
int ssdnn_mma_rate(int dt, int sparse, int n, int iters, void* stream);

/* The same measurement on SM pairs (tcgen05 cta_group::2, the form the large GEMM
 * tiles use): clusters of two CTAs on an even number of SMs, M = 256, N = 256,
 * 128 bytes of K per step; each CTA holds 128 rows of A and 128 columns of B. In
 * the 2:4 form every step also copies its 128 x 16-byte metadata block into TMEM
 * before its instructions, as the GEMM does for each K stage. A step is
 * 2 * 256 * 256 * (128 / elem bytes) dense-equivalent flops per pair. Returns
 * SSDNN_ERR_INVALID_ARG for a bad dtype, flag or step count, else the launch
 * status. */
int ssdnn_mma_rate_pair(int dt, int sparse, int iters, void* stream);

/* ------------------------------------------------------------------ 2:4 ----
 * Compressed 2:4 layouts (Kp = round_up(K, 32)):
 *   values   M x Kp/2 elements, row-major: the kept values of each group in
 *            ascending position order, stored bits copied; zero past K/2.
 *   meta     M x Kp/8 bytes, row-major: group g = k/4 has nibble j0 | j1 << 2
 *            (j0 < j1 its kept positions), at byte g/2, low nibble for even g;
 *            nibble 0x4 past K/4.
 *   meta_hw  the operand order of the sparse tensor core: 2048-byte blocks of
 *            128 rows x 16 bytes, block (mb, kb) at index mb * KB + kb.
 *            e4m3: kb spans 128 columns of K (KB = ceil(K/128)); row r holds the
 *              canonical bytes 16 kb .. 16 kb + 15 of row 128 mb + r.
 *            fp16/bf16: kb spans 64 columns (KB = ceil(K/64)); row r holds four
 *              32-bit words; words 0 and 2 cover the column spans 64 kb .. +31
 *              and 64 kb + 32 .. +63, words 1 and 3 are zero. Rows are paired
 *              (r and r ^ 8): for r with bit 3 clear the word is (canonical
 *              nibbles of groups 0..3 of row r) | (groups 0..3 of row r + 8) << 16;
 *              for r with bit 3 set it is (groups 4..7 of row r - 8) |
 *              (groups 4..7 of row r) << 16 (groups counted within the span).
 *            Rows past M and groups past K hold 0x4 nibbles.
 * Pruning (the pages state no criterion; reading: magnitude): keep the two
 * entries of largest |w| per group, |w| ordered by the stored bits with the sign
 * bit cleared, ties to the lower position. K % 4 == 0 is required.
 */
int sp24_sizes(int dt, int64_t M, int64_t K, size_t* values_bytes, size_t* meta_bytes,
               size_t* meta_hw_bytes);

/* W (M x K, leading dimension ldw) -> values, meta, meta_hw (all three written;
 * meta may be NULL to skip the canonical copy). */
int sp24_prune_compress(int dt, const void* W, int64_t M, int64_t K, int64_t ldw, void* values,
                        uint8_t* meta, uint8_t* meta_hw, void* stream);

/* Y = alpha * decompress(values, meta_hw) . X, fp32 accumulation on the sparse
 * tensor cores, one round-to-nearest-even conversion to out_dt.
 * in_dt in {F16, BF16, E4M3}; out_dt in {F16, BF16}. values has the pitch Kp/2
 * of sp24_prune_compress. ldx >= N, ldy >= N. */
int sp24_gemm(int in_dt, int out_dt, int64_t M, int64_t N, int64_t K, const void* values,
              const uint8_t* meta_hw, const void* X, int64_t ldx, void* Y, int64_t ldy, float alpha,
              void* stream);

/* The dense GEMM of the same kernel family: Y = alpha * W . X. */
int dense_gemm(int in_dt, int out_dt, int64_t M, int64_t N, int64_t K, const void* W, int64_t ldw,
               const void* X, int64_t ldx, void* Y, int64_t ldy, float alpha, void* stream);

/* ------------------------------------------------------------- TW / TVW ----
 * Tiles are 128 consecutive rows of W (and Y): tile t = rows 128 t ..; the
 * number of tiles is nt = ceil(M / 128). keep_counts_host[t] = L_t, 0 <= L_t <= K
 * (TVW: L_t % 4 == 0). dt in {F16, BF16}.
 * Selection (reading of the pages): score s_t[k] = fp32 sum over the tile's rows
 * in ascending order of |w_ik|; the kept set is the first L_t of the order
 * (score descending, k ascending), listed ascending.
 * Layouts (R_t = round_up(L_t, 64), P_t = sum_{s<t} R_s, Q_t = P_t / 64):
 *   offsets   nt + 1 int32: offsets[t] = sum_{s<t} L_s.
 *   indices   offsets[nt] int32: tile t's kept k, ascending, at offsets[t].
 *   schedule  4 * nt int32: entries (t, L_t, P_t, Q_t) for the tiles ordered by
 *             L_t descending, ties by t ascending (tiles of equal length form a
 *             batch; the GEMM hands out work in this order for load balance).
 *   packed    TW:  128 * P_nt elements; element (t, r, j), j < R_t, at
 *                  128 P_t + 8192 (j / 64) + 64 r + j % 64 (zero past L_t and
 *                  past row M).
 *             TVW: 64 * P_nt elements, the 2:4 values of each packed tile:
 *                  (t, r, c), c < R_t / 2, at 64 P_t + 4096 (c / 32) + 32 r + c % 32.
 *   meta      TVW only: 16 * P_nt bytes; byte b < R_t / 8 of tile row r at
 *             16 P_t + r R_t / 8 + b (canonical nibbles along the compacted K).
 *   meta_hw   TVW only: 32 * P_nt bytes; tile t's metadata in the fp16/bf16
 *             operand order of meta_hw above (128 rows, K = R_t), R_t / 64 blocks
 *             starting at block Q_t.
 *   workspace scratch for the scores: nt * K * 4 bytes.
 */
int tw_sizes(int dt, int tvw, int64_t M, int64_t K, const int32_t* keep_counts_host,
             size_t* packed_bytes, size_t* indices_count, size_t* meta_bytes, size_t* meta_hw_bytes,
             size_t* workspace_bytes);

int tw_prune_compress(int dt, int tvw, const void* W, int64_t M, int64_t K, int64_t ldw,
                      const int32_t* keep_counts_host, int32_t* offsets, int32_t* indices,
                      int32_t* schedule, void* packed, uint8_t* meta, uint8_t* meta_hw, void* workspace,
                      void* stream);

/* Y[tile t rows] = W_t . X[indices of t, :] (TW) or the 2:4 product of the TVW
 * values (TVW), fp32 accumulation, one RNE conversion to dt. A tile with L_t = 0
 * writes zeros. keep_counts_host is the array given to tw_prune_compress. */
int tvw_gemm(int dt, int tvw, int64_t M, int64_t N, int64_t K, const int32_t* keep_counts_host,
             const int32_t* offsets, const int32_t* indices, const int32_t* schedule, const void* packed,
             const uint8_t* meta_hw, const void* X, int64_t ldx, void* Y, int64_t ldy, void* stream);

/* sp24_gemm with the activations and the result in host memory. X_host (K x N,
 * pitch ldx) is copied to the caller's device buffer X_dev (same pitch) on
 * `stream`; Y is computed into the caller's device buffer Y_dev (M x N, pitch ldy)
 * in blocks of rows_per_block rows (a multiple of 128; 0 = one block), and each
 * block is copied to Y_host (pitch ldy) on `copy_stream` as soon as its GEMM has
 * finished, while the next block is computed (copy_stream NULL: everything runs
 * on `stream`, in order). The host buffers should be page-locked for the copies
 * to be asynchronous. The call only enqueues; Y_host is complete once `stream`
 * has completed. Returns as sp24_gemm, or SSDNN_ERR_INVALID_ARG for a null host
 * buffer or a block height that is not a multiple of 128.
 * Y_dev NULL: the GEMM's epilogue stores the result straight into Y_host, which
 * must then be page-locked (cudaHostAlloc / cudaHostRegister; anything else is
 * SSDNN_ERR_INVALID_ARG); rows_per_block and copy_stream are ignored and K = 0 is
 * SSDNN_ERR_UNSUPPORTED. The product path refuses host memory for every other
 * operand. The direct form saves the device buffer, not time: the epilogue's
 * row-wise stores cross the host link in small transactions, several times
 * slower than the copy engines for a large Y. */
int sp24_gemm_host(int in_dt, int out_dt, int64_t M, int64_t N, int64_t K, const void* values,
                   const uint8_t* meta_hw, const void* X_host, int64_t ldx, void* Y_host, int64_t ldy, float alpha,
                   void* X_dev, void* Y_dev, int64_t rows_per_block, void* stream, void* copy_stream);

/* ------------------------------------------------------------ block-wise ----
 * Block sparsity, the comparison pattern of the tiled-GEMM page ("Accelerating
 * Sparse DNNs Based on Tiled GEMM", Abstract; Figure 5 caption: BW pruning):
 * whole blocks of W are removed. Readings (the page fixes no block shape): a
 * block is 128 rows (one tile, as for TW) x 64 consecutive columns; K % 64 == 0.
 * Block score = fp32 sum over the block's 64 columns, ascending, of the TW
 * column scores (fp32 sums of |w| over the tile's rows, ascending); tile t keeps
 * the first keep_blocks_host[t] blocks of (score descending, block ascending),
 * listed ascending. The GEMM reads each kept block's 64-row X panel with one TMA
 * box (no gather).
 * Layouts (nt = ceil(M / 128), B_t = keep_blocks_host[t], P_t = sum_{s<t} 64 B_s):
 *   offsets   nt + 1 int32, offsets[t] = sum_{s<t} B_s (in blocks).
 *   indices   sum B_t int32: the kept block indices of each tile, ascending.
 *   schedule  4 nt int32: (t, 64 B_t, P_t, P_t / 64), tiles by B_t descending, as TW.
 *   packed    the TW dense packed operand of the kept columns: element (t, r, j),
 *             j < 64 B_t, at 128 P_t + 8192 (j / 64) + 64 r + j % 64 (rows past M zero).
 *   workspace bw_sizes' workspace_bytes (scores and column lists).
 * fp16/bf16 only (E4M3: SSDNN_ERR_UNSUPPORTED); K % 64 != 0: SSDNN_ERR_UNSUPPORTED. */
int bw_sizes(int dt, int64_t M, int64_t K, const int32_t* keep_blocks_host, size_t* packed_bytes,
             size_t* indices_count, size_t* workspace_bytes);
int bw_prune_compress(int dt, const void* W, int64_t M, int64_t K, int64_t ldw, const int32_t* keep_blocks_host,
                      int32_t* offsets, int32_t* indices, int32_t* schedule, void* packed, void* workspace,
                      void* stream);
/* Y[tile t] = W_t . X[kept rows], fp32 accumulation, one RNE conversion to dt; a
 * tile that keeps no block writes zeros. bw_gemm_ep adds the output type, alpha
 * and the fused epilogue (below). */
int bw_gemm(int dt, int64_t M, int64_t N, int64_t K, const int32_t* keep_blocks_host, const int32_t* offsets,
            const int32_t* indices, const int32_t* schedule, const void* packed, const void* X, int64_t ldx, void* Y,
            int64_t ldy, void* stream);

/* ---------------------------------------------------------- element-wise ----
 * Unstructured sparsity ("SparseRT: Accelerating Unstructured Sparsity on GPUs
 * for Deep Learning Inference", Abstract: individually pruned weights, 90-95 %
 * sparsity, fully connected / 1x1 layers as sparse x dense products; the EW
 * pattern of the tiled-GEMM page, Figure 5 caption). Readings: every row keeps
 * the same count k of its largest |w| (stored bits with the sign cleared, ties to
 * the lower column), listed in ascending column order, as CSR:
 *   row_ptr  M + 1 int32 (row_ptr[i] = i k), col_idx M k int32, vals M k values
 *            (stored bits copied).
 * ew_prune_compress needs ew_sizes' workspace (M x K fp32 magnitudes). ew_spmm
 * takes any CSR (row_ptr non-decreasing, columns ascending within a row, all
 * < K): Y = W_ew . X, fp32 accumulation on the CUDA cores, one RNE conversion to
 * dt. fp16/bf16 only (E4M3: SSDNN_ERR_UNSUPPORTED). */
int ew_sizes(int dt, int64_t M, int64_t K, int64_t k, size_t* vals_bytes, size_t* indices_count,
             size_t* workspace_bytes);
int ew_prune_compress(int dt, const void* W, int64_t M, int64_t K, int64_t ldw, int64_t k, int32_t* row_ptr,
                      int32_t* col_idx, void* vals, void* workspace, void* stream);
int ew_spmm(int dt, int64_t M, int64_t N, int64_t K, const int32_t* row_ptr, const int32_t* col_idx,
            const void* vals, const void* X, int64_t ldx, void* Y, int64_t ldy, void* stream);

/* ------------------------------------------------------ 3x3 convolution ----
 * Sparse 3x3 convolutions (ResNet-50 use cases: "SparseRT: Accelerating
 * Unstructured Sparsity on GPUs for Deep Learning Inference", Abstract) with a
 * 2:4 filter ("Accelerating Sparse Deep Neural Networks", Abstract), run as an
 * implicit GEMM on the (sparse) tensor cores. Stride 1, zero padding 1.
 * Readings: X is NHWC (Nb, H, W, Cin), 16-byte aligned; the filter is
 * (Cout, 3, 3, Cin) flattened to Cout x 9 Cin with column (r 3 + s) Cin + c, so its
 * 2:4 form is sp24_prune_compress of that matrix (K = 9 Cin); Y is Cout x (Nb H W),
 * Y[co, (n H + h) W + w] = alpha sum_{r,s,c} W[co, r, s, c] X[n, h + r - 1, w + s - 1, c]
 * (zero outside the image), pitch ldy >= Nb H W, fp32 accumulation, one RNE
 * conversion to out_dt (fp16 / bf16). Cin % 64 == 0 and W <= 224, else
 * SSDNN_ERR_UNSUPPORTED; 16-bit data only. */
int sp24_conv3x3(int dt, int out_dt, int64_t Cout, int64_t Cin, int64_t Nb, int64_t H, int64_t W, const void* values,
                 const uint8_t* meta_hw, const void* X, void* Y, int64_t ldy, float alpha, void* stream);
/* The same with a dense filter Wf (Cout x 9 Cin, pitch ldw): the same-family baseline. */
int dense_conv3x3(int dt, int out_dt, int64_t Cout, int64_t Cin, int64_t Nb, int64_t H, int64_t W, const void* Wf,
                  int64_t ldw, const void* X, void* Y, int64_t ldy, float alpha, void* stream);

/* The 3x3 convolution with a tile-wise (TW) filter ("Accelerating Sparse DNNs Based
 * on Tiled GEMM", Abstract: whole K-rows pruned per output tile of the GEMM, the
 * skip made where operands are fetched from global memory; "SparseRT", Abstract:
 * sparse 3x3 convolutions). Reading: the implicit GEMM fetches its activation
 * operand in units of one filter tap x 64 input channels (one TMA box of NHWC
 * data), so a 128-channel output tile keeps whole K-row groups of one tap and 64
 * channels; a finer group would need 2-byte strided gathers of NHWC activations.
 * Group g of the flattened filter (Cout x 9 Cin, column (r 3 + s) Cin + c) covers
 * columns 64 g .. 64 g + 63, i.e. tap g / (Cin / 64) and channels
 * 64 (g % (Cin / 64)) ..; its score is the fp32 sum of its 64 columns' TW scores.
 * The compressed filter is exactly bw_prune_compress of the flattened filter with
 * keep_blocks_host = keep_groups_host (kept groups per 128-channel tile); this call
 * takes that form (the same offsets, indices, schedule and packed operand).
 * Y as for sp24_conv3x3; a tile that keeps no group writes zeros. Cin % 64 == 0 and
 * W <= 224, else SSDNN_ERR_UNSUPPORTED; fp16 / bf16 only. */
int tw_conv3x3(int dt, int out_dt, int64_t Cout, int64_t Cin, int64_t Nb, int64_t H, int64_t W,
               const int32_t* keep_groups_host, const int32_t* offsets, const int32_t* indices, const int32_t* schedule,
               const void* packed, const void* X, void* Y, int64_t ldy, float alpha, void* stream);

/* --------------------------------------------------- fused layer epilogue ----
 * A pruned fully connected layer or 1x1 convolution runs as one of the GEMMs
 * above ("Accelerating Sparse DNNs Based on Tiled GEMM", Abstract), and the step
 * that follows it -- bias, activation, quantisation of the layer output -- is
 * fused into the GEMM's epilogue ("kernel fusion", same page, TL;DR). Per output
 * element, in fp32 and in this order:
 *     z = alpha * acc + bias[row]       (one fma; without a bias: alpha * acc)
 *     a = act(z)                        none | ReLU max(z, 0) | GELU 0.5 z (1 + erf(z / sqrt 2))
 *     Y = round_out(y_scale * a)        ties to even; e4m3 saturates to +-448
 * acc is the fp32 tensor-core accumulator; row indexes the output features (rows
 * of W and of Y). For e4m3 output, y_scale is the reciprocal of the output
 * tensor's quantisation scale. With K == 0 (or no kept column at all) acc = 0. */
typedef enum { SSDNN_ACT_NONE = 0, SSDNN_ACT_RELU = 1, SSDNN_ACT_GELU = 2 } ssdnn_act;

typedef struct ssdnn_epilogue {
  const float* bias; /* device, M floats (one per output row), 4-byte aligned; NULL = no bias */
  int act;           /* ssdnn_act */
  float y_scale;     /* finite multiplier after the activation (1.0f = none) */
} ssdnn_epilogue;

/* sp24_gemm / dense_gemm / tvw_gemm / bw_gemm with the fused epilogue `ep` (NULL = the
 * plain conversion). out_dt may also be SSDNN_E4M3 here (ldy * out bytes a
 * multiple of 16). Returns SSDNN_ERR_INVALID_ARG for an unknown activation or a
 * non-finite y_scale, SSDNN_ERR_UNSUPPORTED for a misaligned bias; otherwise as
 * the plain call. tvw_gemm_ep adds the output type and alpha that tvw_gemm
 * fixes to dt and 1. */
int sp24_gemm_ep(int in_dt, int out_dt, int64_t M, int64_t N, int64_t K, const void* values,
                 const uint8_t* meta_hw, const void* X, int64_t ldx, void* Y, int64_t ldy, float alpha,
                 const ssdnn_epilogue* ep, void* stream);
int dense_gemm_ep(int in_dt, int out_dt, int64_t M, int64_t N, int64_t K, const void* W, int64_t ldw,
                  const void* X, int64_t ldx, void* Y, int64_t ldy, float alpha, const ssdnn_epilogue* ep,
                  void* stream);
int tvw_gemm_ep(int dt, int out_dt, int tvw, int64_t M, int64_t N, int64_t K, const int32_t* keep_counts_host,
                const int32_t* offsets, const int32_t* indices, const int32_t* schedule, const void* packed,
                const uint8_t* meta_hw, const void* X, int64_t ldx, void* Y, int64_t ldy, float alpha,
                const ssdnn_epilogue* ep, void* stream);
int bw_gemm_ep(int dt, int out_dt, int64_t M, int64_t N, int64_t K, const int32_t* keep_blocks_host,
               const int32_t* offsets, const int32_t* indices, const int32_t* schedule, const void* packed,
               const void* X, int64_t ldx, void* Y, int64_t ldy, float alpha, const ssdnn_epilogue* ep,
               void* stream);

/* ------------------------------------------------------ tile variants ----
 * sp24_gemm_ep / dense_gemm_ep with an explicit tile variant instead of the one
 * the library picks from the shape (for tuning and for tests that must run
 * every variant; the results are identical up to fp32 summation order):
 *   0      chosen by shape (the plain calls)
 *   1064   128 x 64 tiles, one CTA (fp16/bf16 only)
 *   1128   128 x 128 tiles, one CTA
 *   1256   128 x 256 tiles, one CTA
 *   2192   256 x 192 tiles, one CTA with two M = 128 instructions (2:4 only)
 *   2256   256 x 256 tiles, one CTA with two M = 128 instructions (dense only)
 *   9256   256 x 256 tiles on an SM pair (cta_group::2), one 128-byte K step per stage
 *   19256  the same with two K steps per stage (2:4 only)
 *   11064, 11128  1064 / 1128 with two 128-byte K steps of the compressed weight per
 *          stage (2:4 only; 11064 fp16/bf16 only)
 * (For 2:4, 1064 and 1128 run one K step per stage; the plain calls pick two.)
 * Any other value, or one the operand type does not have: SSDNN_ERR_UNSUPPORTED,
 * before any work is enqueued. The pages have no counterpart: this selects among
 * implementations of the same product. */
int sp24_gemm_variant(int in_dt, int out_dt, int64_t M, int64_t N, int64_t K, const void* values,
                      const uint8_t* meta_hw, const void* X, int64_t ldx, void* Y, int64_t ldy, float alpha,
                      const ssdnn_epilogue* ep, int variant, void* stream);
int dense_gemm_variant(int in_dt, int out_dt, int64_t M, int64_t N, int64_t K, const void* W, int64_t ldw,
                       const void* X, int64_t ldx, void* Y, int64_t ldy, float alpha, const ssdnn_epilogue* ep,
                       int variant, void* stream);

/* ------------------------------------------------- allocation-free variant ----
 * tw_prune_compress_noalloc: tw_prune_compress for callers that cannot allocate
 * device memory. (The pages have no counterpart: this is a deployment aid.)
 * Who needs it: a plugin running inside an inference engine that owns all device
 * memory and hands it only the buffers of its inputs and outputs, or a serving
 * loop that must never call cudaMalloc/cudaFree, which synchronise the device
 * and can fail under memory pressure. Such callers cannot provide the score
 * workspace tw_prune_compress needs.
 * What it does instead: the per-tile scores go to a fixed array in device memory
 * that the library defines (SSDNN_NOALLOC_MAX_SCORES floats = 8 MiB); every GPU
 * that loads the library holds that array until the process exits. The offsets
 * and schedule tables are computed on the device, so no host-to-device copy is
 * made either. The call allocates nothing and calls no allocating routine.
 * Limits: nt = ceil(M/128) <= SSDNN_NOALLOC_MAX_TILES and nt * K <=
 * SSDNN_NOALLOC_MAX_SCORES; beyond them it returns SSDNN_ERR_UNSUPPORTED and does
 * nothing.
 * Set-up: every call looks up the device address of that array with the
 * device current (a lookup that allocates nothing). The first call on a device
 * may also be the first use of the library's kernels there, and with lazy
 * module loading (CUDA_MODULE_LOADING=LAZY, the default) the CUDA runtime then
 * loads the module, which takes device memory once. Callers that may not
 * allocate at all should make one call during their set-up, before any stream
 * capture; later calls allocate nothing. A device reset invalidates nothing the
 * library keeps: the address is looked up again on the next call.
 * Sharing: all calls on a device share the one array, which keeps the last call's
 * scores (every call overwrites the part it reads, so nothing needs clearing).
 * Calls whose work overlaps on the GPU (different streams without ordering) race
 * on it and must be serialised by the caller.
 * Arguments, layouts and results are those of tw_prune_compress (bit-identical
 * outputs), without the workspace. */
#define SSDNN_NOALLOC_MAX_SCORES (1 << 21)
#define SSDNN_NOALLOC_MAX_TILES 2048
int tw_prune_compress_noalloc(int dt, int tvw, const void* W, int64_t M, int64_t K, int64_t ldw,
                              const int32_t* keep_counts_host, int32_t* offsets, int32_t* indices,
                              int32_t* schedule, void* packed, uint8_t* meta, uint8_t* meta_hw, void* stream);

#ifdef __cplusplus
}
#endif
#endif /* SSDNN_H */
