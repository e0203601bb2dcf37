// Tensor-core issue-rate microbenchmark: dense and 2:4-sparse tcgen05.mma with
// operands resident in shared memory and the accumulator (and the sparse
// metadata) in TMEM, so that no global-memory traffic is involved.
//
// It measures the ceiling the GEMM kernels run against. The 2:4 sparse tensor
// core is stated to do twice the math of the dense one ("Accelerating Sparse Deep
// Neural Networks", Abstract; "NVIDIA A100 benchmarks" page, 2:4 paragraph); this
// kernel checks that claim on the device at hand, for the instruction shapes the
// GEMM uses (M = 128 rows, N = 128 / 192 / 256 columns, one stage of K per step).
//
// One CTA per SM. Its first thread issues `iters` steps of MMAS instructions into
// one accumulator (the same operands every step), commits, and waits (bounded)
// for completion. The host times the launch; a step is 2 * 128 * N * BK flops
// of dense-equivalent work (BK = 128 bytes of K).
#include <cuda_runtime.h>

#include "../../include/ssdnn.h"
#include "common.cuh"
#include "kernels.h"

namespace ssdnn {
namespace {

constexpr int kSmemRequest = 160 * 1024;  // forces one CTA per SM

template <int DT, bool SPARSE, int N, int BROW>
struct RateCfg {
  static constexpr int EB = Elem<DT>::bytes;
  static constexpr int BK = 128 / EB;
  static constexpr int A_BYTES = SPARSE ? 128 * 64 : 128 * 128;
  static constexpr int B_BOX_COLS = BROW / EB;
  static constexpr int B_BOXES = N / B_BOX_COLS;
  static constexpr int B_BOX_BYTES = BK * BROW;
  static constexpr int B_BYTES = B_BOXES * B_BOX_BYTES;
  static constexpr uint32_t B_SWZ = BROW == 128 ? 2u : 4u;
  static constexpr int MMA_K = (SPARSE ? 64 : 32) / EB;
  static constexpr int MMAS = BK / MMA_K;
  static constexpr uint32_t IDESC = ptx::idesc(Elem<DT>::mma_fmt, Elem<DT>::mma_fmt, SPARSE, 128, N, false, true);
  static constexpr int USED = 1024 + A_BYTES + B_BYTES + 2048 + 64;
  static_assert(B_BOXES * B_BOX_COLS == N, "N must be a multiple of the B box width");
  static_assert(USED <= kSmemRequest, "operands exceed the shared-memory request");
};

// Finite operand bits of moderate magnitude (|x| in [1, 2)), random signs.
template <int DT>
__device__ __forceinline__ uint32_t operand_word(uint32_t i) {
  uint32_t h = i * 0x9E3779B9u;
  h ^= h >> 15;
  h *= 0x85EBCA6Bu;
  h ^= h >> 13;
  if constexpr (DT == 0) return (h & 0x83FF83FFu) | 0x3C003C00u;   // fp16 pairs
  if constexpr (DT == 1) return (h & 0x807F807Fu) | 0x3F803F80u;   // bf16 pairs
  return (h & 0x87878787u) | 0x38383838u;                          // e4m3 quads
}

template <int DT, bool SPARSE, int N, int BROW>
__global__ void __launch_bounds__(128, 1) k_mma_rate(int iters, uint32_t* err) {
  using C = RateCfg<DT, SPARSE, N, BROW>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = ptx::smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);
  uint8_t* sA = smem;
  uint8_t* sB = sA + C::A_BYTES;
  uint8_t* sM = sB + C::B_BYTES;
  uint64_t* bar = reinterpret_cast<uint64_t*>(sM + 2048);
  uint32_t* slot = reinterpret_cast<uint32_t*>(bar + 1);
  const uint32_t warp = threadIdx.x >> 5;

  uint32_t* ops = reinterpret_cast<uint32_t*>(sA);
  for (int i = threadIdx.x; i < (C::A_BYTES + C::B_BYTES) / 4; i += blockDim.x)
    ops[i] = operand_word<DT>(static_cast<uint32_t>(i) + 7919u * blockIdx.x);
  // metadata: every group keeps positions (0, 1), a valid 2:4 selection
  uint32_t* meta = reinterpret_cast<uint32_t*>(sM);
  for (int i = threadIdx.x; i < 2048 / 4; i += blockDim.x) meta[i] = 0x44444444u;
  ptx::fence_proxy_async_smem();
  if (threadIdx.x == 0) {
    ptx::mbar_init(bar, 1);
    ptx::fence_mbar_init();
  }
  if (warp == 0) {
    ptx::tmem_alloc(slot, 512);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *slot;

  if (threadIdx.x == 0) {
    const uint32_t a = ptx::smem_u32(sA), b = ptx::smem_u32(sB);
    const uint32_t meta_col = tmem + 256u;
    if constexpr (SPARSE) ptx::tmem_cp_128x128b(meta_col, ptx::sdesc(ptx::smem_u32(sM), 128, 128, 0));
    for (int it = 0; it < iters; ++it) {
#pragma unroll
      for (int j = 0; j < C::MMAS; ++j) {
        const uint32_t accum = (it > 0 || j > 0) ? 1u : 0u;
        const uint64_t bdesc = ptx::sdesc(b + j * C::MMA_K * BROW, C::B_BOX_BYTES, 8 * BROW, C::B_SWZ);
        if constexpr (SPARSE) {
          const uint64_t adesc = ptx::sdesc(a + j * 32, 16, 512, 4);
          if constexpr (Elem<DT>::f8)
            ptx::mma_sp_f8(tmem, adesc, bdesc, meta_col + 2u * j, C::IDESC, accum);
          else
            ptx::mma_sp_f16(tmem, adesc, bdesc, meta_col + 2u * j, C::IDESC, accum);
        } else {
          const uint64_t adesc = ptx::sdesc(a + j * 32, 16, 1024, 2);
          if constexpr (Elem<DT>::f8)
            ptx::mma_f8(tmem, adesc, bdesc, C::IDESC, accum);
          else
            ptx::mma_f16(tmem, adesc, bdesc, C::IDESC, accum);
        }
      }
    }
    ptx::mma_commit(bar);
    wait_bounded(bar, 0, err);
  }
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, 512);
  }
}

template <int DT, bool SPARSE, int N, int BROW>
cudaError_t launch_rate(int iters, cudaStream_t s, uint32_t* err) {
  auto kern = k_mma_rate<DT, SPARSE, N, BROW>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemRequest);
  if (e != cudaSuccess) return e;
  int dev = 0, sms = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
  kern<<<sms, 128, kSmemRequest, s>>>(iters, err);
  return cudaGetLastError();
}

template <int DT, bool SPARSE>
cudaError_t launch_rate_n(int n, int iters, cudaStream_t s, uint32_t* err) {
  constexpr int EB = Elem<DT>::bytes;
  switch (n) {
    case 128: return launch_rate<DT, SPARSE, 128, 128>(iters, s, err);
    case 256: return launch_rate<DT, SPARSE, 256, 128>(iters, s, err);
    case 192:
      if constexpr (EB == 2)
        return launch_rate<DT, SPARSE, 192, 128>(iters, s, err);
      else
        return launch_rate<DT, SPARSE, 192, 64>(iters, s, err);
  }
  return cudaErrorInvalidValue;
}

// The same on SM pairs (cta_group::2), the form the large GEMMs run: clusters of two
// CTAs, the even CTA's first thread issuing M = 256, N = 256 instructions whose A
// rows and B columns are split between the two CTAs' shared memory (each CTA: 128
// rows of A, 128 columns of B). For the 2:4 form every step first copies its
// metadata block into one of four TMEM slots, as the GEMM's MMA issuer does. A
// step is 2 * 256 * 256 * (128 / elem bytes) dense-equivalent flops per pair.
template <int DT, bool SPARSE>
__global__ void __launch_bounds__(128, 1) k_mma_rate_pair(int iters, uint32_t* err) {
  using C = RateCfg<DT, SPARSE, 128, 128>;  // this CTA's share: 128 B columns, 128-byte B rows
  constexpr uint32_t IDESC = ptx::idesc(Elem<DT>::mma_fmt, Elem<DT>::mma_fmt, SPARSE, 256, 256, false, true);
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = ptx::smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);
  uint8_t* sA = smem;
  uint8_t* sB = sA + C::A_BYTES;
  uint8_t* sM = sB + C::B_BYTES;
  uint64_t* bar = reinterpret_cast<uint64_t*>(sM + 2048);
  uint32_t* slot = reinterpret_cast<uint32_t*>(bar + 1);
  const uint32_t warp = threadIdx.x >> 5;
  const bool leader = (ptx::cluster_ctarank() & 1u) == 0u;

  uint32_t* ops = reinterpret_cast<uint32_t*>(sA);
  for (int i = threadIdx.x; i < (C::A_BYTES + C::B_BYTES) / 4; i += blockDim.x)
    ops[i] = operand_word<DT>(static_cast<uint32_t>(i) + 7919u * blockIdx.x);
  uint32_t* meta = reinterpret_cast<uint32_t*>(sM);
  for (int i = threadIdx.x; i < 2048 / 4; i += blockDim.x) meta[i] = 0x44444444u;
  ptx::fence_proxy_async_smem();
  if (threadIdx.x == 0) {
    ptx::mbar_init(bar, 1);
    ptx::fence_mbar_init();
  }
  if (warp == 0) {
    ptx::tmem_alloc_pair(slot, 512);
    ptx::tmem_relinquish_pair();
  }
  ptx::tc_fence_before();
  ptx::cluster_sync();  // both CTAs' operands and barriers are ready
  ptx::tc_fence_after();
  const uint32_t tmem = *slot;

  if (threadIdx.x == 0 && leader) {
    const uint32_t a = ptx::smem_u32(sA), b = ptx::smem_u32(sB);
    const uint64_t mdesc = ptx::sdesc(ptx::smem_u32(sM), 128, 128, 0);
    for (int it = 0; it < iters; ++it) {
      const uint32_t meta_col = tmem + 256u + 4u * static_cast<uint32_t>(it & 3);
      if constexpr (SPARSE) ptx::tmem_cp_128x128b_pair(meta_col, mdesc);
#pragma unroll
      for (int j = 0; j < C::MMAS; ++j) {
        const uint32_t accum = (it > 0 || j > 0) ? 1u : 0u;
        const uint64_t bdesc = ptx::sdesc(b + j * C::MMA_K * 128, C::B_BOX_BYTES, 8 * 128, 2);
        if constexpr (SPARSE) {
          const uint64_t adesc = ptx::sdesc(a + j * 32, 16, 512, 4);
          if constexpr (Elem<DT>::f8)
            ptx::mma_sp_f8_pair(tmem, adesc, bdesc, meta_col + 2u * j, IDESC, accum);
          else
            ptx::mma_sp_f16_pair(tmem, adesc, bdesc, meta_col + 2u * j, IDESC, accum);
        } else {
          const uint64_t adesc = ptx::sdesc(a + j * 32, 16, 1024, 2);
          if constexpr (Elem<DT>::f8)
            ptx::mma_f8_pair(tmem, adesc, bdesc, IDESC, accum);
          else
            ptx::mma_f16_pair(tmem, adesc, bdesc, IDESC, accum);
        }
      }
    }
    ptx::mma_commit_pair_multicast(bar, 3);  // both CTAs learn that the MMAs are done
  }
  if (threadIdx.x == 0) wait_bounded(bar, 0, err);
  ptx::tc_fence_before();
  ptx::cluster_sync();
  if (warp == 0) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc_pair(tmem, 512);
  }
  ptx::cluster_sync();  // no CTA leaves while its peer may still address it
}

template <int DT, bool SPARSE>
cudaError_t launch_rate_pair(int iters, cudaStream_t s, uint32_t* err) {
  auto kern = k_mma_rate_pair<DT, SPARSE>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemRequest);
  if (e != cudaSuccess) return e;
  int dev = 0, sms = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
  cudaLaunchConfig_t cfg{};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cfg.gridDim = dim3(static_cast<unsigned>(sms & ~1), 1, 1);
  cfg.blockDim = dim3(128, 1, 1);
  cfg.dynamicSmemBytes = kSmemRequest;
  cfg.stream = s;
  return cudaLaunchKernelEx(&cfg, kern, iters, err);
}

}  // namespace

cudaError_t launch_mma_rate_pair(int dt, int sparse, int iters, cudaStream_t s, uint32_t* err) {
  switch (dt) {
    case SSDNN_F16:
      return sparse ? launch_rate_pair<0, true>(iters, s, err) : launch_rate_pair<0, false>(iters, s, err);
    case SSDNN_BF16:
      return sparse ? launch_rate_pair<1, true>(iters, s, err) : launch_rate_pair<1, false>(iters, s, err);
    case SSDNN_E4M3:
      return sparse ? launch_rate_pair<2, true>(iters, s, err) : launch_rate_pair<2, false>(iters, s, err);
  }
  return cudaErrorInvalidValue;
}

cudaError_t launch_mma_rate(int dt, int sparse, int n, int iters, cudaStream_t s, uint32_t* err) {
  switch (dt) {
    case SSDNN_F16:
      return sparse ? launch_rate_n<0, true>(n, iters, s, err) : launch_rate_n<0, false>(n, iters, s, err);
    case SSDNN_BF16:
      return sparse ? launch_rate_n<1, true>(n, iters, s, err) : launch_rate_n<1, false>(n, iters, s, err);
    case SSDNN_E4M3:
      return sparse ? launch_rate_n<2, true>(n, iters, s, err) : launch_rate_n<2, false>(n, iters, s, err);
  }
  return cudaErrorInvalidValue;
}

}  // namespace ssdnn
