// tw_prune_compress_noalloc: the tile-wise prune for callers that cannot
// allocate device memory.
//
// The ordinary entry point takes its score scratch from the caller and uploads
// its small host tables with a copy from pageable memory. This variant needs
// neither: the scores live in a file-scope device array of fixed size, and the
// offsets and schedule tables are computed on the device from the kept counts,
// which travel as a kernel parameter. Everything else runs the same kernels.
#include <cuda_runtime.h>

#include "../../include/ssdnn.h"
#include "common.cuh"
#include "kernels.h"

namespace ssdnn {
namespace {

// Score scratch shared by every call on a device (kept for the life of the process).
constexpr int64_t kScratchFloats = SSDNN_NOALLOC_MAX_SCORES;
static __device__ __align__(256) float g_noalloc_scores[kScratchFloats];

constexpr int kMaxTiles = SSDNN_NOALLOC_MAX_TILES;
struct KeepCounts {
  int32_t L[kMaxTiles];
};

// Device address of the scratch for the current device. The host-side symbol is
// only a stand-in, so the address is looked up with that device current, on
// every call: the lookup allocates nothing, and an address cached across calls
// would go stale if the device were reset and the module loaded again.
cudaError_t scratch_address(float** out) {
  void* p = nullptr;
  const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scores);
  if (e != cudaSuccess) return e;
  *out = static_cast<float*>(p);
  return cudaSuccess;
}

// offsets[t] = sum_{s<t} L_s; schedule = (t, L_t, P_t, P_t / 64) in the order
// L_t descending, ties by t ascending (the rank of t counts the tiles before it).
__global__ void __launch_bounds__(1024) k_tw_tables(const KeepCounts keep, int nt, int32_t* __restrict__ offsets,
                                                    int32_t* __restrict__ schedule) {
  __shared__ int32_t s_P[kMaxTiles];
  if (threadIdx.x == 0) {
    int32_t o = 0, p = 0;
    for (int t = 0; t < nt; ++t) {
      offsets[t] = o;
      s_P[t] = p;
      o += keep.L[t];
      p += (keep.L[t] + 63) / 64 * 64;
    }
    offsets[nt] = o;
  }
  __syncthreads();
  for (int t = threadIdx.x; t < nt; t += blockDim.x) {
    const int32_t L = keep.L[t];
    int rank = 0;
    for (int s = 0; s < nt; ++s) {
      const int32_t Ls = keep.L[s];
      rank += (Ls > L || (Ls == L && s < t)) ? 1 : 0;
    }
    schedule[4 * rank + 0] = t;
    schedule[4 * rank + 1] = L;
    schedule[4 * rank + 2] = s_P[t];
    schedule[4 * rank + 3] = s_P[t] / 64;
  }
}

}  // namespace
}  // namespace ssdnn

using namespace ssdnn;

extern "C" int tw_prune_compress_noalloc(int dt, int tvw, const void* W, int64_t M, int64_t K, int64_t ldw,
                                         const int32_t* keep_counts_host, int32_t* offsets, int32_t* indices,
                                         int32_t* schedule, void* packed, uint8_t* meta, uint8_t* meta_hw,
                                         void* stream) {
  constexpr int64_t kMaxDim = (int64_t(1) << 31) - 1;
  if ((dt != SSDNN_F16 && dt != SSDNN_BF16) || M < 0 || K < 0 || M > kMaxDim || K > kMaxDim)
    return dt == SSDNN_E4M3 ? SSDNN_ERR_UNSUPPORTED : SSDNN_ERR_INVALID_ARG;
  if (M == 0) return SSDNN_OK;
  if (!keep_counts_host || !offsets || !schedule) return SSDNN_ERR_INVALID_ARG;
  const int64_t nt = ceil_div(M, 128);
  if (nt > kMaxTiles || nt * K > kScratchFloats) return SSDNN_ERR_UNSUPPORTED;  // beyond the fixed scratch
  TwTables tabs{};
  tabs.nt = nt;
  int64_t L_total = 0;
  KeepCounts kc{};
  for (int64_t t = 0; t < nt; ++t) {
    const int64_t L = keep_counts_host[t];
    if (L < 0 || L > K) return SSDNN_ERR_INVALID_ARG;
    if (tvw && (L % 4)) return SSDNN_ERR_UNSUPPORTED;
    const int64_t R = round_up(L, 64);
    tabs.P_total += R;
    tabs.Q_total += R / 64;
    tabs.max_R = R > tabs.max_R ? R : tabs.max_R;
    L_total += L;
    if (L_total > kMaxDim || 128 * tabs.P_total > kMaxDim) return SSDNN_ERR_UNSUPPORTED;
    kc.L[t] = static_cast<int32_t>(L);
  }
  if (K > 0 && (!W || ldw < K)) return SSDNN_ERR_INVALID_ARG;
  if (L_total > 0 && !indices) return SSDNN_ERR_INVALID_ARG;
  if (tabs.P_total > 0 && (!packed || (tvw && (!meta || !meta_hw)))) return SSDNN_ERR_INVALID_ARG;
  auto aligned16 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
  if ((W && (reinterpret_cast<uintptr_t>(W) & 1u)) || (packed && !aligned16(packed)) ||
      (meta && !aligned16(meta)) || (meta_hw && !aligned16(meta_hw)) ||
      (reinterpret_cast<uintptr_t>(offsets) & 3u) || (reinterpret_cast<uintptr_t>(schedule) & 3u) ||
      (indices && (reinterpret_cast<uintptr_t>(indices) & 3u)))
    return SSDNN_ERR_UNSUPPORTED;
  float* scores = nullptr;
  if (scratch_address(&scores) != cudaSuccess) return SSDNN_ERR_CUDA;
  auto s = static_cast<cudaStream_t>(stream);
  k_tw_tables<<<1, 1024, 0, s>>>(kc, static_cast<int>(nt), offsets, schedule);
  if (cudaGetLastError() != cudaSuccess) return SSDNN_ERR_CUDA;
  const cudaError_t e = launch_tw_prune(dt, tvw, W, M, K, ldw, tabs, offsets, indices, schedule, packed, meta,
                                        meta_hw, scores, s, nullptr);
  return e == cudaSuccess ? SSDNN_OK : SSDNN_ERR_CUDA;
}
