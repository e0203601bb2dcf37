// The C ABI: argument validation, host-side tables, and dispatch to the kernels.
// Every entry point returns an ssdnn_status and never throws.
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <atomic>
#include <cstring>
#include <mutex>
#include <vector>

#include "../../include/ssdnn.h"
#include "common.cuh"
#include "kernels.h"

namespace ssdnn {
namespace {

// Per-device error word written by kernels whose bounded waits expire.
__device__ uint32_t g_error_word;

constexpr int kMaxDevices = 64;
std::mutex g_err_mu;
uint32_t* g_err_ptr[kMaxDevices] = {};

uint32_t* error_word() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lk(g_err_mu);
  if (!g_err_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_error_word) != cudaSuccess) return nullptr;
    g_err_ptr[dev] = static_cast<uint32_t*>(p);
  }
  return g_err_ptr[dev];
}

// One thread waits on an mbarrier that nothing ever arrives on, with the given
// limit: the wait must give up, record a timeout in the error word and return.
__global__ void k_selftest_timeout(uint32_t* err, uint64_t limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x != 0) return;
  ptx::mbar_init(&bar, 1);
  ptx::fence_mbar_init();
  wait_bounded(&bar, 0, err, limit_ns);
}

// Ordering events for the host-buffer GEMM: a small per-device pool, created on
// first use and reused (re-recording an event is safe once waits have been
// enqueued against its previous record). Index -1 is the completion event.
constexpr int kCopyEvents = 64;
cudaEvent_t g_events[kMaxDevices][kCopyEvents + 1] = {};

cudaEvent_t copy_event(int64_t i) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  const int slot = i < 0 ? kCopyEvents : static_cast<int>(i % kCopyEvents);
  std::lock_guard<std::mutex> lk(g_err_mu);
  cudaEvent_t& e = g_events[dev][slot];
  if (!e && cudaEventCreateWithFlags(&e, cudaEventDisableTiming) != cudaSuccess) e = nullptr;
  return e;
}

int elem_bytes(int dt) { return dt == SSDNN_E4M3 ? 1 : 2; }
bool valid_dt(int dt) { return dt == SSDNN_F16 || dt == SSDNN_BF16 || dt == SSDNN_E4M3; }
bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
constexpr int64_t kMaxDim = (int64_t(1) << 31) - 1;

int from_cuda(cudaError_t e) {
  if (e == cudaSuccess) return SSDNN_OK;
  return e == cudaErrorInvalidValue ? SSDNN_ERR_INVALID_ARG : SSDNN_ERR_CUDA;
}

int out_bytes(int out_dt) { return out_dt == SSDNN_E4M3 ? 1 : 2; }

// Zero the M x N output (K == 0 or no kept columns anywhere).
int zero_output(void* Y, int64_t ldy, int64_t M, int64_t N, int ob, cudaStream_t s) {
  if (M == 0 || N == 0) return SSDNN_OK;
  return from_cuda(cudaMemset2DAsync(Y, static_cast<size_t>(ldy * ob), 0, static_cast<size_t>(N * ob),
                                     static_cast<size_t>(M), s));
}

// Output checks shared by the GEMMs; e4m3 output only through the epilogue entry points.
int check_gemm_io(int out_dt, bool f8_out_ok, int64_t M, int64_t N, int64_t K, const void* X, int64_t ldx, int eb,
                  void* Y, int64_t ldy) {
  if (out_dt != SSDNN_F16 && out_dt != SSDNN_BF16 && !(f8_out_ok && out_dt == SSDNN_E4M3))
    return SSDNN_ERR_UNSUPPORTED;
  if (M < 0 || N < 0 || K < 0 || M > kMaxDim || N > kMaxDim || K > kMaxDim) return SSDNN_ERR_INVALID_ARG;
  if (M == 0 || N == 0) return SSDNN_OK;
  if (!Y || (K > 0 && !X)) return SSDNN_ERR_INVALID_ARG;
  if (ldy < N || (K > 0 && ldx < N)) return SSDNN_ERR_INVALID_ARG;
  if (!aligned16(Y) || (ldy * out_bytes(out_dt)) % 16) return SSDNN_ERR_UNSUPPORTED;
  if (K > 0 && (!aligned16(X) || (ldx * eb) % 16)) return SSDNN_ERR_UNSUPPORTED;
  return SSDNN_OK;
}

int check_epilogue(const ssdnn_epilogue* ep) {
  if (!ep) return SSDNN_OK;
  if (ep->act < SSDNN_ACT_NONE || ep->act > SSDNN_ACT_GELU || !std::isfinite(ep->y_scale))
    return SSDNN_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(ep->bias) & 3u) return SSDNN_ERR_UNSUPPORTED;
  return SSDNN_OK;
}

void set_epilogue(GemmArgs& a, const ssdnn_epilogue* ep) {
  if (!ep) return;
  a.bias = ep->bias;
  a.act = ep->act;
  a.y_scale = ep->y_scale;
}

// A product with no terms: Y = round(y_scale * act(bias[row])), zeros without a bias
// (every activation maps 0 to 0).
int empty_product(void* Y, int64_t ldy, int64_t M, int64_t N, int out_dt, const ssdnn_epilogue* ep,
                  cudaStream_t s) {
  if (ep && ep->bias)
    return from_cuda(launch_fill_epilogue(Y, ldy, M, N, out_dt, ep->bias, ep->act, ep->y_scale, s));
  return zero_output(Y, ldy, M, N, out_bytes(out_dt), s);
}

struct Tables {
  TwTables t;
  std::vector<int32_t> offsets, schedule;
  int64_t L_total = 0;
};

int build_tables(int tvw, int64_t M, int64_t K, const int32_t* keep, Tables* out) {
  const int64_t nt = ceil_div(M, 128);
  out->t.nt = nt;
  out->offsets.assign(static_cast<size_t>(nt + 1), 0);
  std::vector<int64_t> P(static_cast<size_t>(nt), 0), Q(static_cast<size_t>(nt), 0);
  int64_t p = 0, q = 0, o = 0, maxR = 0;
  for (int64_t t = 0; t < nt; ++t) {
    const int64_t L = keep[t];
    if (L < 0 || L > K) return SSDNN_ERR_INVALID_ARG;
    if (tvw && (L % 4)) return SSDNN_ERR_UNSUPPORTED;
    const int64_t R = round_up(L, 64);
    P[static_cast<size_t>(t)] = p;
    Q[static_cast<size_t>(t)] = p / 64;  // first 2048-byte metadata block of the tile
    p += R;
    q += R / 64;
    o += L;
    maxR = std::max(maxR, R);
    if (o > kMaxDim || 128 * p > kMaxDim) return SSDNN_ERR_UNSUPPORTED;
    out->offsets[static_cast<size_t>(t + 1)] = static_cast<int32_t>(o);
  }
  out->t.P_total = p;
  out->t.Q_total = q;
  out->t.max_R = maxR;
  out->L_total = o;
  std::vector<int32_t> order(static_cast<size_t>(nt));
  for (int64_t t = 0; t < nt; ++t) order[static_cast<size_t>(t)] = static_cast<int32_t>(t);
  std::stable_sort(order.begin(), order.end(), [&](int32_t a, int32_t b) { return keep[a] > keep[b]; });
  out->schedule.resize(static_cast<size_t>(4 * nt));
  for (int64_t e = 0; e < nt; ++e) {
    const int32_t t = order[static_cast<size_t>(e)];
    out->schedule[static_cast<size_t>(4 * e + 0)] = t;
    out->schedule[static_cast<size_t>(4 * e + 1)] = keep[t];
    out->schedule[static_cast<size_t>(4 * e + 2)] = static_cast<int32_t>(P[static_cast<size_t>(t)]);
    out->schedule[static_cast<size_t>(4 * e + 3)] = static_cast<int32_t>(Q[static_cast<size_t>(t)]);
  }
  return SSDNN_OK;
}

// Block-wise tables: per-tile kept block counts -> the tile-wise tables of the kept
// columns (L_t = 64 B_t) plus the block offsets, and the workspace layout.
struct BwTables {
  Tables cols;                      // tile-wise tables of the kept columns
  std::vector<int32_t> blk_offsets;  // nt + 1, in blocks
  int64_t n_blocks = 0;
  size_t ws_scores = 0, ws_bscores = 0, ws_coloff = 0, ws_colidx = 0, ws_bytes = 0;  // byte offsets
};

int build_bw_tables(int64_t M, int64_t K, const int32_t* keep_blocks, BwTables* out) {
  if (K % 64) return SSDNN_ERR_UNSUPPORTED;
  const int64_t nt = ceil_div(M, 128), KB = K / 64;
  std::vector<int32_t> keep_cols(static_cast<size_t>(nt));
  out->blk_offsets.assign(static_cast<size_t>(nt + 1), 0);
  int64_t nb = 0;
  for (int64_t t = 0; t < nt; ++t) {
    const int64_t b = keep_blocks[t];
    if (b < 0 || b > KB) return SSDNN_ERR_INVALID_ARG;
    keep_cols[static_cast<size_t>(t)] = static_cast<int32_t>(64 * b);
    nb += b;
    out->blk_offsets[static_cast<size_t>(t + 1)] = static_cast<int32_t>(nb);
  }
  out->n_blocks = nb;
  const int st = build_tables(0, M, K, keep_cols.data(), &out->cols);
  if (st != SSDNN_OK) return st;
  auto up = [](size_t x) { return (x + 255) / 256 * 256; };
  out->ws_scores = 0;
  out->ws_bscores = up(static_cast<size_t>(nt * K) * 4);
  out->ws_coloff = out->ws_bscores + up(static_cast<size_t>(nt * KB) * 4);
  out->ws_colidx = out->ws_coloff + up(static_cast<size_t>(nt + 1) * 4);
  out->ws_bytes = out->ws_colidx + up(static_cast<size_t>(64 * nb) * 4);
  return SSDNN_OK;
}

}  // namespace
int sp24_gemm_impl(int in_dt, int out_dt, int64_t M, int64_t N, int64_t K, const void* values,
                   const uint8_t* meta_hw, const void* X, int64_t ldx, void* Y, int64_t ldy, float alpha,
                   const ssdnn_epilogue* ep, bool f8_out_ok, void* stream, int variant = 0) {
  if (!valid_dt(in_dt)) return SSDNN_ERR_INVALID_ARG;
  const int eb = elem_bytes(in_dt);
  if (!gemm_variant_ok(variant, true, eb)) return SSDNN_ERR_UNSUPPORTED;
  int st = check_gemm_io(out_dt, f8_out_ok, M, N, K, X, ldx, eb, Y, ldy);
  if (st == SSDNN_OK) st = check_epilogue(ep);
  if (st != SSDNN_OK || M == 0 || N == 0) return st;
  if (K % 4) return SSDNN_ERR_UNSUPPORTED;
  auto s = static_cast<cudaStream_t>(stream);
  if (K == 0) return empty_product(Y, ldy, M, N, out_dt, ep, s);
  if (!values || !meta_hw) return SSDNN_ERR_INVALID_ARG;
  if (!aligned16(values) || !aligned16(meta_hw)) return SSDNN_ERR_UNSUPPORTED;
  GemmArgs a{};
  a.dt = in_dt;
  a.out_dt = out_dt;
  a.M = M;
  a.N = N;
  a.K = K;
  a.A = values;
  a.lda = round_up(K, 32) / 2;
  a.meta_hw = meta_hw;
  a.X = X;
  a.ldx = ldx;
  a.Y = Y;
  a.ldy = ldy;
  a.alpha = alpha;
  a.variant = variant;
  set_epilogue(a, ep);
  return from_cuda(launch_gemm(1, a, s, error_word()));
}

int dense_gemm_impl(int in_dt, int out_dt, int64_t M, int64_t N, int64_t K, const void* W, int64_t ldw,
                    const void* X, int64_t ldx, void* Y, int64_t ldy, float alpha, const ssdnn_epilogue* ep,
                    bool f8_out_ok, void* stream, int variant = 0) {
  if (!valid_dt(in_dt)) return SSDNN_ERR_INVALID_ARG;
  const int eb = elem_bytes(in_dt);
  if (!gemm_variant_ok(variant, false, eb)) return SSDNN_ERR_UNSUPPORTED;
  int st = check_gemm_io(out_dt, f8_out_ok, M, N, K, X, ldx, eb, Y, ldy);
  if (st == SSDNN_OK) st = check_epilogue(ep);
  if (st != SSDNN_OK || M == 0 || N == 0) return st;
  auto s = static_cast<cudaStream_t>(stream);
  if (K == 0) return empty_product(Y, ldy, M, N, out_dt, ep, s);
  if (!W || ldw < K) return SSDNN_ERR_INVALID_ARG;
  if (!aligned16(W) || (ldw * eb) % 16) return SSDNN_ERR_UNSUPPORTED;
  GemmArgs a{};
  a.dt = in_dt;
  a.out_dt = out_dt;
  a.M = M;
  a.N = N;
  a.K = K;
  a.A = W;
  a.lda = ldw;
  a.X = X;
  a.ldx = ldx;
  a.Y = Y;
  a.ldy = ldy;
  a.alpha = alpha;
  a.variant = variant;
  set_epilogue(a, ep);
  return from_cuda(launch_gemm(0, a, s, error_word()));
}

int tvw_gemm_impl(int dt, int out_dt, int tvw, int64_t M, int64_t N, int64_t K, const int32_t* keep_counts_host,
                  const int32_t* offsets, const int32_t* indices, const int32_t* schedule, const void* packed,
                  const uint8_t* meta_hw, const void* X, int64_t ldx, void* Y, int64_t ldy, float alpha,
                  const ssdnn_epilogue* ep, bool f8_out_ok, void* stream) {
  if (dt != SSDNN_F16 && dt != SSDNN_BF16) return dt == SSDNN_E4M3 ? SSDNN_ERR_UNSUPPORTED : SSDNN_ERR_INVALID_ARG;
  int st = check_gemm_io(out_dt, f8_out_ok, M, N, K, X, ldx, 2, Y, ldy);
  if (st == SSDNN_OK) st = check_epilogue(ep);
  if (st != SSDNN_OK || M == 0 || N == 0) return st;
  if (!keep_counts_host) return SSDNN_ERR_INVALID_ARG;
  Tables tb;
  st = build_tables(tvw, M, K, keep_counts_host, &tb);
  if (st != SSDNN_OK) return st;
  auto s = static_cast<cudaStream_t>(stream);
  if (K == 0 || tb.t.P_total == 0) return empty_product(Y, ldy, M, N, out_dt, ep, s);
  if (!offsets || !indices || !schedule || !packed || (tvw && !meta_hw)) return SSDNN_ERR_INVALID_ARG;
  if (!aligned16(packed) || (tvw && !aligned16(meta_hw))) return SSDNN_ERR_UNSUPPORTED;
  GemmArgs a{};
  a.dt = dt;
  a.out_dt = out_dt;
  a.M = M;
  a.N = N;
  a.K = K;
  a.A = packed;
  a.meta_hw = meta_hw;
  a.X = X;
  a.ldx = ldx;
  a.Y = Y;
  a.ldy = ldy;
  a.alpha = alpha;
  a.nt = tb.t.nt;
  a.packed_rows = 2 * tb.t.P_total;
  a.offsets = offsets;
  a.indices = indices;
  a.schedule = schedule;
  set_epilogue(a, ep);
  return from_cuda(launch_gemm(tvw ? 3 : 2, a, s, error_word()));
}

int bw_gemm_impl(int dt, int out_dt, int64_t M, int64_t N, int64_t K, const int32_t* keep_blocks_host,
                 const int32_t* offsets, const int32_t* indices, const int32_t* schedule, const void* packed,
                 const void* X, int64_t ldx, void* Y, int64_t ldy, float alpha, const ssdnn_epilogue* ep,
                 bool f8_out_ok, void* stream) {
  if (dt != SSDNN_F16 && dt != SSDNN_BF16) return dt == SSDNN_E4M3 ? SSDNN_ERR_UNSUPPORTED : SSDNN_ERR_INVALID_ARG;
  int st = check_gemm_io(out_dt, f8_out_ok, M, N, K, X, ldx, 2, Y, ldy);
  if (st == SSDNN_OK) st = check_epilogue(ep);
  if (st != SSDNN_OK || M == 0 || N == 0) return st;
  if (!keep_blocks_host) return SSDNN_ERR_INVALID_ARG;
  BwTables tb;
  st = build_bw_tables(M, K, keep_blocks_host, &tb);
  if (st != SSDNN_OK) return st;
  auto s = static_cast<cudaStream_t>(stream);
  if (K == 0 || tb.n_blocks == 0) return empty_product(Y, ldy, M, N, out_dt, ep, s);
  if (!offsets || !indices || !schedule || !packed) return SSDNN_ERR_INVALID_ARG;
  if (!aligned16(packed)) return SSDNN_ERR_UNSUPPORTED;
  GemmArgs a{};
  a.dt = dt;
  a.out_dt = out_dt;
  a.M = M;
  a.N = N;
  a.K = K;
  a.A = packed;
  a.X = X;
  a.ldx = ldx;
  a.Y = Y;
  a.ldy = ldy;
  a.alpha = alpha;
  a.nt = tb.cols.t.nt;
  a.packed_rows = 2 * tb.cols.t.P_total;
  a.offsets = offsets;
  a.indices = indices;
  a.schedule = schedule;
  set_epilogue(a, ep);
  return from_cuda(launch_gemm(4, a, s, error_word()));
}

}  // namespace ssdnn

using namespace ssdnn;

extern "C" {

const char* ssdnn_status_str(int status) {
  switch (status) {
    case SSDNN_OK: return "ok";
    case SSDNN_ERR_INVALID_ARG: return "invalid argument";
    case SSDNN_ERR_UNSUPPORTED: return "unsupported shape, alignment or dtype";
    case SSDNN_ERR_CUDA: return "CUDA error";
    case SSDNN_ERR_TIMEOUT: return "device-side wait timed out";
    case SSDNN_ERR_DEVICE: return "device error flag set";
  }
  return "unknown status";
}

int ssdnn_version(void) { return 100; }

int ssdnn_check_device_error(void* stream) {
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return SSDNN_ERR_CUDA;
  uint32_t* w = error_word();
  if (!w) return SSDNN_ERR_CUDA;
  uint32_t v = 0;
  if (cudaMemcpy(&v, w, sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess) return SSDNN_ERR_CUDA;
  if (v) {
    const uint32_t zero = 0;
    if (cudaMemcpy(w, &zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess) return SSDNN_ERR_CUDA;
  }
  if (v & kErrTimeout) return SSDNN_ERR_TIMEOUT;
  if (v) return SSDNN_ERR_DEVICE;
  return SSDNN_OK;
}

int ssdnn_mma_rate(int dt, int sparse, int n, int iters, void* stream) {
  if (!valid_dt(dt) || (sparse != 0 && sparse != 1) || iters < 1 || iters > (1 << 18))
    return SSDNN_ERR_INVALID_ARG;
  if (n != 128 && n != 192 && n != 256) return SSDNN_ERR_UNSUPPORTED;
  uint32_t* w = error_word();
  if (!w) return SSDNN_ERR_CUDA;
  return from_cuda(launch_mma_rate(dt, sparse, n, iters, static_cast<cudaStream_t>(stream), w));
}

int ssdnn_mma_rate_pair(int dt, int sparse, int iters, void* stream) {
  if (!valid_dt(dt) || (sparse != 0 && sparse != 1) || iters < 1 || iters > (1 << 18))
    return SSDNN_ERR_INVALID_ARG;
  uint32_t* w = error_word();
  if (!w) return SSDNN_ERR_CUDA;
  return from_cuda(launch_mma_rate_pair(dt, sparse, iters, static_cast<cudaStream_t>(stream), w));
}

int ssdnn_selftest_wait_timeout(uint32_t limit_us, void* stream) {
  if (limit_us == 0 || limit_us > 1000000u) return SSDNN_ERR_INVALID_ARG;
  uint32_t* w = error_word();
  if (!w) return SSDNN_ERR_CUDA;
  k_selftest_timeout<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(w, uint64_t(limit_us) * 1000ull);
  return from_cuda(cudaGetLastError());
}

int sp24_sizes(int dt, int64_t M, int64_t K, size_t* values_bytes, size_t* meta_bytes, size_t* meta_hw_bytes) {
  if (!valid_dt(dt) || M < 0 || K < 0 || M > kMaxDim || K > kMaxDim) return SSDNN_ERR_INVALID_ARG;
  if (K % 4) return SSDNN_ERR_UNSUPPORTED;
  const int64_t Kp = round_up(K, 32);
  if (values_bytes) *values_bytes = static_cast<size_t>(M * (Kp / 2) * elem_bytes(dt));
  if (meta_bytes) *meta_bytes = static_cast<size_t>(M * (Kp / 8));
  const int64_t span = dt == SSDNN_E4M3 ? 128 : 64;  // K columns per operand metadata block
  if (meta_hw_bytes) *meta_hw_bytes = static_cast<size_t>(ceil_div(M, 128) * ceil_div(K, span) * 2048);
  return SSDNN_OK;
}

int sp24_prune_compress(int dt, const void* W, int64_t M, int64_t K, int64_t ldw, void* values, uint8_t* meta,
                        uint8_t* meta_hw, void* stream) {
  if (!valid_dt(dt) || M < 0 || K < 0 || M > kMaxDim || K > kMaxDim) return SSDNN_ERR_INVALID_ARG;
  if (K % 4) return SSDNN_ERR_UNSUPPORTED;
  if (M == 0 || K == 0) return SSDNN_OK;
  if (!W || !values || !meta_hw || ldw < K) return SSDNN_ERR_INVALID_ARG;
  const int eb = elem_bytes(dt);
  if ((reinterpret_cast<uintptr_t>(W) % eb) || !aligned16(values) || !aligned16(meta_hw) ||
      (meta && (reinterpret_cast<uintptr_t>(meta) & 3u)))
    return SSDNN_ERR_UNSUPPORTED;
  return from_cuda(launch_sp24_compress(dt, W, M, K, ldw, values, meta, meta_hw,
                                        static_cast<cudaStream_t>(stream), error_word()));
}

int sp24_gemm(int in_dt, int out_dt, int64_t M, int64_t N, int64_t K, const void* values,
              const uint8_t* meta_hw, const void* X, int64_t ldx, void* Y, int64_t ldy, float alpha,
              void* stream) {
  return sp24_gemm_impl(in_dt, out_dt, M, N, K, values, meta_hw, X, ldx, Y, ldy, alpha, nullptr, false, stream);
}

int sp24_gemm_ep(int in_dt, int out_dt, int64_t M, int64_t N, int64_t K, const void* values,
                 const uint8_t* meta_hw, const void* X, int64_t ldx, void* Y, int64_t ldy, float alpha,
                 const ssdnn_epilogue* ep, void* stream) {
  return sp24_gemm_impl(in_dt, out_dt, M, N, K, values, meta_hw, X, ldx, Y, ldy, alpha, ep, true, stream);
}

int sp24_gemm_host(int in_dt, int out_dt, int64_t M, int64_t N, int64_t K, const void* values,
                   const uint8_t* meta_hw, const void* X_host, int64_t ldx, void* Y_host, int64_t ldy, float alpha,
                   void* X_dev, void* Y_dev, int64_t rows_per_block, void* stream, void* copy_stream) {
  if (!valid_dt(in_dt)) return SSDNN_ERR_INVALID_ARG;
  const int eb = elem_bytes(in_dt);
  const bool direct = Y_dev == nullptr;  // the epilogue writes the page-locked Y_host itself
  int st = check_gemm_io(out_dt, false, M, N, K, X_dev, ldx, eb, direct ? Y_host : Y_dev, ldy);
  if (st != SSDNN_OK || M == 0 || N == 0) return st;
  if (!Y_host || (K > 0 && !X_host)) return SSDNN_ERR_INVALID_ARG;
  if (direct && K == 0) return SSDNN_ERR_UNSUPPORTED;
  if (rows_per_block < 0 || rows_per_block % 128) return SSDNN_ERR_INVALID_ARG;
  if (K % 4) return SSDNN_ERR_UNSUPPORTED;
  auto s = static_cast<cudaStream_t>(stream);
  auto cs = copy_stream ? static_cast<cudaStream_t>(copy_stream) : s;
  const int ob = out_bytes(out_dt);
  const size_t y_pitch = static_cast<size_t>(ldy * ob);
  if (K > 0) {
    const size_t x_pitch = static_cast<size_t>(ldx * eb);
    if (cudaMemcpy2DAsync(X_dev, x_pitch, X_host, x_pitch, static_cast<size_t>(N * eb), static_cast<size_t>(K),
                          cudaMemcpyHostToDevice, s) != cudaSuccess)
      return SSDNN_ERR_CUDA;
  }
  if (direct)
    return sp24_gemm_impl(in_dt, out_dt, M, N, K, values, meta_hw, X_dev, ldx, Y_host, ldy, alpha, nullptr, false,
                          stream);
  const int64_t rb = rows_per_block > 0 ? rows_per_block : M;
  const int64_t Kp = round_up(K, 32), KB = ceil_div(K, in_dt == SSDNN_E4M3 ? 128 : 64);
  for (int64_t r0 = 0; r0 < M; r0 += rb) {
    const int64_t rows = std::min(rb, M - r0);
    const auto* vals = static_cast<const uint8_t*>(values) + r0 * (Kp / 2) * eb;
    const uint8_t* meta = meta_hw + (r0 / 128) * KB * 2048;
    uint8_t* yd = static_cast<uint8_t*>(Y_dev) + r0 * ldy * ob;
    st = sp24_gemm_impl(in_dt, out_dt, rows, N, K, K > 0 ? vals : nullptr, K > 0 ? meta : nullptr, X_dev, ldx, yd, ldy,
                        alpha, nullptr, false, stream);
    if (st != SSDNN_OK) return st;
    if (cs != s) {  // the copy stream takes this block as soon as its GEMM has finished
      cudaEvent_t ev = copy_event(r0 / rb);
      if (!ev || cudaEventRecord(ev, s) != cudaSuccess || cudaStreamWaitEvent(cs, ev, 0) != cudaSuccess)
        return SSDNN_ERR_CUDA;
    }
    if (cudaMemcpy2DAsync(static_cast<uint8_t*>(Y_host) + r0 * y_pitch, y_pitch, yd, y_pitch,
                          static_cast<size_t>(N * ob), static_cast<size_t>(rows), cudaMemcpyDeviceToHost,
                          cs) != cudaSuccess)
      return SSDNN_ERR_CUDA;
  }
  if (cs != s) {  // the caller's stream completes only after the last copy
    cudaEvent_t ev = copy_event(-1);
    if (!ev || cudaEventRecord(ev, cs) != cudaSuccess || cudaStreamWaitEvent(s, ev, 0) != cudaSuccess)
      return SSDNN_ERR_CUDA;
  }
  return SSDNN_OK;
}

int dense_gemm(int in_dt, int out_dt, int64_t M, int64_t N, int64_t K, const void* W, int64_t ldw,
               const void* X, int64_t ldx, void* Y, int64_t ldy, float alpha, void* stream) {
  return dense_gemm_impl(in_dt, out_dt, M, N, K, W, ldw, X, ldx, Y, ldy, alpha, nullptr, false, stream);
}

int dense_gemm_ep(int in_dt, int out_dt, int64_t M, int64_t N, int64_t K, const void* W, int64_t ldw,
                  const void* X, int64_t ldx, void* Y, int64_t ldy, float alpha, const ssdnn_epilogue* ep,
                  void* stream) {
  return dense_gemm_impl(in_dt, out_dt, M, N, K, W, ldw, X, ldx, Y, ldy, alpha, ep, true, stream);
}

int sp24_gemm_variant(int in_dt, int out_dt, int64_t M, int64_t N, int64_t K, const void* values,
                      const uint8_t* meta_hw, const void* X, int64_t ldx, void* Y, int64_t ldy, float alpha,
                      const ssdnn_epilogue* ep, int variant, void* stream) {
  return sp24_gemm_impl(in_dt, out_dt, M, N, K, values, meta_hw, X, ldx, Y, ldy, alpha, ep, true, stream, variant);
}

int dense_gemm_variant(int in_dt, int out_dt, int64_t M, int64_t N, int64_t K, const void* W, int64_t ldw,
                       const void* X, int64_t ldx, void* Y, int64_t ldy, float alpha, const ssdnn_epilogue* ep,
                       int variant, void* stream) {
  return dense_gemm_impl(in_dt, out_dt, M, N, K, W, ldw, X, ldx, Y, ldy, alpha, ep, true, stream, variant);
}

int tw_sizes(int dt, int tvw, int64_t M, int64_t K, const int32_t* keep_counts_host, size_t* packed_bytes,
             size_t* indices_count, size_t* meta_bytes, size_t* meta_hw_bytes, size_t* workspace_bytes) {
  if ((dt != SSDNN_F16 && dt != SSDNN_BF16) || M < 0 || K < 0 || M > kMaxDim || K > kMaxDim)
    return dt == SSDNN_E4M3 ? SSDNN_ERR_UNSUPPORTED : SSDNN_ERR_INVALID_ARG;
  if (M > 0 && !keep_counts_host) return SSDNN_ERR_INVALID_ARG;
  Tables tb;
  int st = build_tables(tvw, M, K, keep_counts_host, &tb);
  if (st != SSDNN_OK) return st;
  const int64_t P = tb.t.P_total;
  if (packed_bytes) *packed_bytes = static_cast<size_t>((tvw ? 64 : 128) * P * 2);
  if (indices_count) *indices_count = static_cast<size_t>(tb.L_total);
  if (meta_bytes) *meta_bytes = tvw ? static_cast<size_t>(16 * P) : 0;
  if (meta_hw_bytes) *meta_hw_bytes = tvw ? static_cast<size_t>(2048 * tb.t.Q_total) : 0;
  if (workspace_bytes) *workspace_bytes = static_cast<size_t>(tb.t.nt * K * 4);
  return SSDNN_OK;
}

int tw_prune_compress(int dt, int tvw, const void* W, int64_t M, int64_t K, int64_t ldw,
                      const int32_t* keep_counts_host, int32_t* offsets, int32_t* indices, int32_t* schedule,
                      void* packed, uint8_t* meta, uint8_t* meta_hw, void* workspace, void* stream) {
  if ((dt != SSDNN_F16 && dt != SSDNN_BF16) || M < 0 || K < 0 || M > kMaxDim || K > kMaxDim)
    return dt == SSDNN_E4M3 ? SSDNN_ERR_UNSUPPORTED : SSDNN_ERR_INVALID_ARG;
  if (M == 0) return SSDNN_OK;
  if (!keep_counts_host || !offsets || !schedule) return SSDNN_ERR_INVALID_ARG;
  Tables tb;
  int st = build_tables(tvw, M, K, keep_counts_host, &tb);
  if (st != SSDNN_OK) return st;
  if (K > 0 && (!W || ldw < K || !workspace)) return SSDNN_ERR_INVALID_ARG;
  if (tb.L_total > 0 && !indices) return SSDNN_ERR_INVALID_ARG;
  if (tb.t.P_total > 0 && (!packed || (tvw && (!meta || !meta_hw)))) return SSDNN_ERR_INVALID_ARG;
  if ((W && (reinterpret_cast<uintptr_t>(W) & 1u)) || (packed && !aligned16(packed)) ||
      (meta && !aligned16(meta)) || (meta_hw && !aligned16(meta_hw)) || (workspace && !aligned16(workspace)) ||
      (reinterpret_cast<uintptr_t>(offsets) & 3u) || (reinterpret_cast<uintptr_t>(schedule) & 3u) ||
      (indices && (reinterpret_cast<uintptr_t>(indices) & 3u)))
    return SSDNN_ERR_UNSUPPORTED;
  auto s = static_cast<cudaStream_t>(stream);
  // Host tables (pageable source: the copy is staged before the call returns).
  cudaError_t e = cudaMemcpyAsync(offsets, tb.offsets.data(), tb.offsets.size() * sizeof(int32_t),
                                  cudaMemcpyHostToDevice, s);
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(schedule, tb.schedule.data(), tb.schedule.size() * sizeof(int32_t),
                        cudaMemcpyHostToDevice, s);
  if (e != cudaSuccess) return SSDNN_ERR_CUDA;
  return from_cuda(launch_tw_prune(dt, tvw, W, M, K, ldw, tb.t, offsets, indices, schedule, packed, meta, meta_hw,
                                   static_cast<float*>(workspace), s, error_word()));
}

int tvw_gemm(int dt, int tvw, int64_t M, int64_t N, int64_t K, const int32_t* keep_counts_host,
             const int32_t* offsets, const int32_t* indices, const int32_t* schedule, const void* packed,
             const uint8_t* meta_hw, const void* X, int64_t ldx, void* Y, int64_t ldy, void* stream) {
  return tvw_gemm_impl(dt, dt, tvw, M, N, K, keep_counts_host, offsets, indices, schedule, packed, meta_hw, X, ldx,
                       Y, ldy, 1.0f, nullptr, false, stream);
}

int tvw_gemm_ep(int dt, int out_dt, int tvw, int64_t M, int64_t N, int64_t K, const int32_t* keep_counts_host,
                const int32_t* offsets, const int32_t* indices, const int32_t* schedule, const void* packed,
                const uint8_t* meta_hw, const void* X, int64_t ldx, void* Y, int64_t ldy, float alpha,
                const ssdnn_epilogue* ep, void* stream) {
  return tvw_gemm_impl(dt, out_dt, tvw, M, N, K, keep_counts_host, offsets, indices, schedule, packed, meta_hw, X,
                       ldx, Y, ldy, alpha, ep, true, stream);
}

int bw_sizes(int dt, int64_t M, int64_t K, const int32_t* keep_blocks_host, size_t* packed_bytes,
             size_t* indices_count, size_t* workspace_bytes) {
  if ((dt != SSDNN_F16 && dt != SSDNN_BF16) || M < 0 || K < 0 || M > kMaxDim || K > kMaxDim)
    return dt == SSDNN_E4M3 ? SSDNN_ERR_UNSUPPORTED : SSDNN_ERR_INVALID_ARG;
  if (M > 0 && !keep_blocks_host) return SSDNN_ERR_INVALID_ARG;
  BwTables tb;
  const int st = build_bw_tables(M, K, keep_blocks_host, &tb);
  if (st != SSDNN_OK) return st;
  if (packed_bytes) *packed_bytes = static_cast<size_t>(128 * 64 * tb.n_blocks * 2);
  if (indices_count) *indices_count = static_cast<size_t>(tb.n_blocks);
  if (workspace_bytes) *workspace_bytes = tb.ws_bytes;
  return SSDNN_OK;
}

int bw_prune_compress(int dt, const void* W, int64_t M, int64_t K, int64_t ldw, const int32_t* keep_blocks_host,
                      int32_t* offsets, int32_t* indices, int32_t* schedule, void* packed, void* workspace,
                      void* stream) {
  if ((dt != SSDNN_F16 && dt != SSDNN_BF16) || M < 0 || K < 0 || M > kMaxDim || K > kMaxDim)
    return dt == SSDNN_E4M3 ? SSDNN_ERR_UNSUPPORTED : SSDNN_ERR_INVALID_ARG;
  if (M == 0) return SSDNN_OK;
  if (!keep_blocks_host || !offsets || !schedule) return SSDNN_ERR_INVALID_ARG;
  BwTables tb;
  int st = build_bw_tables(M, K, keep_blocks_host, &tb);
  if (st != SSDNN_OK) return st;
  if (K > 0 && (!W || ldw < K || !workspace)) return SSDNN_ERR_INVALID_ARG;
  if (tb.n_blocks > 0 && (!indices || !packed)) return SSDNN_ERR_INVALID_ARG;
  if ((W && (reinterpret_cast<uintptr_t>(W) & 1u)) || (packed && !aligned16(packed)) ||
      (workspace && !aligned16(workspace)) || (reinterpret_cast<uintptr_t>(offsets) & 3u) ||
      (reinterpret_cast<uintptr_t>(schedule) & 3u) || (indices && (reinterpret_cast<uintptr_t>(indices) & 3u)))
    return SSDNN_ERR_UNSUPPORTED;
  auto s = static_cast<cudaStream_t>(stream);
  auto* ws = static_cast<uint8_t*>(workspace);
  auto* col_off = reinterpret_cast<int32_t*>(ws + tb.ws_coloff);
  // Host tables (pageable source: the copy is staged before the call returns).
  cudaError_t e = cudaMemcpyAsync(offsets, tb.blk_offsets.data(), tb.blk_offsets.size() * sizeof(int32_t),
                                  cudaMemcpyHostToDevice, s);
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(schedule, tb.cols.schedule.data(), tb.cols.schedule.size() * sizeof(int32_t),
                        cudaMemcpyHostToDevice, s);
  if (e == cudaSuccess && K > 0)
    e = cudaMemcpyAsync(col_off, tb.cols.offsets.data(), tb.cols.offsets.size() * sizeof(int32_t),
                        cudaMemcpyHostToDevice, s);
  if (e != cudaSuccess) return SSDNN_ERR_CUDA;
  if (K == 0) return SSDNN_OK;
  return from_cuda(launch_bw_prune(dt, W, M, K, ldw, tb.cols.t, offsets, indices, tb.n_blocks, col_off,
                                   reinterpret_cast<int32_t*>(ws + tb.ws_colidx), schedule, packed,
                                   reinterpret_cast<float*>(ws + tb.ws_scores),
                                   reinterpret_cast<float*>(ws + tb.ws_bscores), s));
}

int bw_gemm(int dt, int64_t M, int64_t N, int64_t K, const int32_t* keep_blocks_host, const int32_t* offsets,
            const int32_t* indices, const int32_t* schedule, const void* packed, const void* X, int64_t ldx, void* Y,
            int64_t ldy, void* stream) {
  return bw_gemm_impl(dt, dt, M, N, K, keep_blocks_host, offsets, indices, schedule, packed, X, ldx, Y, ldy, 1.0f,
                      nullptr, false, stream);
}

int bw_gemm_ep(int dt, int out_dt, int64_t M, int64_t N, int64_t K, const int32_t* keep_blocks_host,
               const int32_t* offsets, const int32_t* indices, const int32_t* schedule, const void* packed,
               const void* X, int64_t ldx, void* Y, int64_t ldy, float alpha, const ssdnn_epilogue* ep,
               void* stream) {
  return bw_gemm_impl(dt, out_dt, M, N, K, keep_blocks_host, offsets, indices, schedule, packed, X, ldx, Y, ldy, alpha,
                      ep, true, stream);
}

int ew_sizes(int dt, int64_t M, int64_t K, int64_t k, size_t* vals_bytes, size_t* indices_count,
             size_t* workspace_bytes) {
  if ((dt != SSDNN_F16 && dt != SSDNN_BF16) || M < 0 || K < 0 || k < 0 || M > kMaxDim || K > kMaxDim || k > K)
    return dt == SSDNN_E4M3 ? SSDNN_ERR_UNSUPPORTED : SSDNN_ERR_INVALID_ARG;
  if (M * k > kMaxDim) return SSDNN_ERR_UNSUPPORTED;
  if (vals_bytes) *vals_bytes = static_cast<size_t>(M * k * 2);
  if (indices_count) *indices_count = static_cast<size_t>(M * k);
  if (workspace_bytes) *workspace_bytes = static_cast<size_t>(M * K * 4);
  return SSDNN_OK;
}

int ew_prune_compress(int dt, const void* W, int64_t M, int64_t K, int64_t ldw, int64_t k, int32_t* row_ptr,
                      int32_t* col_idx, void* vals, void* workspace, void* stream) {
  int st = ew_sizes(dt, M, K, k, nullptr, nullptr, nullptr);
  if (st != SSDNN_OK) return st;
  if (!row_ptr) return SSDNN_ERR_INVALID_ARG;
  if (M > 0 && k > 0 && (!W || ldw < K || !col_idx || !vals || !workspace)) return SSDNN_ERR_INVALID_ARG;
  if ((W && (reinterpret_cast<uintptr_t>(W) & 1u)) || (vals && (reinterpret_cast<uintptr_t>(vals) & 1u)) ||
      (workspace && !aligned16(workspace)) || (reinterpret_cast<uintptr_t>(row_ptr) & 3u) ||
      (col_idx && (reinterpret_cast<uintptr_t>(col_idx) & 3u)))
    return SSDNN_ERR_UNSUPPORTED;
  return from_cuda(launch_ew_prune(dt, W, M, K, ldw, k, row_ptr, col_idx, vals, static_cast<float*>(workspace),
                                   static_cast<cudaStream_t>(stream)));
}

int ew_spmm(int dt, int64_t M, int64_t N, int64_t K, const int32_t* row_ptr, const int32_t* col_idx,
            const void* vals, const void* X, int64_t ldx, void* Y, int64_t ldy, void* stream) {
  if (dt != SSDNN_F16 && dt != SSDNN_BF16) return dt == SSDNN_E4M3 ? SSDNN_ERR_UNSUPPORTED : SSDNN_ERR_INVALID_ARG;
  const int st = check_gemm_io(dt, false, M, N, K, X, ldx, 2, Y, ldy);
  if (st != SSDNN_OK || M == 0 || N == 0) return st;
  if (!row_ptr || (K > 0 && (!col_idx || !vals))) return SSDNN_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(row_ptr) & 3u) || (col_idx && (reinterpret_cast<uintptr_t>(col_idx) & 3u)) ||
      (vals && (reinterpret_cast<uintptr_t>(vals) & 1u)))
    return SSDNN_ERR_UNSUPPORTED;
  auto s = static_cast<cudaStream_t>(stream);
  if (K == 0) return zero_output(Y, ldy, M, N, 2, s);
  return from_cuda(launch_ew_spmm(dt, M, N, K, row_ptr, col_idx, vals, X, ldx, Y, ldy, s));
}

// 3x3 convolution (implicit GEMM), shared checks: 16-bit data, C_in a multiple of 64,
// image width at most 224, output C_out x (N H W) with a 16-byte-aligned pitch.
static int conv_impl(int sparse, int dt, int out_dt, int64_t Cout, int64_t Cin, int64_t Nb, int64_t H, int64_t W,
                     const void* A, int64_t lda, const uint8_t* meta_hw, const void* X, void* Y, int64_t ldy,
                     float alpha, void* stream) {
  if (dt != SSDNN_F16 && dt != SSDNN_BF16) return dt == SSDNN_E4M3 ? SSDNN_ERR_UNSUPPORTED : SSDNN_ERR_INVALID_ARG;
  if (Cout < 0 || Cin < 0 || Nb < 0 || H < 0 || W < 0) return SSDNN_ERR_INVALID_ARG;
  if (Cout > kMaxDim || Nb * H * W > kMaxDim || 9 * Cin > kMaxDim || H > kMaxDim) return SSDNN_ERR_INVALID_ARG;
  if (Cin % 64 || W > 224) return SSDNN_ERR_UNSUPPORTED;
  const int64_t M = Cout, N = Nb * H * W, K = 9 * Cin;
  // X is NHWC, not an N-pitch matrix: only its base alignment applies (passed as a pitch that checks clean)
  int st = check_gemm_io(out_dt, false, M, N, K, X, round_up(N, 8), 2, Y, ldy);
  if (st != SSDNN_OK || M == 0 || N == 0) return st;
  auto s = static_cast<cudaStream_t>(stream);
  if (K == 0) return zero_output(Y, ldy, M, N, 2, s);
  if (!A || (sparse && !meta_hw) || (!sparse && lda < K)) return SSDNN_ERR_INVALID_ARG;
  if (!aligned16(A) || (sparse && !aligned16(meta_hw)) || (!sparse && (lda * 2) % 16)) return SSDNN_ERR_UNSUPPORTED;
  GemmArgs a{};
  a.dt = dt;
  a.out_dt = out_dt;
  a.M = M;
  a.N = N;
  a.K = K;
  a.A = A;
  a.lda = sparse ? K / 2 : lda;
  a.meta_hw = meta_hw;
  a.X = X;
  a.ldx = N;
  a.Y = Y;
  a.ldy = ldy;
  a.alpha = alpha;
  a.conv_cin = Cin;
  a.conv_h = H;
  a.conv_w = W;
  a.conv_nb = Nb;
  return from_cuda(launch_gemm(sparse ? 5 : 6, a, s, error_word()));
}

int tw_conv3x3(int dt, int out_dt, int64_t Cout, int64_t Cin, int64_t Nb, int64_t H, int64_t W,
               const int32_t* keep_groups_host, const int32_t* offsets, const int32_t* indices, const int32_t* schedule,
               const void* packed, const void* X, void* Y, int64_t ldy, float alpha, void* stream) {
  if (dt != SSDNN_F16 && dt != SSDNN_BF16) return dt == SSDNN_E4M3 ? SSDNN_ERR_UNSUPPORTED : SSDNN_ERR_INVALID_ARG;
  if (Cout < 0 || Cin < 0 || Nb < 0 || H < 0 || W < 0) return SSDNN_ERR_INVALID_ARG;
  if (Cout > kMaxDim || Nb * H * W > kMaxDim || 9 * Cin > kMaxDim || H > kMaxDim) return SSDNN_ERR_INVALID_ARG;
  if (Cin % 64 || W > 224) return SSDNN_ERR_UNSUPPORTED;
  const int64_t M = Cout, N = Nb * H * W, K = 9 * Cin;
  int st = check_gemm_io(out_dt, false, M, N, K, X, round_up(N, 8), 2, Y, ldy);
  if (st != SSDNN_OK || M == 0 || N == 0) return st;
  if (!keep_groups_host) return SSDNN_ERR_INVALID_ARG;
  BwTables tb;
  st = build_bw_tables(M, K, keep_groups_host, &tb);  // a group is one tap x 64 channels: 64 columns of K
  if (st != SSDNN_OK) return st;
  auto s = static_cast<cudaStream_t>(stream);
  if (K == 0 || tb.n_blocks == 0) return zero_output(Y, ldy, M, N, 2, s);
  if (!offsets || !indices || !schedule || !packed) return SSDNN_ERR_INVALID_ARG;
  if (!aligned16(packed)) return SSDNN_ERR_UNSUPPORTED;
  GemmArgs a{};
  a.dt = dt;
  a.out_dt = out_dt;
  a.M = M;
  a.N = N;
  a.K = K;
  a.A = packed;
  a.X = X;
  a.ldx = N;
  a.Y = Y;
  a.ldy = ldy;
  a.alpha = alpha;
  a.nt = tb.cols.t.nt;
  a.packed_rows = 2 * tb.cols.t.P_total;
  a.offsets = offsets;
  a.indices = indices;
  a.schedule = schedule;
  a.conv_cin = Cin;
  a.conv_h = H;
  a.conv_w = W;
  a.conv_nb = Nb;
  return from_cuda(launch_gemm(7, a, s, error_word()));
}

int sp24_conv3x3(int dt, int out_dt, int64_t Cout, int64_t Cin, int64_t Nb, int64_t H, int64_t W, const void* values,
                 const uint8_t* meta_hw, const void* X, void* Y, int64_t ldy, float alpha, void* stream) {
  return conv_impl(1, dt, out_dt, Cout, Cin, Nb, H, W, values, 0, meta_hw, X, Y, ldy, alpha, stream);
}

int dense_conv3x3(int dt, int out_dt, int64_t Cout, int64_t Cin, int64_t Nb, int64_t H, int64_t W, const void* Wf,
                  int64_t ldw, const void* X, void* Y, int64_t ldy, float alpha, void* stream) {
  return conv_impl(0, dt, out_dt, Cout, Cin, Nb, H, W, Wf, ldw, nullptr, X, Y, ldy, alpha, stream);
}

}  // extern "C"
