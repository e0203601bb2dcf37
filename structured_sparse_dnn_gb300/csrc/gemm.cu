// The tensor-core GEMM family: dense, 2:4 sparse, tile-wise (TW) and
// tile-vector-wise (TVW), one persistent warp-specialised kernel template.
//
// Y = alpha * A . X with A the weight operand (M x K, K-major) and X the
// activations (K x N, N contiguous, i.e. an MN-major B operand).
//   dense : A = W.
//   sp24  : A = the 2:4-compressed values (K/2 wide) and its position metadata;
//           the sparse tensor core skips the zero half ("Accelerating Sparse Deep
//           Neural Networks", Abstract: twice the math rate of dense units).
//   TW    : per 128-row tile, A = the packed kept columns and the B rows are
//           gathered from X by the tile's index list -- the tile-wise pattern is
//           applied where operands come from global memory ("Accelerating Sparse
//           DNNs Based on Tiled GEMM", Abstract).
//   TVW   : TW with the packed tile in 2:4 form, executed on the sparse tensor
//           core (same page: 2:4 inside the tensor core, TW at global memory).
// Tiles are handed out in the schedule order (longest kept length first, equal
// lengths adjacent: "load-balancing through batching", same page, TL;DR), and the
// gather, MMA and epilogue run fused in one kernel ("kernel fusion", same TL;DR).
//
// Roles (256 threads, one CTA per SM, persistent over work units):
//   warp 0      producer: TMA tiles of A and B (B by 4-row gathers for TW/TVW),
//               1-D bulk copy of the 2:4 metadata blocks, into a ring of stages.
//   warp 1      MMA issuer: tcgen05.cp of metadata to TMEM, tcgen05.mma(.sp) into
//               a TMEM fp32 accumulator, commits release stages / publish tiles.
//   warp 2      TMEM allocator.
//   warps 4..7  epilogue: tcgen05.ld the accumulator (warp w reads TMEM lanes
//               32 (w % 4) ..), scale by alpha, round to the output type, store.
//
// Stage geometry (bytes are the same for 16-bit and 8-bit inputs):
//   BK = 128 / elem_bytes dense K per stage (64 fp16/bf16, 128 e4m3).
//   A  : 128 rows x 128 B (dense, 128B swizzle) or 128 rows x 64 B (sparse
//        values, 64B swizzle).
//   B  : BK rows x BN columns, as BN*eb/128 boxes of BK rows x 128 B, 128B swizzle
//        (MN-major canonical layout: 8-row atoms of 1024 B, boxes BK*128 B apart).
//   meta (sparse): one 2048-byte block per stage = 128 rows x 16 B, copied to
//        four TMEM columns; instruction j reads its metadata at column 2 j.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include <algorithm>

#include "common.cuh"
#include "kernels.h"

namespace ssdnn {
namespace {

struct Params {
  int32_t M, N;
  int32_t MB, NB;           // BM-row blocks (BM = 128 MT), BN-column blocks
  int32_t MB128;            // 128-row blocks (the metadata's row blocks)
  int32_t MG;               // groups of CLUSTER consecutive BM-row blocks (one group per cluster pass)
  int32_t GR;               // rasterisation: M groups per band; work sweeps a band's N blocks
  int32_t num_units;        // work items: (M group, N block) pairs, or (schedule entry, N block)
  int32_t nk;               // k stages per unit (dense / sp24)
  int32_t meta_kb;          // 2048-byte metadata blocks per 128-row block (one per 128 bytes of K)
  int32_t out_dt;           // 0 f16, 1 bf16, 2 e4m3
  int32_t act;              // fused epilogue: 0 none, 1 ReLU, 2 GELU
  const float* bias;        // fused epilogue: one fp32 bias per output row, or null
  float y_scale;            // fused epilogue: multiplier after the activation
  int32_t nstages;          // stages of the shared-memory ring in use (<= the compiled count)
  float alpha;
  const uint8_t* meta_hw;
  const int32_t* schedule;  // TW/TVW: (t, L, P, Q) per tile, in work order
  const int32_t* offsets;
  const int32_t* indices;
  const void* X;            // TW/TVW: the activations, gathered row by row
  int64_t ldx;              // elements
  uint8_t* Y;
  int64_t ldy;              // elements
  uint32_t* err;
  // 3x3 convolution: image geometry and the pixel patch of one work unit
  int32_t conv_cin, conv_h, conv_w, conv_rows;  // C_in, H, W, image rows per patch
  int32_t conv_patches;                         // patches per image
  int32_t conv_nb;                              // images
  uint32_t conv_box_bytes;                      // bytes one activation box delivers
  int32_t y_direct;                             // Y is page-locked host memory: plain stores, no TMA
  int32_t b3d;      // SM pairs: the B map is 3-D (64 columns, K rows, 64-column blocks), one box per stage
};

template <int DT, bool SPARSE, bool GATHER, int BN, int MT, int BROW = 128, bool PAIR = false,
          bool BLOCKW = false, bool CONV = false, int KX = 1>
struct Cfg {
  // CONV: 3x3 convolution as an implicit GEMM -- the B operand of a K stage is one
  // tap (r, s) and 64 input channels of a patch of image rows, loaded K-major by one
  // 4-D TMA box of the NHWC activations (the zero padding is the box's out-of-range fill).
  static constexpr bool CONVOLUTION = CONV;
  // BLOCKW: block-wise sparsity -- per 128-row tile, the packed kept 64-column blocks
  // of W against the matching 64-row panels of X, each loaded by one TMA box.
  static constexpr bool BLOCKWISE = BLOCKW;
  static constexpr bool SCHEDULED = GATHER || BLOCKW;         // work follows the tile schedule
  // PAIR: the two CTAs of a cluster form an SM pair running M = 256 MMAs (each CTA
  // holds 128 rows of A, BN/2 columns of B and its 128 accumulator rows); every
  // CTA loads its own operands (no multicast).
  static constexpr bool PAIRED = PAIR;
  static constexpr int CLUSTER = PAIR ? 2 : 1;              // CTAs per cluster
  static constexpr int BN_CTA = PAIR ? BN / 2 : BN;         // B columns held by this CTA
  static constexpr int SUB = MT;                            // 128-row sub-tiles per CTA tile
  static constexpr int BM = 128 * MT;
  // 4 control warps, 4 epilogue warps per sub-tile, and for TW/TVW 4 warps that
  // gather the kept X rows with 16-byte cp.async
  static constexpr int GATHER_WARPS = 16;
  static constexpr int GATHER_THREADS = GATHER ? 32 * GATHER_WARPS : 0;
  // SM pairs drain their 128 x 256 accumulator with eight epilogue warps (two per
  // TMEM lane quadrant, each taking half of the columns)
  static constexpr int EPI_SPLIT = PAIR ? 2 : 1;
  static constexpr int EPI_WARPS = 4 * MT * EPI_SPLIT;
  static constexpr int EPI_WARP0 = 4;
  static constexpr int GATHER_WARP0 = 4 + EPI_WARPS;
  static constexpr int THREADS = 128 + 32 * EPI_WARPS + GATHER_THREADS;
  static constexpr int EB = Elem<DT>::bytes;
  static constexpr bool F8 = Elem<DT>::f8;
  // KX = 2 (2:4 on SM pairs): a stage holds two 128-byte K steps, so every
  // compressed weight row of the stage is one 128-byte (128B-swizzled) row and the
  // ring turns over half as often
  static constexpr int BK = KX * 128 / EB;                  // dense K per stage
  static constexpr int A_SUB_BYTES = KX * (SPARSE ? 128 * 64 : 128 * 128);
  static constexpr int A_BYTES = MT * A_SUB_BYTES;
  static constexpr int B_BYTES = KX * 128 * BN_CTA;         // BK * BN_CTA * EB
  static constexpr int META_BYTES = SPARSE ? 2048 * MT * KX : 0;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES + META_BYTES;
  // Output staging (all but TW/TVW): each epilogue warp converts a 32 x 32 chunk
  // into one of two 2 KB shared-memory buffers and a TMA store writes it out, so
  // the accumulator is drained without waiting on global stores.
  static constexpr bool STAGED = !GATHER && !CONV;
  // two 2 KB buffers per epilogue warp; one for the 52 KB two-step stages, whose ring
  // then gets a fourth stage within the 227 KB a CTA may hold
  static constexpr int STAGING_BUFS = KX == 2 ? 1 : 2;
  static constexpr int STAGING_BYTES = STAGED ? EPI_WARPS * 2048 * STAGING_BUFS : 0;
  static constexpr int SMEM_BUDGET = KX == 2 ? 227 * 1024 - 1024 - 256 : 220 * 1024;
  static constexpr int STAGES_RAW = (SMEM_BUDGET - STAGING_BYTES) / STAGE_BYTES;
  static constexpr int STAGES = STAGES_RAW > 8 ? 8 : STAGES_RAW;
  static constexpr int MMA_K = (SPARSE ? 64 : 32) / EB;      // dense K per instruction
  static constexpr int MMAS = BK / MMA_K;                    // instructions per stage
  // B boxes are BK rows of BROW bytes (128: 128B swizzle; 64: 64B swizzle, which
  // lets an e4m3 N tile be a multiple of 64 columns)
  static constexpr int B_ROW = BROW;
  static constexpr int B_BOX_COLS = BROW / EB;               // columns per B box
  static constexpr int B_BOXES = BN_CTA / B_BOX_COLS;
  static constexpr int B_BOX_BYTES = BK * BROW;
  static constexpr int B_SBO = 8 * BROW;                     // 8-row swizzle atom
  static constexpr uint32_t B_SWZ = BROW == 128 ? 2u : 4u;
  static_assert(BROW == 128 || (BROW == 64 && !GATHER), "the gather writes 128-byte rows");
  static constexpr int ACC_COLS = MT * BN;                  // fp32 accumulator columns of one tile
  static constexpr int META_SLOTS = 4;
  static constexpr int META_SLOT_COLS = 4 * MT * KX;        // one 128x128b copy per sub-tile and K step
  static constexpr int META_COLS = SPARSE ? META_SLOTS * META_SLOT_COLS : 0;
  static constexpr int NACC = (2 * ACC_COLS + META_COLS <= 512) ? 2 : 1;
  static constexpr int META_COL0 = NACC * ACC_COLS;         // TMEM columns after the accumulators
  // the epilogue drains a single accumulator into registers before storing (at most
  // four 32-column chunks per warp: 64 packed words per thread)
  static constexpr bool EARLY_RELEASE = NACC == 1 && STAGED && BN / 32 / EPI_SPLIT <= 4;
  static constexpr uint32_t TMEM_COLS = 512;
  static constexpr uint32_t IDESC = ptx::idesc(Elem<DT>::mma_fmt, Elem<DT>::mma_fmt, SPARSE, PAIR ? 256 : 128,
                                               BN, false, !CONV);
  static constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + STAGING_BYTES + 1024 /*align*/ + 256 /*barriers*/;
  static_assert(STAGES >= 2, "the shared-memory ring needs two stages");
  static_assert(SMEM_BYTES <= 227 * 1024, "more shared memory than a CTA may hold");
  static_assert(CONV || B_BOXES * B_BOX_COLS == BN_CTA, "BN must be a multiple of the B box width");
  static_assert(BN % 32 == 0, "the epilogue drains 32-column chunks");
  static_assert(!PAIR || (MT == 1 && !GATHER), "SM pairs: one 128-row sub-tile per CTA");
  static_assert(!BLOCKW || (!SPARSE && !GATHER && !PAIR && MT == 1), "block-wise: dense 128-row tiles");
  static_assert(!CONV || (!GATHER && !PAIR && MT == 1 && Elem<DT>::bytes == 2),
                "convolution: 16-bit, 128-row tiles");
  static_assert(META_COL0 + META_COLS <= 512, "accumulators and metadata exceed TMEM");
  static_assert(KX == 1 || (KX == 2 && SPARSE && MT == 1 && !GATHER && !BLOCKW),
                "double K stages: 2:4 tiles of 128 rows (one CTA, an SM pair or a convolution)");
  // SM pairs with two-step stages take their X boxes on a second barrier
  static constexpr bool B_OWN_BARRIER = PAIR && KX == 2;
  static_assert(MT == 1 || !GATHER, "256-row tiles: no gather");
};

// N width of one output tile (both CTAs of a pair write all of it for their rows).
template <typename C>
__device__ __forceinline__ constexpr int BN_OF() {
  return C::BN_CTA * (C::PAIRED ? 2 : 1);
}

struct UnitInfo {
  int32_t m0, n0, nk;
  int32_t subs;       // 128-row sub-tiles of this tile that hold rows of W (the rest are zero)
  bool phantom;       // a cluster member past the last 128-row block: loads B, writes nothing
  int32_t a_row0;     // packed-operand row of the first chunk (TW/TVW)
  int32_t meta_blk0;  // first metadata block index
  int32_t idx_base;   // offsets[t] (TW/TVW)
  int32_t L;          // kept count (TW/TVW)
  int32_t ncols;      // valid output columns from n0 (convolution patches)
  int32_t img, h0;    // convolution: image and first image row of the patch
};

template <typename C, bool GATHER>
__device__ __forceinline__ UnitInfo decode_unit(const Params& p, int32_t u, uint32_t crank) {
  UnitInfo ui;
  ui.ncols = 0;
  ui.img = 0;
  ui.h0 = 0;
  if constexpr (C::CONVOLUTION) {
    int32_t mb, patch;
    if constexpr (C::BLOCKWISE) {
      // tile-wise filter: units are (schedule entry, pixel patch), entries (tiles by
      // kept group count, longest first) outermost
      const int32_t np = p.conv_nb * p.conv_patches;
      const int32_t e = u / np;
      patch = u - e * np;
      const int32_t* sch = p.schedule + 4 * e;
      const int32_t t = __ldg(sch + 0), L = __ldg(sch + 1), P = __ldg(sch + 2);
      mb = t;
      ui.nk = (L + C::BK - 1) / C::BK;    // kept (tap, 64-channel) groups
      ui.a_row0 = 2 * P;                  // packed chunks of 128 rows, tile t from row 2 P
      ui.idx_base = __ldg(p.offsets + t);
      ui.L = L;
    } else {
      // units: 128-row blocks of C_out fastest, then pixel patches (image, row block)
      mb = u % p.MB;
      patch = u / p.MB;
      ui.nk = p.nk;
      ui.a_row0 = mb * 128;
      ui.idx_base = 0;
      ui.L = 0;
    }
    ui.img = patch / p.conv_patches;
    ui.h0 = (patch - ui.img * p.conv_patches) * p.conv_rows;
    ui.phantom = false;
    ui.m0 = mb * 128;
    ui.n0 = (ui.img * p.conv_h + ui.h0) * p.conv_w;
    ui.ncols = min(p.conv_rows, p.conv_h - ui.h0) * p.conv_w;
    ui.meta_blk0 = mb * p.meta_kb;
    ui.subs = 1;
    return ui;
  }
  if constexpr (!GATHER) {
    // Bands of GR M groups: inside a band the M index runs fastest, then N, so the
    // CTAs in flight share a few weight rows and a few X panels and both stay in
    // L2 (plain M-fastest order streams all of W once per wave of N blocks).
    const int32_t band = u / (p.GR * p.NB), r = u - band * (p.GR * p.NB);
    const int32_t gh = min(p.GR, p.MG - band * p.GR);
    const int32_t nb = r / gh, mg = band * p.GR + (r - nb * gh);
    const int32_t mb = mg * C::CLUSTER + static_cast<int32_t>(crank);
    ui.phantom = mb >= p.MB;
    ui.m0 = mb * C::BM;
    ui.n0 = nb * BN_OF<C>();
    ui.nk = p.nk;
    ui.a_row0 = ui.m0;
    // one 2048-byte metadata block per (128-row block, 128 bytes of K)
    ui.meta_blk0 = mb * C::SUB * p.meta_kb;
    ui.subs = ui.phantom ? 0 : min(C::SUB, p.MB128 - mb * C::SUB);
    ui.idx_base = 0;
    ui.L = 0;
  } else {
    const int32_t e = u / p.NB, nb = u % p.NB;
    const int32_t* s = p.schedule + 4 * e;
    const int32_t t = __ldg(s + 0), L = __ldg(s + 1), P = __ldg(s + 2), Q = __ldg(s + 3);
    ui.phantom = false;
    ui.subs = 1;
    ui.m0 = t * 128;
    ui.n0 = nb * BN_OF<C>();
    ui.nk = (L + C::BK - 1) / C::BK;
    ui.a_row0 = 2 * P;  // packed chunks: 128 rows each, tile t starts at row 2 P
    ui.meta_blk0 = Q;
    ui.idx_base = __ldg(p.offsets + t);
    ui.L = L;
  }
  return ui;
}

// GELU in its exact form x Phi(x) = 0.5 x (1 + erf(x / sqrt 2)), with erf from the
// rational approximation of Abramowitz and Stegun, Handbook of Mathematical
// Functions, formula 7.1.26 (|error| <= 1.5e-7 for z >= 0):
//   erf(z) = 1 - (a1 t + a2 t^2 + a3 t^3 + a4 t^4 + a5 t^5) exp(-z^2), t = 1 / (1 + p z).
// With q = (a1 t + ... + a5 t^5) exp(-z^2) and z = |x| / sqrt 2, 1 + erf(x / sqrt 2) is
// 2 - q for x >= 0 and q for x < 0 (taken as q itself, so no cancellation there).
__device__ __forceinline__ float gelu_exact(float x) {
  constexpr float kP = 0.3275911f, kA1 = 0.254829592f, kA2 = -0.284496736f, kA3 = 1.421413741f,
                  kA4 = -1.453152027f, kA5 = 1.061405429f;
  const float z = fabsf(x) * 0.70710678118654752f;
  const float t = __fdividef(1.f, fmaf(kP, z, 1.f));
  const float poly = t * fmaf(fmaf(fmaf(fmaf(kA5, t, kA4), t, kA3), t, kA2), t, kA1);
  const float q = poly * __expf(-z * z);
  return 0.5f * x * (x >= 0.f ? 2.f - q : q);
}

// The same GELU epilogue on two accumulator values at once (alpha times the value
// plus the bias, GELU, the output scale), with the fp32 arithmetic on packed pairs:
// half the instructions of two scalar calls, the same results (0.5 x r y_scale is
// taken as (x r)(0.5 y_scale), equal to (0.5 x) r y_scale since halving is exact).
__device__ __forceinline__ void gelu_epilogue_pair(float a0, float a1, float alpha, float b, bool has_bias,
                                                   float y_scale, float& o0, float& o1) {
  constexpr float kP = 0.3275911f, kA1 = 0.254829592f, kA2 = -0.284496736f, kA3 = 1.421413741f,
                  kA4 = -1.453152027f, kA5 = 1.061405429f;
  using namespace ptx;
  const uint64_t acc = f2_pack(a0, a1), al = f2_pack(alpha, alpha);
  const uint64_t x = has_bias ? f2_fma(acc, al, f2_pack(b, b)) : f2_mul(acc, al);
  const uint64_t z = f2_mul(x & 0x7FFFFFFF7FFFFFFFull, f2_pack(0.70710678118654752f, 0.70710678118654752f));
  const uint64_t d = f2_fma(f2_pack(kP, kP), z, f2_pack(1.f, 1.f));
  const uint64_t t = f2_pack(__fdividef(1.f, f2_lo(d)), __fdividef(1.f, f2_hi(d)));
  uint64_t poly = f2_fma(f2_pack(kA5, kA5), t, f2_pack(kA4, kA4));
  poly = f2_fma(poly, t, f2_pack(kA3, kA3));
  poly = f2_fma(poly, t, f2_pack(kA2, kA2));
  poly = f2_fma(poly, t, f2_pack(kA1, kA1));
  poly = f2_mul(poly, t);
  const uint64_t zz = f2_mul(z, z);
  const uint64_t q = f2_mul(poly, f2_pack(__expf(-f2_lo(zz)), __expf(-f2_hi(zz))));
  const float q0 = f2_lo(q), q1 = f2_hi(q);
  const uint64_t r = f2_pack(f2_lo(x) >= 0.f ? 2.f - q0 : q0, f2_hi(x) >= 0.f ? 2.f - q1 : q1);
  const float hs = 0.5f * y_scale;
  const uint64_t o = f2_mul(f2_mul(x, r), f2_pack(hs, hs));
  o0 = f2_lo(o);
  o1 = f2_hi(o);
}

// The fused layer epilogue on one fp32 accumulator value, in this order: alpha
// times the accumulator plus the row's bias (one fma), the activation, the
// output scale.
__device__ __forceinline__ float epilogue_value(float acc, float alpha, float b, bool has_bias, int act,
                                               float y_scale) {
  float x = has_bias ? fmaf(acc, alpha, b) : acc * alpha;  // has_bias is uniform: no divergence
  if (act == 1) {
    x = x > 0.f ? x : 0.f;
  } else if (act == 2) {
    x = gelu_exact(x);
  }
  return x * y_scale;
}

// Rounds 32 consecutive outputs of one row to the output type (ties to even; e4m3
// saturating) and packs them: 16 words of fp16/bf16 pairs, or 8 words of e4m3
// quads (words 8..15 unused).
__device__ __forceinline__ void pack_row32(int out_dt, const float (&x)[32], uint32_t (&w)[16]) {
  if (out_dt == 2) {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const uint32_t lo = __nv_cvt_float2_to_fp8x2(make_float2(x[4 * i], x[4 * i + 1]), __NV_SATFINITE, __NV_E4M3);
      const uint32_t hi =
          __nv_cvt_float2_to_fp8x2(make_float2(x[4 * i + 2], x[4 * i + 3]), __NV_SATFINITE, __NV_E4M3);
      w[i] = (lo & 0xFFFFu) | (hi << 16);
    }
#pragma unroll
    for (int i = 8; i < 16; ++i) w[i] = 0u;
    return;
  }
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    if (out_dt == 1) {
      const __nv_bfloat162 h = __floats2bfloat162_rn(x[2 * i], x[2 * i + 1]);
      w[i] = *reinterpret_cast<const uint32_t*>(&h);
    } else {
      const __half2 h = __floats2half2_rn(x[2 * i], x[2 * i + 1]);
      w[i] = *reinterpret_cast<const uint32_t*>(&h);
    }
  }
}

// Stores 32 packed outputs of one row at columns n0 .. n0 + 31 (those below N).
__device__ __forceinline__ void store_packed_row32(uint8_t* dst_row, int32_t n0, int32_t N, int out_dt,
                                                   const uint32_t (&w)[16], uint64_t pol) {
  if (out_dt == 2) {
    uint8_t* dst = dst_row + n0;
    if (n0 + 32 <= N && (reinterpret_cast<uintptr_t>(dst) & 15u) == 0) {
      ptx::st_global_v4_hint(dst, w[0], w[1], w[2], w[3], pol);
      ptx::st_global_v4_hint(dst + 16, w[4], w[5], w[6], w[7], pol);
    } else {
#pragma unroll
      for (int i = 0; i < 32; ++i)
        if (n0 + i < N) dst[i] = static_cast<uint8_t>(w[i >> 2] >> (8 * (i & 3)));
    }
    return;
  }
  uint16_t* dst = reinterpret_cast<uint16_t*>(dst_row) + n0;
  if (n0 + 32 <= N && (reinterpret_cast<uintptr_t>(dst) & 15u) == 0) {
#pragma unroll
    for (int v = 0; v < 4; ++v)
      ptx::st_global_v4_hint(reinterpret_cast<uint4*>(dst) + v, w[4 * v], w[4 * v + 1], w[4 * v + 2], w[4 * v + 3],
                             pol);
  } else {
#pragma unroll
    for (int i = 0; i < 32; ++i)
      if (n0 + i < N) dst[i] = static_cast<uint16_t>(w[i >> 1] >> (16 * (i & 1)));
  }
}

// The same for the output of a convolution unit, whose columns start at any
// offset of the row (patches of W-wide image rows).
__device__ __forceinline__ void store_packed_row32_any(uint8_t* dst_row, int32_t n0, int32_t N, int out_dt,
                                                       const uint32_t (&w)[16], uint64_t pol) {
  if (out_dt == 2) {
    uint8_t* dst = dst_row + n0;
    const uintptr_t a = reinterpret_cast<uintptr_t>(dst);
    if (n0 + 32 <= N && (a & 15u) == 0) {
      ptx::st_global_v4_hint(dst, w[0], w[1], w[2], w[3], pol);
      ptx::st_global_v4_hint(dst + 16, w[4], w[5], w[6], w[7], pol);
    } else if (n0 + 32 <= N && (a & 3u) == 0) {
#pragma unroll
      for (int k = 0; k < 8; ++k) reinterpret_cast<uint32_t*>(dst)[k] = w[k];
    } else {
#pragma unroll
      for (int i = 0; i < 32; ++i)
        if (n0 + i < N) dst[i] = static_cast<uint8_t>(w[i >> 2] >> (8 * (i & 3)));
    }
    return;
  }
  uint16_t* dst = reinterpret_cast<uint16_t*>(dst_row) + n0;
  const uintptr_t a = reinterpret_cast<uintptr_t>(dst);
  if (n0 + 32 <= N && (a & 15u) == 0) {
#pragma unroll
    for (int v = 0; v < 4; ++v)
      ptx::st_global_v4_hint(reinterpret_cast<uint4*>(dst) + v, w[4 * v], w[4 * v + 1], w[4 * v + 2], w[4 * v + 3],
                             pol);
    return;
  }
  // A column range at another offset (convolution patches of W-wide image rows, a
  // ragged row end): element pairs as 32-bit stores from the first 4-byte boundary
  // on, with a 2-byte store at either end where needed (n0 < N, so cnt >= 1).
  const int32_t cnt = min(32, N - n0);
  if (cnt == 32 && (a & 7u) == 0) {
#pragma unroll
    for (int k = 0; k < 8; ++k) reinterpret_cast<uint2*>(dst)[k] = make_uint2(w[2 * k], w[2 * k + 1]);
  } else if ((a & 2u) == 0) {
#pragma unroll
    for (int k = 0; k < 16; ++k) {
      if (2 * k + 1 < cnt)
        reinterpret_cast<uint32_t*>(dst)[k] = w[k];
      else if (2 * k < cnt)
        dst[2 * k] = static_cast<uint16_t>(w[k]);
    }
  } else {
    dst[0] = static_cast<uint16_t>(w[0]);
    uint32_t* d32 = reinterpret_cast<uint32_t*>(dst + 1);  // elements 2k + 1 and 2k + 2
#pragma unroll
    for (int k = 0; k < 16; ++k) {
      const uint32_t lo = w[k] >> 16, hi = k < 15 ? (w[k + 1] & 0xFFFFu) : 0u;
      if (2 * k + 2 < cnt)
        d32[k] = lo | (hi << 16);
      else if (2 * k + 1 < cnt)
        dst[2 * k + 1] = static_cast<uint16_t>(lo);
    }
  }
}

// Writes 32 packed outputs as row `lane` of a 32 x 32 staging box: 64-byte rows
// with the 64B swizzle (fp16/bf16) or 32-byte rows with the 32B swizzle (e4m3),
// the layouts the output tensor map stores from, without bank conflicts between
// the lanes of a quarter warp.
__device__ __forceinline__ void stage_packed_row32(uint8_t* buf, uint32_t lane, int out_dt, const uint32_t (&w)[16]) {
  if (out_dt == 2) {
    uint8_t* row = buf + lane * 32;
#pragma unroll
    for (int v = 0; v < 2; ++v)
      *reinterpret_cast<uint4*>(row + ((v ^ ((lane >> 2) & 1)) << 4)) =
          make_uint4(w[4 * v], w[4 * v + 1], w[4 * v + 2], w[4 * v + 3]);
    return;
  }
  uint8_t* row = buf + lane * 64;
#pragma unroll
  for (int v = 0; v < 4; ++v)
    *reinterpret_cast<uint4*>(row + ((v ^ ((lane >> 1) & 3)) << 4)) =
        make_uint4(w[4 * v], w[4 * v + 1], w[4 * v + 2], w[4 * v + 3]);
}

template <int DT, bool SPARSE, bool GATHER, int BN, int MT, int BROW, bool PAIR, bool BLOCKW, bool CONV, int KX>
__global__ void __launch_bounds__(Cfg<DT, SPARSE, GATHER, BN, MT, BROW, PAIR, BLOCKW, CONV, KX>::THREADS, 1)
    k_gemm(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
           const __grid_constant__ CUtensorMap tmM, const __grid_constant__ CUtensorMap tmY, const Params p) {
  using C = Cfg<DT, SPARSE, GATHER, BN, MT, BROW, PAIR, BLOCKW, CONV, KX>;
  // SM pairs (PAIR): both CTAs load their own A rows, metadata and B columns, all
  // counted on the even CTA's full barrier; the even CTA's MMA thread issues the
  // M = 256 MMAs and its commits release both CTAs' stages and accumulators; the odd
  // CTA's epilogue releases the accumulator on the even CTA's barrier.
  constexpr int CL = C::CLUSTER;
  const uint32_t crank = (CL > 1) ? ptx::cluster_ctarank() : 0u;
  const bool leader = !PAIR || (crank & 1u) == 0u;
  // Work units are dealt in rounds of one unit per cluster, alternating direction
  // (round r gives unit r S + c to cluster c for even r, r S + S - 1 - c for odd
  // r): with tiles ordered by kept count descending, a cluster that took a long
  // unit in one round takes a short one in the next.
  const int32_t unit_c = static_cast<int32_t>(blockIdx.x) / CL;
  const int32_t unit_S = static_cast<int32_t>(gridDim.x) / CL;
  auto unit_at = [&](int32_t r) -> int32_t {
    const int32_t base = r * unit_S;
    if (base >= p.num_units) return -1;
    const int32_t u = base + ((r & 1) ? unit_S - 1 - unit_c : unit_c);
    return u < p.num_units ? u : -1;
  };
  constexpr uint16_t kMask = static_cast<uint16_t>((1u << CL) - 1u);
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = ptx::smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);
  uint8_t* staging = smem + C::STAGES * C::STAGE_BYTES;
  uint64_t* bars = reinterpret_cast<uint64_t*>(staging + C::STAGING_BYTES);
  uint64_t* full = bars;
  uint64_t* empty = bars + C::STAGES;
  uint64_t* acc_full = bars + 2 * C::STAGES;
  uint64_t* acc_empty = acc_full + C::NACC;
  uint64_t* drain = acc_empty + C::NACC;
  // KX = 2: the X boxes of a stage complete on a second barrier, so that neither
  // barrier expects more than 64 KB per phase
  uint64_t* full_b = drain + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(full_b + (C::B_OWN_BARRIER ? C::STAGES : 0));
  volatile uint32_t* abort_flag = tmem_slot + 1;

  const uint32_t warp = threadIdx.x >> 5;
  const uint32_t lane = threadIdx.x & 31u;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      ptx::mbar_init(&full[s], 1 + C::GATHER_THREADS);
      ptx::mbar_init(&empty[s], 1);
      if constexpr (C::B_OWN_BARRIER) ptx::mbar_init(&full_b[s], 1);
    }
    for (int a = 0; a < C::NACC; ++a) {
      ptx::mbar_init(&acc_full[a], 1);
      ptx::mbar_init(&acc_empty[a], 32 * C::EPI_WARPS * (PAIR ? 2 : 1));
    }
    ptx::mbar_init(drain, 1);
    *abort_flag = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    ptx::prefetch_tmap(&tmA);
    ptx::prefetch_tmap(&tmB);
    if constexpr (PAIR && SPARSE) ptx::prefetch_tmap(&tmM);
  }
  if (warp == 2) {
    if constexpr (PAIR) {
      ptx::tmem_alloc_pair(tmem_slot, C::TMEM_COLS);
      ptx::tmem_relinquish_pair();
    } else {
      ptx::tmem_alloc(tmem_slot, C::TMEM_COLS);
      ptx::tmem_relinquish();
    }
  }
  ptx::tc_fence_before();
  if constexpr (CL > 1)
    ptx::cluster_sync();  // the peer's barriers are initialised before any arrival reaches them
  else
    __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    const uint64_t pol_a = ptx::policy_evict_last();
    const uint64_t pol_b = ptx::policy_evict_normal();
    int stage = 0;
    uint32_t phase = 0;
    int issued = 0;
    bool ok = true;
    for (int32_t r = 0, u = unit_at(0); u >= 0 && ok; u = unit_at(++r)) {
      const UnitInfo ui = decode_unit<C, C::SCHEDULED>(p, u, crank);
      for (int32_t kb = 0; kb < ui.nk; ++kb) {
        if (*abort_flag) { ok = false; break; }
        if (lane == 0) ok = wait_bounded(&empty[stage], phase ^ 1u, p.err);
        ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
        if (!ok) { *abort_flag = 1; break; }
        uint8_t* sA = smem + stage * C::STAGE_BYTES;
        uint8_t* sB = sA + C::A_BYTES;
        uint8_t* sM = sB + C::B_BYTES;
        if (lane == 0) {
          if constexpr (PAIR) {
            // both CTAs' bytes complete on the even CTA's full barrier
            constexpr uint32_t kTx = 2u * (C::A_BYTES + (KX == 2 ? 0 : C::B_BYTES) + C::META_BYTES);
            if (leader) ptx::mbar_arrive_expect_tx(&full[stage], kTx);
            if (KX == 2 && leader) ptx::mbar_arrive_expect_tx(&full_b[stage], 2u * C::B_BYTES);
            const uint32_t bar = ptx::mapa(ptx::smem_u32(&full[stage]), crank & ~1u);
            const uint32_t bar_b = KX == 2 ? ptx::mapa(ptx::smem_u32(&full_b[stage]), crank & ~1u) : bar;
            // the X panel, the stage's largest copy, first
            const int32_t n_half = ui.n0 + static_cast<int32_t>(crank & 1u) * C::BN_CTA;
            if (C::B_BOXES > 1 && p.b3d) {
              // all of this CTA's B boxes of the stage as one 3-D box: the layout
              // [64-column block][K row][128 B] is the boxes' layout, B_BOX_BYTES apart
              ptx::tma_load_3d_pair(sB, &tmB, bar_b, 0, kb * C::BK, n_half / C::B_BOX_COLS, pol_b);
            } else {
#pragma unroll
              for (int bx = 0; bx < C::B_BOXES; ++bx)
                ptx::tma_load_2d_pair(sB + bx * C::B_BOX_BYTES, &tmB, bar_b, n_half + bx * C::B_BOX_COLS,
                                      kb * C::BK, pol_b);
            }
            ptx::tma_load_2d_pair(sA, &tmA, bar, kb * (SPARSE ? C::BK / 2 : C::BK), ui.m0, pol_a);
            if constexpr (SPARSE)  // one metadata block; past the last row block it reads zeros
              ptx::tma_load_2d_pair(sM, &tmM, bar, 0, (ui.meta_blk0 + KX * kb) * 16, pol_a);
          } else {
          // 2:4 metadata blocks of the stage (KX per sub-tile; the last stage of a row
          // block may cover only one of two)
          const int32_t meta_n = SPARSE ? min(KX, p.meta_kb - KX * kb) : 0;
          ptx::mbar_arrive_expect_tx(&full[stage], C::A_BYTES +
                                                       (GATHER ? 0u : (CONV ? KX * p.conv_box_bytes : C::B_BYTES)) +
                                                       static_cast<uint32_t>(2048 * meta_n * ui.subs));
          // the X operand first (the stage's largest copy), then A and the metadata
          if constexpr (CONV) {
            // tap (r, s) and 64 input channels of each K step of stage kb, for the patch's
            // image rows shifted by the tap (out-of-range rows and columns read as zeros)
            // (tile-wise filter: the kb-th kept (tap, 64-channel) group of the tile)
            const int32_t cblocks = p.conv_cin / 64;
#pragma unroll
            for (int x = 0; x < KX; ++x) {
              const int32_t g = BLOCKW ? __ldg(p.indices + ui.idx_base + kb) : KX * kb + x;
              const int32_t tap = g / cblocks, c0 = (g - tap * cblocks) * 64;
              const int32_t r = tap / 3, sx = tap - 3 * r;
              ptx::tma_load_4d(sB + x * (C::B_BYTES / KX), &tmB, &full[stage], c0, sx - 1, ui.h0 + r - 1, ui.img,
                               pol_b);
            }
          } else if constexpr (!GATHER) {
            // block-wise: the X panel of the kb-th kept block of this tile
            const int32_t krow = BLOCKW ? __ldg(p.indices + ui.idx_base + kb) * C::BK : kb * C::BK;
#pragma unroll
            for (int bx = 0; bx < C::B_BOXES; ++bx)
              ptx::tma_load_2d(sB + bx * C::B_BOX_BYTES, &tmB, &full[stage], ui.n0 + bx * C::B_BOX_COLS, krow,
                               pol_b);
          }
          // A: dense W / 2:4 values / packed tile box (inner coordinate in elements);
          // rows past M read as zeros
          const int32_t a_col = C::SCHEDULED ? 0 : kb * (SPARSE ? C::BK / 2 : C::BK);
          const int32_t a_row = C::SCHEDULED ? ui.a_row0 + 128 * kb : ui.m0;
          ptx::tma_load_2d(sA, &tmA, &full[stage], a_col, a_row, pol_a);
          if constexpr (SPARSE) {
            for (int mt = 0; mt < ui.subs; ++mt) {
              // sub-tile mt's blocks follow the row block's meta_kb blocks (TW/TVW tiles: nk)
              const int32_t stride = C::SCHEDULED ? ui.nk : p.meta_kb;
              const uint8_t* src = p.meta_hw + static_cast<int64_t>(ui.meta_blk0 + mt * stride + KX * kb) * 2048;
              ptx::bulk_load(sM + mt * 2048 * KX, src, static_cast<uint32_t>(2048 * meta_n), &full[stage], pol_a);
            }
          }
          }
        }
        __syncwarp();
        ++issued;
        if (++stage == p.nstages) { stage = 0; phase ^= 1u; }
      }
    }
    if (ok && lane == 0) {
      // Tail: every stage this CTA filled has been released by all consumers of
      // the cluster, so no remote arrival or multicast write is still due here.
      int s = stage;
      uint32_t ph = phase;
      const int pending = issued < p.nstages ? issued : p.nstages;
      for (int n = 0; n < pending; ++n) {
        if (--s < 0) { s = p.nstages - 1; ph ^= 1u; }
        wait_bounded(&empty[s], ph, p.err);
      }
    }
    // On abort, wait (bounded) for the copies still in flight before exiting.
    if (!ok && lane == 0) {
      int s = stage;
      uint32_t ph = phase;
      const int pending = issued < p.nstages ? issued : p.nstages;
      for (int n = 0; n < pending; ++n) {
        if (--s < 0) { s = p.nstages - 1; ph ^= 1u; }
        wait_bounded(&full[s], ph, nullptr);
        if constexpr (C::B_OWN_BARRIER) wait_bounded(&full_b[s], ph, nullptr);
      }
    }
  } else if (warp == 1 && leader) {
    // ------------------------------------------------------------ MMA issuer
    // (of an SM pair, only the even CTA issues)
    int stage = 0;
    uint32_t phase = 0;
    int acc = 0;
    uint32_t acc_phase = 0;
    int meta_slot = 0;
    bool ok = true;
    for (int32_t r = 0, u = unit_at(0); u >= 0 && ok; u = unit_at(++r)) {
      const UnitInfo ui = decode_unit<C, C::SCHEDULED>(p, u, crank);
      if (lane == 0) ok = wait_bounded(&acc_empty[acc], acc_phase ^ 1u, p.err);
      ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
      if (!ok || *abort_flag) { *abort_flag = 1; ok = false; break; }
      ptx::tc_fence_after();
      const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * C::ACC_COLS);
      uint32_t cur_meta = 0;
      for (int32_t kb = 0; kb < ui.nk; ++kb) {
        if (lane == 0) ok = wait_bounded(&full[stage], phase, p.err);
        if (C::B_OWN_BARRIER && lane == 0 && ok) ok = wait_bounded(&full_b[stage], phase, p.err);
        ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
        if (!ok) { *abort_flag = 1; break; }
        // TW/TVW: the gathered rows were written by cp.async (generic proxy); order them
        // before the tensor core's reads (async proxy)
        if constexpr (GATHER) ptx::fence_proxy_async_smem();
        ptx::tc_fence_after();
        if (lane == 0) {
          const uint32_t sA = ptx::smem_u32(smem + stage * C::STAGE_BYTES);
          const uint32_t sB = sA + C::A_BYTES;
          if constexpr (SPARSE) {
            const uint32_t sM = sB + C::B_BYTES;
            cur_meta = tmem_base + C::META_COL0 + static_cast<uint32_t>(C::META_SLOT_COLS * meta_slot);
            meta_slot = (meta_slot + 1) % C::META_SLOTS;
            // per sub-tile: 128 rows x 16 B, rows contiguous (8-row core matrices 128 B apart)
#pragma unroll
            for (int mt = 0; mt < MT * KX; ++mt) {  // sub-tiles, or (KX = 2) the stage's two K steps
              if constexpr (PAIR)  // each CTA's block into its own TMEM
                ptx::tmem_cp_128x128b_pair(cur_meta + 4u * mt, ptx::sdesc(sM + 2048u * mt, 128, 128, 0));
              else
                ptx::tmem_cp_128x128b(cur_meta + 4u * mt, ptx::sdesc(sM + 2048u * mt, 128, 128, 0));
            }
          }
#pragma unroll
          for (int j = 0; j < C::MMAS; ++j)
#pragma unroll
          for (int mt = 0; mt < MT; ++mt) {
            const uint32_t accum = (kb > 0 || j > 0) ? 1u : 0u;
            // B: MN-major boxes, or (convolution) K-major pixel rows of 128 bytes
            // (KX = 2: the stage's second K step in the second box)
            constexpr int kJPS = C::MMAS / KX;  // instructions per K step
            const uint64_t bdesc =
                CONV ? ptx::sdesc(sB + (j / kJPS) * (C::B_BYTES / KX) + (j % kJPS) * C::MMA_K * C::EB, 16, 1024, 2)
                     : ptx::sdesc(sB + j * C::MMA_K * C::B_ROW, C::B_BOX_BYTES, C::B_SBO, C::B_SWZ);
            const uint32_t d_sub = d_tmem + static_cast<uint32_t>(mt * BN);
            const uint32_t a_sub = sA + static_cast<uint32_t>(mt * C::A_SUB_BYTES);
            if constexpr (SPARSE) {
              // 64-byte rows, 64B swizzle; (KX = 2) 128-byte rows, 128B swizzle
              const uint64_t adesc = KX == 1 ? ptx::sdesc(a_sub + j * 32, 16, 512, 4)
                                             : ptx::sdesc(a_sub + j * 32, 16, 1024, 2);
              // the metadata of instruction j starts at column 2 j of the stage's
              // 4 KX (the sparse MMA reads it from an even column: one column for a
              // 16-bit K = 32 step, two for an e4m3 K = 64 step)
              const uint32_t col = 4u * KX * mt + 2u * j;
              if constexpr (PAIR && C::F8)
                ptx::mma_sp_f8_pair(d_sub, adesc, bdesc, cur_meta + col, C::IDESC, accum);
              else if constexpr (PAIR)
                ptx::mma_sp_f16_pair(d_sub, adesc, bdesc, cur_meta + col, C::IDESC, accum);
              else if constexpr (C::F8)
                ptx::mma_sp_f8(d_sub, adesc, bdesc, cur_meta + col, C::IDESC, accum);
              else
                ptx::mma_sp_f16(d_sub, adesc, bdesc, cur_meta + col, C::IDESC, accum);
            } else {
              const uint64_t adesc = ptx::sdesc(a_sub + j * 32, 16, 1024, 2);
              if constexpr (PAIR && C::F8)
                ptx::mma_f8_pair(d_sub, adesc, bdesc, C::IDESC, accum);
              else if constexpr (PAIR)
                ptx::mma_f16_pair(d_sub, adesc, bdesc, C::IDESC, accum);
              else if constexpr (C::F8)
                ptx::mma_f8(d_sub, adesc, bdesc, C::IDESC, accum);
              else
                ptx::mma_f16(d_sub, adesc, bdesc, C::IDESC, accum);
            }
          }
          if constexpr (PAIR)
            ptx::mma_commit_pair_multicast(&empty[stage], kMask);
          else
            ptx::mma_commit(&empty[stage]);
        }
        __syncwarp();
        if (++stage == p.nstages) { stage = 0; phase ^= 1u; }
      }
      if (!ok) break;
      if (lane == 0) {
        if constexpr (PAIR)
          ptx::mma_commit_pair_multicast(&acc_full[acc], kMask);
        else
          ptx::mma_commit(&acc_full[acc]);
      }
      __syncwarp();
      if (++acc == C::NACC) { acc = 0; acc_phase ^= 1u; }
    }
    // Make sure no MMA is still writing TMEM when the allocation is released.
    if (lane == 0) {
      if constexpr (PAIR)
        ptx::mma_commit_pair(drain);
      else
        ptx::mma_commit(drain);
      wait_bounded(drain, 0, nullptr);
    }
    __syncwarp();
  } else if (GATHER && warp >= C::GATHER_WARP0) {
    // ------------------------------------------------------------ X-row gather (TW/TVW)
    // Gather warp w copies stage rows r = GW i + w (i < 64 / GW). Lanes take consecutive
    // 16-byte chunks of a row (a warp instruction copies 512 contiguous bytes of X:
    // one row for a 256-wide N tile, two rows for 128), straight into the
    // 128B-swizzled MN-major operand layout; rows past L_t and columns past N are
    // zero-filled. Each thread's copies of a stage complete on the stage's full
    // barrier by themselves (cp.async.mbarrier.arrive), so the gather runs ahead
    // by the whole ring; the MMA thread fences them for the tensor core's async
    // proxy after its wait.
    const int w = warp - C::GATHER_WARP0;
    constexpr int CPR = BN / 8;                      // 16-byte chunks per row
    constexpr int RPI = 32 / CPR;                    // rows per warp instruction
    constexpr int GW = C::GATHER_WARPS;
    constexpr int ROWS_W = 64 / GW;                  // stage rows per gather warp
    constexpr int ITERS = ROWS_W / RPI;              // instructions per stage
    const int sub = static_cast<int>(lane) / CPR, q = static_cast<int>(lane) % CPR;
    const int col = 8 * q;                           // column within the N tile
    const int bx = col >> 6, cc = (col & 63) >> 3;   // 64-column box, 16-byte chunk in its row
    constexpr int kIdxAhead = 3;
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    const uint16_t* X = static_cast<const uint16_t*>(p.X);
    int32_t idx_ring[kIdxAhead];                     // lane l < ROWS_W: X row of stage row GW l + w
    for (int32_t r = 0, u = unit_at(0); u >= 0 && ok; u = unit_at(++r)) {
      const UnitInfo ui = decode_unit<C, C::SCHEDULED>(p, u, crank);
      const int32_t gcol = ui.n0 + col;
      const uint32_t col_bytes = gcol >= p.N ? 0u : static_cast<uint32_t>(min(8, p.N - gcol) * 2);
      auto row_of = [&](int32_t kb) -> int32_t {
        const int32_t j = kb * C::BK + GW * static_cast<int32_t>(lane) + w;
        return (lane < ROWS_W && kb < ui.nk && j < ui.L) ? __ldg(p.indices + ui.idx_base + j) : -1;
      };
#pragma unroll
      for (int d = 0; d < kIdxAhead; ++d) idx_ring[d] = row_of(d);
      for (int32_t kb = 0; kb < ui.nk; ++kb) {
        if (*abort_flag) { ok = false; break; }
        if (lane == 0) ok = wait_bounded(&empty[stage], phase ^ 1u, p.err);
        ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
        if (!ok) { *abort_flag = 1; break; }
        uint8_t* sB = smem + stage * C::STAGE_BYTES + C::A_BYTES;
#pragma unroll
        for (int i = 0; i < ITERS; ++i) {
          const int ri = i * RPI + sub;              // warp-local row 0 .. ROWS_W - 1
          const int r = GW * ri + w;                 // stage row 0..63
          const int32_t xrow = __shfl_sync(0xffffffffu, idx_ring[0], ri);
          const uint32_t bytes = xrow < 0 ? 0u : col_bytes;
          const uint16_t* src = bytes ? X + static_cast<int64_t>(xrow) * p.ldx + gcol : X;
          ptx::cp_async_16(sB + bx * C::B_BOX_BYTES + r * 128 + ((cc ^ (r & 7)) << 4), src, bytes);
        }
        ptx::cp_async_mbar_arrive_noinc(&full[stage]);
#pragma unroll
        for (int d = 0; d + 1 < kIdxAhead; ++d) idx_ring[d] = idx_ring[d + 1];
        idx_ring[kIdxAhead - 1] = row_of(kb + kIdxAhead);
        if (++stage == p.nstages) { stage = 0; phase ^= 1u; }
      }
    }
    ptx::cp_async_wait<0>();  // no copy of this thread is still writing shared memory
  } else if (warp >= C::EPI_WARP0 && warp < C::EPI_WARP0 + C::EPI_WARPS) {
    // ------------------------------------------------------------ epilogue
    const uint32_t q = warp & 3u;                 // TMEM lane quadrant this warp may read
    const uint32_t mt = PAIR ? 0u : (warp - 4u) >> 2;  // sub-tile this warp drains
    const int half = PAIR ? static_cast<int>((warp - 4u) >> 2) : 0;  // column half (SM pairs)
    const uint64_t pol_y = ptx::policy_evict_first();  // the output is not re-read here
    uint32_t chunk_seq = 0;                            // staging buffer alternation
    const bool plain_epilogue = p.bias == nullptr && p.act == 0 && p.y_scale == 1.0f;
    int acc = 0;
    uint32_t acc_phase = 0;
    bool ok = true;
    for (int32_t r = 0, u = unit_at(0); u >= 0 && ok; u = unit_at(++r)) {
      const UnitInfo ui = decode_unit<C, C::SCHEDULED>(p, u, crank);
      ok = wait_bounded(&acc_full[acc], acc_phase, p.err);
      if (!ok || *abort_flag) { *abort_flag = 1; break; }
      ptx::tc_fence_after();
      const int32_t row = ui.m0 + static_cast<int32_t>(128 * mt + 32 * q + lane);
      const bool row_ok = row < p.M && !ui.phantom;
      uint8_t* yrow = p.Y + static_cast<int64_t>(row) * p.ldy * (p.out_dt == 2 ? 1 : 2);
      const bool has_bias = p.bias != nullptr;
      const float bias = (has_bias && row_ok) ? __ldg(p.bias + row) : 0.f;
      constexpr int NCH = BN / 32 / C::EPI_SPLIT;   // 32-column chunks this warp drains
      const int c0 = half * NCH;
      const bool ragged_end = ((p.N * (p.out_dt == 2 ? 1 : 2)) & 15) != 0;
      const int32_t wrow0 = ui.m0 + static_cast<int32_t>(128 * mt + 32 * q);
      // chunk c of this warp's rows: TMEM -> raw fp32 accumulator bits (call
      // tmem_ld_wait before using them)
      auto load_chunk = [&](int c, uint32_t (&r)[32]) {
        if (ui.nk > 0) {
          ptx::tmem_ld_32x32b_x32(
              tmem_base + ((32u * q) << 16) + static_cast<uint32_t>(acc * C::ACC_COLS + mt * BN + 32 * c), r);
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) r[i] = 0u;
        }
      };
      // raw accumulator bits -> fp32 epilogue -> packed output words
      auto convert_raw = [&](const uint32_t (&r)[32], uint32_t (&w)[16]) {
        float x[32];
        // the activation is chosen once per chunk, so each branch is straight-line
        // code over 32 independent values
        if (plain_epilogue) {  // no bias, no activation, no output scale: one multiply
#pragma unroll
          for (int i = 0; i < 32; ++i) x[i] = __uint_as_float(r[i]) * p.alpha;
        } else if (p.act == 2) {
#pragma unroll
          for (int i = 0; i < 32; i += 2)
            gelu_epilogue_pair(__uint_as_float(r[i]), __uint_as_float(r[i + 1]), p.alpha, bias, has_bias, p.y_scale,
                               x[i], x[i + 1]);
        } else if (p.act == 1) {
#pragma unroll
          for (int i = 0; i < 32; ++i) x[i] = epilogue_value(__uint_as_float(r[i]), p.alpha, bias, has_bias, 1, p.y_scale);
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) x[i] = epilogue_value(__uint_as_float(r[i]), p.alpha, bias, has_bias, 0, p.y_scale);
        }
        pack_row32(p.out_dt, x, w);
      };
      // this warp's part of the accumulator has been read (its tcgen05.ld have
      // completed: tmem_ld_wait precedes every call): release it
      auto release = [&]() {
        ptx::tc_fence_before();
        if (leader)
          ptx::mbar_arrive(&acc_empty[acc]);
        else  // the odd CTA of a pair releases its rows on the even CTA's barrier. The
              // arrive is relaxed: the reads it signals are complete, and with
              // release semantics at cluster scope the arrive took about 0.4 us longer
              // per tile
          ptx::mbar_arrive_cluster_relaxed(ptx::mapa(ptx::smem_u32(&acc_empty[acc]), crank & ~1u));
      };
      auto store_chunk = [&](int c, const uint32_t (&w)[16]) {
        const int32_t n0 = ui.n0 + 32 * c;
        if constexpr (C::STAGED) {
          if (p.y_direct) {  // host-memory output: each thread stores its row's chunk
            if (row_ok && n0 < p.N) store_packed_row32(yrow, n0, p.N, p.out_dt, w, pol_y);
            return;
          }
          // this warp's 32 rows x 32 columns go through a staging buffer and a TMA
          // store, which clips rows past M and columns past N
          if (ui.phantom || wrow0 >= p.M || n0 >= p.N) return;  // uniform over the warp
          if (ragged_end && n0 + 32 > p.N) {
            // a row end that is not a multiple of 16 bytes: the copy engine writes
            // whole 16-byte units there, so that chunk is stored directly
            if (row_ok) store_packed_row32(yrow, n0, p.N, p.out_dt, w, pol_y);
            return;
          }
          uint8_t* buf = staging + (warp - C::EPI_WARP0) * (2048 * C::STAGING_BUFS) +
                         (C::STAGING_BUFS == 2 ? (chunk_seq & 1) * 2048 : 0);
          ++chunk_seq;
          // the store that last used this buffer has read it
          if (lane == 0) {
            if constexpr (C::STAGING_BUFS == 2)
              ptx::bulk_wait_read<1>();
            else
              ptx::bulk_wait_read<0>();
          }
          __syncwarp();
          stage_packed_row32(buf, lane, p.out_dt, w);
          ptx::fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            ptx::tma_store_2d(&tmY, buf, n0, wrow0);
            ptx::bulk_commit();
          }
        } else {
          // convolution patches end at their last valid image row
          const int32_t n_lim = CONV ? ui.n0 + ui.ncols : p.N;
          if (!row_ok || n0 >= n_lim) return;
          if constexpr (CONV)
            store_packed_row32_any(yrow, n0, n_lim, p.out_dt, w, pol_y);
          else
            store_packed_row32(yrow, n0, n_lim, p.out_dt, w, pol_y);
        }
      };
      if constexpr (C::EARLY_RELEASE) {
        // single accumulator: read all of this warp's chunks raw into registers and
        // release the accumulator before the epilogue arithmetic and the stores, so
        // the next tile's MMAs (and the producer behind them) wait only for the
        // TMEM reads
        uint32_t raw[NCH][32];
#pragma unroll
        for (int i = 0; i < NCH; ++i) load_chunk(c0 + i, raw[i]);
        ptx::tmem_ld_wait();
        release();
        // the epilogue arithmetic starts after the release: the raw values pass through
        // an (empty) volatile asm placed after it, so the compiler cannot hoist the
        // arithmetic above the release
#pragma unroll
        for (int i = 0; i < NCH; ++i)
#pragma unroll
          for (int j = 0; j < 32; ++j) asm volatile("" : "+r"(raw[i][j]));
#pragma unroll
        for (int i = 0; i < NCH; ++i) {
          uint32_t w[16];
          convert_raw(raw[i], w);
          store_chunk(c0 + i, w);
        }
      } else {
#pragma unroll 1
        for (int c = c0; c < c0 + NCH; ++c) {
          uint32_t r[32], w[16];
          load_chunk(c, r);
          ptx::tmem_ld_wait();
          if (c == c0 + NCH - 1) release();
          convert_raw(r, w);
          store_chunk(c, w);
        }
      }
      if (++acc == C::NACC) { acc = 0; acc_phase ^= 1u; }
    }
    if constexpr (C::STAGED) {
      if (lane == 0) ptx::bulk_wait<0>();  // this warp's output stores have completed
      __syncwarp();
    }
  }

  ptx::tc_fence_before();
  if constexpr (PAIR)
    ptx::cluster_sync();  // the even CTA's MMAs into both CTAs' TMEM have drained
  else
    __syncthreads();
  if (warp == 2) {
    ptx::tc_fence_after();
    if constexpr (PAIR)
      ptx::tmem_dealloc_pair(tmem_base, C::TMEM_COLS);
    else
      ptx::tmem_dealloc(tmem_base, C::TMEM_COLS);
  }
}

// ------------------------------------------------------------------ host side
}  // namespace

// (The tensor-map encoder and the 2-D map are shared with the other kernel files.)
using EncodeFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                              const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                              CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeFn encode_fn() {
  static EncodeFn fn = nullptr;
  if (!fn) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeFn>(ptr);
  }
  return fn;
}

// 2-D tensor map over a row-major matrix (rows x cols elements, pitch in bytes).
bool make_map(CUtensorMap* m, const void* base, int eb, uint64_t cols, uint64_t rows, uint64_t pitch_bytes,
              uint32_t box_cols, uint32_t box_rows, CUtensorMapSwizzle swz) {
  EncodeFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {pitch_bytes};
  const cuuint32_t box[2] = {box_cols, box_rows};
  const cuuint32_t es[2] = {1, 1};
  const CUresult r = fn(m, eb == 2 ? CU_TENSOR_MAP_DATA_TYPE_UINT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8, 2,
                        const_cast<void*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

namespace {

// 4-D tensor map over NHWC activations seen innermost-first as (C, W, H, N),
// one box = 64 channels x box_w columns x box_h rows x 1 image, 128B swizzle.
bool make_map_nhwc(CUtensorMap* m, const void* base, uint64_t C_, uint64_t W_, uint64_t H_, uint64_t N_,
                   uint32_t box_w, uint32_t box_h) {
  EncodeFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[4] = {C_, W_, H_, N_};
  const cuuint64_t strides[3] = {C_ * 2, W_ * C_ * 2, H_ * W_ * C_ * 2};
  const cuuint32_t box[4] = {64, box_w, box_h, 1};
  const cuuint32_t es[4] = {1, 1, 1, 1};
  const CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT16, 4, const_cast<void*>(base), dims, strides, box, es,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// 3-D tensor map over a row-major 16-bit matrix of K rows seen as (64 columns,
// K rows, nblk 64-column blocks) -- strides row pitch and 128 bytes -- with boxes of
// 64 x box_rows x box_blks, 128B swizzle: one box lands as box_blks 64-column boxes
// of box_rows 128-byte rows, one after another.
bool make_map_3d_blocks(CUtensorMap* m, const void* base, uint64_t rows, uint64_t nblk, uint64_t pitch_bytes,
                        uint32_t box_rows, uint32_t box_blks) {
  EncodeFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[3] = {64, rows, nblk};
  const cuuint64_t strides[2] = {pitch_bytes, 128};
  const cuuint32_t box[3] = {64, box_rows, box_blks};
  const cuuint32_t es[3] = {1, 1, 1};
  const CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT16, 3, const_cast<void*>(base), dims, strides, box, es,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

int sm_count() {
  int dev = 0, n = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
  return n > 0 ? n : 1;
}

template <int DT, bool SPARSE, bool GATHER, int BN, int MT = 1, int BROW = 128, bool PAIR = false,
          bool BLOCKW = false, bool CONV = false, int KX = 1>
cudaError_t run(const GemmArgs& a, cudaStream_t s, uint32_t* err) {
  using C = Cfg<DT, SPARSE, GATHER, BN, MT, BROW, PAIR, BLOCKW, CONV, KX>;
  const int eb = C::EB;
  CUtensorMap tA, tB, tM;
  bool ok;
  bool b3d = false;
  int32_t conv_rows = 0;
  if constexpr (CONV) {
    // A as for the 2:4 / dense GEMM over the flattened filter; X as NHWC boxes of
    // BN / W whole image rows
    conv_rows = static_cast<int32_t>(BN / a.conv_w);
    if constexpr (BLOCKW)  // tile-wise filter: the packed kept groups seen as (packed_rows x 64)
      ok = make_map(&tA, a.A, eb, 64, a.packed_rows, 128, 64, 128, CU_TENSOR_MAP_SWIZZLE_128B);
    else if constexpr (SPARSE && KX == 2)  // two K steps: 128-byte rows of compressed values
      ok = make_map(&tA, a.A, eb, static_cast<uint64_t>(a.K / 2), a.M, a.lda * eb, 128 / eb, C::BM,
                    CU_TENSOR_MAP_SWIZZLE_128B);
    else if constexpr (SPARSE)
      ok = make_map(&tA, a.A, eb, static_cast<uint64_t>(a.K / 2), a.M, a.lda * eb, 64 / eb, C::BM,
                    CU_TENSOR_MAP_SWIZZLE_64B);
    else
      ok = make_map(&tA, a.A, eb, a.K, a.M, a.lda * eb, 128 / eb, C::BM, CU_TENSOR_MAP_SWIZZLE_128B);
    ok = ok && conv_rows >= 1 &&
         make_map_nhwc(&tB, a.X, a.conv_cin, a.conv_w, a.conv_h, a.conv_nb, static_cast<uint32_t>(a.conv_w),
                       static_cast<uint32_t>(conv_rows));
  } else if constexpr (BLOCKW) {
    // the packed kept blocks seen as (packed_rows x 64); X as for the dense GEMM
    ok = make_map(&tA, a.A, eb, 64, a.packed_rows, 128, 64, 128, CU_TENSOR_MAP_SWIZZLE_128B);
    ok = ok && make_map(&tB, a.X, eb, a.N, a.K, a.ldx * eb, C::B_BOX_COLS, C::BK,
                        CU_TENSOR_MAP_SWIZZLE_128B);
  } else if constexpr (!GATHER) {
    if constexpr (SPARSE && KX == 2)
      ok = make_map(&tA, a.A, eb, static_cast<uint64_t>(a.K / 2), a.M, a.lda * eb, 128 / eb, C::BM,
                    CU_TENSOR_MAP_SWIZZLE_128B);
    else if constexpr (SPARSE)
      ok = make_map(&tA, a.A, eb, static_cast<uint64_t>(a.K / 2), a.M, a.lda * eb, 64 / eb, C::BM,
                    CU_TENSOR_MAP_SWIZZLE_64B);
    else
      ok = make_map(&tA, a.A, eb, a.K, a.M, a.lda * eb, 128 / eb, C::BM, CU_TENSOR_MAP_SWIZZLE_128B);
    if (PAIR && C::B_BOXES > 1 && BROW == 128 && a.N % C::B_BOX_COLS == 0) {
      // X seen as (64 columns, K rows, N / 64 blocks): one box per stage brings all of
      // this CTA's B boxes; every element it addresses lies inside the matrix
      b3d = ok && make_map_3d_blocks(&tB, a.X, a.K, a.N / C::B_BOX_COLS, a.ldx * eb, C::BK, C::B_BOXES);
    }
    if (!b3d) {
      ok = ok && make_map(&tB, a.X, eb, a.N, a.K, a.ldx * eb, C::B_BOX_COLS, C::BK,
                          BROW == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B);
    }
  } else {
    // packed operand seen as (packed_rows x 64) dense or (packed_rows x 32) values
    if constexpr (SPARSE)
      ok = make_map(&tA, a.A, eb, 32, a.packed_rows, 64, 32, 128, CU_TENSOR_MAP_SWIZZLE_64B);
    else
      ok = make_map(&tA, a.A, eb, 64, a.packed_rows, 128, 64, 128, CU_TENSOR_MAP_SWIZZLE_128B);
    ok = ok && make_map(&tB, a.X, eb, a.N, a.K, a.ldx * eb, 128 / eb, 1, CU_TENSOR_MAP_SWIZZLE_128B);
  }
  if constexpr (PAIR && SPARSE) {
    // the 2048-byte metadata blocks as a (blocks * 16) x 128-byte matrix: one 16-row
    // box per stage (long rows: the copy engine's cost grows with the rows of a box)
    const uint64_t rows = static_cast<uint64_t>(ceil_div(a.M, 128)) * ceil_div(a.K, 128 / eb) * 16;
    ok = ok && make_map(&tM, a.meta_hw, 1, 128, rows, 128, 128, 16 * KX, CU_TENSOR_MAP_SWIZZLE_NONE);
  } else {
    tM = tA;  // unused
  }
  // Y in page-locked host memory is written by plain stores from the epilogue (the
  // copy engine is not used on host memory); other host memory is refused.
  bool y_host = false;
  {
    cudaPointerAttributes attr{};
    if (cudaPointerGetAttributes(&attr, a.Y) != cudaSuccess) {
      (void)cudaGetLastError();
      return cudaErrorInvalidValue;
    }
    if (attr.type == cudaMemoryTypeUnregistered) return cudaErrorInvalidValue;
    y_host = attr.type == cudaMemoryTypeHost;
    for (const void* in : {a.A, a.X, static_cast<const void*>(a.meta_hw)}) {
      if (!in) continue;
      if (cudaPointerGetAttributes(&attr, in) != cudaSuccess) {
        (void)cudaGetLastError();
        return cudaErrorInvalidValue;
      }
      if (attr.type == cudaMemoryTypeHost || attr.type == cudaMemoryTypeUnregistered) return cudaErrorInvalidValue;
    }
  }
  CUtensorMap tY;
  if (C::STAGED && !y_host) {
    // the output as 32 x 32 boxes (64-byte rows with the 64B swizzle; e4m3: 32-byte rows, 32B swizzle)
    const bool f8_out = a.out_dt == SSDNN_E4M3;
    ok = ok && make_map(&tY, a.Y, f8_out ? 1 : 2, a.N, a.M, a.ldy * (f8_out ? 1 : 2), 32, 32,
                        f8_out ? CU_TENSOR_MAP_SWIZZLE_32B : CU_TENSOR_MAP_SWIZZLE_64B);
  } else {
    tY = tA;  // unused
  }
  if (!ok) return cudaErrorInvalidValue;

  Params p{};
  p.M = static_cast<int32_t>(a.M);
  p.N = static_cast<int32_t>(a.N);
  p.MB = static_cast<int32_t>(ceil_div(a.M, C::BM));
  p.MB128 = static_cast<int32_t>(ceil_div(a.M, 128));
  p.NB = static_cast<int32_t>(ceil_div(a.N, BN));
  p.MG = static_cast<int32_t>(ceil_div(p.MB, C::CLUSTER));
  {
    // bands of at most ~32 M groups, balanced
    const int64_t bands = ceil_div(p.MG, 32);
    p.GR = static_cast<int32_t>(ceil_div(p.MG, bands));
  }
  p.nk = static_cast<int32_t>(ceil_div(a.K, C::BK));
  p.meta_kb = static_cast<int32_t>(ceil_div(a.K, 128 / eb));
  p.num_units = C::SCHEDULED ? static_cast<int32_t>(a.nt) * p.NB : p.MG * p.NB;
  if constexpr (CONV) {
    p.conv_cin = static_cast<int32_t>(a.conv_cin);
    p.conv_h = static_cast<int32_t>(a.conv_h);
    p.conv_w = static_cast<int32_t>(a.conv_w);
    p.conv_rows = conv_rows;
    p.conv_patches = static_cast<int32_t>(ceil_div(a.conv_h, conv_rows));
    p.conv_box_bytes = static_cast<uint32_t>(128 * conv_rows * a.conv_w);
    p.conv_nb = static_cast<int32_t>(a.conv_nb);
    p.num_units = (BLOCKW ? static_cast<int32_t>(a.nt) : p.MB) * p.conv_nb * p.conv_patches;
  }
  p.out_dt = a.out_dt == SSDNN_BF16 ? 1 : (a.out_dt == SSDNN_E4M3 ? 2 : 0);
  p.act = a.act;
  p.bias = a.bias;
  p.y_scale = a.y_scale;
  p.nstages = C::STAGES;
  p.alpha = a.alpha;
  p.meta_hw = a.meta_hw;
  p.schedule = a.schedule;
  p.offsets = a.offsets;
  p.indices = a.indices;
  p.X = a.X;
  p.ldx = a.ldx;
  p.Y = static_cast<uint8_t*>(a.Y);
  p.ldy = a.ldy;
  p.err = err;
  p.y_direct = y_host ? 1 : 0;
  p.b3d = b3d ? 1 : 0;
  if (p.num_units == 0) return cudaSuccess;

  auto kern = k_gemm<DT, SPARSE, GATHER, BN, MT, BROW, PAIR, BLOCKW, CONV, KX>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  constexpr int CL = C::CLUSTER;
  if constexpr (CL == 1) {
    const int grid = std::min(p.num_units, sm_count());
    kern<<<grid, C::THREADS, C::SMEM_BYTES, s>>>(tA, tB, tM, tY, p);
    return cudaGetLastError();
  } else {
    if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 0)) != cudaSuccess)
      return e;
    cudaLaunchConfig_t cfg{};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = CL;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cfg.blockDim = dim3(C::THREADS, 1, 1);
    cfg.dynamicSmemBytes = C::SMEM_BYTES;
    cfg.stream = s;
    // persistent: as many clusters as can be resident at once, at most one per work item
    cfg.gridDim = dim3(static_cast<unsigned>(sm_count() / CL * CL), 1, 1);
    int max_clusters = 0;
    if ((e = cudaOccupancyMaxActiveClusters(&max_clusters, kern, &cfg)) != cudaSuccess) return e;
    if (max_clusters < 1) return cudaErrorInvalidConfiguration;
    const int clusters = std::min(p.num_units, max_clusters);
    cfg.gridDim = dim3(static_cast<unsigned>(clusters * CL), 1, 1);
    return cudaLaunchKernelEx(&cfg, kern, tA, tB, tM, tY, p);
  }
}

// Tile choice by a fill-rate model: a CTA's time is its stage count times the
// bytes one stage brings into shared memory, and the kernel's time is the number
// of waves of CTAs (persistent, one per SM) times that. Candidates are
// (sub-tiles of 128 rows, N tile).
struct TileChoice {
  int mt, bn;
  bool pair;  // an SM pair (two CTAs, M = 256 MMAs) per 256 x bn tile
};
TileChoice choose_tile(bool sparse, int eb, int64_t M, int64_t N) {
  // 16-bit inputs also have 128x64 tiles, which give small-M shapes (a BERT FFN
  // down projection: 768 rows) twice the work units of 128x128
  // dense: large problems run on SM pairs (256 x 256 tiles, double-buffered accumulator)
  const TileChoice dense_c[] = {{1, 64, false}, {1, 128, false}, {1, 256, false}, {1, 256, true}};
  // 16-bit 2:4: SM pairs also for mid-size shapes (a BERT FFN up projection, 3072 x
  // 1024 x 768: 14.3 us on pairs against 16.4 on 128 x 256 tiles)
  const TileChoice sp16_c[] = {{1, 64, false}, {1, 128, false}, {1, 256, false}, {2, 192, false}, {1, 256, true}};
  // e4m3 2:4: SM-pair 256x256 tiles for large problems (measured ahead of 256x192
  // tiles with 64-byte B boxes, which stay ahead for fp16/bf16)
  const TileChoice sp8_c[] = {{1, 128, false}, {1, 256, false}, {2, 192, false}, {1, 256, true}};
  const TileChoice dense8_c[] = {{1, 128, false}, {1, 256, false}, {1, 256, true}};
  const TileChoice* cand = !sparse ? (eb == 2 ? dense_c : dense8_c) : (eb == 2 ? sp16_c : sp8_c);
  const int n_cand = !sparse ? (eb == 2 ? 4 : 3) : (eb == 2 ? 5 : 4);
  const int64_t sms = sm_count();
  TileChoice best = cand[0];
  double best_cost = 1e300;
  for (int i = 0; i < n_cand; ++i) {
    const TileChoice c = cand[i];
    // an SM pair covers 256 rows with two CTAs, each filling 128 rows and half of the X panel
    const int64_t units = ceil_div(M, c.pair ? 256 : 128 * c.mt) * ceil_div(N, c.bn) * (c.pair ? 2 : 1);
    const int64_t waves = ceil_div(units, sms);
    const int64_t stage = c.pair ? (sparse ? 8192 + 2048 : 16384) + 64 * c.bn
                                 : c.mt * (sparse ? 8192 + 2048 : 16384) + 128 * c.bn;
    const double cost = static_cast<double>(waves) * static_cast<double>(stage) * (1.0 + 0.02 * (c.pair ? 2 : c.mt));
    if (cost < best_cost) { best_cost = cost; best = c; }
  }
  return best;
}

template <int DT>
cudaError_t dispatch_dt(int mode, const GemmArgs& a, cudaStream_t s, uint32_t* err) {
  constexpr int EB = Elem<DT>::bytes;
  if (mode == 0 || mode == 1) {
    const bool sparse = mode == 1;
    TileChoice c = choose_tile(sparse, EB, a.M, a.N);
    // large 16-bit 2:4 problems: SM pairs with two-step stages (measured ahead of
    // the 256 x 192 single-CTA tiles the fill model picks there)
    if (sparse && EB == 2 && c.mt == 2 && c.bn == 192) c = TileChoice{1, 256, true};
    // 2:4 tiles of 128 rows: stages of two 128-byte K steps (half the serial K loop of
    // one-step stages) on SM pairs and on single CTAs up to 128 columns
    int kx = 2;
    if (a.variant) {  // an explicit tile variant (validated by the caller)
      const int v = a.variant % 10000;
      c = TileChoice{v / 1000 == 9 ? 1 : v / 1000, v % 1000, v / 1000 == 9};
      kx = a.variant >= 10000 ? 2 : 1;
    }
    if (c.pair && sparse) {
      // the metadata tensor map addresses 128-row blocks by an int32 row coordinate
      const int64_t meta_rows = ceil_div(a.M, 128) * ceil_div(a.K, 128 / EB) * 16;
      if (meta_rows > INT32_MAX) c = TileChoice{2, 192, false};
    }
    if (c.pair) {
      if (c.bn != 256) return cudaErrorInvalidValue;
      // 2:4: stages of two 128-byte K steps halve the ring's turnovers (each stage
      // costs a fixed share of the operand stream, whatever its size)
      if (sparse)
        return kx == 1 ? run<DT, true, false, 256, 1, 128, true>(a, s, err)
                                  : run<DT, true, false, 256, 1, 128, true, false, false, 2>(a, s, err);
      return run<DT, false, false, 256, 1, 128, true>(a, s, err);
    }
    if (c.mt == 2) {
      if (!sparse && c.bn == 256) return run<DT, false, false, 256, 2>(a, s, err);
      if (sparse && EB == 2 && c.bn == 192) {
        if constexpr (EB == 2) return run<DT, true, false, 192, 2>(a, s, err);
      }
      if (sparse && EB == 1 && c.bn == 192) {
        if constexpr (EB == 1) return run<DT, true, false, 192, 2, 64>(a, s, err);
      }
      return cudaErrorInvalidValue;
    }
    if (c.bn == 64) {
      if constexpr (EB == 2) {
        if (sparse)
          return kx == 2 ? run<DT, true, false, 64, 1, 128, false, false, false, 2>(a, s, err)
                         : run<DT, true, false, 64>(a, s, err);
        return run<DT, false, false, 64>(a, s, err);
      }
      return cudaErrorInvalidValue;
    }
    if (c.bn == 128) {
      if (sparse)
        return kx == 2 ? run<DT, true, false, 128, 1, 128, false, false, false, 2>(a, s, err)
                       : run<DT, true, false, 128>(a, s, err);
      return run<DT, false, false, 128>(a, s, err);
    }
    return sparse ? run<DT, true, false, 256>(a, s, err) : run<DT, false, false, 256>(a, s, err);
  }
  if (mode == 5 || mode == 6 || mode == 7) {
    // 3x3 convolution: N tiles of whole image rows, 128 or 224 columns, whichever takes
    // fewer rounds of units over the SMs, a 224-column unit costing about 1.35 times a
    // 128-column one (measured on ResNet-50 layers, dense, 2:4 and tile-wise filters)
    if constexpr (EB == 2) {
      const int64_t sms = sm_count();
      auto rounds = [&](int64_t bn) {
        return ceil_div(ceil_div(a.M, 128) * a.conv_nb * ceil_div(a.conv_h, bn / a.conv_w), sms);
      };
      const bool narrow_c = a.conv_w <= 128 && 100 * rounds(128) < 135 * rounds(224);
      if (mode == 7)  // tile-wise filter
        return narrow_c ? run<DT, false, false, 128, 1, 128, false, true, true>(a, s, err)
                        : run<DT, false, false, 224, 1, 128, false, true, true>(a, s, err);
      if (mode == 5) {
        // 128-column tiles over whole 128-channel K pairs: two K steps per stage
        if (narrow_c && a.conv_cin % 128 == 0)
          return run<DT, true, false, 128, 1, 128, false, false, true, 2>(a, s, err);
        return narrow_c ? run<DT, true, false, 128, 1, 128, false, false, true>(a, s, err)
                        : run<DT, true, false, 224, 1, 128, false, false, true>(a, s, err);
      }
      return narrow_c ? run<DT, false, false, 128, 1, 128, false, false, true>(a, s, err)
                      : run<DT, false, false, 224, 1, 128, false, false, true>(a, s, err);
    }
    return cudaErrorInvalidValue;
  }
  // tile-wise and block-wise: 128-row tiles follow the pattern's tiles
  const bool narrow = a.N <= 128 || a.nt * ceil_div(a.N, 256) < 2 * sm_count();
  if constexpr (DT != 2) {
    if (mode == 2) return narrow ? run<DT, false, true, 128>(a, s, err) : run<DT, false, true, 256>(a, s, err);
    if (mode == 3) return narrow ? run<DT, true, true, 128>(a, s, err) : run<DT, true, true, 256>(a, s, err);
    if (mode == 4)
      return narrow ? run<DT, false, false, 128, 1, 128, false, true>(a, s, err)
                    : run<DT, false, false, 256, 1, 128, false, true>(a, s, err);
  }
  return cudaErrorInvalidValue;
}

__global__ void k_fill_epilogue(uint8_t* __restrict__ Y, int64_t ldy, int64_t M, int64_t N, int out_dt,
                                const float* __restrict__ bias, int act, float y_scale) {
  const bool hb = bias != nullptr;
  for (int64_t row = blockIdx.y; row < M; row += gridDim.y) {
    const float v = epilogue_value(0.f, 1.f, hb ? __ldg(bias + row) : 0.f, hb, act, y_scale);
    for (int64_t j = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; j < N;
         j += static_cast<int64_t>(gridDim.x) * blockDim.x) {
      if (out_dt == 2) {
        Y[row * ldy + j] = static_cast<uint8_t>(__nv_cvt_float_to_fp8(v, __NV_SATFINITE, __NV_E4M3));
      } else if (out_dt == 1) {
        const __nv_bfloat16 h = __float2bfloat16_rn(v);
        reinterpret_cast<__nv_bfloat16*>(Y)[row * ldy + j] = h;
      } else {
        const __half h = __float2half_rn(v);
        reinterpret_cast<__half*>(Y)[row * ldy + j] = h;
      }
    }
  }
}

}  // namespace

cudaError_t launch_fill_epilogue(void* Y, int64_t ldy, int64_t M, int64_t N, int out_dt, const float* bias, int act,
                                 float y_scale, cudaStream_t s) {
  if (M == 0 || N == 0) return cudaSuccess;
  const int code = out_dt == SSDNN_BF16 ? 1 : (out_dt == SSDNN_E4M3 ? 2 : 0);
  const dim3 grid(static_cast<unsigned>(std::min<int64_t>(ceil_div(N, 256), 64)),
                  static_cast<unsigned>(std::min<int64_t>(M, 65535)));
  k_fill_epilogue<<<grid, 256, 0, s>>>(static_cast<uint8_t*>(Y), ldy, M, N, code, bias, act, y_scale);
  return cudaGetLastError();
}

bool gemm_variant_ok(int variant, bool sparse, int elem_bytes) {
  switch (variant) {
    case 0: case 1128: case 1256: case 9256: return true;
    case 1064: return elem_bytes == 2;
    case 11064: return sparse && elem_bytes == 2;
    case 2192: case 11128: case 19256: return sparse;
    case 2256: return !sparse;
  }
  return false;
}

cudaError_t launch_gemm(int mode, const GemmArgs& a, cudaStream_t s, uint32_t* err) {
  switch (a.dt) {
    case SSDNN_F16: return dispatch_dt<0>(mode, a, s, err);
    case SSDNN_BF16: return dispatch_dt<1>(mode, a, s, err);
    case SSDNN_E4M3: return dispatch_dt<2>(mode, a, s, err);
  }
  return cudaErrorInvalidValue;
}

}  // namespace ssdnn
