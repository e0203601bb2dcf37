// 2:4 magnitude prune + compress.
//
// The 2:4 pattern: in each contiguous group of four values along K two are zero,
// and the matrix is kept as its nonzero values plus small position metadata
// ("NVIDIA A100 benchmarks" blog page, 2:4 paragraph and Figure 1 caption).
// Criterion (reading): keep the two largest |w| of each group, ties to the lower
// position, comparing the stored bits with the sign cleared as integers.
//
// A thread owns 32 consecutive elements of a row (8 groups; e4m3: two adjacent such
// chunks): 64 B of fp16/bf16 or 2 x 32 B of e4m3 read with 16-byte loads, 32 B /
// 2 x 16 B of values and 4 B of canonical metadata per chunk written, plus its part
// of the tensor-core operand layout of the metadata. The grid also covers the 128-row and K-block padding of that
// layout, which it fills with the (0,1) pattern. A group's kept pair comes from six
// pairwise magnitude comparisons, looked up in a 64-entry table of kept pairs. For
// e4m3 the comparisons of four groups are made together: their four words are
// transposed (word p = position p of each group) and each comparison is one
// byte-parallel subtraction; the table is of byte selectors, and four groups'
// selectors are combined in one word. For fp16/bf16 the comparisons are made on the
// 16-bit lanes of one group's two words.
#include "common.cuh"
#include "kernels.h"

namespace ssdnn {
namespace {

// The order of a group's four magnitudes m0..m3 as six comparison bits:
//   b0 = [m0 >= m1]  b1 = [m1 >= m2]  b2 = [m2 >= m3]  b3 = [m3 > m0]
//   b4 = [m0 >= m2]  b5 = [m1 >= m3]
// (ties count for the lower position; the pair (3, 0) is compared strictly for that
// reason). Entry idx of the shared table is, for the group's kept pair j0 < j1: the
// metadata nibble j0 | j1 << 2 in bits 0..3, the byte selector of the pair within its
// own word(s) in bits 8..23, and (e4m3) the selector of the pair as the high half of
// a two-group output word in bits 24..31.
__device__ __forceinline__ uint32_t kept_pair_entry(uint32_t idx, int eb) {
  const uint32_t w01 = idx & 1u, w12 = (idx >> 1) & 1u, w23 = (idx >> 2) & 1u, w03 = 1u - ((idx >> 3) & 1u),
                 w02 = (idx >> 4) & 1u, w13 = (idx >> 5) & 1u;
  const uint32_t wins[4] = {w01 + w02 + w03, (1u - w01) + w12 + w13, (1u - w02) + (1u - w12) + w23,
                            (1u - w03) + (1u - w13) + (1u - w23)};
  // the two positions with the most wins, ties to the lower position
  uint32_t a = 0;
  for (uint32_t i = 1; i < 4; ++i)
    if (wins[i] > wins[a]) a = i;
  uint32_t b = a == 0 ? 1u : 0u;
  for (uint32_t i = 0; i < 4; ++i)
    if (i != a && wins[i] > wins[b]) b = i;
  const uint32_t j0 = min(a, b), j1 = max(a, b);
  const uint32_t nib = j0 | (j1 << 2);
  if (eb == 1) return nib | ((j0 | (j1 << 4)) << 8) | (((j0 + 4) | ((j1 + 4) << 4)) << 24);
  return nib | (((2 * j0) | ((2 * j0 + 1) << 4) | ((2 * j1) << 8) | ((2 * j1 + 1) << 12)) << 8);
}

// The order indices of four groups of four e4m3 codes (one group per word, byte i =
// code i), one per byte of the result: byte g = r_g = b5 | b4 << 1 | b3 << 2 | b2 << 3 |
// b1 << 4 | b0 << 5, group g's order bits in reversed order. The words are
// transposed so that t_p holds the code at position p of all four groups; each
// comparison is then one byte-parallel subtraction with a guard bit (magnitudes are
// 7 bits, so 0x80 + m_a - m_b never borrows across bytes and its bit 7 is
// [m_a >= m_b]; with 0x7F it is [m_a > m_b]).
__device__ __forceinline__ uint32_t order_index4_e4m3(uint32_t w0, uint32_t w1, uint32_t w2, uint32_t w3) {
  const uint32_t x01l = __byte_perm(w0, w1, 0x5140), x01h = __byte_perm(w0, w1, 0x7362);
  const uint32_t x23l = __byte_perm(w2, w3, 0x5140), x23h = __byte_perm(w2, w3, 0x7362);
  const uint32_t t0 = __byte_perm(x01l, x23l, 0x5410) & 0x7F7F7F7Fu;
  const uint32_t t1 = __byte_perm(x01l, x23l, 0x7632) & 0x7F7F7F7Fu;
  const uint32_t t2 = __byte_perm(x01h, x23h, 0x5410) & 0x7F7F7F7Fu;
  const uint32_t t3 = __byte_perm(x01h, x23h, 0x7632) & 0x7F7F7F7Fu;
  const uint32_t e01 = t0 - t1 + 0x80808080u, e12 = t1 - t2 + 0x80808080u, e23 = t2 - t3 + 0x80808080u;
  const uint32_t e30 = t3 - t0 + 0x7F7F7F7Fu, e02 = t0 - t2 + 0x80808080u, e13 = t1 - t3 + 0x80808080u;
  // bit 7 of each byte of e01, e12, e23, e30, e02, e13 to bits 5..0
  uint32_t v = (e01 >> 2) & 0x20202020u;
  v = (v & 0x20202020u) | ((e12 >> 3) & 0x1F1F1F1Fu);
  v = (v & 0x30303030u) | ((e23 >> 4) & 0x0F0F0F0Fu);
  v = (v & 0x38383838u) | ((e30 >> 5) & 0x07070707u);
  v = (v & 0x3C3C3C3Cu) | ((e02 >> 6) & 0x03030303u);
  v = (v & 0x3E3E3E3Eu) | ((e13 >> 7) & 0x01010101u);
  return v;
}

// The same for a group of four 16-bit codes in two words (lo = v0 | v1 << 16,
// hi = v2 | v3 << 16): lane-parallel subtractions with a guard bit (15-bit magnitudes).
__device__ __forceinline__ uint32_t order_bits_16(uint32_t lo, uint32_t hi) {
  const uint32_t ml = lo & 0x7FFF7FFFu, mh = hi & 0x7FFF7FFFu;
  const uint32_t gl = ml | 0x80008000u, gh = mh | 0x80008000u;
  const uint32_t da = gl - __byte_perm(ml, 0u, 0x1032);  // bit 15: [m0 >= m1]
  const uint32_t db = gh - __byte_perm(mh, 0u, 0x1032);  // bit 15: [m2 >= m3]
  const uint32_t dc = gl - mh;                           // bits 15, 31: [m0 >= m2], [m1 >= m3]
  // lanes (m1, m3) against (m2, m0), the upper lane strictly: bits 15, 31: [m1 >= m2], [m3 > m0]
  const uint32_t x = __byte_perm(ml, mh, 0x7632) | 0x80008000u;
  const uint32_t y = __byte_perm(mh, ml, 0x5410);
  const uint32_t dd = x - y - 0x00010000u;
  // b0, b1, b2, b3 to bits 7, 15, 23, 31 (bytes da.1, dd.1, db.1, dd.3) and b4, b5 to
  // bits 7, 15 (bytes dc.1, dc.3), then gathered as for e4m3
  const uint32_t v = (__byte_perm(da, dd, 0x7051) & 0x80008080u) | ((db << 8) & 0x00800000u);
  const uint32_t u = __byte_perm(dc, 0u, 0x0031) & 0x00008080u;
  const uint32_t z = (v >> 7) | (u >> 3);
  return (z * 0x01020408u) >> 24;
}

// Shared-memory tables of a block: the kept-pair entries (fp16/bf16), the e4m3 byte
// selectors at the bit-reversed order index, and the rows' metadata words exchanged
// for the 16-bit operand order.
struct CompressShared {
  uint32_t tab[64];
  uint8_t sel[64];
  uint32_t nib[16][17];
};

// Threads 0..63 fill the tables (the caller synchronises before use).
__device__ __forceinline__ void build_tables(CompressShared& sh, int eb) {
  if (threadIdx.x < 64) {
    const uint32_t e = kept_pair_entry(threadIdx.x, eb);
    sh.tab[threadIdx.x] = e;
    // e4m3: the same entry at the bit-reversed index (the four-group order index)
    sh.sel[__brev(threadIdx.x) >> 26] = static_cast<uint8_t>(e >> 8);
  }
}

// The work of one thread on the codes it holds: w[cc] = chunk c0 + cc of row i (32
// elements, zero past K and M, so that such groups take the (0, 1) entry: nibble 0x4
// and zero values). Writes the kept values, the canonical nibbles (if meta) and the
// operand-order metadata. A thread is (tr, tc) of a 16 x 16 block that covers 16
// consecutive rows; every thread of the block calls it (16-bit: one barrier inside).
template <int EB>
__device__ __forceinline__ void compress_store(const uint32_t (&w)[EB == 1 ? 2 : 1][16], int64_t i, int64_t c0,
                                               int tr, int tc, int64_t M, int64_t Kp, uint8_t* __restrict__ values,
                                               int64_t ldv_b, uint8_t* __restrict__ meta, int64_t ldm,
                                               uint8_t* __restrict__ meta_hw, int64_t KBhw, int64_t chunks_pad,
                                               CompressShared& sh) {
  constexpr int CPT = EB == 1 ? 2 : 1;
  uint32_t nib[CPT];
  uint32_t outv[CPT][8];  // 16 kept values (EB bytes each) per chunk
#pragma unroll
  for (int cc = 0; cc < CPT; ++cc) {
    uint32_t nw = 0;
    if constexpr (EB == 1) {
      // the groups' selector bytes j0 | j1 << 4, four to a word
      uint32_t sb[8];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const uint32_t v = order_index4_e4m3(w[cc][4 * h], w[cc][4 * h + 1], w[cc][4 * h + 2], w[cc][4 * h + 3]);
        sb[4 * h] = sh.sel[v & 0xFFu];
        sb[4 * h + 1] = sh.sel[__byte_perm(v, 0u, 0x4441)];
        sb[4 * h + 2] = sh.sel[__byte_perm(v, 0u, 0x4442)];
        sb[4 * h + 3] = sh.sel[v >> 24];
      }
      const uint32_t S0 = __byte_perm(__byte_perm(sb[0], sb[1], 0x0040), __byte_perm(sb[2], sb[3], 0x0040), 0x5410);
      const uint32_t S1 = __byte_perm(__byte_perm(sb[4], sb[5], 0x0040), __byte_perm(sb[6], sb[7], 0x0040), 0x5410);
      // output word of groups (g, g + 1): selector j0 | j1 << 4 | (j0' + 4) << 8 | (j1' + 4) << 12
      outv[cc][0] = __byte_perm(w[cc][0], w[cc][1], S0 + 0x4400u);
      outv[cc][1] = __byte_perm(w[cc][2], w[cc][3], (S0 >> 16) + 0x4400u);
      outv[cc][2] = __byte_perm(w[cc][4], w[cc][5], S1 + 0x4400u);
      outv[cc][3] = __byte_perm(w[cc][6], w[cc][7], (S1 >> 16) + 0x4400u);
#pragma unroll
      for (int q = 4; q < 8; ++q) outv[cc][q] = 0u;
      // nibble j0 | j1 << 2 of each selector byte, then the bytes' nibbles packed in order
      auto nibbles = [](uint32_t S) {
        const uint32_t n = (S | (S >> 2)) & 0x0F0F0F0Fu;
        const uint32_t t = (n | (n >> 4)) & 0x00FF00FFu;
        return (t | (t >> 8)) & 0xFFFFu;
      };
      nw = nibbles(S0) | (nibbles(S1) << 16);
    } else {
#pragma unroll
      for (int g = 0; g < 8; ++g) {
        const uint32_t e = sh.tab[order_bits_16(w[cc][2 * g], w[cc][2 * g + 1])];
        nw |= (e & 0xFu) << (4 * g);
        outv[cc][g] = __byte_perm(w[cc][2 * g], w[cc][2 * g + 1], e >> 8);
      }
    }
    nib[cc] = nw;
  }
  if (i < M) {
#pragma unroll
    for (int cc = 0; cc < CPT; ++cc) {
      const int64_t c = c0 + cc;
      if (c * 32 >= Kp) break;
      uint8_t* dv = values + i * ldv_b + c * 16 * EB;
      reinterpret_cast<uint4*>(dv)[0] = make_uint4(outv[cc][0], outv[cc][1], outv[cc][2], outv[cc][3]);
      if constexpr (EB == 2)
        reinterpret_cast<uint4*>(dv)[1] = make_uint4(outv[cc][4], outv[cc][5], outv[cc][6], outv[cc][7]);
      if (meta) *reinterpret_cast<uint32_t*>(meta + i * ldm + c * 4) = nib[cc];
    }
  }
  const int64_t mb = i >> 7, r = i & 127;
  if constexpr (EB == 1) {
    // e4m3 operand order = canonical nibbles, 16 bytes per row per 128 columns of K
    // (the thread's two chunks are adjacent: 8 bytes, one store)
    if (c0 < chunks_pad)
      *reinterpret_cast<uint2*>(meta_hw + ((mb * KBhw + (c0 >> 2)) * 128 + r) * 16 + (c0 & 3) * 4) =
          make_uint2(nib[0], nib[1]);
  } else {
    // 16-bit operand order: rows r and r ^ 8 share one 32-bit word per 32-column
    // span (lower row: groups 0..3 of both rows; upper row: groups 4..7 of both),
    // each span in its own even TMEM column (odd words zero).
    sh.nib[tr][tc] = nib[0];
    __syncthreads();
    const uint32_t partner = sh.nib[tr ^ 8][tc];
    const uint32_t hw =
        (tr & 8) ? ((partner >> 16) | (nib[0] & 0xFFFF0000u)) : ((nib[0] & 0xFFFFu) | (partner << 16));
    if (c0 < chunks_pad)
      *reinterpret_cast<uint2*>(meta_hw + ((mb * KBhw + (c0 >> 1)) * 128 + r) * 16 + (c0 & 1) * 8) =
          make_uint2(hw, 0u);
  }
}

// A thread owns CPT chunks of 32 consecutive elements of a row (8 groups each): 64 B
// (fp16/bf16, one chunk) or 2 x 32 B (e4m3, two adjacent chunks), all loaded before
// any is processed; block = 16 rows x 16 threads, eight blocks per SM (at most 32
// registers a thread); grid.y walks 16-row groups of the 128-row-padded matrix.
template <int EB>
__global__ void __launch_bounds__(256, 8) k_sp24_compress(const uint8_t* __restrict__ W, int64_t M, int64_t K,
                                                       int64_t ldw_b, uint8_t* __restrict__ values,
                                                       int64_t ldv_b, uint8_t* __restrict__ meta, int64_t ldm,
                                                       uint8_t* __restrict__ meta_hw, int64_t KBhw,
                                                       int64_t chunks_pad, bool vec_ok) {
  constexpr int CPT = EB == 1 ? 2 : 1;  // chunks per thread
  __shared__ CompressShared sh;
  const int tr = threadIdx.x >> 4, tc = threadIdx.x & 15;
  const int64_t i = static_cast<int64_t>(blockIdx.y) * 16 + tr;
  const int64_t c0 = (static_cast<int64_t>(blockIdx.x) * 16 + tc) * CPT;  // first chunk

  uint32_t w[CPT][16];
#pragma unroll
  for (int cc = 0; cc < CPT; ++cc) {
    const int64_t k0 = (c0 + cc) * 32;
#pragma unroll
    for (int q = 0; q < 16; ++q) w[cc][q] = 0;
    if (i >= M || k0 >= K) continue;
    const uint8_t* src = W + i * ldw_b + k0 * EB;
    if (vec_ok && k0 + 32 <= K) {
#pragma unroll
      for (int q = 0; q < 2 * EB; ++q) {  // 32 elements = 2 * EB 16-byte loads
        const uint4 v = __ldg(reinterpret_cast<const uint4*>(src) + q);
        w[cc][4 * q + 0] = v.x;
        w[cc][4 * q + 1] = v.y;
        w[cc][4 * q + 2] = v.z;
        w[cc][4 * q + 3] = v.w;
      }
    } else {
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        if (k0 + j >= K) break;
        const uint32_t e = (EB == 2) ? static_cast<uint32_t>(reinterpret_cast<const uint16_t*>(src)[j])
                                     : static_cast<uint32_t>(src[j]);
        if constexpr (EB == 2)
          w[cc][j >> 1] |= e << ((j & 1) * 16);
        else
          w[cc][j >> 2] |= e << ((j & 3) * 8);
      }
    }
  }
  build_tables(sh, EB);  // while the loads are in flight
  __syncthreads();
  compress_store<EB>(w, i, c0, tr, tc, M, (K + 31) / 32 * 32, values, ldv_b, meta, ldm, meta_hw, KBhw, chunks_pad,
                     sh);
}

}  // namespace

cudaError_t launch_sp24_compress(int dt, const void* W, int64_t M, int64_t K, int64_t ldw, void* values,
                                 uint8_t* meta, uint8_t* meta_hw, cudaStream_t s, uint32_t* err) {
  (void)err;  // no waits in this kernel
  const int EB = (dt == SSDNN_E4M3) ? 1 : 2;
  const int64_t span = (EB == 1) ? 128 : 64;          // K columns per operand metadata block
  const int64_t MB = ceil_div(M, 128), KBhw = ceil_div(K, span);
  const int64_t chunks_pad = KBhw * (span / 32);
  if (MB == 0 || KBhw == 0) return cudaSuccess;
  const int64_t Kp = round_up(K, 32);
  const int64_t ldv_b = Kp / 2 * EB;
  const bool vec_ok = (reinterpret_cast<uintptr_t>(W) % 16 == 0) && ((ldw * EB) % 16 == 0);
  const int64_t cpt = EB == 1 ? 2 : 1;  // chunks per thread (chunks_pad is a multiple of 4 for e4m3)
  const int64_t tiles_x = ceil_div(chunks_pad, 16 * cpt), tiles_y = MB * 8;
  const dim3 grid(static_cast<unsigned>(tiles_x), static_cast<unsigned>(tiles_y));
  if (EB == 2)
    k_sp24_compress<2><<<grid, 256, 0, s>>>(static_cast<const uint8_t*>(W), M, K, ldw * 2,
                                            static_cast<uint8_t*>(values), ldv_b, meta, Kp / 8, meta_hw, KBhw,
                                            chunks_pad, vec_ok);
  else
    k_sp24_compress<1><<<grid, 256, 0, s>>>(static_cast<const uint8_t*>(W), M, K, ldw,
                                            static_cast<uint8_t*>(values), ldv_b, meta, Kp / 8, meta_hw, KBhw,
                                            chunks_pad, vec_ok);
  return cudaGetLastError();
}

}  // namespace ssdnn
