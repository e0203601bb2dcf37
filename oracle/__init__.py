"""CPU oracle for the structured-sparse weight GEMM.

TEST INFRASTRUCTURE ONLY. Only the test suite, the package smoke check and the
benchmark's CPU-baseline leg may import or call anything in this directory.
The product path (the CUDA library and its binding) never imports it, and this
oracle imports nothing from the product.

What it computes, each function citing the page passage it follows:
  * codecs      -- fp16 / bf16 / OCP e4m3 decoding and RNE encoding, from the
                   format definitions.
  * sp24        -- magnitude 2:4 pruning and the compressed representation
                   (kept values plus 2-bit positions), decompression.
  * gemm        -- Y = alpha * decompress(W) . X in fp64, rounded once to the
                   output type; the elementwise error bound sum_k |w_ik x_kj|.
  * epilogue    -- the fused layer epilogue: per-row bias, ReLU / GELU,
                   output scaling and rounding (e4m3 output included).
  * bw          -- block-wise sparsity (128 x 64 blocks of a tile row kept by
                   block score), packing and the block-sparse GEMM.
  * ew          -- element-wise (unstructured) magnitude pruning to CSR and the
                   sparse x dense product.
  * conv        -- 3x3 convolution (stride 1, padding 1) of NHWC activations with a
                   2:4-sparse or dense filter, through the im2col matrix.
  * tw          -- tile-wise scores, per-tile top-L selection, packing of the
                   kept columns, the tile-vector-wise hybrid, the tile schedule.

Numerics: the GEMM accumulates in fp64 (library matmul as a step) because the
pages fix no precision. The tile-wise scores are fp32 sums in ascending row
order, because they decide an integer result (which K indices a tile keeps) and
the CUDA path decides it in fp32 in that order.

Every function has a pin in tests/ other than itself (closed forms, brute force
on tiny inputs, invariants, hand-derived fixtures in tests/golden/).
"""
from . import codecs, sp24, gemm, tw, epilogue, bw, ew, conv  # noqa: F401
