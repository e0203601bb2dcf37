"""GPU parity of the 3x3 convolution (implicit GEMM, stride 1, zero padding)
through the C ABI, with a 2:4 and a dense filter, against the oracle's im2col
convolution: small and ragged images (H not a multiple of the row patch, C_out
not a multiple of 128), both N tile widths, one and two K steps per stage, and the
ResNet-50 layers of the benchmark."""
import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import REL, bits_of, canary_intact, dev_tensor, guarded_output, lib, rand_bits

pytestmark = pytest.mark.gpu

# (Nb, H, W, Cin, Cout)
# (C_in a multiple of 128 with 128-column tiles: the 2:4 filter's stages carry two K steps;
# odd image widths put a unit's first output column at an odd offset; the last two are the
# ResNet-50 layers of the benchmark at its batch of 32)
CASES = [(1, 5, 7, 64, 128), (2, 14, 14, 128, 256), (1, 28, 28, 64, 200), (3, 9, 30, 64, 64), (1, 3, 224, 64, 128),
         (1, 28, 28, 128, 200), (2, 9, 30, 256, 64), (3, 7, 7, 128, 128), (1, 11, 13, 64, 64),
         (1, 1, 1, 128, 128), (2, 3, 5, 128, 64),
         (32, 28, 28, 128, 128), (32, 14, 14, 256, 256)]


@pytest.mark.parametrize("dt", ["f16", "bf16"])
@pytest.mark.parametrize("case", CASES)
@pytest.mark.parametrize("sparse", [True, False])
def test_conv3x3(dt, case, sparse):
    ss = lib()
    Nb, H, W, Cin, Cout = case
    X = rand_bits(1100 + H + W, (Nb * H * W, Cin), dt, 1.0).reshape(Nb, H, W, Cin)
    Wf = rand_bits(1110 + Cout + Cin, (Cout, 9 * Cin), dt, 0.2)
    Xd = dev_tensor(X.reshape(-1, Cin), dt).reshape(Nb, H, W, Cin)
    N = Nb * H * W
    pad = 8 + (-N) % 8                                   # a 16-byte output pitch
    Y, buf = guarded_output(Cout, N, torch.bfloat16 if dt == "bf16" else torch.float16, pad_cols=pad)
    if sparse:
        f = ss.sp24_prune_compress(dev_tensor(Wf, dt), canonical_meta=False)
        ss.conv3x3(f, Xd, out=Y)
    else:
        ss.conv3x3(dev_tensor(Wf, dt), Xd, out=Y)
    torch.cuda.synchronize()
    assert ss.check_device_error() == 0
    Y_ref, B = oracle.conv.conv3x3(Wf, X, dt, dt, sparse=sparse)
    ok = oracle.gemm.within_bound(bits_of(Y), Y_ref, B, dt, REL[dt])
    assert ok.all(), f"{(~ok).sum()} of {ok.size} outside the bound"
    assert canary_intact(buf, Cout, N)


# (Nb, H, W, Cin, Cout, kept groups per 128-channel tile); a group is one tap x 64
# input channels, 9 Cin / 64 groups per tile
TW_CASES = [(1, 5, 7, 64, 128, [3]), (2, 14, 14, 128, 256, [5, 0]), (1, 28, 28, 64, 200, [9, 2]),
            (3, 9, 30, 64, 64, [1]), (1, 3, 224, 128, 128, [18])]


@pytest.mark.parametrize("dt", ["f16", "bf16"])
@pytest.mark.parametrize("case", TW_CASES)
def test_conv3x3_tile_wise_filter(dt, case):
    """The tile-wise filter: bw_prune_compress of the flattened filter (indices and
    packed operand bit-exact against the oracle) and tw_conv3x3 within the bound of
    the oracle's convolution with the masked filter; a tile that keeps no group
    writes zeros, a tile that keeps all groups is the dense convolution."""
    ss = lib()
    Nb, H, W, Cin, Cout, keep = case
    keep = np.array(keep, dtype=np.int32)
    X = rand_bits(1200 + H + W, (Nb * H * W, Cin), dt, 1.0).reshape(Nb, H, W, Cin)
    Wf = rand_bits(1210 + Cout + Cin, (Cout, 9 * Cin), dt, 0.2)
    Xd = dev_tensor(X.reshape(-1, Cin), dt).reshape(Nb, H, W, Cin)
    N = Nb * H * W
    pad = 8 + (-N) % 8
    Y, buf = guarded_output(Cout, N, torch.bfloat16 if dt == "bf16" else torch.float16, pad_cols=pad)
    f = ss.bw_prune_compress(dev_tensor(Wf, dt), keep)
    ss.conv3x3(f, Xd, out=Y)
    torch.cuda.synchronize()
    assert ss.check_device_error() == 0
    Y_ref, B, form = oracle.conv.conv3x3_tw(Wf, X, dt, dt, keep)
    assert np.array_equal(f.indices.cpu().numpy()[:int(keep.sum())], form["indices"])
    ok = oracle.gemm.within_bound(bits_of(Y), Y_ref, B, dt, REL[dt])
    assert ok.all(), f"{(~ok).sum()} of {ok.size} outside the bound"
    assert canary_intact(buf, Cout, N)
