"""GPU parity of the element-wise (unstructured) path through the C ABI: the
CSR prune bit-exact against the oracle (row pointers, columns, values), and the
CSR x dense product within the bound, on ragged shapes (rows, columns, K not a
multiple of the 128-row chunk), the limits (k = 0, k = K) and a 90 %-sparse
4096^3 case on sampled rows."""
import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import REL, bits_of, canary_intact, dev_padded, dev_tensor, guarded_output, lib, rand_bits

pytestmark = pytest.mark.gpu

CASES = [(300, 200, 40, 20), (64, 1000, 264, 100), (129, 256, 512, 256), (200, 72, 136, 0), (128, 512, 64, 51)]


@pytest.mark.parametrize("dt", ["f16", "bf16"])
@pytest.mark.parametrize("case", CASES)
def test_ew_prune_and_spmm(dt, case):
    ss = lib()
    M, K, N, k = case
    W = rand_bits(1000 + M + K, (M, K), dt, 0.5)
    W[1, : min(K, 16)] = W[1, 0]                       # ties inside a row
    X = rand_bits(1010 + N, (K, N), dt, 1.0)
    form = ss.ew_prune_compress(dev_tensor(W, dt), k)
    Y, buf = guarded_output(M, N, torch.bfloat16 if dt == "bf16" else torch.float16)
    ss.ew_spmm(form, dev_padded(X, dt), out=Y)
    torch.cuda.synchronize()
    assert ss.check_device_error() == 0
    ref = oracle.ew.prune(W, dt, k)
    assert np.array_equal(form.row_ptr.cpu().numpy(), ref["row_ptr"])
    assert np.array_equal(form.col_idx.cpu().numpy(), ref["col_idx"])
    assert np.array_equal(bits_of(form.vals), ref["vals"])
    Y_ref, B = oracle.ew.spmm(ref, M, K, X, dt, dt)
    ok = oracle.gemm.within_bound(bits_of(Y), Y_ref, B, dt, REL[dt])
    assert ok.all(), f"{(~ok).sum()} outside the bound"
    assert canary_intact(buf, M, N)


def test_ew_spmm_90_percent_sparse_4096():
    ss = lib()
    M = K = N = 4096
    k = round(0.1 * K)
    W = rand_bits(1020, (M, K), "bf16", 0.02)
    X = rand_bits(1021, (K, N), "bf16", 1.0)
    form = ss.ew_prune_compress(dev_tensor(W, "bf16"), k)
    Y = ss.ew_spmm(form, dev_tensor(X, "bf16"))
    torch.cuda.synchronize()
    assert ss.check_device_error() == 0
    rows = np.unique(np.concatenate([np.arange(64), np.arange(M - 64, M),
                                     np.random.default_rng(0).choice(M, 64, replace=False)]))
    ref = {"k": k, "col_idx": form.col_idx.cpu().numpy(), "vals": bits_of(form.vals)}
    # the selection of the sampled rows against the oracle's, then the product on them
    for i in rows[:16]:
        assert np.array_equal(ref["col_idx"][i * k:(i + 1) * k], oracle.ew.select_row(W[i], k, "bf16"))
    Y_ref, B = oracle.ew.spmm(ref, M, K, X, "bf16", "bf16", rows=rows)
    ok = oracle.gemm.within_bound(bits_of(Y[torch.from_numpy(rows).cuda()]), Y_ref, B, "bf16", REL["bf16"])
    assert ok.all(), f"{(~ok).sum()} outside the bound"
