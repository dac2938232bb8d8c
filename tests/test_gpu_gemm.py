"""The tensor-core head GEMM through the C ABI against float64 products of the same bf16 values.

bf16 x bf16 products are exact in fp32; the fp32 sums may lose at most the dot-product
bound K * 2^-24 * sum_k |a_k b_k| (doubled here for the tensor cores' summation order).
"""
import numpy as np
import pytest

from tests import gpu_harness as H

pytestmark = pytest.mark.gpu


def bf16_bits(x):
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    return ((b + 0x7FFF + ((b >> 16) & 1)) >> 16).astype(np.uint16)


def bf16_value(bits):
    return (bits.astype(np.uint32) << 16).view(np.float32)


@pytest.mark.parametrize("M,N,K,ldd,alpha", [
    (128, 256, 64, 256, 1.0),          # one tile, one stage
    (200, 300, 72, 300, 0.5),          # ragged M, N and K (the TMA fills zeros past the edges)
    (1000, 1300, 256, 1304, 1.0),      # several tiles, a wider output stride
    (256, 4096, 1024, 4096, 2.0),      # many stages: the ring wraps
    (40, 32000, 256, 32000, 1.0),      # the head's shape: a few rows by a vocabulary
    (7, 9, 8, 11, 1.0),                # smaller than a tile, unaligned output rows
])
def test_gemm_bf16_tn(M, N, K, ldd, alpha):
    torch = H.torch_cuda()
    from top_kl_distill_gb300 import vloss as vl
    g = np.random.default_rng(M * 7 + N * 3 + K)
    a = bf16_bits(g.standard_normal((M, K)).astype(np.float32))
    b = bf16_bits(g.standard_normal((N, K)).astype(np.float32))
    A64, B64 = bf16_value(a).astype(np.float64), bf16_value(b).astype(np.float64)
    da = torch.from_numpy(a.view(np.int16)).cuda().view(torch.bfloat16)
    db = torch.from_numpy(b.view(np.int16)).cuda().view(torch.bfloat16)
    D = torch.full((M, ldd), float("nan"), device="cuda")
    vl.vl_gemm_bf16_tn(da, db, D, M, N, K, ldd, alpha)
    torch.cuda.synchronize()
    got = H.host(D).astype(np.float64)
    want = alpha * (A64 @ B64.T)
    bound = 2 * K * 2.0 ** -24 * abs(alpha) * (np.abs(A64) @ np.abs(B64).T) + 1e-30
    err = np.abs(got[:, :N] - want)
    assert np.all(err <= bound), (f"{int((err > bound).sum())} of {err.size} off; worst err/bound "
                                  f"{np.max(err / bound):.3g} at {np.unravel_index(np.argmax(err / bound), err.shape)}")
    if ldd > N:
        assert np.isnan(got[:, N:]).all(), "columns past N were written"
    H.report("tensor-core GEMM", "max err / bound", float(np.max(err / bound)))
