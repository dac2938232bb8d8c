"""acc_add through the C ABI: bit-exact fp32 sums at any alignment and length."""
import numpy as np
import pytest

from oracle import vloss_oracle as O
from tests import gpu_harness as H

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("n", [1, 3, 4, 5, 1000, (1 << 20) + 3])
@pytest.mark.parametrize("offs", [(0, 0), (1, 1), (3, 1), (2, 0)])
def test_acc_add_bit_exact(n, offs):
    torch = H.torch_cuda()
    from top_kl_distill_gb300 import vloss as vl
    g = np.random.default_rng(n + 7 * offs[0] + offs[1])
    a = (g.standard_normal(n) * 10.0 ** g.integers(-3, 3, n)).astype(np.float32)
    b = (g.standard_normal(n) * 10.0 ** g.integers(-3, 3, n)).astype(np.float32)
    da = H.dev(a, offset=offs[0])
    db = H.dev(b, offset=offs[1])
    vl.vl_acc_add(da, db, n)
    torch.cuda.synchronize()
    assert np.array_equal(H.host(da).view(np.uint32), O.acc_add(a, b).view(np.uint32))


def test_acc_add_zero_length_and_errors():
    torch = H.torch_cuda()
    from top_kl_distill_gb300 import vloss as vl
    a = torch.ones(8, device="cuda")
    vl.vl_acc_add(a, a, 0)
    with pytest.raises(vl.VlossError):
        vl.vl_acc_add(a[0:6], a[2:8], 6)        # overlapping ranges
    vl.vl_acc_add(a, a, 8)                       # a == b is allowed: doubles
    torch.cuda.synchronize()
    assert np.all(H.host(a) == 2.0)
