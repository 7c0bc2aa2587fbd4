"""Failure detection without a GPU fault: an internal pipeline wait that can
never be satisfied (its loads are withheld) runs out after a short limit, the
kernel winds down and the status KD_ERR_TIMEOUT reaches the host; the context
stays usable for the next call.  Bad teacher ids are reported the same way."""
import numpy as np
import pytest
import torch

from lm_head_top_tma_b300 import _native as N
from lm_head_top_tma_b300 import api

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("pair", [False, True])
def test_wait_timeout_is_reported_and_context_survives(cuda_device, pair):
    assert api.debug_wait_timeout(50, cuda_device, cta_pair=pair) == N.KD_ERR_TIMEOUT
    A = torch.ones(256, 64, device=cuda_device, dtype=torch.bfloat16)
    D = api.gemm_bf16(A, A, 256, 256, 64, cta_pair=pair)
    torch.cuda.synchronize()
    assert torch.all(D == 64.0)


def test_bad_index_is_reported(cuda_device):
    T, d, V, K = 130, 64, 512, 8
    rng = np.random.default_rng(0)
    H = torch.randn(T, d, device=cuda_device).to(torch.bfloat16)
    W = (0.1 * torch.randn(V, d, device=cuda_device)).to(torch.bfloat16)
    idx = torch.tensor(rng.integers(0, V, size=(T, K)), dtype=torch.int32, device=cuda_device)
    p = torch.full((T, K), 1.0 / K, device=cuda_device)
    idx[5, 3] = V          # out of range
    idx[77, 0] = -1
    with pytest.raises(N.KDError) as e:
        api.forward(H, W, idx, p, 64)
    assert e.value.code == N.KD_ERR_BAD_INDEX
    # unchecked call: the two rows contribute nothing, the others are intact
    loss, lse, rows = api.forward(H, W, idx, p, 64, loss_rows=True, check=False)
    torch.cuda.synchronize()
    assert rows[5].item() == 0.0 and rows[77].item() == 0.0
    assert rows[6].item() != 0.0
