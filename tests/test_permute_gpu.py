"""seq->head permutation on the GPU against the oracle's index loop:
bit-exact, every element, small shapes (ragged chunk sizes, 1/2/4/8-byte
elements) and the full [131072, 32, 128] bf16 tensor with 8 groups."""
import numpy as np
import pytest
import torch

import oracle
from gpu_common import timed, workload

pytestmark = pytest.mark.gpu

_INT = {1: (torch.uint8, np.uint8), 2: (torch.int16, np.int16), 4: (torch.int32, np.int32),
        8: (torch.int64, np.int64)}


@pytest.mark.parametrize("T,H,d,P,eb", [
    (1, 8, 128, 8, 2), (7, 8, 3, 4, 2), (64, 8, 8, 2, 4), (33, 6, 5, 3, 1),
    (100, 32, 128, 8, 2), (129, 4, 64, 1, 4), (17, 16, 2, 16, 8), (50, 12, 7, 4, 1),
])
def test_permute_small_bit_exact(nsp, T, H, d, P, eb):
    tdt, ndt = _INT[eb]
    rng = np.random.default_rng(T * 1000 + H)
    x_np = rng.integers(np.iinfo(ndt).min, np.iinfo(ndt).max, size=(T, H, d), dtype=ndt)
    x = torch.from_numpy(x_np).cuda()
    y = torch.empty((P, T, H // P, d), dtype=tdt, device="cuda")
    nsp.nsp_seq2head_permute(x, y, T, H, d, P, inverse=False)
    ref = oracle.seq2head(x_np, P)
    assert np.array_equal(y.cpu().numpy(), ref)
    back = torch.empty_like(x)
    nsp.nsp_seq2head_permute(y, back, T, H, d, P, inverse=True)
    assert np.array_equal(back.cpu().numpy(), oracle.head2seq(ref, P))
    assert np.array_equal(back.cpu().numpy(), x_np)


def test_permute_full_config3_bit_exact(nsp):
    w = workload(3)
    T, H, d = w.q.shape
    P = w.cfg.permute_groups
    x = w.q.cuda()
    y = nsp.seq2head(x, P)
    torch.cuda.synchronize()
    bits = w.q.view(torch.int16).numpy()
    ref = timed("oracle seq2head C3", oracle.seq2head, bits, P)
    assert np.array_equal(y.view(torch.int16).cpu().numpy(), ref)
    back = nsp.head2seq(y)
    assert torch.equal(back.view(torch.int16), x.view(torch.int16))
