"""seq->head permutation on the GPU against the oracle's index loop:
bit-exact, every element, small shapes (ragged chunk sizes, 1/2/4/8-byte
elements) and the full [131072, 32, 128] bf16 tensor with 8 groups; the
batch-aware subgroup form (B sequences, K ranks each) against the oracle's
grouped loop, and config 3's tensor as 4 sequences of 32768 tokens on
4 x 2 ranks."""
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


@pytest.mark.parametrize("B,L,H,d,K,eb", [
    (1, 100, 32, 128, 8, 2), (2, 64, 8, 128, 4, 2), (3, 33, 6, 5, 3, 1), (4, 17, 16, 2, 8, 8),
    (5, 7, 12, 7, 2, 4), (8, 1, 8, 128, 1, 2),
])
def test_permute_groups_bit_exact(nsp, B, L, H, d, K, eb):
    tdt, ndt = _INT[eb]
    rng = np.random.default_rng(B * 100 + L)
    x_np = rng.integers(np.iinfo(ndt).min, np.iinfo(ndt).max, size=(B * L, H, d), dtype=ndt)
    x = torch.from_numpy(x_np).cuda()
    y = nsp.seq2head_groups(x, B, K)
    ref = oracle.seq2head_groups(x_np, B, K)
    assert np.array_equal(y.cpu().numpy(), ref)
    back = nsp.head2seq_groups(y)
    assert np.array_equal(back.cpu().numpy(), oracle.head2seq_groups(ref, B, K))
    assert torch.equal(back, x)
    if B == 1:
        assert torch.equal(y[0], nsp.seq2head(x, K))


def test_permute_groups_config3_tensor(nsp):
    """Config 3's [131072, 32, 128] bf16 q as a micro-batch of 4 sequences of
    32768 tokens, each on its own group of 2 ranks (N = 8 = B K)."""
    w = workload(3)
    x = w.q.cuda()
    y = nsp.seq2head_groups(x, 4, 2)
    torch.cuda.synchronize()
    bits = w.q.view(torch.int16).numpy()
    ref = timed("oracle seq2head_groups C3", oracle.seq2head_groups, bits, 4, 2)
    assert np.array_equal(y.view(torch.int16).cpu().numpy(), ref)
    assert torch.equal(nsp.head2seq_groups(y).view(torch.int16), x.view(torch.int16))
