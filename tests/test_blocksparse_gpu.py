"""GPU parity of the block-sparse forward (fa_fwd_blocksparse, through the C
ABI) against the float64 oracle's block-mask forward."""
import math

import numpy as np
import pytest
import torch

import oracle
from tests.guards import Guarded, check_all
from tests.parity import assert_close, assert_lse_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fa(cuda_device):
    import exact_io_aware_35_gb300 as fa
    fa.load_library()
    return fa


def inputs(B, N, Hq, Hkv, d, seed, s=0.5):
    g = torch.Generator().manual_seed(seed)
    q = (torch.randn(B, N, Hq, d, generator=g) * s).to(torch.bfloat16)
    k = (torch.randn(B, N, Hkv, d, generator=g) * s).to(torch.bfloat16)
    v = torch.randn(B, N, Hkv, d, generator=g).to(torch.bfloat16)
    return q, k, v


def random_mask(Hq, nb, seed, density):
    m = torch.rand(Hq, nb, nb, generator=torch.Generator().manual_seed(seed)) < density
    return m.to(torch.uint8)


def local_mask(Hq, nb, width):
    i = torch.arange(nb)
    m = ((i[:, None] - i[None, :]).abs() <= width).to(torch.uint8)
    return m.expand(Hq, nb, nb).contiguous()


def run(fa, q, k, v, mask, causal, scale):
    """fa_fwd_blocksparse with NaN-filled outputs between guard canaries
    (tests/guards.py)."""
    qd = q.cuda()
    B, N, Hq, d = q.shape
    o = Guarded(qd.shape, qd.dtype, qd.device)
    lse = Guarded((B, Hq, N), torch.float32, qd.device)
    fa.fa_fwd_blocksparse(qd, k.cuda(), v.cuda(), mask.cuda(), causal=causal, scale=scale, o=o.t,
                          lse=lse.t)
    assert fa.fa_get_device_error() == fa.FA_OK
    check_all(o=o, lse=lse)
    return o.t.cpu(), lse.t.cpu()


def check(o, lse, o_ref, lse_ref):
    assert_close(o, o_ref, "o")
    lse, lse_ref = lse.double().numpy(), np.asarray(lse_ref)
    empty = np.isneginf(lse_ref)
    assert (np.isneginf(lse) == empty).all(), "rows with no visible key must give lse = -inf"
    assert_lse_close(lse[~empty], lse_ref[~empty])


# (B, N, Hq, Hkv, d, causal, mask kind)
CASES = [
    (1, 1000, 4, 2, 128, False, "random"),
    (1, 1000, 4, 2, 128, True, "random"),
    (2, 512, 2, 1, 64, True, "local"),
    (1, 300, 8, 8, 64, False, "random"),
    (1, 100, 2, 1, 128, True, "ones"),
    (1, 640, 4, 1, 128, True, "diagonal"),
]


@pytest.mark.parametrize("B,N,Hq,Hkv,d,causal,kind", CASES)
def test_blocksparse_matches_oracle(fa, B, N, Hq, Hkv, d, causal, kind):
    nb = (N + 127) // 128
    q, k, v = inputs(B, N, Hq, Hkv, d, seed=N + Hq)
    if kind == "random":
        mask = random_mask(Hq, nb, seed=N, density=0.5)
    elif kind == "local":
        mask = local_mask(Hq, nb, 1)
    elif kind == "diagonal":
        mask = local_mask(Hq, nb, 0)
    else:
        mask = torch.ones(Hq, nb, nb, dtype=torch.uint8)
    scale = 1 / math.sqrt(d)
    o, lse = run(fa, q, k, v, mask, causal, scale)
    o_ref, lse_ref = oracle.attn_fwd_blockmask(q, k, v, mask.numpy(), 128, causal, scale)
    check(o, lse, o_ref, lse_ref)


def test_all_ones_mask_is_the_dense_forward(fa):
    q, k, v = inputs(1, 700, 4, 2, 128, seed=21)
    mask = torch.ones(4, 6, 6, dtype=torch.uint8)
    o, lse = run(fa, q, k, v, mask, True, 0.09)
    o_ref, lse_ref = oracle.attn_fwd(q, k, v, True, 0.09)
    assert_close(o, o_ref, "o")
    assert_lse_close(lse, lse_ref)


def test_empty_mask_rows(fa):
    # head 1 sees nothing from query block 2 on; head 0 under causal loses its
    # diagonal in block 0, so query block 0 has no visible key at all
    q, k, v = inputs(1, 400, 2, 1, 128, seed=22)
    mask = torch.ones(2, 4, 4, dtype=torch.uint8)
    mask[1, 2:, :] = 0
    mask[0, 0, 0] = 0
    o, lse = run(fa, q, k, v, mask, True, 0.1)
    o_ref, lse_ref = oracle.attn_fwd_blockmask(q, k, v, mask.numpy(), 128, True, 0.1)
    check(o, lse, o_ref, lse_ref)
    assert (o[0, 256:, 1] == 0).all() and (o[0, :128, 0] == 0).all()


@pytest.mark.parametrize("causal", [False, True])
def test_staggered_masks_of_one_thread_block(fa, causal):
    # a thread block holds two query tiles (query blocks 2i and 2i+1) and
    # streams the union of their key blocks: here the even query blocks see
    # only their first and last visible key blocks while the odd ones see all,
    # so one tile's blocks lie far apart in the union (longer than the K/V
    # ring), and some tiles see nothing at all
    N, Hq = 1400, 2
    nb = (N + 127) // 128
    q, k, v = inputs(1, N, Hq, 1, 128, seed=25)
    mask = torch.ones(Hq, nb, nb, dtype=torch.uint8)
    for i in range(0, nb, 2):
        last = i if causal else nb - 1
        mask[:, i, :] = 0
        mask[:, i, 0] = 1
        mask[:, i, last] = 1
    mask[1, 4, :] = 0  # an empty tile beside a full one (query blocks 4, 5)
    mask[1, 7, :] = 0  # and the other way round (query blocks 6, 7)
    o, lse = run(fa, q, k, v, mask, causal, 1 / math.sqrt(128))
    o_ref, lse_ref = oracle.attn_fwd_blockmask(q, k, v, mask.numpy(), 128, causal,
                                               1 / math.sqrt(128))
    check(o, lse, o_ref, lse_ref)


def test_blocksparse_bench_shape_sampled(fa):
    # the block-sparse bench shape: gqa8k's head layout (Hq32 Hkv8, N 8192,
    # d 128, causal) with a local-window-plus-random mask; oracle on one head
    from fa_workloads import block_sparse_mask
    N, Hq, Hkv, d = 8192, 32, 8, 128
    q, k, v = inputs(1, N, Hq, Hkv, d, seed=23)
    mask = block_sparse_mask(Hq, N, seed=24)
    o, lse = run(fa, q, k, v, mask, True, 1 / math.sqrt(d))
    for h in (0, 17):
        hk = h // (Hq // Hkv)
        o_ref, lse_ref = oracle.attn_fwd_blockmask(q[:, :, h:h + 1], k[:, :, hk:hk + 1],
                                                   v[:, :, hk:hk + 1], mask[h:h + 1].numpy(),
                                                   128, True, 1 / math.sqrt(d))
        check(o[:, :, h:h + 1], lse[:, h:h + 1], o_ref, lse_ref)
