"""Block-sparse forward and backward parity: the CUDA path vs the dense oracle
with the masked 128 x 128 blocks set to -inf."""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from _util import check_fwd, check_grads, cuda, f64

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("N", [512, 1000])
def test_sparse_small_random_masks(fa, d, N):
    w = W.Workload("generic", 2, 2, N, d, causal=False, backward=False)
    x = W.make_inputs(w, 21)
    nb = (N + 127) // 128
    g = np.random.default_rng(N + d)
    mask = (g.random((nb, nb)) < 0.5).astype(np.uint8)
    mask[1, :] = 0            # a query block that sees nothing: O = 0, LSE = -inf
    mask[0, :] = 1
    o, lse = fa.blocksparse_forward(cuda(x["q"]), cuda(x["k"]), cuda(x["v"]),
                                    torch.from_numpy(mask).cuda(), scale=w.scale)
    torch.cuda.synchronize()
    assert fa.device_status() == 0
    o_ref, l_ref = oracle.forward(x["q"], x["k"], x["v"], w.scale, block_mask=mask)
    check_fwd(o, lse, o_ref, l_ref, f"sparse d={d} N={N}")
    assert np.all(f64(o)[:, :, 128:256] == 0)
    assert np.all(np.isneginf(f64(lse)[:, :, 128:256]))


def test_sparse_all_ones_equals_dense_bitwise(fa):
    w = W.Workload("generic", 1, 3, 640, 64, causal=False, backward=False)
    x = W.make_inputs(w, 22)
    q, k, v = cuda(x["q"]), cuda(x["k"]), cuda(x["v"])
    ones = torch.ones(5, 5, dtype=torch.uint8, device="cuda")
    o1, l1 = fa.blocksparse_forward(q, k, v, ones)
    o2, l2 = fa.forward(q, k, v)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_sparse_full_size_workload(fa):
    w = W.WORKLOADS["blocksparse"]
    x = W.make_inputs(w, 0)
    mask = x["block_mask"]
    o, lse = fa.blocksparse_forward(cuda(x["q"]), cuda(x["k"]), cuda(x["v"]), mask.cuda(),
                                    scale=w.scale)
    torch.cuda.synchronize()
    assert fa.device_status() == 0
    # whole query blocks: first, last, and two with random off-band blocks
    m = mask.numpy()
    offband = [r for r in range(m.shape[0]) if m[r].sum() > (3 if 0 < r < m.shape[0] - 1 else 2)]
    blocks = sorted({0, m.shape[0] - 1, *offband[:2]})
    rows = np.concatenate([np.arange(b * 128, (b + 1) * 128) for b in blocks])
    o_ref, l_ref = oracle.forward(x["q"], x["k"], x["v"], w.scale, block_mask=m, rows=rows)
    check_fwd(f64(o)[:, :, rows], f64(lse)[:, :, rows], o_ref, l_ref, "blocksparse full size")


# ---------------------------------------------------------------- backward
def _sparse_bwd(fa, x, mask, scale):
    q, k, v, do = cuda(x["q"]), cuda(x["k"]), cuda(x["v"]), cuda(x["dout"])
    m = torch.from_numpy(mask).cuda()
    o, lse = fa.blocksparse_forward(q, k, v, m, scale=scale)
    g = fa.blocksparse_backward(q, k, v, o, do, lse, m, scale=scale)
    torch.cuda.synchronize()
    assert fa.device_status() == 0
    return g


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("N", [512, 1000])
def test_sparse_bwd_small_random_masks(fa, d, N):
    w = W.Workload("generic", 2, 2, N, d, causal=False, backward=True)
    x = W.make_inputs(w, 31)
    nb = (N + 127) // 128
    g = np.random.default_rng(N + d + 1)
    mask = (g.random((nb, nb)) < 0.5).astype(np.uint8)
    mask[0, :] = 1
    mask[1, :] = 0            # a query block that sees nothing: its dQ rows are 0
    mask[:, 2] = 0            # a key block no query block keeps: its dK, dV rows are 0
    grads = _sparse_bwd(fa, x, mask, w.scale)
    ref = oracle.backward(x["q"], x["k"], x["v"], x["dout"], w.scale, block_mask=mask)
    check_grads(grads, ref, f"sparse bwd d={d} N={N}")
    dq, dk, dv = (f64(t) for t in grads)
    assert np.all(dq[:, :, 128:256] == 0)
    assert np.all(dk[:, :, 256:384] == 0) and np.all(dv[:, :, 256:384] == 0)


def test_sparse_bwd_all_ones_equals_dense(fa):
    w = W.Workload("generic", 1, 3, 640, 64, causal=False, backward=True)
    x = W.make_inputs(w, 32)
    ones = np.ones((5, 5), dtype=np.uint8)
    gs = _sparse_bwd(fa, x, ones, w.scale)
    q, k, v, do = cuda(x["q"]), cuda(x["k"]), cuda(x["v"]), cuda(x["dout"])
    o, lse = fa.forward(q, k, v)
    gd = fa.backward(q, k, v, o, do, lse)
    torch.cuda.synchronize()
    assert torch.equal(gs[1], gd[1]) and torch.equal(gs[2], gd[2])
    # dQ sums tiles with fp32 reduce-adds: equal up to reduction order
    assert torch.allclose(gs[0].float(), gd[0].float(), rtol=0, atol=1e-2)


def test_sparse_bwd_full_size_workload(fa):
    w = W.WORKLOADS["blocksparse"]
    x = W.make_inputs(w, 0)
    mask = x["block_mask"].numpy()
    grads = _sparse_bwd(fa, x, mask, w.scale)
    heads = [(1, 3)]
    ref = oracle.backward(x["q"], x["k"], x["v"], x["dout"], w.scale, block_mask=mask,
                          heads=heads)
    for b, h in heads:
        check_grads([f64(t)[b, h] for t in grads], [r[b, h] for r in ref], f"blocksparse bwd {(b, h)}")


@pytest.mark.parametrize("d", [64, 128])
def test_sparse_kept_tiles_far_apart(fa, d):
    """Every mask row and column keeps two blocks 33 tiles apart (the walks over
    a mask scan 32 tiles per step): forward over all rows, backward of one head."""
    N = 128 * 40
    w = W.Workload("generic", 1, 2, N, d, causal=False, backward=True)
    x = W.make_inputs(w, 41 + d)
    nb = N // 128
    mask = np.zeros((nb, nb), dtype=np.uint8)
    for r in range(nb):
        mask[r, r] = 1
        mask[r, (r + 33) % nb] = 1
    q, k, v = cuda(x["q"]), cuda(x["k"]), cuda(x["v"])
    m = torch.from_numpy(mask).cuda()
    o, lse = fa.blocksparse_forward(q, k, v, m, scale=w.scale)
    torch.cuda.synchronize()
    assert fa.device_status() == 0
    o_ref, l_ref = oracle.forward(x["q"], x["k"], x["v"], w.scale, block_mask=mask)
    check_fwd(o, lse, o_ref, l_ref, f"sparse far apart d={d}")
    grads = _sparse_bwd(fa, x, mask, w.scale)
    ref = oracle.backward(x["q"], x["k"], x["v"], x["dout"], w.scale, block_mask=mask,
                          heads=[(0, 1)])
    check_grads([f64(t)[0, 1] for t in grads], [r[0, 1] for r in ref], f"sparse far apart bwd d={d}")


@pytest.mark.parametrize("d,causal", [(64, False), (128, False), (64, True)])
def test_sparse_skewed_costs(fa, d, causal):
    """Mask rows and columns that keep very different numbers of blocks (the
    items are dealt out heaviest first, from a per-CTA sort of the mask's rows
    or columns): a diagonal, two full rows and two full columns, a row and a
    column that keep nothing; more items than one wave of CTAs."""
    N = 128 * 40
    nb = N // 128
    w = W.Workload("generic", 2, 4, N, d, causal=causal, backward=True)
    x = W.make_inputs(w, 51 + d + int(causal))
    mask = np.zeros((nb, nb), dtype=np.uint8)
    np.fill_diagonal(mask, 1)
    mask[5, :] = 1
    mask[30, :] = 1
    mask[:, 7] = 1
    mask[:, 33] = 1
    mask[12, :] = 0
    mask[:, 20] = 0
    q, k, v, do = cuda(x["q"]), cuda(x["k"]), cuda(x["v"]), cuda(x["dout"])
    m = torch.from_numpy(mask).cuda()
    o, lse = fa.attention_forward(q, k, v, causal=causal, scale=w.scale, block_mask=m)
    g = fa.attention_backward(q, k, v, o, do, lse, causal=causal, scale=w.scale, block_mask=m)
    torch.cuda.synchronize()
    assert fa.device_status() == 0
    blocks = [0, 5, 7, 12, 30, 39]
    rows = np.concatenate([np.arange(b * 128, (b + 1) * 128) for b in blocks])
    o_ref, l_ref = oracle.forward(x["q"], x["k"], x["v"], w.scale, causal=causal, block_mask=mask,
                                  rows=rows)
    check_fwd(f64(o)[:, :, rows], f64(lse)[:, :, rows], o_ref, l_ref, f"skewed d={d} causal={causal}")
    assert np.all(f64(o)[:, :, 12 * 128:13 * 128] == 0)
    ref = oracle.backward(x["q"], x["k"], x["v"], x["dout"], w.scale, causal=causal, block_mask=mask,
                          heads=[(1, 2)])
    check_grads([f64(t)[1, 2] for t in g], [r[1, 2] for r in ref], f"skewed bwd d={d} causal={causal}")
    dk, dv = f64(g[1]), f64(g[2])
    assert np.all(dk[:, :, 20 * 128:21 * 128] == 0) and np.all(dv[:, :, 20 * 128:21 * 128] == 0)
