"""Block-sparse forward parity: the CUDA path vs the dense oracle with the
masked 128 x 128 blocks set to -inf."""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from _util import check_fwd, cuda, f64

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
