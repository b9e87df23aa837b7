"""Full-size consistency checks of the bench workloads, beyond the sampled
oracle comparisons of the other test files: every CTA's later items run, and
a race or an item run twice or not at all would show as a difference.

- Repeats: the same call twice gives the same bits for O, LSE, dK and dV
  (dQ sums its tiles with fp32 reduce-adds in any order: equal to 1e-2).
- Layouts: the same values stored as [B, N, H, d] give the same bits for O,
  LSE, dK and dV as the row-major call (a different memory access pattern and
  timing on every tile).
- Split of the last wave: with and without the split workspace the results
  agree to the parity bars (the merge sums partial results in another order).
- Key tiles that no query tile keeps (block mask) and rows of no valid key
  give exact zeros."""
import pytest
import torch

import workloads as W
from _util import O_ATOL, cuda

pytestmark = pytest.mark.gpu


def as_bnhd(t):
    """The same values stored as [B, N, H, d], returned as a [B, H, N, d] view."""
    return t.transpose(1, 2).contiguous().transpose(1, 2)


def _inputs(name):
    w = W.WORKLOADS[name]
    x = W.make_inputs(w, 0)
    q, k, v, do = (cuda(x[t]) for t in ("q", "k", "v", "dout"))
    kv = cuda(x.get("kv_len"))
    m = x.get("block_mask")
    m = None if m is None else m.cuda().contiguous()
    return w, q, k, v, do, kv, m


def _run(fa, w, q, k, v, do, kv, m, split=True):
    o, lse = fa.attention_forward(q, k, v, causal=w.causal, scale=w.scale, kv_len=kv, block_mask=m,
                                  split=split)
    g = fa.attention_backward(q, k, v, o, do, lse, causal=w.causal, scale=w.scale, kv_len=kv,
                              block_mask=m, split=split)
    torch.cuda.synchronize()
    assert fa.device_status() == 0
    return (o, lse, *g)


def _same(a, b, what):
    o1, l1, dq1, dk1, dv1 = a
    o2, l2, dq2, dk2, dv2 = b
    assert torch.equal(o1, o2), f"{what}: O differs"
    assert torch.equal(l1, l2), f"{what}: LSE differs"
    assert torch.equal(dk1, dk2), f"{what}: dK differs"
    assert torch.equal(dv1, dv2), f"{what}: dV differs"
    assert torch.allclose(dq1.float(), dq2.float(), rtol=0, atol=1e-2), f"{what}: dQ differs"


@pytest.mark.parametrize("name", ["long_n16384_noncausal", "gpt2_small", "bert_large", "blocksparse"])
def test_fullsize_repeat_and_layout(fa, name):
    w, q, k, v, do, kv, m = _inputs(name)
    a = _run(fa, w, q, k, v, do, kv, m)
    b = _run(fa, w, q, k, v, do, kv, m)
    _same(a, b, f"{name} repeated")
    for t in (a[0], *a[2:]):
        assert torch.isfinite(t.float()).all()
    assert not torch.isnan(a[1]).any()  # LSE: -inf only for rows that see no key
    c = _run(fa, w, as_bnhd(q), as_bnhd(k), as_bnhd(v), as_bnhd(do), kv, m)
    _same(a, c, f"{name} as [B,N,H,d]")
    if m is not None:  # key tiles no query tile keeps: dK = dV = 0 exactly
        dead = (m.sum(0) == 0).nonzero().flatten().tolist()
        for j in dead:
            assert not a[3][:, :, j * 128:(j + 1) * 128].any() and not a[4][:, :, j * 128:(j + 1) * 128].any()
    if kv is not None:  # keys past the valid length: dK = dV = 0 exactly
        for bi, n in enumerate(kv.tolist()):
            assert not a[3][bi, :, n:].any() and not a[4][bi, :, n:].any()


@pytest.mark.parametrize("name", ["long_n16384_noncausal", "long_n8192_noncausal", "long_n4096_noncausal"])
def test_fullsize_split_matches_unsplit(fa, name):
    w, q, k, v, do, kv, m = _inputs(name)
    a = _run(fa, w, q, k, v, do, kv, m, split=True)
    b = _run(fa, w, q, k, v, do, kv, m, split=False)
    assert (a[0].float() - b[0].float()).abs().max().item() <= O_ATOL
    assert (a[1] - b[1]).abs().max().item() <= 1e-3
    for x, y, nm in zip(a[2:], b[2:], ("dQ", "dK", "dV")):
        err = (x.float() - y.float()).abs().max().item()
        assert err <= 2e-2 * y.float().abs().max().item(), f"{name} {nm}: split vs unsplit {err}"
