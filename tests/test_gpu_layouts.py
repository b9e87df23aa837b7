"""General entry points (fa_attention_fwd / fa_attention_bwd): strided layouts
and every mask option at once, against the oracle on the same seeded inputs.

Layout is data movement only, so a strided call must give the same bits as
the row-major call on the same values (dQ up to the order of its fp32
additions); the oracle then checks the row-major result, and the combined
options are checked against the oracle directly."""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from _util import GRAD_REL, O_ATOL, check_fwd, check_grads, cuda, f64

pytestmark = pytest.mark.gpu


def as_bnhd(t):
    """The same values stored as [B, N, H, d], returned as a [B, H, N, d] view."""
    return t.transpose(1, 2).contiguous().transpose(1, 2)


def as_padded(t, pad):
    """The same values in rows of d + pad elements, as a [B, H, N, d] view."""
    B, H, N, d = t.shape
    s = torch.zeros((B, H, N, d + pad), dtype=t.dtype, device=t.device)
    s[..., :d] = t
    return s[..., :d]


def generic(B, H, N, d, causal, seed):
    w = W.Workload("generic", B, H, N, d, causal=causal, backward=True)
    return w, W.make_inputs(w, seed)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("layout", ["bnhd", "padded"])
def test_strided_equals_row_major_and_oracle(fa, d, causal, layout):
    w, x = generic(2, 3, 1000, d, causal, seed=40 + d)
    q, k, v, do = cuda(x["q"]), cuda(x["k"]), cuda(x["v"]), cuda(x["dout"])
    o, lse = fa.forward(q, k, v, causal=causal)
    g = fa.backward(q, k, v, o, do, lse, causal=causal)
    conv = as_bnhd if layout == "bnhd" else (lambda t: as_padded(t, 64))
    qs, ks, vs, dos = conv(q), conv(k), conv(v), conv(do)
    assert not qs.is_contiguous()
    os_, lses = fa.attention_forward(qs, ks, vs, causal=causal)
    gs = fa.attention_backward(qs, ks, vs, os_, dos, lses, causal=causal)
    torch.cuda.synchronize()
    assert fa.device_status() == 0
    assert os_.stride() == qs.stride() and gs[0].stride() == qs.stride()
    assert torch.equal(os_, o) and torch.equal(lses, lse)
    assert torch.equal(gs[1], g[1]) and torch.equal(gs[2], g[2])
    assert torch.allclose(gs[0].float(), g[0].float(), rtol=0, atol=1e-2)
    o_ref, l_ref = oracle.forward(x["q"], x["k"], x["v"], w.scale, causal=causal)
    check_fwd(os_, lses, o_ref, l_ref, f"{layout} d={d} causal={causal}")
    ref = oracle.backward(x["q"], x["k"], x["v"], x["dout"], w.scale, causal=causal)
    check_grads(gs, ref, f"{layout} d={d} causal={causal}")


def test_default_options_equal_plain_calls(fa):
    w, x = generic(2, 2, 640, 64, True, seed=44)
    q, k, v, do = cuda(x["q"]), cuda(x["k"]), cuda(x["v"]), cuda(x["dout"])
    o1, l1 = fa.attention_forward(q, k, v, causal=True)
    o2, l2 = fa.forward(q, k, v, causal=True)
    g1 = fa.attention_backward(q, k, v, o1, do, l1, causal=True)
    g2 = fa.backward(q, k, v, o2, do, l2, causal=True)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    assert torch.equal(g1[1], g2[1]) and torch.equal(g1[2], g2[2])


def _random_mask(nb, seed, empty_row=None, empty_col=None):
    g = np.random.default_rng(seed)
    m = (g.random((nb, nb)) < 0.5).astype(np.uint8)
    np.fill_diagonal(m, 1)
    if empty_row is not None:
        m[empty_row, :] = 0
    if empty_col is not None:
        m[:, empty_col] = 0
    return m


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("N", [640, 1000])
def test_causal_block_sparse(fa, d, N):
    w, x = generic(2, 2, N, d, True, seed=N + d + 5)
    nb = (N + 127) // 128
    m = _random_mask(nb, N + d, empty_row=2, empty_col=1)
    m[3, 3] = 0                      # a diagonal block dropped: row tile 3 sees only j < 3
    q, k, v, do = cuda(x["q"]), cuda(x["k"]), cuda(x["v"]), cuda(x["dout"])
    mt = torch.from_numpy(m).cuda()
    o, lse = fa.attention_forward(q, k, v, causal=True, block_mask=mt)
    g = fa.attention_backward(q, k, v, o, do, lse, causal=True, block_mask=mt)
    torch.cuda.synchronize()
    assert fa.device_status() == 0
    o_ref, l_ref = oracle.forward(x["q"], x["k"], x["v"], w.scale, causal=True, block_mask=m)
    check_fwd(o, lse, o_ref, l_ref, f"causal sparse d={d} N={N}")
    ref = oracle.backward(x["q"], x["k"], x["v"], x["dout"], w.scale, causal=True, block_mask=m)
    check_grads(g, ref, f"causal sparse d={d} N={N}")
    assert np.all(np.isneginf(f64(lse)[:, :, 256:384]))          # the empty row tile
    assert np.all(f64(g[1])[:, :, 128:256] == 0) and np.all(f64(g[2])[:, :, 128:256] == 0)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_every_option_at_once(fa, d, causal):
    # [B, N, H, d] storage + key padding + block mask + dropout (+ causal).
    # Rows that see exactly one key are left to the next test: there the
    # exact softmax gradient is zero and what remains is the rounding of D.
    kv = torch.tensor([2, 300, 777], dtype=torch.int32)
    w, x = generic(3, 2, 777, d, causal, seed=50 + d)
    nb = 7
    m = _random_mask(nb, d + int(causal), empty_row=4)
    p, seed, off = 0.25, 0xABCDEF0123, 17
    p32 = float(np.float32(p))
    q, k, v, do = (as_bnhd(cuda(x[n])) for n in ("q", "k", "v", "dout"))
    mt, kvt = torch.from_numpy(m).cuda(), kv.cuda()
    kw = dict(causal=causal, kv_len=kvt, block_mask=mt, dropout_p=p, seed=seed, offset=off)
    o, lse = fa.attention_forward(q, k, v, **kw)
    g = fa.attention_backward(q, k, v, o, do, lse, **kw)
    torch.cuda.synchronize()
    assert fa.device_status() == 0
    r = oracle.rescale(oracle.threshold(p32))
    drop = (p32, seed, off)
    o_ref, l_ref = oracle.forward(x["q"], x["k"], x["v"], w.scale, causal=causal,
                                  kv_len=kv.numpy(), block_mask=m, dropout=drop)
    # O is stored in bf16: beyond the plain bar scaled by r, the rounding of
    # the exact value itself (unit roundoff 2^-8 of |O|) can not be avoided
    # once r |v| passes 2 (kv_len 2 rows with one key dropped give O = r v_j).
    err = np.abs(f64(o) - o_ref)
    assert np.all(err <= O_ATOL * r + 2.0 ** -8 * np.abs(o_ref)), err.max()
    check_fwd(o, lse, o_ref, l_ref, f"all options d={d} causal={causal}", np.inf)
    ref = oracle.backward(x["q"], x["k"], x["v"], x["dout"], w.scale, causal=causal,
                          kv_len=kv.numpy(), block_mask=m, dropout=drop)
    check_grads(g, ref, f"all options d={d} causal={causal}", GRAD_REL * r)


@pytest.mark.parametrize("d", [64, 128])
def test_single_visible_key_with_dropout(fa, d):
    # Batch 0 sees only key 0 (kv_len = 1), so P = 1 there, O_i = Z_i0 r v_0,
    # and the exact dS of every row is 0: dQ = 0 for the batch and dK is 0
    # except that the kernel forms D = rowsum(dO * O) from the bf16 O, so each
    # kept row adds dO_i . (r v_0 - bf16(r v_0)) to dS_i0. That is bounded by
    # |delta D_i| <= sum_c |dO_ic| * 2^-8 |O_ic| (bf16 half-ulp), which gives
    # |dK_0| <= scale * sum_i |delta D_i| |q_i| per column (plus fp32 and the
    # bf16 rounding of dS and dK). The other batch is checked against the oracle.
    kv = torch.tensor([1, 400], dtype=torch.int32)
    w, x = generic(2, 2, 400, d, False, seed=60 + d)
    p, seed, off = 0.2, 77, 0
    q, k, v, do = cuda(x["q"]), cuda(x["k"]), cuda(x["v"]), cuda(x["dout"])
    kw = dict(kv_len=kv.cuda(), dropout_p=p, seed=seed, offset=off)
    o, lse = fa.attention_forward(q, k, v, **kw)
    dq, dk, dv = fa.attention_backward(q, k, v, o, do, lse, **kw)
    torch.cuda.synchronize()
    assert fa.device_status() == 0
    assert torch.count_nonzero(dk[0, :, 1:]) == 0 and torch.count_nonzero(dv[0, :, 1:]) == 0
    qq, kk, oo, dd = f64(q[0]), f64(k[0]), f64(o[0]), f64(do[0])
    delta = (np.abs(dd) * np.abs(oo) * 2.0 ** -8).sum(-1)              # [H, N] bound on |delta D|
    bound_k = w.scale * (delta[..., None] * np.abs(qq)).sum(1)         # [H, d]: |dK_0|
    bound_q = w.scale * delta[..., None] * np.abs(kk[:, :1, :])        # [H, N, d]: |dQ_i|
    got_k, got_q = np.abs(f64(dk[0, :, 0])), np.abs(f64(dq[0]))
    assert np.all(got_k <= 1.02 * bound_k + 1e-3), (got_k / (bound_k + 1e-9)).max()
    assert np.all(got_q <= 1.02 * bound_q + 1e-3), (got_q / (bound_q + 1e-9)).max()
    ref = oracle.backward(x["q"], x["k"], x["v"], x["dout"], w.scale, kv_len=kv.numpy(),
                          heads=[(1, 0), (1, 1)], dropout=(float(np.float32(p)), seed, off))
    r = oracle.rescale(oracle.threshold(float(np.float32(p))))
    check_grads([f64(t)[1] for t in (dq, dk, dv)], [g[1] for g in ref], "kv_len 400 batch",
                GRAD_REL * r)
