"""Fused-dropout parity: the CUDA path (through the C-ABI) against the oracle
with the same (p, seed, offset).

The keep decisions are integer work and must match bit for bit
(fa_dropout_mask against oracle.keep_mask, over ragged sizes and every head).
O and LSE and the gradients are held to the bars of the pass without dropout
with the O and gradient bars multiplied by r = 1 / (1 - p'): every kept
probability, the output O and the kept entries of dS carry that factor, and
so does their bf16 rounding (the output O is bf16; an exact O of 4.18 already
rounds by 1.2e-2 at r = 1.25). A CPU emulation of the kernels' roundings
(bf16 P, dS and O, fp32 elsewhere) reproduces the measured errors. The dropout
probability is passed to the oracle as the float32 value that the library
receives, so both sides take the threshold from the same number."""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from _util import GRAD_REL, O_ATOL, check_fwd, check_grads, cuda, f64

pytestmark = pytest.mark.gpu


def p32(p):
    return float(np.float32(p))


def bars(p):
    """(O max-abs bar, gradient relative bar) at drop probability p."""
    r = oracle.rescale(oracle.threshold(p32(p)))
    return O_ATOL * r, GRAD_REL * r


def run(fa, x, causal, scale, p, seed, offset, kv_len=None, backward=True):
    q, k, v = cuda(x["q"]), cuda(x["k"]), cuda(x["v"])
    kv = cuda(kv_len)
    o, lse = fa.dropout_forward(q, k, v, p, seed, offset, causal=causal, scale=scale, kv_len=kv)
    g = None
    if backward:
        g = fa.dropout_backward(q, k, v, o, cuda(x["dout"]), lse, p, seed, offset, causal=causal,
                                scale=scale, kv_len=kv)
    torch.cuda.synchronize()
    assert fa.device_status() == 0
    return o, lse, g


def generic(B, H, N, d, causal, seed, backward=True):
    w = W.Workload("generic", B, H, N, d, causal=causal, backward=backward)
    return w, W.make_inputs(w, seed)


# ---------------------------------------------------------------- keep decisions
@pytest.mark.parametrize("N,p", [(1, 0.5), (17, 0.1), (300, 0.5), (1000, 0.9)])
def test_mask_matches_oracle_bitwise(fa, N, p):
    B, H, seed, off = 2, 3, 0xDEADBEEF12345678, 77
    keep = fa.dropout_mask(B, H, N, p, seed, off).cpu().numpy().astype(bool)
    for b in range(B):
        for h in range(H):
            ref = oracle.keep_mask(b * H + h, np.arange(N), N, seed, off, p32(p))
            assert np.array_equal(keep[b, h], ref), (b, h)


def test_mask_full_size_heads(fa):
    # gpt2_small shape (B=8, H=12, N=1024): the whole mask on the device,
    # three heads and the kept fraction checked against the oracle.
    B, H, N, p, seed, off = 8, 12, 1024, 0.1, 1234, 5
    keep = fa.dropout_mask(B, H, N, p, seed, off)
    frac = keep.float().mean().item()
    t = oracle.threshold(p32(p))
    n = keep.numel()
    assert abs(frac - (1 - t / 256)) < 6 * np.sqrt((t / 256) * (1 - t / 256) / n)
    for b, h in [(0, 0), (3, 7), (7, 11)]:
        ref = oracle.keep_mask(b * H + h, np.arange(N), N, seed, off, p32(p))
        assert np.array_equal(keep[b, h].cpu().numpy().astype(bool), ref), (b, h)


# ---------------------------------------------------------------- forward
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N", [128, 384, 1000])
def test_fwd_small_sweep(fa, d, causal, N):
    w, x = generic(2, 2, N, d, causal, seed=N + d, backward=False)
    p, seed, off = 0.2, 42 + N, 3
    o, lse, _ = run(fa, x, causal, w.scale, p, seed, off, backward=False)
    o_ref, l_ref = oracle.forward(x["q"], x["k"], x["v"], w.scale, causal=causal,
                                  dropout=(p32(p), seed, off))
    check_fwd(o, lse, o_ref, l_ref, f"dropout fwd d={d} causal={causal} N={N}", bars(p)[0])


@pytest.mark.parametrize("d", [64, 128])
def test_fwd_high_drop_rate_and_kv_len(fa, d):
    kv = torch.tensor([1, 129, 500], dtype=torch.int32)
    w, x = generic(3, 2, 500, d, False, seed=7, backward=False)
    p, seed, off = 0.75, 99, 0
    o, lse, _ = run(fa, x, False, w.scale, p, seed, off, kv_len=kv, backward=False)
    o_ref, l_ref = oracle.forward(x["q"], x["k"], x["v"], w.scale, kv_len=kv.numpy(),
                                  dropout=(p32(p), seed, off))
    check_fwd(o, lse, o_ref, l_ref, f"dropout fwd p=0.75 kv_len d={d}", bars(p)[0])


def test_p_zero_equals_plain_bitwise(fa):
    w, x = generic(2, 3, 640, 64, True, seed=8)
    q, k, v, do = cuda(x["q"]), cuda(x["k"]), cuda(x["v"]), cuda(x["dout"])
    o1, l1 = fa.dropout_forward(q, k, v, 0.0, 5, 0, causal=True)
    o2, l2 = fa.forward(q, k, v, causal=True)
    g1 = fa.dropout_backward(q, k, v, o1, do, l1, 0.0, 5, 0, causal=True)
    g2 = fa.backward(q, k, v, o2, do, l2, causal=True)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    assert torch.equal(g1[1], g2[1]) and torch.equal(g1[2], g2[2])
    assert torch.allclose(g1[0].float(), g2[0].float(), rtol=0, atol=1e-2)  # dQ: atomic order


def test_same_arguments_same_result_new_offset_new_mask(fa):
    w, x = generic(1, 2, 384, 64, False, seed=9, backward=False)
    a = run(fa, x, False, w.scale, 0.3, 11, 0, backward=False)[0]
    b = run(fa, x, False, w.scale, 0.3, 11, 0, backward=False)[0]
    c = run(fa, x, False, w.scale, 0.3, 11, 1, backward=False)[0]
    assert torch.equal(a, b)
    assert not torch.equal(a, c)


# ---------------------------------------------------------------- backward
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N", [128, 1000])
def test_bwd_small_sweep(fa, d, causal, N):
    w, x = generic(2, 2, N, d, causal, seed=N + d + 3)
    p, seed, off = 0.2, 1000 + N, 9
    _, _, g = run(fa, x, causal, w.scale, p, seed, off)
    ref = oracle.backward(x["q"], x["k"], x["v"], x["dout"], w.scale, causal=causal,
                          dropout=(p32(p), seed, off))
    check_grads(g, ref, f"dropout bwd d={d} causal={causal} N={N}", bars(p)[1])


@pytest.mark.parametrize("d", [64, 128])
def test_bwd_kv_len_and_high_drop_rate(fa, d):
    kv = torch.tensor([1, 128, 300, 429], dtype=torch.int32)
    w, x = generic(4, 2, 429, d, True, seed=12)
    p, seed, off = 0.6, 2024, 1
    _, _, g = run(fa, x, True, w.scale, p, seed, off, kv_len=kv)
    ref = oracle.backward(x["q"], x["k"], x["v"], x["dout"], w.scale, causal=True,
                          kv_len=kv.numpy(), dropout=(p32(p), seed, off))
    check_grads(g, ref, f"dropout bwd kv_len d={d}", bars(p)[1])
    dk, dv = f64(g[1]), f64(g[2])
    for b, L in enumerate(kv.tolist()):
        assert np.all(dk[b, :, L:] == 0) and np.all(dv[b, :, L:] == 0)


def test_full_size_gpt2_small(fa):
    # The GPT-2 small workload (B=8, H=12, N=1024, d=64, causal) with p = 0.1:
    # forward and gradients of three heads against the oracle.
    w = W.WORKLOADS["gpt2_small"]
    x = W.make_inputs(w, 0)
    p, seed, off = 0.1, 0x5EED, 0
    o, lse, g = run(fa, x, True, w.scale, p, seed, off)
    heads = [(0, 0), (4, 6), (7, 11)]
    o_ref, l_ref = oracle.forward(x["q"], x["k"], x["v"], w.scale, causal=True, heads=heads,
                                  dropout=(p32(p), seed, off))
    ref = oracle.backward(x["q"], x["k"], x["v"], x["dout"], w.scale, causal=True, heads=heads,
                          dropout=(p32(p), seed, off))
    for b, h in heads:
        check_fwd(f64(o)[b, h], f64(lse)[b, h], o_ref[b, h], l_ref[b, h], f"gpt2 head {(b, h)}",
                  bars(p)[0])
        check_grads([f64(t)[b, h] for t in g], [r[b, h] for r in ref], f"gpt2 head {(b, h)}",
                    bars(p)[1])
