"""Where the dropout bars come from, checked on the CPU.

A rounding model of the kernels (NumPy; it shares nothing with the CUDA code):
P is rounded to bf16 before it meets V or dS, O and dS are rounded to bf16,
everything else is exact. On the GPU parity cases it predicts the measured
errors; here it shows, against the oracle, the two facts the dropout bars rest
on:

* rounding the exact O to bf16 already misses an O bar of 1e-2 once |O|
  passes 2.56, which dropout's 1 / (1 - p') makes common (the O bar is scaled
  by that factor and gets the bf16 unit roundoff 2^-8 |O| where |O| is large);
* with D = rowsum(dO * O) taken from the bf16 O, rows that see a single key
  put the rounding of O straight into dS (their exact dS is 0), and dK sums it
  over the rows: far above the gradient bar at kv_len = 1, yet near the bar
  with an exact D and at kv_len = 2. Hence the separate bound for that case.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from oracle import dropout as od


def bf16(x):
    return torch.from_numpy(np.asarray(x, np.float32)).to(torch.bfloat16).double().numpy()


def model_dk(x, w, kv, p, seed, off, exact_d=False):
    """dK of the rounding model for a [B, H, N, d] problem with key padding and dropout."""
    q, k, v, do = (oracle.to_f64(x[n]) for n in ("q", "k", "v", "dout"))
    B, H, N, _ = q.shape
    r = od.rescale(od.threshold(p))
    dk = np.zeros_like(k)
    for b in range(B):
        for h in range(H):
            P = oracle.head_probs(q[b, h], k[b, h], w.scale, w.causal, int(kv[b]))
            Z = od.keep_mask(b * H + h, np.arange(N), N, seed, off, p)
            dpd = np.where(Z, (do[b, h] @ v[b, h].T) * r, 0.0)
            if exact_d:
                D = (P * dpd).sum(1)
            else:
                O = bf16((bf16(P) * Z) @ v[b, h] * r)
                D = (O * do[b, h]).sum(1)
            dS = bf16(bf16(P) * (dpd - D[:, None]))
            dk[b, h] = w.scale * dS.T @ q[b, h]
    return bf16(dk)


def rel(g, ref):
    return np.abs(g - ref).max() / np.abs(ref).max()


def test_bf16_rounding_of_the_exact_output_exceeds_the_plain_o_bar():
    # the forward case measured on the GPU (d = 64, causal, N = 1000, p = 0.2)
    w = W.Workload("generic", 2, 2, 1000, 64, causal=True, backward=False)
    x = W.make_inputs(w, 1064)
    p = float(np.float32(0.2))
    o, _ = oracle.forward(x["q"], x["k"], x["v"], w.scale, causal=True, dropout=(p, 1042, 3))
    err = np.abs(bf16(o) - o).max()
    r = od.rescale(od.threshold(p))
    assert 1e-2 < err <= 1e-2 * r                      # beyond the plain bar, inside the scaled one
    assert np.all(np.abs(bf16(o) - o) <= 2.0 ** -8 * np.abs(o) + 1e-12)   # unit roundoff


@pytest.mark.parametrize("d", [64, 128])
def test_single_visible_key_rows_need_their_own_bound(d):
    kv1 = np.array([1, 300, 777])
    w = W.Workload("generic", 3, 2, 777, d, causal=False, backward=True)
    x = W.make_inputs(w, 50 + d)
    p = float(np.float32(0.25))
    seed, off = 0xABCDEF0123, 17
    r = od.rescale(od.threshold(p))
    bar = 2e-2 * r
    ref1 = oracle.backward(x["q"], x["k"], x["v"], x["dout"], w.scale, kv_len=kv1,
                           dropout=(p, seed, off))[1]
    e_model = rel(model_dk(x, w, kv1, p, seed, off), ref1)
    e_exact = rel(model_dk(x, w, kv1, p, seed, off, exact_d=True), ref1)
    assert e_exact < 0.5 * bar                          # the kernels' other roundings are small
    assert e_model > 4 * e_exact                        # D from the bf16 O dominates
    kv2 = np.array([2, 300, 777])
    ref2 = oracle.backward(x["q"], x["k"], x["v"], x["dout"], w.scale, kv_len=kv2,
                           dropout=(p, seed, off))[1]
    assert rel(model_dk(x, w, kv2, p, seed, off), ref2) < bar
