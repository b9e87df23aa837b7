"""Pins of the CPU fp64 oracle against facts that do not come from the oracle.

Each check is chosen so that a plausible slip in the oracle (a dropped scale,
a transposed operand, a wrong mask direction, a wrong log base, a sign error in
the softmax Jacobian) fails at least one of them:

* a hand-derived worked example (tests/golden/) of the attention definition;
* closed forms: identical keys give the mean of the visible values and
  LSE = scale*q.k + ln(n); a single dominant logit returns that value row;
  N = 1 gives O = V;
* invariants: rows of P are probability vectors, zero where masked;
* special cases that reduce to smaller dense problems (key padding, causal
  prefix, block masks, permutation of keys, shift of a row's logits);
* central finite differences of L = sum(dO * O) for the backward pass, and the
  explicit-Jacobian route against the vector route.
"""
import json
import math
import os

import numpy as np
import pytest

import oracle
from oracle import attention as oa

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "worked_example_n3_d2.json")


def rng(seed=0):
    return np.random.default_rng(seed)


# --------------------------------------------------------------- worked example
@pytest.fixture(scope="module")
def golden():
    with open(GOLDEN) as f:
        return json.load(f)


def test_golden_noncausal(golden):
    q, k, v = (np.array(golden[x]) for x in ("q", "k", "v"))
    o, lse = oracle.head_forward(q, k, v, golden["scale"])
    ref = golden["noncausal"]
    np.testing.assert_allclose(o, ref["O"], rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, ref["LSE"], rtol=0, atol=1e-12)
    p = oracle.head_probs(q, k, golden["scale"])
    np.testing.assert_allclose(p, ref["P"], rtol=0, atol=1e-12)


def test_golden_causal(golden):
    q, k, v = (np.array(golden[x]) for x in ("q", "k", "v"))
    o, lse = oracle.head_forward(q, k, v, golden["scale"], causal=True)
    np.testing.assert_allclose(o, golden["causal"]["O"], rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, golden["causal"]["LSE"], rtol=0, atol=1e-12)


def test_golden_kv_len(golden):
    q, k, v = (np.array(golden[x]) for x in ("q", "k", "v"))
    o, lse = oracle.head_forward(q, k, v, golden["scale"], kv_len=2)
    np.testing.assert_allclose(o, golden["kv_len_2"]["O"], rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, golden["kv_len_2"]["LSE"], rtol=0, atol=1e-12)


def test_golden_scale_enters_logits(golden):
    # Doubling the scale equals doubling q: S = scale * q.k (reading of where the scale applies).
    q, k, v = (np.array(golden[x]) for x in ("q", "k", "v"))
    o2, l2 = oracle.head_forward(q, k, v, 2.0)
    o1, l1 = oracle.head_forward(2.0 * q, k, v, 1.0)
    np.testing.assert_allclose(o2, o1, atol=1e-12)
    np.testing.assert_allclose(l2, l1, atol=1e-12)
    # and row 0 with scale 2: exp(2 ln3) = 9 -> P = [9/11, 1/11, 1/11], LSE = ln 11
    np.testing.assert_allclose(l2[0], math.log(11.0), atol=1e-12)


# --------------------------------------------------------------- closed forms
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("kv_len", [None, 5])
def test_identical_keys(causal, kv_len):
    r = rng(1)
    n, d, s = 9, 4, 0.37
    q = r.normal(size=(n, d))
    kvec = r.normal(size=d)
    k = np.tile(kvec, (n, 1))
    v = r.normal(size=(n, 3))
    o, lse = oracle.head_forward(q, k, v, s, causal=causal, kv_len=kv_len)
    for i in range(n):
        hi = n
        if kv_len is not None:
            hi = min(hi, kv_len)
        if causal:
            hi = min(hi, i + 1)
        np.testing.assert_allclose(o[i], v[:hi].mean(axis=0), atol=1e-12)
        np.testing.assert_allclose(lse[i], s * q[i] @ kvec + math.log(hi), atol=1e-12)
    if causal:
        np.testing.assert_allclose(o[0], v[0], atol=1e-15)


def test_dominant_logit():
    r = rng(2)
    n, d = 16, 8
    k = r.normal(size=(n, d))
    k /= np.linalg.norm(k, axis=1, keepdims=True)
    v = r.normal(size=(n, 5))
    target = r.integers(0, n, size=n)
    # q_i = c * k_t: logit of key t is c, of any other key c*cos < c - margin
    cos = k @ k.T
    gap = 1.0 - np.max(np.where(np.eye(n, dtype=bool), -np.inf, cos))
    c = 80.0 / gap
    q = c * k[target]
    o, lse = oracle.head_forward(q, k, v, 1.0)
    np.testing.assert_allclose(o, v[target], atol=1e-20 + 1e-12)
    np.testing.assert_allclose(lse, c * np.ones(n), rtol=1e-12)


def test_single_key():
    r = rng(3)
    q, k, v = r.normal(size=(1, 6)), r.normal(size=(1, 6)), r.normal(size=(1, 6))
    o, lse = oracle.head_forward(q, k, v, 0.5)
    np.testing.assert_allclose(o, v, atol=1e-15)
    np.testing.assert_allclose(lse, 0.5 * q[0] @ k[0], atol=1e-15)


# --------------------------------------------------------------- invariants
@pytest.mark.parametrize("causal", [False, True])
def test_probability_rows(causal):
    r = rng(4)
    n = 300
    q, k = r.normal(size=(n, 16)), r.normal(size=(n, 16))
    bm = np.array([[1, 0, 1], [0, 1, 0], [1, 1, 1]], dtype=np.uint8)
    p = oracle.head_probs(q, k, 0.25, causal=causal, kv_len=270, block_mask=bm)
    keep = oracle.visible(np.arange(n), n, causal, 270, bm)
    assert np.all(p >= 0)
    assert np.all(p[~keep] == 0)
    sums = p.sum(axis=1)
    live = keep.any(axis=1)
    np.testing.assert_allclose(sums[live], 1.0, atol=1e-12)
    assert np.all(sums[~live] == 0)


def test_visible_mask_semantics():
    keep = oracle.visible(np.arange(4), 4, causal=True)
    np.testing.assert_array_equal(keep, np.tril(np.ones((4, 4), bool)))
    keep = oracle.visible(np.arange(3), 5, causal=False, kv_len=2)
    assert keep[:, :2].all() and not keep[:, 2:].any()
    # asymmetric block mask: block (row 0, col 1) dropped, (row 1, col 0) kept
    bm = np.array([[1, 0], [1, 1]], dtype=np.uint8)
    keep = oracle.visible(np.arange(256), 256, False, None, bm)
    assert keep[0, 0] and not keep[0, 200] and keep[200, 0] and keep[200, 200]


# --------------------------------------------------------------- special cases
def test_kv_len_equals_truncated_dense():
    r = rng(5)
    n, L = 40, 23
    q, k, v = r.normal(size=(n, 8)), r.normal(size=(n, 8)), r.normal(size=(n, 8))
    o, lse = oracle.head_forward(q, k, v, 0.3, kv_len=L)
    o2, lse2 = oracle.head_forward(q, k[:L], v[:L], 0.3)
    np.testing.assert_allclose(o, o2, atol=1e-13)
    np.testing.assert_allclose(lse, lse2, atol=1e-13)
    o3, _ = oracle.head_forward(q, k, v, 0.3, kv_len=n)
    o4, _ = oracle.head_forward(q, k, v, 0.3)
    np.testing.assert_array_equal(o3, o4)


def test_causal_row_is_prefix_dense():
    r = rng(6)
    n = 30
    q, k, v = r.normal(size=(n, 8)), r.normal(size=(n, 8)), r.normal(size=(n, 8))
    o, lse = oracle.head_forward(q, k, v, 0.4, causal=True)
    for i in (0, 1, 7, 29):
        oi, li = oracle.head_forward(q[i:i + 1], k[:i + 1], v[:i + 1], 0.4)
        np.testing.assert_allclose(o[i], oi[0], atol=1e-13)
        np.testing.assert_allclose(lse[i], li[0], atol=1e-13)


def test_block_mask_reduces_to_dense_subsets():
    r = rng(7)
    n = 3 * oracle.BLOCK
    q, k, v = r.normal(size=(n, 8)), r.normal(size=(n, 8)), r.normal(size=(n, 8))
    bm = np.array([[1, 0, 0], [1, 0, 1], [1, 1, 1]], dtype=np.uint8)
    o, lse = oracle.head_forward(q, k, v, 0.2, block_mask=bm)
    B = oracle.BLOCK
    for rb in range(3):
        cols = np.concatenate([np.arange(c * B, (c + 1) * B) for c in range(3) if bm[rb, c]])
        rows = np.arange(rb * B, (rb + 1) * B)
        o2, l2 = oracle.head_forward(q[rows], k[cols], v[cols], 0.2)
        np.testing.assert_allclose(o[rows], o2, atol=1e-13)
        np.testing.assert_allclose(lse[rows], l2, atol=1e-13)
    ones = np.ones((3, 3), np.uint8)
    o3, _ = oracle.head_forward(q, k, v, 0.2, block_mask=ones)
    o4, _ = oracle.head_forward(q, k, v, 0.2)
    np.testing.assert_array_equal(o3, o4)


def test_empty_row_convention():
    r = rng(8)
    n = 2 * oracle.BLOCK
    q, k, v, do = (r.normal(size=(n, 4)) for _ in range(4))
    bm = np.array([[0, 0], [1, 1]], dtype=np.uint8)
    o, lse = oracle.head_forward(q, k, v, 0.5, block_mask=bm)
    assert np.all(o[:oracle.BLOCK] == 0) and np.all(np.isneginf(lse[:oracle.BLOCK]))
    assert np.all(np.isfinite(lse[oracle.BLOCK:]))
    dq, dk, dv = oracle.head_backward(q, k, v, do, 0.5, block_mask=bm)
    assert np.all(dq[:oracle.BLOCK] == 0)
    assert np.all(np.isfinite(dk)) and np.all(np.isfinite(dv))


def test_key_permutation_invariance():
    r = rng(9)
    n = 50
    q, k, v = r.normal(size=(n, 8)), r.normal(size=(n, 8)), r.normal(size=(n, 6))
    perm = r.permutation(n)
    o, lse = oracle.head_forward(q, k, v, 0.3)
    o2, lse2 = oracle.head_forward(q, k[perm], v[perm], 0.3)
    np.testing.assert_allclose(o, o2, atol=1e-13)
    np.testing.assert_allclose(lse, lse2, atol=1e-13)


def test_row_logit_shift():
    # Give every key a constant last coordinate 1: adding c to q_i's last
    # coordinate adds scale*c to every logit of row i.
    r = rng(10)
    n, s = 20, 0.6
    q, k, v = r.normal(size=(n, 5)), r.normal(size=(n, 5)), r.normal(size=(n, 3))
    k[:, -1] = 1.0
    shift = r.normal(size=n) * 10
    q2 = q.copy()
    q2[:, -1] += shift
    o, lse = oracle.head_forward(q, k, v, s)
    o2, lse2 = oracle.head_forward(q2, k, v, s)
    np.testing.assert_allclose(o, o2, atol=1e-12)
    np.testing.assert_allclose(lse2 - lse, s * shift, atol=1e-12)


def test_chunking_does_not_change_results(monkeypatch):
    r = rng(11)
    n = 70
    q, k, v, do = (r.normal(size=(n, 8)) for _ in range(4))
    full = oracle.head_forward(q, k, v, 0.3, causal=True)
    gfull = oracle.head_backward(q, k, v, do, 0.3, causal=True)
    monkeypatch.setattr(oa, "_CHUNK_ELEMS", 3 * n)       # 3 rows per chunk
    part = oracle.head_forward(q, k, v, 0.3, causal=True)
    gpart = oracle.head_backward(q, k, v, do, 0.3, causal=True)
    for a, b in zip(full + gfull, part + gpart):
        np.testing.assert_allclose(a, b, atol=1e-13)


def test_batched_wrappers_apply_per_batch_kv_len():
    r = rng(12)
    B, H, N, d = 2, 2, 12, 4
    q, k, v, do = (r.normal(size=(B, H, N, d)) for _ in range(4))
    kv = np.array([5, 12], np.int32)
    o, lse = oracle.forward(q, k, v, 0.5, kv_len=kv)
    dq, dk, dv = oracle.backward(q, k, v, do, 0.5, kv_len=kv)
    for b in range(B):
        for h in range(H):
            ob, lb = oracle.head_forward(q[b, h], k[b, h], v[b, h], 0.5, kv_len=int(kv[b]))
            np.testing.assert_array_equal(o[b, h], ob)
            np.testing.assert_array_equal(lse[b, h], lb)
            g = oracle.head_backward(q[b, h], k[b, h], v[b, h], do[b, h], 0.5, kv_len=int(kv[b]))
            np.testing.assert_array_equal(dq[b, h], g[0])
            np.testing.assert_array_equal(dv[b, h], g[2])
    # sampled heads / rows leave the rest NaN and match the full answer
    o2, l2 = oracle.forward(q, k, v, 0.5, kv_len=kv, heads=[(1, 0)], rows=[0, 7, 11])
    np.testing.assert_array_equal(o2[1, 0], o[1, 0][[0, 7, 11]])
    assert np.isnan(o2[0, 0]).all()


# --------------------------------------------------------------- backward
def _fd_grads(q, k, v, do, s, **kw):
    h = 1e-6
    out = []
    for which, x in enumerate((q, k, v)):
        g = np.zeros_like(x)
        for idx in np.ndindex(x.shape):
            args = [q.copy(), k.copy(), v.copy()]
            args[which][idx] += h
            lp = oracle.loss(*args, do, s, **kw)
            args[which][idx] -= 2 * h
            lm = oracle.loss(*args, do, s, **kw)
            g[idx] = (lp - lm) / (2 * h)
        out.append(g)
    return out


@pytest.mark.parametrize("causal,kv_len", [(False, None), (True, None), (False, 5), (True, 4)])
def test_backward_finite_differences(causal, kv_len):
    r = rng(13)
    n, d = 7, 3
    q, k, v, do = (r.normal(size=(n, d)) for _ in range(4))
    s = 0.7
    got = oracle.head_backward(q, k, v, do, s, causal=causal, kv_len=kv_len)
    ref = _fd_grads(q, k, v, do, s, causal=causal, kv_len=kv_len)
    for g, f in zip(got, ref):
        err = np.max(np.abs(g - f)) / max(1e-12, np.max(np.abs(f)))
        assert err < 1e-6, err


def test_backward_masked_keys_get_zero_gradient():
    r = rng(14)
    n = 10
    q, k, v, do = (r.normal(size=(n, 4)) for _ in range(4))
    dq, dk, dv = oracle.head_backward(q, k, v, do, 0.5, kv_len=6)
    assert np.all(dk[6:] == 0) and np.all(dv[6:] == 0)
    assert np.any(dk[:6] != 0)


@pytest.mark.parametrize("causal", [False, True])
def test_jacobian_route_equals_vector_route(causal):
    r = rng(15)
    n, d = 16, 6
    q, k, v, do = (r.normal(size=(n, d)) for _ in range(4))
    a = oracle.head_backward(q, k, v, do, 0.4, causal=causal, kv_len=13)
    b = oracle.head_backward_jacobian(q, k, v, do, 0.4, causal=causal, kv_len=13)
    for x, y in zip(a, b):
        np.testing.assert_allclose(x, y, atol=1e-12)


def test_backward_single_key_closed_form():
    # N = 1: O = v, so dV = dO and dQ = dK = 0.
    r = rng(16)
    q, k, v, do = (r.normal(size=(1, 4)) for _ in range(4))
    dq, dk, dv = oracle.head_backward(q, k, v, do, 0.9)
    np.testing.assert_allclose(dv, do, atol=1e-15)
    assert np.all(np.abs(dq) < 1e-15) and np.all(np.abs(dk) < 1e-15)


def test_to_f64_is_exact_for_bf16():
    torch = pytest.importorskip("torch")
    x = torch.randn(64, generator=torch.Generator().manual_seed(0)).to(torch.bfloat16)
    y = oracle.to_f64(x)
    assert y.dtype == np.float64
    assert np.array_equal(y.astype(np.float32), x.float().numpy())
