"""CPU fp64 oracle for exact scaled-dot-product attention.

TEST INFRASTRUCTURE. Only the tests, the smoke check and the bench's CPU
baseline may import this module; the product path never does. It shares no
code with the CUDA library: it materialises the score matrix S and the
probability matrix P in full (row chunk by row chunk, each chunk holding whole
rows), which is exactly the "standard attention" that the method replaces.

What is computed (per batch b and head h, with Q, K, V, dO in R^{N x d}):

  S  = scale * Q K^T + M            M_ij in {0, -inf}  (mask, see ``visible``)
  m_i = max_j S_ij
  LSE_i = m_i + ln sum_j exp(S_ij - m_i)          natural log, scale included
  P  = exp(S - LSE)                               masked entries are exactly 0
  O  = P V

Sources: the problem statement of standard attention -- S = QK^T, P =
softmax(S), O = PV, all N x N intermediates in HBM -- in the condensed
FlashAttention paper page (sample_paper.md), section 2 "Background: GPU Memory
Hierarchy", and the shape caption "Q: N x d, K^T: d x N, QK^T: N x N,
sm(QK^T)V: N x d" on the aggregator page's figure captions. The method is
"exact" (FlashAttention abstract; sample_paper.md section 5, "numerically
exact"), so its result is this definition evaluated without rounding.

The backward pass is the explicit derivative of L = sum(dO * O):

  dV = P^T dO ;  dP = dO V^T ;  dS_i = J_i dP_i with J_i = diag(P_i) - P_i P_i^T
  dQ = scale * dS K ;  dK = scale * dS^T Q

``head_backward`` applies J_i as P_i * (dP_i - <P_i, dP_i>) (the same linear
map); ``head_backward_jacobian`` builds J_i as a matrix (tiny inputs only). The
row dot <P_i, dP_i> is taken from P and dP, never from dO.O.

Readings taken where the pages are silent (all stated in the design notes):
the stored per-row statistic is the natural-log logsumexp including the scale;
causal keeps j <= i (square); key padding masks keys j >= kv_len[b] for every
query row; a block mask (block size 128) masks whole 128 x 128 blocks; a row
with no visible key gives O = 0, LSE = -inf and zero gradients. Dropout, when
asked for, follows oracle/dropout.py (inverted dropout on P, Philox draws).

Pins: every function here is checked in tests/test_oracle.py against closed
forms, invariants, special cases, a hand-derived worked example
(tests/golden/) and central finite differences.
"""
from __future__ import annotations

import numpy as np

BLOCK = 128
_CHUNK_ELEMS = 1 << 23          # fp64 elements of S held per row chunk (64 MB)


def to_f64(x) -> np.ndarray:
    """Exact upcast of a torch tensor (any float dtype, incl. bf16) or array."""
    if hasattr(x, "detach"):
        x = x.detach().cpu().float().numpy()
    return np.asarray(x, dtype=np.float64)


def visible(rows: np.ndarray, n_k: int, causal: bool, kv_len=None,
            block_mask=None, block: int = BLOCK) -> np.ndarray:
    """Boolean [len(rows), n_k]: True where key j is visible to query row i.

    causal: j <= i.  kv_len: j < kv_len.  block_mask: block
    (i // block, j // block) nonzero."""
    i = np.asarray(rows)[:, None]
    j = np.arange(n_k)[None, :]
    keep = np.ones((i.shape[0], n_k), dtype=bool)
    if causal:
        keep &= j <= i
    if kv_len is not None:
        keep &= j < int(kv_len)
    if block_mask is not None:
        bm = np.asarray(block_mask).astype(bool)
        keep &= bm[i // block, j // block]
    return keep


def _chunks(rows: np.ndarray, n_k: int):
    step = max(1, _CHUNK_ELEMS // max(1, n_k))
    for r0 in range(0, len(rows), step):
        yield rows[r0:r0 + step]


def _probs(q_rows, k, scale, keep):
    """P and LSE for a chunk of full rows (standard softmax with max shift)."""
    s = scale * (q_rows @ k.T)
    s = np.where(keep, s, -np.inf)
    m = s.max(axis=1)
    live = np.isfinite(m)
    e = np.exp(s - np.where(live, m, 0.0)[:, None])
    l = e.sum(axis=1)
    lse = np.where(live, m + np.log(np.where(live, l, 1.0)), -np.inf)
    p = np.where(live[:, None], e / np.where(live, l, 1.0)[:, None], 0.0)
    return p, lse


def head_forward(q, k, v, scale, causal=False, kv_len=None, block_mask=None, rows=None,
                 drop=None):
    """One head. q [Nq,d], k [Nk,d], v [Nk,dv] fp64. Returns O [r,dv], LSE [r]
    for the requested query rows (all rows by default).

    ``drop``: optional function (rows, n_k) -> [len(rows), n_k] multiplier
    Z / (1 - p') (oracle.dropout.multiplier); then O = (P * drop) V while LSE
    stays that of the undropped scores."""
    q, k, v = to_f64(q), to_f64(k), to_f64(v)
    rows = np.arange(q.shape[0]) if rows is None else np.asarray(rows)
    o = np.empty((len(rows), v.shape[1]))
    lse = np.empty(len(rows))
    pos = 0
    for rr in _chunks(rows, k.shape[0]):
        keep = visible(rr, k.shape[0], causal, kv_len, block_mask)
        p, l = _probs(q[rr], k, scale, keep)
        if drop is not None:
            p = p * drop(rr, k.shape[0])
        o[pos:pos + len(rr)] = p @ v
        lse[pos:pos + len(rr)] = l
        pos += len(rr)
    return o, lse


def head_probs(q, k, scale, causal=False, kv_len=None, block_mask=None):
    """The full probability matrix P [Nq, Nk] of one head (small inputs)."""
    q, k = to_f64(q), to_f64(k)
    keep = visible(np.arange(q.shape[0]), k.shape[0], causal, kv_len, block_mask)
    return _probs(q, k, scale, keep)[0]


def head_backward(q, k, v, dout, scale, causal=False, kv_len=None, block_mask=None, drop=None):
    """One head's gradients of L = sum(dO * O): returns dQ, dK, dV (fp64).

    With ``drop`` (as in head_forward) O = Pd V with Pd = P * drop, so
    dV = Pd^T dO and the gradient reaching P is dP = (dO V^T) * drop; the
    softmax Jacobian is then applied to that dP exactly as without dropout."""
    q, k, v, dout = to_f64(q), to_f64(k), to_f64(v), to_f64(dout)
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    for rr in _chunks(np.arange(q.shape[0]), k.shape[0]):
        keep = visible(rr, k.shape[0], causal, kv_len, block_mask)
        p, _ = _probs(q[rr], k, scale, keep)
        dp = dout[rr] @ v.T
        pd = p
        if drop is not None:
            mult = drop(rr, k.shape[0])
            dp = dp * mult
            pd = p * mult
        rowdot = (p * dp).sum(axis=1)
        ds = p * (dp - rowdot[:, None])
        dv += pd.T @ dout[rr]
        dk += scale * (ds.T @ q[rr])
        dq[rr] = scale * (ds @ k)
    return dq, dk, dv


def head_backward_jacobian(q, k, v, dout, scale, causal=False, kv_len=None, block_mask=None,
                           drop=None):
    """Same gradients, with each row's softmax Jacobian built as a matrix.
    Quadratic memory per row: tiny inputs only."""
    q, k, v, dout = to_f64(q), to_f64(k), to_f64(v), to_f64(dout)
    p = head_probs(q, k, scale, causal, kv_len, block_mask)
    mult = np.ones_like(p) if drop is None else drop(np.arange(p.shape[0]), p.shape[1])
    dv = (p * mult).T @ dout
    dp = (dout @ v.T) * mult
    ds = np.empty_like(p)
    for i in range(p.shape[0]):
        jac = np.diag(p[i]) - np.outer(p[i], p[i])
        ds[i] = jac @ dp[i]
    return scale * ds @ k, scale * ds.T @ q, dv


def _kvl(kv_len, b):
    return None if kv_len is None else int(np.asarray(kv_len).reshape(-1)[b])


def _drop(dropout, bh):
    if dropout is None:
        return None
    from .dropout import multiplier
    p, seed, offset = dropout
    return multiplier(bh, seed, offset, p)


def forward(q, k, v, scale, causal=False, kv_len=None, block_mask=None, heads=None, rows=None,
            dropout=None):
    """Batched forward over [B,H,N,d]. Returns O [B,H,r,d], LSE [B,H,r].
    ``heads``: optional list of (b, h) to compute (others left NaN).
    ``rows``: optional query-row subset (same for every head).
    ``dropout``: optional (p, seed, offset); head (b, h) uses the keep mask of
    problem b*H + h (oracle.dropout)."""
    q, k, v = to_f64(q), to_f64(k), to_f64(v)
    B, H, N, _ = q.shape
    nr = N if rows is None else len(rows)
    o = np.full((B, H, nr, v.shape[-1]), np.nan)
    lse = np.full((B, H, nr), np.nan)
    todo = heads if heads is not None else [(b, h) for b in range(B) for h in range(H)]
    for b, h in todo:
        o[b, h], lse[b, h] = head_forward(q[b, h], k[b, h], v[b, h], scale, causal,
                                          _kvl(kv_len, b), block_mask, rows,
                                          _drop(dropout, b * H + h))
    return o, lse


def backward(q, k, v, dout, scale, causal=False, kv_len=None, block_mask=None, heads=None,
             dropout=None):
    """Batched backward over [B,H,N,d]. Returns dQ, dK, dV (NaN outside ``heads``).
    ``dropout``: as in forward."""
    q, k, v, dout = to_f64(q), to_f64(k), to_f64(v), to_f64(dout)
    B, H = q.shape[:2]
    dq = np.full(q.shape, np.nan)
    dk = np.full(k.shape, np.nan)
    dv = np.full(v.shape, np.nan)
    todo = heads if heads is not None else [(b, h) for b in range(B) for h in range(H)]
    for b, h in todo:
        dq[b, h], dk[b, h], dv[b, h] = head_backward(q[b, h], k[b, h], v[b, h], dout[b, h],
                                                     scale, causal, _kvl(kv_len, b), block_mask,
                                                     _drop(dropout, b * H + h))
    return dq, dk, dv


def loss(q, k, v, dout, scale, causal=False, kv_len=None, block_mask=None, drop=None):
    """L = sum(dO * O) for one head (the function the backward differentiates)."""
    o, _ = head_forward(q, k, v, scale, causal, kv_len, block_mask, drop=drop)
    return float((to_f64(dout) * o).sum())
