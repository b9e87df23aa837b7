"""Seeded synthetic inputs for the exact-attention workloads.

This module draws random numbers and nothing else: it holds none of the
attention arithmetic. Both the CPU oracle checks and the CUDA path consume the
tensors it returns, so the two sides always see identical bf16 values.

Recipe (the same for every workload):
  * ``torch.Generator('cpu').manual_seed(seed)``;
  * fp32 ``randn`` drawn in the order Q, K, V, then dO (fwd+bwd workloads only),
    each of shape [B, H, N, d], multiplied by the workload's standard deviation;
  * then the optional low-rank bias draws, the key-padding lengths and the
    block-mask draws, in that order;
  * finally Q, K, V, dO are rounded to bfloat16 (round-to-nearest-even).

The shapes stand in for the pages' workloads (GPT-2 small at sequence 1K,
BERT-large at sequence 512, long-context 4K-16K, block-sparse at 16K;
FlashAttention abstract and the condensed paper's section 4, Experiments).
No dataset is read: values are i.i.d. Gaussian.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import torch

BLOCK = 128


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    N: int
    d: int
    causal: bool
    backward: bool                  # fwd+bwd (True) or forward only
    std: float = 1.0                # standard deviation of Q, K, V, dO
    lowrank_rank: int = 0           # per-head low-rank bias added to Q and K
    lowrank_alpha: float = 0.0
    kv_len_range: Optional[tuple] = None   # inclusive [lo, hi] for key padding
    sparse: bool = False            # block-sparse forward (band + random blocks)
    sparse_band: int = 1            # |r - c| <= band is kept
    sparse_frac: float = 0.02       # fraction of off-band blocks kept
    dropout: float = 0.0            # dropout probability on P (0: none)
    dropout_seed: int = 0x5EED      # Philox key of the dropout draws
    layout: str = "bhnd"            # storage order of Q, K, V, dO, O, dQ, dK, dV: bhnd or bnhd

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)

    def with_(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


def _long(N: int, causal: bool) -> Workload:
    return Workload(name=f"long_n{N}_{'causal' if causal else 'noncausal'}",
                    B=1, H=16, N=N, d=128, causal=causal, backward=True, std=0.5,
                    lowrank_rank=8, lowrank_alpha=4.0)


WORKLOADS = {
    # B=1 H=1 N=128 d=64, non-causal, forward only.
    "tiny_fwd": Workload("tiny_fwd", 1, 1, 128, 64, causal=False, backward=False),
    # GPT-2 small shaped attention: 12 heads of 64, sequence 1K, causal.
    "gpt2_small": Workload("gpt2_small", 8, 12, 1024, 64, causal=True, backward=True),
    # BERT-large shaped attention: 16 heads of 64, sequence 512, key padding.
    "bert_large": Workload("bert_large", 16, 16, 512, 64, causal=False, backward=True,
                           kv_len_range=(256, 512)),
    # GPT-2 small with attention dropout 0.1, the rate GPT-2 trains with.
    "gpt2_small_dropout": Workload("gpt2_small_dropout", 8, 12, 1024, 64, causal=True,
                                   backward=True, dropout=0.1),
    # GPT-2 small with Q, K, V, O and gradients stored as [B, N, H, d].
    "gpt2_small_bnhd": Workload("gpt2_small_bnhd", 8, 12, 1024, 64, causal=True, backward=True,
                                layout="bnhd"),
    # Block-sparse forward and backward at sequence 16K.
    "blocksparse": Workload("blocksparse", 2, 8, 16384, 64, causal=False, backward=True,
                            sparse=True),
}
for _n in (4096, 8192, 16384):
    for _c in (False, True):
        _w = _long(_n, _c)
        WORKLOADS[_w.name] = _w
# Long context (N = 8192, d = 128, non-causal) with attention dropout 0.1.
WORKLOADS["long_n8192_noncausal_dropout"] = _long(8192, False).with_(
    name="long_n8192_noncausal_dropout", dropout=0.1)


def block_mask_for(w: Workload, g: torch.Generator) -> torch.Tensor:
    """uint8 [nb, nb] block mask: a band |r-c| <= band plus a seeded random
    choice of round(frac * #off-band) off-band blocks (without replacement)."""
    nb = (w.N + BLOCK - 1) // BLOCK
    r = torch.arange(nb)[:, None]
    c = torch.arange(nb)[None, :]
    band = (r - c).abs() <= w.sparse_band
    mask = band.to(torch.uint8)
    off = (~band).flatten().nonzero().flatten()
    count = int(round(w.sparse_frac * off.numel()))
    if count:
        pick = torch.randperm(off.numel(), generator=g)[:count]
        mask.view(-1)[off[pick]] = 1
    return mask


def make_inputs(w: Workload, seed: int = 0) -> dict:
    """Draw one workload's inputs. Returns CPU tensors:
    q, k, v (and dout for fwd+bwd) bf16 [B,H,N,d]; kv_len int32 [B] or None;
    block_mask uint8 [nb,nb] or None; scale (float)."""
    g = torch.Generator(device="cpu").manual_seed(seed)
    shape = (w.B, w.H, w.N, w.d)
    q = torch.randn(shape, generator=g) * w.std
    k = torch.randn(shape, generator=g) * w.std
    v = torch.randn(shape, generator=g) * w.std
    dout = torch.randn(shape, generator=g) * w.std if w.backward else None
    if w.lowrank_rank:
        rk = w.lowrank_rank
        for b in range(w.B):
            for h in range(w.H):
                basis, _ = torch.linalg.qr(torch.randn(w.d, rk, generator=g))  # d x rk, orthonormal columns
                cq = torch.randn(w.N, rk, generator=g)
                ck = torch.randn(w.N, rk, generator=g)
                q[b, h] += w.lowrank_alpha * cq @ basis.T
                k[b, h] += w.lowrank_alpha * ck @ basis.T
    kv_len = None
    if w.kv_len_range is not None:
        lo, hi = w.kv_len_range
        kv_len = torch.randint(lo, hi + 1, (w.B,), generator=g, dtype=torch.int64).to(torch.int32)
    block_mask = block_mask_for(w, g) if w.sparse else None
    out = {
        "q": q.to(torch.bfloat16), "k": k.to(torch.bfloat16), "v": v.to(torch.bfloat16),
        "dout": None if dout is None else dout.to(torch.bfloat16),
        "kv_len": kv_len, "block_mask": block_mask, "scale": w.scale,
    }
    return out
