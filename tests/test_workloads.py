"""Host-side checks of the seeded synthetic input generator."""
import math

import numpy as np
import pytest
import torch

import workloads as W


def test_catalogue_shapes():
    assert set(W.WORKLOADS) >= {"tiny_fwd", "gpt2_small", "bert_large", "blocksparse",
                                "long_n4096_causal", "long_n16384_noncausal"}
    w = W.WORKLOADS["gpt2_small"]
    assert (w.B, w.H, w.N, w.d, w.causal, w.backward) == (8, 12, 1024, 64, True, True)
    w = W.WORKLOADS["long_n8192_noncausal"]
    assert (w.B, w.H, w.N, w.d, w.std) == (1, 16, 8192, 128, 0.5)
    assert math.isclose(w.scale, 1 / math.sqrt(128))


def test_deterministic_and_bf16():
    w = W.WORKLOADS["bert_large"].with_(B=3, H=2, N=256)
    a = W.make_inputs(w, seed=1)
    b = W.make_inputs(w, seed=1)
    c = W.make_inputs(w, seed=2)
    for key in ("q", "k", "v", "dout"):
        assert a[key].dtype == torch.bfloat16 and a[key].shape == (3, 2, 256, 64)
        assert torch.equal(a[key], b[key])
        assert not torch.equal(a[key], c[key])
    assert a["kv_len"].dtype == torch.int32
    assert torch.all((a["kv_len"] >= 256) & (a["kv_len"] <= 512))


def test_kv_len_range_inclusive():
    w = W.WORKLOADS["bert_large"].with_(B=4000, H=1, N=128, d=64, backward=False)
    kv = W.make_inputs(w, 0)["kv_len"]
    assert int(kv.min()) == 256 and int(kv.max()) == 512


def test_block_mask_counts():
    w = W.WORKLOADS["blocksparse"]
    g = torch.Generator().manual_seed(0)
    m = W.block_mask_for(w, g)
    nb = 128
    assert m.shape == (nb, nb) and m.dtype == torch.uint8
    band = (np.abs(np.arange(nb)[:, None] - np.arange(nb)[None, :]) <= 1)
    assert band.sum() == 382
    assert np.all(m.numpy()[band] == 1)
    assert int(m.sum()) == 382 + round(0.02 * (nb * nb - 382)) == 702
    assert m[0, 0] == 1


def test_lowrank_bias_peaks_logits():
    w = W.WORKLOADS["long_n4096_noncausal"].with_(N=512, H=2)
    x = W.make_inputs(w, 0)
    q = x["q"][0, 0].double()
    k = x["k"][0, 0].double()
    logits = (q @ k.T) * w.scale
    # bias term std = alpha^2 * sqrt(rank) * scale = 16*sqrt(8)/sqrt(128) = 4; the
    # Gaussian part adds 0.25*sqrt(128)*scale = 0.25
    assert 3.0 < float(logits.std()) < 5.0
    w0 = w.with_(lowrank_rank=0)
    y = W.make_inputs(w0, 0)
    l0 = (y["q"][0, 0].double() @ y["k"][0, 0].double().T) * w.scale
    assert float(l0.std()) < 0.5
