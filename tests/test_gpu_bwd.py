"""Backward parity: dQ, dK, dV from the CUDA path (through the C-ABI) vs the
oracle's explicit differentiation, on the same seeded bf16 inputs. The GPU
backward consumes the GPU forward's O and LSE, as a user would."""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from _util import check_grads, cuda, f64

pytestmark = pytest.mark.gpu


def run(fa, x, causal, scale, kv_len=None):
    q, k, v, do = cuda(x["q"]), cuda(x["k"]), cuda(x["v"]), cuda(x["dout"])
    kv = cuda(kv_len)
    o, lse = fa.forward(q, k, v, causal=causal, scale=scale, kv_len=kv)
    dq, dk, dv = fa.backward(q, k, v, o, do, lse, causal=causal, scale=scale, kv_len=kv)
    torch.cuda.synchronize()
    assert fa.device_status() == 0
    return dq, dk, dv


def generic(B, H, N, d, causal, seed):
    w = W.Workload("generic", B, H, N, d, causal=causal, backward=True)
    return w, W.make_inputs(w, seed)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N", [128, 384, 1000, 1])
def test_bwd_small_sweep(fa, d, causal, N):
    w, x = generic(2, 2, N, d, causal, seed=N + d + 1)
    g = run(fa, x, causal, w.scale)
    ref = oracle.backward(x["q"], x["k"], x["v"], x["dout"], w.scale, causal=causal)
    check_grads(g, ref, f"d={d} causal={causal} N={N}")


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_bwd_kv_len_edges(fa, d, causal):
    kv = torch.tensor([1, 127, 128, 129, 300, 512], dtype=torch.int32)
    w, x = generic(len(kv), 2, 512, d, causal, seed=11)
    g = run(fa, x, causal, w.scale, kv)
    ref = oracle.backward(x["q"], x["k"], x["v"], x["dout"], w.scale, causal=causal,
                          kv_len=kv.numpy())
    check_grads(g, ref, f"kv_len d={d} causal={causal}")
    # keys beyond kv_len get exactly zero gradient
    dk, dv = f64(g[1]), f64(g[2])
    for b, L in enumerate(kv.tolist()):
        assert np.all(dk[b, :, L:] == 0) and np.all(dv[b, :, L:] == 0)


@pytest.mark.parametrize("name", ["gpt2_small", "bert_large"])
def test_bwd_full_size_short_sequences(fa, name):
    w = W.WORKLOADS[name]
    x = W.make_inputs(w, 0)
    g = run(fa, x, w.causal, w.scale, x["kv_len"])
    kvn = None if x["kv_len"] is None else x["kv_len"].numpy()
    ref = oracle.backward(x["q"], x["k"], x["v"], x["dout"], w.scale, causal=w.causal, kv_len=kvn)
    check_grads(g, ref, name)


@pytest.mark.parametrize("N,heads", [(4096, [(0, 0), (0, 9)]), (8192, [(0, 5)]), (16384, [(0, 13)])])
@pytest.mark.parametrize("causal", [False, True])
def test_bwd_full_size_long_context(fa, N, heads, causal):
    w = W.WORKLOADS[f"long_n{N}_{'causal' if causal else 'noncausal'}"]
    x = W.make_inputs(w, 0)
    g = run(fa, x, causal, w.scale)
    ref = oracle.backward(x["q"], x["k"], x["v"], x["dout"], w.scale, causal=causal, heads=heads)
    for b, h in heads:
        check_grads([f64(t)[b, h] for t in g], [r[b, h] for r in ref], f"{w.name} head {(b, h)}")


def test_bwd_dk_dv_deterministic(fa):
    w, x = generic(2, 2, 512, 64, True, seed=5)
    a = run(fa, x, True, w.scale)
    b = run(fa, x, True, w.scale)
    assert torch.equal(a[1], b[1]) and torch.equal(a[2], b[2])
    # dQ sums tiles with fp32 atomics: equal up to reduction order
    assert torch.allclose(a[0].float(), b[0].float(), rtol=0, atol=1e-2)


def test_bwd_workspace_contents_ignored(fa):
    w, x = generic(1, 2, 256, 64, False, seed=6)
    q, k, v, do = cuda(x["q"]), cuda(x["k"]), cuda(x["v"]), cuda(x["dout"])
    o, lse = fa.forward(q, k, v)
    need = fa.bwd_workspace_bytes(1, 2, 256, 64)
    ws = torch.full((need,), 0x7F, dtype=torch.uint8, device="cuda")   # garbage floats
    g1 = fa.backward(q, k, v, o, do, lse, workspace=ws)
    g2 = fa.backward(q, k, v, o, do, lse)
    torch.cuda.synchronize()
    for a, b in zip(g1[1:], g2[1:]):
        assert torch.equal(a, b)
    assert torch.allclose(g1[0].float(), g2[0].float(), rtol=0, atol=1e-2)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_bwd_many_items_per_cta(fa, causal, d):
    # 64 x 5 heads x 3 key tiles = 960 work items, so every CTA handles
    # several, and consecutive items of one CTA mix key tiles that see every
    # Q tile, tiles that see one, and tiles with no valid key at all (key
    # padding down to a single key): their dK/dV must come out as zeros.
    B, H, N = 64, 5, 300
    w = W.Workload("generic", B, H, N, d, causal=causal, backward=True, std=0.5)
    x = W.make_inputs(w, 10)
    g = np.random.default_rng(10)
    kv = torch.from_numpy(g.integers(1, N + 1, B).astype(np.int32))
    kv[3] = N
    kv[7] = 1
    kv[11] = 129
    kv[12] = 128
    grads = run(fa, x, causal, w.scale, kv)
    ref = oracle.backward(x["q"], x["k"], x["v"], x["dout"], w.scale, causal=causal,
                          kv_len=kv.numpy())
    check_grads(grads, ref, f"many items d={d} causal={causal}")
    dk, dv = f64(grads[1]), f64(grads[2])
    for b, L in enumerate(kv.tolist()):
        assert np.all(dk[b, :, L:] == 0) and np.all(dv[b, :, L:] == 0)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_bwd_kv_len_zero_gives_zero_grads(fa, d, causal):
    # A batch with no valid key: its rows see nothing, so every gradient of
    # that batch is exactly zero (no key tile contributes to its dQ tiles).
    kv = torch.tensor([0, 5, 300], dtype=torch.int32)
    w, x = generic(len(kv), 2, 300, d, causal, seed=21)
    g = run(fa, x, causal, w.scale, kv)
    ref = oracle.backward(x["q"], x["k"], x["v"], x["dout"], w.scale, causal=causal,
                          kv_len=kv.numpy())
    check_grads(g, ref, f"kv_len 0 d={d} causal={causal}")
    for t in g:
        assert torch.count_nonzero(t[0]) == 0


def test_bwd_stages_match_fused_call(fa):
    # fa_bwd_preprocess, fa_bwd_main, fa_bwd_dq_convert on one stream is fa_bwd.
    import ctypes
    w, x = generic(2, 3, 700, 64, True, seed=22)
    q, k, v, do = cuda(x["q"]), cuda(x["k"]), cuda(x["v"]), cuda(x["dout"])
    o, lse = fa.forward(q, k, v, causal=True, scale=w.scale)
    ref = fa.backward(q, k, v, o, do, lse, causal=True, scale=w.scale)
    need = fa.bwd_workspace_bytes(2, 3, 700, 64)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    dq, dk, dv = (torch.empty_like(q) for _ in range(3))
    L = fa.lib()
    s = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    assert L.fa_bwd_preprocess(o.data_ptr(), do.data_ptr(), lse.data_ptr(), 2, 3, 700, 64,
                               ws.data_ptr(), need, s) == 0
    assert L.fa_bwd_main(q.data_ptr(), k.data_ptr(), v.data_ptr(), do.data_ptr(), dk.data_ptr(),
                         dv.data_ptr(), 2, 3, 700, 64, 1, w.scale, None, ws.data_ptr(), need,
                         s) == 0
    assert L.fa_bwd_dq_convert(dq.data_ptr(), 2, 3, 700, 64, ws.data_ptr(), need, s) == 0
    torch.cuda.synchronize()
    assert fa.device_status() == 0
    assert torch.equal(dk, ref[1]) and torch.equal(dv, ref[2])
    assert torch.allclose(dq.float(), ref[0].float(), rtol=0, atol=1e-2)
