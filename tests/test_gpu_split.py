"""Split of the last wave of work (stream-K): parity of the split forward and
backward with the CPU oracle, and agreement with the unsplit schedule.

Each case first asks the library whether it plans a split for the sizes on
this GPU (fwd_workspace_bytes / bwd_split_workspace_bytes > 0), so that none
of them passes vacuously. Shapes: few (b, h) problems with long sequences
(every work item is cut into parts), a ragged last tile, a whole first wave
followed by a short tail, causal items of every length, dropout, and a
[B, N, H, d] layout."""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from _util import O_ATOL, check_fwd, check_grads, cuda, f64

pytestmark = pytest.mark.gpu


def inputs(B, H, N, d, causal, seed, backward=True):
    w = W.Workload("split", B, H, N, d, causal=causal, backward=backward)
    return w, W.make_inputs(w, seed)


def assert_fwd_split(fa, B, H, N, d, causal):
    n = fa.fwd_workspace_bytes(B, H, N, d, causal)
    assert n > 0, f"no forward split planned for B={B} H={H} N={N} d={d} causal={causal}"


def assert_bwd_split(fa, B, H, N, d, causal):
    n = fa.bwd_split_workspace_bytes(B, H, N, d, causal)
    assert n > fa.bwd_workspace_bytes(B, H, N, d), "no backward split planned"


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N", [4096, 4000])
def test_split_forward_few_problems(fa, d, causal, N):
    """B*H = 2: every item is cut into parts spread over all SMs (N = 4000
    also has a ragged last tile)."""
    assert_fwd_split(fa, 1, 2, N, d, causal)
    w, x = inputs(1, 2, N, d, causal, seed=N + d + int(causal), backward=False)
    q, k, v = cuda(x["q"]), cuda(x["k"]), cuda(x["v"])
    o, lse = fa.forward(q, k, v, causal=causal, scale=w.scale)
    o2, lse2 = fa.forward(q, k, v, causal=causal, scale=w.scale, split=False)
    torch.cuda.synchronize()
    assert fa.device_status() == 0
    o_ref, l_ref = oracle.forward(x["q"], x["k"], x["v"], w.scale, causal=causal)
    check_fwd(o, lse, o_ref, l_ref, f"split d={d} causal={causal} N={N}")
    check_fwd(o2, lse2, o_ref, l_ref, f"unsplit d={d} causal={causal} N={N}")
    # the two schedules differ only in the order of the final additions
    assert float(np.max(np.abs(f64(o) - f64(o2)))) <= 2 ** -7
    assert float(np.max(np.abs(f64(lse) - f64(lse2)))) <= 1e-5


def test_split_forward_whole_wave_then_tail(fa):
    """More items than SMs: a whole first wave on the plain kernel, then the
    tail -- the last heads' items -- cut into parts on the split kernel. Rows
    sampled across every Q tile of the first head (whole items) and of the
    last head (cut items)."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    N, d = 8192, 128
    H = sms // 32 + 2  # 32 Q-tile pairs per head; items = 32 H > sms
    assert_fwd_split(fa, 1, H, N, d, False)
    w, x = inputs(1, H, N, d, False, seed=5, backward=False)
    o, lse = fa.forward(cuda(x["q"]), cuda(x["k"]), cuda(x["v"]), scale=w.scale)
    torch.cuda.synchronize()
    assert fa.device_status() == 0
    heads = [0, H - 1]
    rows = np.arange(5, N, 61)
    o_ref, l_ref = oracle.forward(x["q"][:, heads], x["k"][:, heads], x["v"][:, heads], w.scale,
                                  rows=rows)
    check_fwd(f64(o)[:, heads][:, :, rows], f64(lse)[:, heads][:, :, rows], o_ref, l_ref,
              "wave + tail")


def test_split_forward_workspace_contents_ignored(fa):
    B, H, N, d = 1, 2, 4096, 128
    assert_fwd_split(fa, B, H, N, d, True)
    w, x = inputs(B, H, N, d, True, seed=9, backward=False)
    q, k, v = cuda(x["q"]), cuda(x["k"]), cuda(x["v"])
    n = fa.fwd_workspace_bytes(B, H, N, d, True)
    ws = torch.full((n,), 0xFF, dtype=torch.uint8, device="cuda")  # NaN patterns everywhere
    o1, l1 = fa.forward(q, k, v, causal=True, scale=w.scale, workspace=ws)
    ws.fill_(0x7F)
    o2, l2 = fa.forward(q, k, v, causal=True, scale=w.scale, workspace=ws)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_split_forward_ignores_workspace_with_kv_len(fa):
    B, H, N, d = 2, 1, 4096, 64
    w, x = inputs(B, H, N, d, False, seed=3, backward=False)
    q, k, v = cuda(x["q"]), cuda(x["k"]), cuda(x["v"])
    kv = torch.tensor([4000, 1000], dtype=torch.int32, device="cuda")
    ws = torch.empty(fa.fwd_workspace_bytes(1, 2, N, d, False) or 1 << 20, dtype=torch.uint8,
                     device="cuda")
    o1, l1 = fa.forward(q, k, v, scale=w.scale, kv_len=kv, workspace=ws)
    o2, l2 = fa.forward(q, k, v, scale=w.scale, kv_len=kv, split=False)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


@pytest.mark.parametrize("causal", [False, True])
def test_split_forward_dropout_and_layout(fa, causal):
    """Dropout draws and [B, N, H, d] strides are unchanged by the split: the
    split result matches the unsplit one and the oracle."""
    B, H, N, d = 1, 2, 4096, 64
    assert_fwd_split(fa, B, H, N, d, causal)
    w, x = inputs(B, H, N, d, causal, seed=17, backward=False)
    t = lambda a: a.cuda().transpose(1, 2).contiguous().transpose(1, 2)  # [B,N,H,d] storage
    q, k, v = t(x["q"]), t(x["k"]), t(x["v"])
    p, seed, off = 0.1, 1234, 7
    o, lse = fa.attention_forward(q, k, v, causal=causal, scale=w.scale, dropout_p=p, seed=seed,
                                  offset=off)
    o2, lse2 = fa.attention_forward(q, k, v, causal=causal, scale=w.scale, dropout_p=p, seed=seed,
                                    offset=off, split=False)
    torch.cuda.synchronize()
    assert fa.device_status() == 0
    assert float(np.max(np.abs(f64(o) - f64(o2)))) <= 2 ** -6
    assert float(np.max(np.abs(f64(lse) - f64(lse2)))) <= 1e-5
    rows = np.concatenate([np.arange(0, 130), np.arange(N - 130, N)])
    p32 = float(np.float32(p))  # the value the library receives
    o_ref, l_ref = oracle.forward(x["q"], x["k"], x["v"], w.scale, causal=causal, rows=rows,
                                  dropout=(p32, seed, off))
    r = oracle.rescale(oracle.threshold(p32))  # the dropout bar: O_ATOL x 1 / (1 - p')
    check_fwd(f64(o)[:, :, rows], f64(lse)[:, :, rows], o_ref, l_ref, "split dropout",
              o_atol=O_ATOL * r)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_split_backward_few_problems(fa, d, causal):
    """B*H = 2 at N = 4096: every key-tile item is cut into runs of Q tiles;
    dK, dV of the parts are summed by the merge kernel, dQ accumulates as usual."""
    B, H, N = 1, 2, 4096
    assert_bwd_split(fa, B, H, N, d, causal)
    w, x = inputs(B, H, N, d, causal, seed=40 + d + int(causal))
    q, k, v, do = cuda(x["q"]), cuda(x["k"]), cuda(x["v"]), cuda(x["dout"])
    o, lse = fa.forward(q, k, v, causal=causal, scale=w.scale)
    g = fa.backward(q, k, v, o, do, lse, causal=causal, scale=w.scale)
    g2 = fa.backward(q, k, v, o, do, lse, causal=causal, scale=w.scale, split=False)
    torch.cuda.synchronize()
    assert fa.device_status() == 0
    ref = oracle.backward(x["q"], x["k"], x["v"], x["dout"], w.scale, causal=causal)
    check_grads(g, ref, f"split bwd d={d} causal={causal}")
    check_grads(g2, ref, f"unsplit bwd d={d} causal={causal}")
    for a, b in zip(g[1:], g2[1:]):  # dK, dV: the same sums in another order
        assert float(np.max(np.abs(f64(a) - f64(b)))) <= 2 ** -6 * float(np.max(np.abs(f64(b))))


def test_split_backward_whole_wave_then_tail(fa):
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    H = sms // 16 + 2  # key tiles per head at N = 2048: 16; items = 16 H > sms
    B, N, d = 1, 2048, 128
    assert_bwd_split(fa, B, H, N, d, False)
    w, x = inputs(B, H, N, d, False, seed=6)
    q, k, v, do = cuda(x["q"]), cuda(x["k"]), cuda(x["v"]), cuda(x["dout"])
    o, lse = fa.forward(q, k, v, scale=w.scale)
    g = fa.backward(q, k, v, o, do, lse, scale=w.scale)
    torch.cuda.synchronize()
    assert fa.device_status() == 0
    heads = [0, H - 1]
    ref = oracle.backward(x["q"], x["k"], x["v"], x["dout"], w.scale, heads=[(0, h) for h in heads])
    check_grads([f64(t)[:, heads] for t in g], [r[:, heads] for r in ref], "bwd wave + tail")


def test_split_backward_deterministic(fa):
    B, H, N, d = 1, 2, 4096, 64
    assert_bwd_split(fa, B, H, N, d, True)
    w, x = inputs(B, H, N, d, True, seed=8)
    q, k, v, do = cuda(x["q"]), cuda(x["k"]), cuda(x["v"]), cuda(x["dout"])
    o, lse = fa.forward(q, k, v, causal=True, scale=w.scale)
    a = fa.backward(q, k, v, o, do, lse, causal=True, scale=w.scale)
    b = fa.backward(q, k, v, o, do, lse, causal=True, scale=w.scale)
    torch.cuda.synchronize()
    assert torch.equal(a[1], b[1]) and torch.equal(a[2], b[2])


def test_split_decisions_of_the_bench_workloads(fa):
    """The plan's decisions where its estimate is near the margin, as measured
    on GB300 (152 SMs): the 16K non-causal forward splits (1430 -> 1407 us),
    the 4K non-causal forward does not (forced, 122 -> 129 us), the 4K
    non-causal backward and the 8K non-causal forward do."""
    if torch.cuda.get_device_properties(0).multi_processor_count != 152:
        pytest.skip("the decisions were measured on 152 SMs")
    assert fa.fwd_workspace_bytes(1, 16, 16384, 128, False) > 0
    assert fa.fwd_workspace_bytes(1, 16, 4096, 128, False) == 0
    assert fa.fwd_workspace_bytes(1, 16, 8192, 128, False) > 0
    assert fa.bwd_split_workspace_bytes(1, 16, 4096, 128, False) > fa.bwd_workspace_bytes(1, 16, 4096, 128)
