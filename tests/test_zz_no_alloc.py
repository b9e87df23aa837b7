"""fa_bwd_noalloc: the backward entry point for callers that cannot allocate
device memory (graph captures that must not allocate, frameworks that own
every allocation, plugins without an allocator). It runs the same backward
pass on a static scratch buffer inside the library instead of a
caller-provided workspace.

Checks, through the C-ABI: two calls in a row agree with fa_bwd (the entry
point that takes a workspace) within the backward's tolerance, a second
shape reuses the shared scratch correctly, and sizes beyond the scratch are
rejected before anything is launched. This file is collected last on purpose.
"""
import ctypes

import pytest
import torch

import workloads as W
from _util import GRAD_REL, grad_rel, f64

pytestmark = pytest.mark.gpu


def _inputs(B, H, N, d, causal, seed):
    w = W.Workload("noalloc", B, H, N, d, causal=causal, backward=True)
    x = W.make_inputs(w, seed)
    return w, {n: x[n].cuda() for n in ("q", "k", "v", "dout")}


def _noalloc(fa, w, t, o, lse):
    dq, dk, dv = (torch.empty_like(t["q"]) for _ in range(3))
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    rc = fa.lib().fa_bwd_noalloc(t["q"].data_ptr(), t["k"].data_ptr(), t["v"].data_ptr(),
                                 o.data_ptr(), t["dout"].data_ptr(), lse.data_ptr(),
                                 dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), w.B, w.H, w.N, w.d,
                                 int(w.causal), w.scale, None, stream)
    assert rc == fa.FA_OK, fa.status_string(rc)
    return dq, dk, dv


def _with_workspace(fa, w, t, o, lse):
    return fa.backward(t["q"], t["k"], t["v"], o, t["dout"], lse, causal=w.causal, scale=w.scale)


@pytest.mark.parametrize("first,second", [((2, 3, 640, 64, True), (1, 4, 1000, 128, False))])
def test_noalloc_matches_workspace_entry_point(fa, first, second):
    for shape, seed in ((first, 31), (second, 32)):
        w, t = _inputs(*shape, seed=seed)
        o, lse = fa.forward(t["q"], t["k"], t["v"], causal=w.causal, scale=w.scale)
        ref = _with_workspace(fa, w, t, o, lse)
        for _ in range(2):                       # two calls in a row share the scratch
            got = _noalloc(fa, w, t, o, lse)
            torch.cuda.synchronize()
            assert fa.device_status() == fa.FA_OK
            for g, r in zip(got, ref):
                e = grad_rel(g, f64(r))
                assert e <= GRAD_REL, e


def test_noalloc_rejects_sizes_beyond_scratch(fa):
    limit = 64 * 1024 * 1024
    B, H, N, d = 1, 1, 1 << 20, 128
    assert fa.bwd_workspace_bytes(B, H, N, d) > limit
    x = torch.zeros(16, dtype=torch.bfloat16, device="cuda")     # never read: rejected first
    lse = torch.zeros(16, dtype=torch.float32, device="cuda")
    p = x.data_ptr()
    rc = fa.lib().fa_bwd_noalloc(p, p, p, p, p, lse.data_ptr(), p, p, p, B, H, N, d, 0, 0.1,
                                 None, None)
    assert rc == fa.FA_ERR_INVALID_ARG
