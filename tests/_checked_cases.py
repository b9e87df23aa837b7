"""Representative calls shared by the checked-build test's parent (default
library) and child (checked library) processes. Every input is seeded."""
import numpy as np
import torch

import workloads as W


def _cuda(t):
    return t.cuda()


def run_cases(fa):
    out = {}

    def status(tag):
        s = fa.device_status()
        assert s == 0, f"{tag}: device status {s} ({fa.status_string(s)})"

    # 1. d = 64 causal, ragged N
    w = W.Workload("generic", 2, 3, 700, 64, causal=True, backward=True)
    x = W.make_inputs(w, 61)
    q, k, v, do = (_cuda(x[n]) for n in ("q", "k", "v", "dout"))
    o, lse = fa.forward(q, k, v, causal=True, scale=w.scale)
    g = fa.backward(q, k, v, o, do, lse, causal=True, scale=w.scale)
    torch.cuda.synchronize()
    status("d64 causal")
    out["c1"] = [o, lse, *g]
    # 2. d = 128 non-causal with key padding
    w = W.Workload("generic", 2, 2, 1000, 128, causal=False, backward=True)
    x = W.make_inputs(w, 62)
    q, k, v, do = (_cuda(x[n]) for n in ("q", "k", "v", "dout"))
    kv = torch.tensor([1000, 333], dtype=torch.int32, device="cuda")
    o, lse = fa.forward(q, k, v, scale=w.scale, kv_len=kv)
    g = fa.backward(q, k, v, o, do, lse, scale=w.scale, kv_len=kv)
    torch.cuda.synchronize()
    status("d128 kv_len")
    out["c2"] = [o, lse, *g]
    # 3. [B, N, H, d] storage, d = 64, causal, dropout
    w = W.Workload("generic", 2, 2, 640, 64, causal=True, backward=True)
    x = W.make_inputs(w, 63)
    t = lambda a: a.cuda().transpose(1, 2).contiguous().transpose(1, 2)
    q, k, v, do = (t(x[n]) for n in ("q", "k", "v", "dout"))
    kw = dict(causal=True, scale=w.scale, dropout_p=0.1, seed=77, offset=3)
    o, lse = fa.attention_forward(q, k, v, **kw)
    g = fa.attention_backward(q, k, v, o, do, lse, **kw)
    torch.cuda.synchronize()
    status("bnhd dropout")
    out["c3"] = [o, lse, *g]
    # 4. block mask, d = 128 and d = 64
    for d in (128, 64):
        w = W.Workload("generic", 1, 2, 1024, d, causal=False, backward=True)
        x = W.make_inputs(w, 64 + d)
        q, k, v, do = (_cuda(x[n]) for n in ("q", "k", "v", "dout"))
        rng = np.random.default_rng(d)
        m = (rng.random((8, 8)) < 0.4).astype(np.uint8)
        m[np.arange(8), np.arange(8)] = 1
        mask = torch.from_numpy(m).cuda()
        o, lse = fa.blocksparse_forward(q, k, v, mask, scale=w.scale)
        g = fa.blocksparse_backward(q, k, v, o, do, lse, mask, scale=w.scale)
        torch.cuda.synchronize()
        status(f"sparse d{d}")
        out[f"c4_{d}"] = [o, lse, *g]
    # 5. split of the last wave (few problems, long rows), d = 128 causal
    w = W.Workload("generic", 1, 2, 4096, 128, causal=True, backward=True)
    x = W.make_inputs(w, 65)
    q, k, v, do = (_cuda(x[n]) for n in ("q", "k", "v", "dout"))
    o, lse = fa.forward(q, k, v, causal=True, scale=w.scale, split=True)
    g = fa.backward(q, k, v, o, do, lse, causal=True, scale=w.scale, split=True)
    torch.cuda.synchronize()
    status("split")
    out["c5"] = [o, lse, *g]
    return {key: [t.detach().cpu() for t in ts] for key, ts in out.items()}
