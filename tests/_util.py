"""Shared helpers of the GPU parity tests: run the CUDA path through the
binding, compare with the CPU fp64 oracle under the stated tolerances.

Tolerances (bf16 inputs, fp32 accumulation on the GPU):
  O      max-abs error            <= 1e-2
  LSE    max-abs error            <= 1e-3   (-inf must match -inf exactly)
  dQ/dK/dV  max-abs error / max-abs of the oracle gradient <= 2e-2 per tensor
With dropout the O and gradient bars are multiplied by the rescale factor
r = 1 / (1 - p') (see tests/test_gpu_dropout.py).
"""
import numpy as np
import torch

O_ATOL = 1e-2
LSE_ATOL = 1e-3
GRAD_REL = 2e-2


def f64(t) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


def cuda(x):
    return None if x is None else x.cuda()


def fwd_errors(o_gpu, lse_gpu, o_ref, lse_ref):
    o = f64(o_gpu) if isinstance(o_gpu, torch.Tensor) else o_gpu
    l = f64(lse_gpu) if isinstance(lse_gpu, torch.Tensor) else lse_gpu
    inf_gpu, inf_ref = np.isneginf(l), np.isneginf(lse_ref)
    assert np.array_equal(inf_gpu, inf_ref), "rows with no visible key differ"
    assert np.all(np.isfinite(o)), "non-finite output"
    err_o = float(np.max(np.abs(o - o_ref))) if o.size else 0.0
    diff = np.where(inf_ref, 0.0, l - np.where(inf_ref, 0.0, lse_ref))
    err_l = float(np.max(np.abs(diff))) if l.size else 0.0
    return err_o, err_l


def check_fwd(o_gpu, lse_gpu, o_ref, lse_ref, tag="", o_atol=O_ATOL):
    err_o, err_l = fwd_errors(o_gpu, lse_gpu, o_ref, lse_ref)
    assert err_o <= o_atol, f"{tag} O max-abs error {err_o:.3e}"
    assert err_l <= LSE_ATOL, f"{tag} LSE max-abs error {err_l:.3e}"
    return err_o, err_l


def grad_rel(g, ref) -> float:
    g = f64(g) if isinstance(g, torch.Tensor) else g
    assert np.all(np.isfinite(g)), "non-finite gradient"
    scale = float(np.max(np.abs(ref))) if ref.size else 0.0
    err = float(np.max(np.abs(g - ref))) if ref.size else 0.0
    return err / scale if scale > 0 else err


def check_grads(grads_gpu, grads_ref, tag="", rel=GRAD_REL):
    out = []
    for name, g, r in zip(("dQ", "dK", "dV"), grads_gpu, grads_ref):
        e = grad_rel(g, r)
        assert e <= rel, f"{tag} {name} relative-to-max error {e:.3e}"
        out.append(e)
    return out
