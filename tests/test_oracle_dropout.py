"""Pins of the oracle's dropout (oracle/dropout.py) against facts that do not
come from the oracle:

* the Philox4x32-10 generator against the cuRAND host generator
  CURAND_RNG_PSEUDO_PHILOX4_32_10 (a library implementation of the same
  published bijection): a wrong multiplier, key increment, round count, word
  order or key split changes every word;
* the statistics the reading fixes: bytes uniform on 0..255, keep fraction
  1 - t/256, masks of different problems / offsets / seeds uncorrelated;
* special cases: p = 0 is plain attention; LSE does not depend on dropout;
* unbiasedness: the mean of the dropped O over many offsets tends to the
  undropped O (a missing or wrong 1 / (1 - p') fails it);
* central finite differences of the dropped loss for a fixed mask, and the
  explicit-Jacobian route against the vector route.
"""
import ctypes
import ctypes.util
import glob
import os

import numpy as np
import pytest

import oracle
from oracle import dropout as od


def rng(seed=0):
    return np.random.default_rng(seed)


# --------------------------------------------------------------- generator
def _load_curand():
    cands = [ctypes.util.find_library("curand")]
    for root in (os.environ.get("CUDA_HOME"), os.environ.get("CUDA_PATH"), "/usr/local/cuda"):
        if root:
            cands += sorted(glob.glob(os.path.join(root, "lib64", "libcurand.so*")))
            cands += sorted(glob.glob(os.path.join(root, "targets", "*", "lib", "libcurand.so*")))
    try:
        import nvidia  # pip-packaged CUDA libraries, when present
        for p in getattr(nvidia, "__path__", []):
            cands += sorted(glob.glob(os.path.join(p, "curand", "lib", "libcurand.so*")))
    except ImportError:
        pass
    for c in cands:
        if not c:
            continue
        try:
            return ctypes.CDLL(c)
        except OSError:
            continue
    return None


def _curand_philox_host(seed: int, n_words: int) -> np.ndarray:
    lib = _load_curand()
    if lib is None:
        pytest.skip("libcurand not found")
    gen = ctypes.c_void_p()
    rc = lib.curandCreateGeneratorHost(ctypes.byref(gen), 161)  # CURAND_RNG_PSEUDO_PHILOX4_32_10
    if rc != 0:
        pytest.skip(f"curandCreateGeneratorHost returned {rc}")
    try:
        assert lib.curandSetPseudoRandomGeneratorSeed(gen, ctypes.c_ulonglong(seed)) == 0
        buf = (ctypes.c_uint32 * n_words)()
        assert lib.curandGenerate(gen, buf, ctypes.c_size_t(n_words)) == 0
        return np.frombuffer(buf, dtype=np.uint32).copy()
    finally:
        lib.curandDestroyGenerator(gen)


@pytest.mark.parametrize("seed", [0x0123456789ABCDEF, 0x9E3779B97F4A7C15, 7])
def test_philox_matches_curand_host_generator(seed):
    # The host generator's first 16384 blocks of four words: block n is
    # Philox of counter (0, 0, n, 0) under key (seed lo, seed hi). Every
    # counter word is non-zero after the first round, so all ten rounds, both
    # multipliers and both key words are exercised.
    nb = 16384
    ref = _curand_philox_host(seed, 4 * nb).reshape(nb, 4)
    n = np.arange(nb, dtype=np.uint64)
    got = np.stack(od.philox4x32_10(0, 0, n, 0, seed & 0xFFFFFFFF, seed >> 32), -1)
    np.testing.assert_array_equal(got, ref)


def test_philox_is_a_bijection_on_a_sample():
    # Distinct counters under one key give distinct outputs (no collisions
    # among 2^18 128-bit outputs; a collision would have probability ~2^-91).
    n = np.arange(1 << 18, dtype=np.uint64)
    w = np.stack(od.philox4x32_10(n & 0xFF, n >> 8, 3, 9, 11, 12), -1)
    assert len(np.unique(w.view([("", np.uint32)] * 4))) == len(n)


# --------------------------------------------------------------- keep decisions
def test_threshold_reading():
    assert od.threshold(0.0) == 0
    assert od.threshold(0.5) == 128
    assert od.threshold(0.1) == 26            # 25.6 rounds to 26
    assert od.threshold(0.25) == 64
    assert od.threshold(0.999) == 255         # 255.74 rounds to 256, capped
    assert od.rescale(64) == pytest.approx(4.0 / 3.0, rel=0, abs=1e-15)
    for bad in (1.0, -0.01, float("nan")):
        with pytest.raises(ValueError):
            od.threshold(bad)


def test_bytes_uniform_and_keep_fraction():
    by = od.draw_bytes(5, np.arange(1024), 1024, seed=1234, offset=0).ravel()
    n = by.size
    hist = np.bincount(by, minlength=256)
    chi2 = ((hist - n / 256) ** 2 / (n / 256)).sum()
    assert abs(chi2 - 255) < 8 * np.sqrt(2 * 255), chi2   # 255 degrees of freedom
    for p in (0.1, 0.5, 0.9):
        t = od.threshold(p)
        frac = (by >= t).mean()
        q = 1 - t / 256
        assert abs(frac - q) < 6 * np.sqrt(q * (1 - q) / n), (p, frac)


def test_masks_of_different_streams_are_uncorrelated():
    rows = np.arange(256)
    base = od.keep_mask(0, rows, 512, 42, 0, 0.5).astype(float)
    for other in (od.keep_mask(1, rows, 512, 42, 0, 0.5), od.keep_mask(0, rows, 512, 42, 1, 0.5),
                  od.keep_mask(0, rows, 512, 43, 0, 0.5), od.keep_mask(0, rows + 1, 512, 42, 0, 0.5)):
        c = np.corrcoef(base.ravel(), other.astype(float).ravel())[0, 1]
        assert abs(c) < 6 / np.sqrt(base.size), c


def test_keep_mask_depends_only_on_its_indices():
    # A row subset and a key prefix read the same draws as the full matrix.
    full = od.draw_bytes(3, np.arange(300), 200, 9, 2)
    sub = od.draw_bytes(3, np.array([5, 299, 17]), 37, 9, 2)
    np.testing.assert_array_equal(sub, full[[5, 299, 17], :37])


# --------------------------------------------------------------- attention with dropout
def test_p_zero_is_plain_attention():
    r = rng(1)
    B, H, N, d = 2, 2, 40, 8
    q, k, v, do = (r.normal(size=(B, H, N, d)) for _ in range(4))
    o0, l0 = oracle.forward(q, k, v, 0.3, causal=True)
    o1, l1 = oracle.forward(q, k, v, 0.3, causal=True, dropout=(0.0, 5, 6))
    np.testing.assert_array_equal(o0, o1)
    np.testing.assert_array_equal(l0, l1)
    g0 = oracle.backward(q, k, v, do, 0.3, causal=True)
    g1 = oracle.backward(q, k, v, do, 0.3, causal=True, dropout=(0.0, 5, 6))
    for a, b in zip(g0, g1):
        np.testing.assert_array_equal(a, b)


def test_lse_does_not_depend_on_dropout():
    r = rng(2)
    q, k, v = (r.normal(size=(1, 1, 50, 8)) for _ in range(3))
    _, l0 = oracle.forward(q, k, v, 0.4)
    _, l1 = oracle.forward(q, k, v, 0.4, dropout=(0.3, 1, 1))
    np.testing.assert_array_equal(l0, l1)


def test_dropped_output_is_unbiased():
    # E[O_dropout] = O: the mean over many independent masks converges to the
    # undropped output within a few standard errors.
    r = rng(3)
    n, d, p = 24, 6, 0.25
    q, k, v = (r.normal(size=(n, d)) for _ in range(3))
    o_ref, _ = oracle.head_forward(q, k, v, 0.5)
    reps = 3000
    acc = np.zeros((reps, n, d))
    for t in range(reps):
        acc[t], _ = oracle.head_forward(q, k, v, 0.5, drop=od.multiplier(0, 77, t, p))
    mean = acc.mean(0)
    se = acc.std(0) / np.sqrt(reps)
    z = np.abs(mean - o_ref) / se
    assert z.max() < 6, z.max()
    # without the 1 / (1 - p') factor the mean would be (1 - p') O: far outside
    assert np.abs(mean * (1 - od.threshold(p) / 256) - o_ref).max() > 10 * se.max()


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


@pytest.mark.parametrize("causal,kv_len,p", [(False, None, 0.3), (True, None, 0.5), (False, 5, 0.2)])
def test_dropout_backward_finite_differences(causal, kv_len, p):
    r = rng(4)
    n, d = 9, 3
    q, k, v, do = (r.normal(size=(n, d)) for _ in range(4))
    drop = od.multiplier(2, 1234, 5, p)
    assert 0 < (drop(np.arange(n), n) == 0).sum() < n * n   # some, not all, dropped
    got = oracle.head_backward(q, k, v, do, 0.7, causal=causal, kv_len=kv_len, drop=drop)
    ref = _fd_grads(q, k, v, do, 0.7, causal=causal, kv_len=kv_len, drop=drop)
    for g, f in zip(got, ref):
        err = np.max(np.abs(g - f)) / max(1e-12, np.max(np.abs(f)))
        assert err < 1e-6, err


def test_dropout_jacobian_route_equals_vector_route():
    r = rng(5)
    n, d = 20, 5
    q, k, v, do = (r.normal(size=(n, d)) for _ in range(4))
    drop = od.multiplier(1, 99, 0, 0.4)
    a = oracle.head_backward(q, k, v, do, 0.4, causal=True, drop=drop)
    b = oracle.head_backward_jacobian(q, k, v, do, 0.4, causal=True, drop=drop)
    for x, y in zip(a, b):
        np.testing.assert_allclose(x, y, atol=1e-12)


def test_batched_dropout_uses_problem_index():
    # forward() over [B, H] draws head (b, h) from problem b*H + h.
    r = rng(6)
    B, H, N, d = 2, 3, 20, 4
    q, k, v = (r.normal(size=(B, H, N, d)) for _ in range(3))
    o, _ = oracle.forward(q, k, v, 0.5, dropout=(0.5, 8, 3))
    oh, _ = oracle.head_forward(q[1, 2], k[1, 2], v[1, 2], 0.5, drop=od.multiplier(5, 8, 3, 0.5))
    np.testing.assert_array_equal(o[1, 2], oh)
