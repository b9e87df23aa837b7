"""Host-side checks of the C-ABI: the library builds and loads, exports every
symbol include/fa.h declares, and rejects invalid arguments before touching
the GPU. Fake pointers are used only in calls that must fail validation, so
these tests are skipped where a GPU is present (the GPU tests cover the
valid paths with real buffers)."""
import ctypes
import os
import re
import subprocess

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fa.h")


@pytest.fixture(scope="module")
def L():
    from exact_io_aware_11_gb300 import build
    build.build()
    import exact_io_aware_11_gb300 as fa
    return fa.lib()


def declared_symbols():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"^[a-z][\w\s\*]*?\b(fa_\w+)\(", text, flags=re.M)))


def test_header_declares_the_boundary():
    names = declared_symbols()
    for n in ("fa_fwd", "fa_fwd_kpad", "fa_bwd", "fa_bwd_workspace_bytes", "fa_blocksparse_fwd",
              "fa_blocksparse_bwd", "fa_dropout_fwd", "fa_dropout_bwd", "fa_dropout_mask",
              "fa_device_status", "fa_status_string", "fa_selftest_wait_timeout"):
        assert n in names


def test_library_exports_every_declared_symbol(L):
    from exact_io_aware_11_gb300 import library_path
    out = subprocess.run(["nm", "-D", "--defined-only", library_path()], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r"\sT\s(fa_\w+)$", out, flags=re.M))
    missing = [n for n in declared_symbols() if n not in exported]
    assert not missing, missing
    for n in declared_symbols():
        assert hasattr(L, n)


def test_status_strings(L):
    import exact_io_aware_11_gb300 as fa
    assert fa.status_string(0) == "FA_OK"
    assert fa.status_string(4) == "FA_ERR_DEVICE_TIMEOUT"
    assert fa.status_string(5) == "FA_ERR_DEVICE_CHECK"
    assert fa.status_string(99) == "FA_UNKNOWN_STATUS"


def test_checked_build_exports_every_declared_symbol():
    """The FA_CHECKS build (device-side checks of every TMA copy) compiles and
    exports the same boundary; the GPU test runs it."""
    from exact_io_aware_11_gb300 import build
    path = build.build(checked=True)
    out = subprocess.run(["nm", "-D", "--defined-only", path], capture_output=True, text=True,
                         check=True).stdout
    exported = set(re.findall(r"\sT\s(fa_\w+)$", out, flags=re.M))
    missing = [n for n in declared_symbols() if n not in exported]
    assert not missing, missing


def test_workspace_bytes_is_linear_in_n(L):
    import exact_io_aware_11_gb300 as fa
    for d in (64, 128):
        a = fa.bwd_workspace_bytes(2, 3, 1024, d)
        b = fa.bwd_workspace_bytes(2, 3, 2048, d)
        assert a == 2 * 3 * 1024 * (4 * d + 8)
        assert b == 2 * a
    # ragged N is padded to whole 128-row tiles
    assert fa.bwd_workspace_bytes(1, 1, 130, 64) == fa.bwd_workspace_bytes(1, 1, 256, 64)
    assert fa.bwd_workspace_bytes(1, 1, 0, 64) == 0
    assert fa.bwd_workspace_bytes(1, 1, 128, 96) == 0


needs_cpu = pytest.mark.skipif(torch.cuda.is_available(),
                               reason="fake-pointer validation tests run on CPU-only hosts")

A = 1 << 20          # fake, 16-byte aligned "device" addresses, never dereferenced
SPAN = 1 << 28


def ptrs(n):
    return [A + i * SPAN for i in range(n)]


@needs_cpu
@pytest.mark.parametrize("case,expect", [
    (dict(B=0), 1), (dict(H=0), 1), (dict(N=0), 1), (dict(d=96), 2), (dict(d=32), 2),
    (dict(causal=2), 1), (dict(scale=float("nan")), 1), (dict(scale=float("inf")), 1),
    (dict(scale=-0.125), 1), (dict(scale=0.0), 1),
    (dict(q=None), 1), (dict(o=None), 1), (dict(lse=None), 1), (dict(q=A + 8), 1),
    (dict(o=A + 4 * SPAN + 2), 1),
    (dict(o=A), 1),                         # output aliases q
    (dict(lse=A + 3 * SPAN + 64), 1),        # lse overlaps o
])
def test_fwd_rejects_invalid(L, case, expect):
    q, k, v, o, lse = ptrs(5)
    args = dict(q=q, k=k, v=v, o=o, lse=lse, B=2, H=2, N=256, d=64, causal=0, scale=0.125)
    args.update(case)
    rc = L.fa_fwd(args["q"], args["k"], args["v"], args["o"], args["lse"], args["B"], args["H"],
                  args["N"], args["d"], args["causal"], args["scale"], None)
    assert rc == expect


@needs_cpu
def test_kpad_rejects_misaligned_kv_len(L):
    q, k, v, o, lse, kv = ptrs(6)
    assert L.fa_fwd_kpad(q, k, v, o, lse, 1, 1, 128, 64, 0, 0.125, kv + 2, None) == 1


@needs_cpu
@pytest.mark.parametrize("case,expect", [
    (dict(block_mask=None), 1), (dict(block_size=64), 2), (dict(d=80), 2), (dict(N=-1), 1),
])
def test_blocksparse_rejects_invalid(L, case, expect):
    q, k, v, o, lse, m = ptrs(6)
    args = dict(B=1, H=1, N=256, d=64, scale=0.125, block_mask=m, block_size=128)
    args.update(case)
    rc = L.fa_blocksparse_fwd(q, k, v, o, lse, args["B"], args["H"], args["N"], args["d"],
                              args["scale"], args["block_mask"], args["block_size"], None)
    assert rc == expect


@needs_cpu
@pytest.mark.parametrize("case,expect", [
    (dict(ws_bytes=-1), 1),                  # one byte short
    (dict(workspace=None), 1), (dict(dout=None), 1), (dict(dq=A), 1),   # dq aliases q
    (dict(dk=A + 6 * SPAN), 1),              # dk aliases dq
    (dict(workspace=A + 8 * SPAN + 8), 1),   # misaligned workspace
    (dict(workspace=A + SPAN), 1),           # workspace overlaps k
    (dict(d=256), 2), (dict(causal=-1), 1),
])
def test_bwd_rejects_invalid(L, case, expect):
    q, k, v, o, do, lse, dq, dk, dv, ws = ptrs(10)
    B, H, N, d = 2, 2, 256, case.get("d", 64)
    need = L.fa_bwd_workspace_bytes(B, H, N, 64)
    args = dict(q=q, k=k, v=v, o=o, dout=do, lse=lse, dq=dq, dk=dk, dv=dv, workspace=ws,
                ws_bytes=0, causal=0)
    args.update(case)
    rc = L.fa_bwd(args["q"], args["k"], args["v"], args["o"], args["dout"], args["lse"],
                  args["dq"], args["dk"], args["dv"], B, H, N, d, args["causal"], 0.125, None,
                  args["workspace"], need + args["ws_bytes"], None)
    assert rc == expect


@needs_cpu
def test_python_binding_refuses_cpu_tensors(L):
    import exact_io_aware_11_gb300 as fa
    x = torch.zeros(1, 1, 128, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        fa.forward(x, x, x)


@needs_cpu
def test_device_calls_fail_cleanly_without_gpu(L):
    import exact_io_aware_11_gb300 as fa
    # No device: status cannot be read, the self-test cannot launch.
    assert fa.device_status() in (fa.FA_ERR_CUDA, fa.FA_ERR_UNSUPPORTED)
    assert L.fa_selftest_wait_timeout(0, None) == fa.FA_ERR_INVALID_ARG


@needs_cpu
@pytest.mark.parametrize("p,expect", [(1.0, 1), (-0.01, 1), (float("nan"), 1), (1.5, 1)])
def test_dropout_rejects_invalid_probability(L, p, expect):
    q, k, v, o, lse, do, dq, dk, dv, ws, keep = ptrs(11)
    assert L.fa_dropout_fwd(q, k, v, o, lse, 1, 1, 128, 64, 0, 0.125, None, p, 1, 0, None) == expect
    need = L.fa_bwd_workspace_bytes(1, 1, 128, 64)
    assert L.fa_dropout_bwd(q, k, v, o, do, lse, dq, dk, dv, 1, 1, 128, 64, 0, 0.125, None, p, 1,
                            0, ws, need, None) == expect
    assert L.fa_dropout_mask(1, 1, 128, p, 1, 0, keep, None) == expect


@needs_cpu
def test_dropout_validates_like_the_plain_calls(L):
    q, k, v, o, lse, keep = ptrs(6)
    assert L.fa_dropout_fwd(q, k, v, o, lse, 1, 1, 128, 96, 0, 0.125, None, 0.1, 1, 0, None) == 2
    assert L.fa_dropout_fwd(q, k, v, q, lse, 1, 1, 128, 64, 0, 0.125, None, 0.1, 1, 0, None) == 1
    assert L.fa_dropout_mask(0, 1, 128, 0.1, 1, 0, keep, None) == 1
    assert L.fa_dropout_mask(1, 1, 128, 0.1, 1, 0, None, None) == 1


def test_python_dropout_arguments_checked_before_any_call():
    import exact_io_aware_11_gb300 as fa
    with pytest.raises(ValueError):
        fa._lib._check_dropout(1.0, 0, 0)
    with pytest.raises(ValueError):
        fa._lib._check_dropout(0.1, -1, 0)
    with pytest.raises(ValueError):
        fa._lib._check_dropout(0.1, 0, 2 ** 32)
    assert fa._lib._check_dropout(0.25, 2 ** 64 - 1, 2 ** 32 - 1) == (0.25, 2 ** 64 - 1, 2 ** 32 - 1)


def _opts(**kw):
    from exact_io_aware_11_gb300 import AttentionOptions
    o = AttentionOptions()
    o.scale = 0.125
    o.block_size = 128
    for k_, v_ in kw.items():
        setattr(o, k_, v_)
    return o


@needs_cpu
@pytest.mark.parametrize("strides,expect", [
    ((0, 0, 0), 3),                                   # row-major [B,H,N,d]: valid (no device here)
    ((256 * 4 * 64, 64, 4 * 64), 3),                  # [B,N,H,d]
    ((4 * 256 * 128, 256 * 128, 128), 3),             # rows padded to 128 elements
    ((4 * 256 * 64, 256 * 64, 68), 1),                # row stride not a multiple of 8
    ((4 * 256 * 64, 256 * 64 - 8, 64), 1),            # heads overlap
    ((4 * 256 * 64, 64, 64), 1),                      # rows of different heads overlap
    ((-4 * 256 * 64, 256 * 64, 64), 1),               # negative
    ((4 * 256 * 64, 256 * 64, 56), 1),                # row stride < d
])
def test_attention_strides_validated(L, strides, expect):
    import ctypes
    q, k, v, o, lse = ptrs(5)
    opt = _opts(stride_b=strides[0], stride_h=strides[1], stride_n=strides[2])
    assert L.fa_attention_fwd(q, k, v, o, lse, 2, 4, 256, 64, ctypes.byref(opt), None) == expect


@needs_cpu
def test_attention_options_validated(L):
    import ctypes
    q, k, v, o, lse, m = ptrs(6)
    assert L.fa_attention_fwd(q, k, v, o, lse, 1, 1, 128, 64, None, None) == 1
    for kw, expect in [(dict(dropout_p=1.0), 1), (dict(dropout_p=-0.5), 1), (dict(causal=3), 1),
                       (dict(scale=0.0), 1), (dict(block_mask=m, block_size=64), 2),
                       (dict(block_mask=m, causal=1, dropout_p=0.3), 3)]:
        opt = _opts(**kw)
        assert L.fa_attention_fwd(q, k, v, o, lse, 1, 1, 128, 64, ctypes.byref(opt), None) == expect, kw


@needs_cpu
def test_attention_strides_reject_huge_spans(L):
    import ctypes
    q, k, v, o, lse = ptrs(5)
    # a row stride whose span over N rows passes 2^36 elements (and whose
    # product with N would overflow 64 bits if it were formed unchecked)
    opt = _opts(stride_b=0, stride_h=0, stride_n=(1 << 35))
    assert L.fa_attention_fwd(q, k, v, o, lse, 1, 1, 1 << 30, 64, ctypes.byref(opt), None) == 1
    opt = _opts(stride_b=(1 << 35) - 8, stride_h=64, stride_n=128)
    assert L.fa_attention_fwd(q, k, v, o, lse, 4, 2, 16, 64, ctypes.byref(opt), None) == 1


@needs_cpu
@pytest.mark.parametrize("B,H,N", [(65535, 65535, 128), (4096, 4096, 1 << 14), (1, 1, (1 << 31) - 1)])
def test_sizes_beyond_32_bit_work_counts_rejected(L, B, H, N):
    # B*H*ceil(N/128) work items (or N rounded up to whole tiles) past 2^31 - 1
    q, k, v, o, lse, keep = ptrs(6)
    assert L.fa_fwd(q, k, v, o, lse, B, H, N, 64, 0, 0.125, None) == 1
    assert L.fa_dropout_mask(B, H, N, 0.1, 1, 0, keep, None) == 1



def test_split_workspace_queries(L):
    import exact_io_aware_11_gb300 as fa
    for d in (64, 128):
        # one 128-row Q tile: nothing to split
        assert fa.fwd_workspace_bytes(1, 1, 128, d, False) == 0
        # two (b, h) problems of 4096 rows: 32 items for over a hundred SMs
        assert fa.fwd_workspace_bytes(1, 2, 4096, d, True) > 0
        base = fa.bwd_workspace_bytes(1, 2, 4096, d)
        assert fa.bwd_split_workspace_bytes(1, 2, 4096, d, False) > base
        assert fa.bwd_split_workspace_bytes(1, 1, 128, d, False) == fa.bwd_workspace_bytes(1, 1, 128, d)
    for args in [(0, 1, 128, 64, 0), (1, 1, 128, 96, 0), (1, 1, 128, 64, 2), (1, 1, 0, 64, 0)]:
        assert L.fa_fwd_workspace_bytes(*args) == 0
        assert L.fa_bwd_split_workspace_bytes(*args) == 0


def test_workspace_bytes_zero_for_unrepresentable_sizes(L):
    # N near INT_MAX would overflow the tile rounding; B or H beyond 65535 is
    # rejected by every entry point, so no workspace size exists for them.
    assert L.fa_bwd_workspace_bytes(1, 1, (1 << 31) - 1, 64) == 0
    assert L.fa_bwd_workspace_bytes(65536, 1, 128, 64) == 0
    assert L.fa_bwd_workspace_bytes(1, 1, (1 << 31) - 256, 128) > 0


@needs_cpu
def test_noalloc_boundary_at_the_scratch_size(L):
    # rows = B*H*Npad; d = 64 needs 4*64 + 8 bytes a row: 1985 heads of 128
    # rows fit in 64 MiB, 1986 do not. The size check runs before any CUDA
    # call, so without a GPU the call that fits reaches the device query
    # (FA_ERR_CUDA) and the one that does not is rejected (FA_ERR_INVALID_ARG).
    limit = 64 * 1024 * 1024
    assert L.fa_bwd_workspace_bytes(1, 1985, 128, 64) <= limit
    assert L.fa_bwd_workspace_bytes(1, 1986, 128, 64) > limit
    assert L.fa_bwd_workspace_bytes(1, 1008, 128, 128) <= limit
    assert L.fa_bwd_workspace_bytes(1, 1009, 128, 128) > limit
    q, k, v, o, do, lse, dq, dk, dv = ptrs(9)
    assert L.fa_bwd_noalloc(q, k, v, o, do, lse, dq, dk, dv, 1, 1986, 128, 64, 0, 0.125, None,
                            None) == 1
    assert L.fa_bwd_noalloc(None, k, v, o, do, lse, dq, dk, dv, 1, 1985, 128, 64, 0, 0.125, None,
                            None) == 1
    assert L.fa_bwd_noalloc(q, k, v, o, do, lse, dq, dk, dv, 1, 1985, 128, 64, 0, 0.125, None,
                            None) == 3


@needs_cpu
def test_interleaved_views_accepted_overlapping_rejected(L):
    """q, k, v (and dq, dk, dv) as the three slices of one packed [B, N, 3, H, d]
    buffer share no element, so validation accepts them (and then fails only for
    want of a device); outputs that do share elements are rejected."""
    import ctypes
    B, H, N, d = 2, 4, 256, 64
    sb, sh, sn = N * 3 * H * d, d, 3 * H * d          # element strides of each slice
    opt = _opts(stride_b=sb, stride_h=sh, stride_n=sn)
    P, G, O, DO, LSE, WS = ptrs(6)                    # packed inputs, packed gradients, ...
    q, k, v = P, P + 2 * H * d, P + 4 * H * d         # byte offsets of the slices
    dq, dk, dv = G, G + 2 * H * d, G + 4 * H * d
    o, do = O, O + 2 * H * d
    need = L.fa_bwd_workspace_bytes(B, H, N, d)
    rc = L.fa_attention_fwd(q, k, v, o, LSE, B, H, N, d, ctypes.byref(opt), None)
    assert rc == 3
    rc = L.fa_attention_bwd(q, k, v, o, do, LSE, dq, dk, dv, B, H, N, d, ctypes.byref(opt), WS,
                            need, None)
    assert rc == 3
    # dk shifted by half a row onto dq's elements, or equal to dq: rejected
    for bad_dk in (G + d, G):
        rc = L.fa_attention_bwd(q, k, v, o, do, LSE, dq, bad_dk, dv, B, H, N, d,
                                ctypes.byref(opt), WS, need, None)
        assert rc == 1
    # an output on an input's elements (o on k's slice): rejected
    assert L.fa_attention_fwd(q, k, v, k, LSE, B, H, N, d, ctypes.byref(opt), None) == 1
