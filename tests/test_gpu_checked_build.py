"""The checked build (-DFA_CHECKS=1): on the device, every TMA copy checks its
coordinates and addresses before it is issued and reports a failure as
FA_ERR_DEVICE_CHECK instead of issuing it. Representative calls -- ragged N,
key padding, a [B, N, H, d] layout with dropout, block masks at d = 64 and
128, split workspaces -- run with it in a child process; the device status
must stay clean and the results must equal the default build's (dQ, summed by
reduce-adds in any order, to 1e-2)."""
import os
import subprocess
import sys

import pytest
import torch

import _checked_cases

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
TESTS = os.path.join(ROOT, "tests")

CHILD = """
import sys, torch
sys.path.insert(0, {root!r}); sys.path.insert(0, {tests!r})
from exact_io_aware_11_gb300 import _lib
_lib._LIB_PATH = {lib!r}
import exact_io_aware_11_gb300 as fa
import _checked_cases
assert fa.lib()._name == {lib!r}
torch.save(_checked_cases.run_cases(fa), {out!r})
"""


def test_checked_build_matches_default(fa, tmp_path):
    from exact_io_aware_11_gb300 import build
    lib = build.build(checked=True)
    out = str(tmp_path / "checked.pt")
    code = CHILD.format(root=ROOT, tests=TESTS, lib=lib, out=out)
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-3000:]
    checked = torch.load(out)
    ref = _checked_cases.run_cases(fa)
    assert set(checked) == set(ref)
    for key in ref:
        for idx, (a, b) in enumerate(zip(checked[key], ref[key])):
            if idx == 2:  # dQ
                assert torch.allclose(a.float(), b.float(), rtol=0, atol=1e-2), key
            else:
                assert torch.equal(a, b), (key, idx)
