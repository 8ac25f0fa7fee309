"""The checked build (KIVI_DEBUG_CHECKS=1, libkivi_debug.so).

In a child process that loads the checked library, a cache runs appends,
fused steps, decodes and chunked prefill at 2, 3 and 4 bits (one with a
window) and must match the oracle with an empty error word; then inputs with
a NaN key, an inf value and an inf query element are planted, and each call
that read one must report bit 3 (non-finite input) while nothing sets bit 2
(an address outside the cache region).  The product library is untouched.
"""
import json
import os
import subprocess
import sys

import pytest
import torch

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))


def test_checked_build_is_clean_and_flags_non_finite_inputs():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    env = dict(os.environ, KIVI_DEBUG_CHECKS="1")
    r = subprocess.run([sys.executable, os.path.join(HERE, "debug_checks_run.py")], env=env, capture_output=True,
                       text=True, timeout=900)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-4000:]
    res = json.loads([line for line in r.stdout.splitlines() if line.startswith("{")][-1])
    print(res)
    assert res["lib"] == "libkivi_debug.so"
    for key in ("clean_b4", "clean_b3", "clean_b2", "before", "after"):
        assert res[key] == 0, (key, res[key])
    for key in ("nan_key_append", "inf_value_append", "inf_query"):
        assert res[key] == 8, (key, res[key])
