"""bench.py's algorithmic byte and FLOP counts (CPU only).

The byte counts are checked against the library's own counts at run time on
the GPU; here they are pinned against the oracle's layout and its count of
decode bytes, and the prefill FLOP count against a brute-force count of the
(query row, visible token) pairs under the causal and window rules.
"""
import numpy as np
import pytest

import bench
from kivi_quantized_kv_gb300.synth import Workload


def W(**kw):
    base = dict(name="t", batch=2, h_q=8, h_kv=2, head_dim=64, tokens=300, bits=4, group=16, residual=32,
                sinks=3, window=0)
    base.update(kw)
    return Workload(**base)


def n_slots(oracle_lib, w, T):
    p = oracle_lib.Params(bits=w.bits, group=w.group, residual=w.residual, sinks=w.sinks, h_q=w.h_q,
                          h_kv=w.h_kv, head_dim=w.head_dim, batch=w.batch, max_tokens=0 if w.window else T,
                          window=w.window, outlier_permille=w.outlier_permille)
    return oracle_lib.layout(p)["n_slots"], p


@pytest.mark.parametrize("window,T,pm", [(0, 1, 0), (0, 3, 0), (0, 35, 0), (0, 300, 0), (48, 300, 0), (48, 1000, 0),
                                         (64, 77, 0), (0, 300, 10), (48, 1000, 37)])
def test_decode_bytes_match_the_oracle(oracle_lib, window, T, pm):
    w = W(window=window, group=32, outlier_permille=pm) if pm else W(window=window)
    ns, p = n_slots(oracle_lib, w, T)
    c = oracle_lib.Cache(p)
    rng = np.random.default_rng(T)
    k = rng.standard_normal((w.batch, w.h_kv, T, w.head_dim)).astype(np.float16)
    assert c.append(k, k) == 0
    assert bench.decode_bytes_at(w, T, ns) == c.decode_bytes()


@pytest.mark.parametrize("window,T,m", [(0, 300, 1), (0, 300, 64), (0, 40, 40), (48, 300, 20), (48, 300, 200),
                                        (64, 1000, 150)])
def test_prefill_flops_count_visible_pairs(oracle_lib, window, T, m):
    w = W(window=window)
    ns, _ = n_slots(oracle_lib, w, T)
    _, ng, _ = bench.state_at(w, T)
    pos = np.arange(T)
    resident = np.ones(T, bool)
    if window:
        first = max(ng - ns, 0)
        resident = (pos < w.sinks) | (pos >= w.sinks + first * w.group)
    pairs = 0
    for j in range(m):
        P = T - m + j
        vis = resident & (pos <= P)
        if window:
            vis &= (pos < w.sinks) | (pos >= P + 1 - window)
        pairs += int(vis.sum())
    assert bench.prefill_flops_at(w, T, m, ns) == 4 * w.head_dim * pairs * w.batch * w.h_q


def test_prefill_bytes_of_one_query_are_decode_bytes():
    for window, T in ((0, 300), (48, 300), (48, 1000)):
        w = W(window=window)
        ns = 1000 if not window else -(-window // w.group) + 1
        assert bench.prefill_bytes_at(w, T, 1, ns) == bench.decode_bytes_at(w, T, ns)
