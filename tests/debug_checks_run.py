"""Child-process body of test_gpu_debug_checks.py (not a test module).

Run with KIVI_DEBUG_CHECKS=1 in the environment, so the binding loads the
checked build libkivi_debug.so (which this script builds first).  It drives
one small cache through appends, fused steps, decodes and chunked prefill,
checks bytes and outputs against the oracle as the other GPU tests do, and
reads the error word after each phase; it prints one JSON line of what the
word held.  Non-finite inputs are a precondition of the method; here they
are planted deliberately, in the inputs only, and the checked build must
report them (bit 3) without touching anything it should not.
"""
import json
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(HERE))
sys.path.insert(0, HERE)

import numpy as np  # noqa: E402
import torch  # noqa: E402

from kivi_quantized_kv_gb300 import build as kbuild  # noqa: E402

kbuild.build(debug_checks=True)

from kivi_quantized_kv_gb300 import KiviConfig, _abi  # noqa: E402
from gpu_util import TOL, Pair, random_q, random_stream, row_rel_err  # noqa: E402


def main():
    res = {"lib": os.path.basename(_abi.lib_path())}
    dev = torch.device("cuda")
    for bits, window in ((4, 0), (3, 0), (2, 160)):
        cfg = KiviConfig(bits=bits, group=32, residual=64, sinks=3, h_q=8, h_kv=2, head_dim=128, batch=2,
                         max_tokens=1024, window=window)
        p = Pair(cfg)
        k, v = random_stream(cfg, 300, seed=11 + bits)
        p.append(k[:, :, :290], v[:, :, :290])
        for t in range(290, 300):   # fused steps over a freeze
            q = random_q(cfg, seed=t)
            out = p.gpu.append_decode(k[:, :, t:t + 1].to(dev), v[:, :, t:t + 1].to(dev), q.to(dev))
            assert p.ref.append(k[:, :, t:t + 1].numpy(), v[:, :, t:t + 1].numpy()) == 0
            err = row_rel_err(out.float().cpu().numpy(), p.ref.decode_attn(q.numpy(), threads=8))
            assert err <= TOL, (bits, t, err)
        assert p.bytes_equal()
        m = 16
        qm = torch.randn((cfg.batch, m, cfg.h_q, cfg.head_dim), generator=torch.Generator().manual_seed(5)).half()
        got = p.gpu.prefill(qm.to(dev)).float().cpu().numpy()
        err = row_rel_err(got, p.ref.prefill_attn(qm.numpy()))
        assert err <= TOL, (bits, "prefill", err)
        res[f"clean_b{bits}"] = p.gpu.read_error()

    # planted non-finite inputs: a NaN key, an inf value, an inf query element
    cfg = KiviConfig(bits=4, group=32, residual=64, sinks=3, h_q=8, h_kv=2, head_dim=128, batch=2, max_tokens=512)
    p = Pair(cfg)
    k, v = random_stream(cfg, 200, seed=3)
    p.append(k, v)
    res["before"] = p.gpu.read_error()
    k1, v1 = random_stream(cfg, 1, seed=4)
    k1[1, 0, 0, 7] = float("nan")
    p.gpu.append(k1.to(dev), v1.to(dev))
    res["nan_key_append"] = p.gpu.read_error()
    k2, v2 = random_stream(cfg, 40, seed=5)   # a chunk (its append also freezes a group) with an inf value
    v2[0, 1, 3, 100] = float("inf")
    p.gpu.append(k2.to(dev), v2.to(dev))
    res["inf_value_append"] = p.gpu.read_error()
    q = random_q(cfg, seed=6)
    q[1, 5, 9] = float("-inf")
    p.gpu.decode(q.to(dev))
    res["inf_query"] = p.gpu.read_error()
    q = random_q(cfg, seed=7)
    p.gpu.decode(q.to(dev))
    res["after"] = p.gpu.read_error()
    print(json.dumps(res), flush=True)


if __name__ == "__main__":
    main()
