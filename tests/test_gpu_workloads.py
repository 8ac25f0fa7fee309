"""Parity at the workloads' full sizes, in the launch configuration the
benchmark times (automatic split count).

The CUDA cache is filled with the whole workload (every sequence and kv
head) from the seeded generator on the GPU.  The oracle cannot afford every
unit, so it rebuilds a few sampled (sequence, kv head) units from the same
input chunks: units never interact, so each sampled unit's bytes and its
query heads' attention rows must match exactly / within 2e-3.
"""
import numpy as np
import pytest
import torch

import oracle
from kivi_quantized_kv_gb300 import KiviCache, KiviConfig
from kivi_quantized_kv_gb300.synth import KVStream, WORKLOADS, queries, sweep_workload
from gpu_util import TOL, oparams, row_rel_err

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__ as ge
    ge.build()
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def run_sampled(w, units, chunk=2048, layer=0):
    dev = torch.device("cuda")
    cfg = KiviConfig.from_workload(w)
    cache = KiviCache(cfg, device=dev)
    stream = KVStream(w, layer=layer, device=dev)
    ks = {u: [] for u in units}
    vs = {u: [] for u in units}
    t = 0
    while t < w.tokens:
        n = min(chunk, w.tokens - t)
        k, v = stream.next(n)
        cache.append(k, v)
        for (b, h) in units:
            ks[(b, h)].append(k[b, h].cpu())
            vs[(b, h)].append(v[b, h].cpu())
        t += n
    q = queries(w, layer=layer, device=dev)
    out = cache.decode(q).float().cpu().numpy()
    torch.cuda.synchronize()
    arena = cache.cache_region()
    L = cache.layout()
    rep = w.h_q // w.h_kv
    worst = 0.0
    for (b, h) in units:
        p1 = oparams(cfg, batch=1, h_kv=1, h_q=rep)
        ref = oracle.Cache(p1)
        kk = torch.cat(ks[(b, h)], dim=0)[None, None].numpy()
        vv = torch.cat(vs[(b, h)], dim=0)[None, None].numpy()
        assert ref.append(kk, vv) == 0
        u = b * w.h_kv + h
        got = arena[u * L["unit_bytes"]:(u + 1) * L["unit_bytes"]].cpu().numpy()
        assert np.array_equal(got, ref.arena()), (w.name, b, h)
        qq = q[b, h * rep:(h + 1) * rep].cpu()[None].numpy()
        exp = ref.decode_attn(qq)
        err = row_rel_err(out[b, h * rep:(h + 1) * rep][None], exp)
        assert err <= TOL, (w.name, b, h, err)
        worst = max(worst, err)
    return worst


@pytest.mark.parametrize("name", ["tiny", "mha7b", "gqa8b_b4", "gqa8b_b2", "swa_mistral", "mha7b_b3", "gqa8b_b3",
                                  "mha_d64_b3", "mha7b_o10", "mha7b_b3_o10", "gqa8b_b4_prerope"])
def test_workload_full_size_sampled_units(name):
    """Sixteen (sequence, kv head) units per workload (all of them when it has
    fewer), the first and the last among them.  With 304 CTAs over at most
    256 units, nearly every unit's positions are cut between CTAs, so the
    sampled units go through the cross-CTA merge."""
    w = WORKLOADS[name]
    units = sampled_units(w.batch, w.h_kv, 16, seed=len(name))
    err = run_sampled(w, units)
    print(f"{name}: worst row error {err:.2e}")


def sampled_units(batch, h_kv, n, seed):
    """n distinct (sequence, kv head) units, the first and last among them."""
    g = np.random.default_rng(seed)
    total = batch * h_kv
    others = [int(u) for u in g.permutation(total) if u not in (0, total - 1)]
    pick = sorted({0, total - 1} | set(others[:max(0, n - 2)]))
    return [(u // h_kv, u % h_kv) for u in pick]


@pytest.mark.parametrize("batch,tokens,bits,layer", [(16, 16384, 4, 0), (1, 131072, 2, 31), (128, 1024, 8, 5),
                                                     (16, 1024, 2, 17)])
def test_sweep_cells_sampled(batch, tokens, bits, layer):
    """Cells of the 32-layer decode-step sweep at full size, 16 sampled
    (sequence, kv head) units each (every unit when a cell has fewer)."""
    w = sweep_workload(batch, tokens, bits)
    run_sampled(w, sampled_units(batch, w.h_kv, 16, seed=batch * 7 + bits), chunk=4096, layer=layer)


@pytest.mark.parametrize("bits", [2, 4, 8])
def test_sweep_full_32_layer_step(bits):
    """One whole decode step of the smallest sweep cell (B 1, T 1024): each of
    the 32 layers holds its own cache (seeded per layer) and takes its fused
    append + decode call; every layer's bytes and every head's output are
    checked against an oracle cache of that layer."""
    from kivi_quantized_kv_gb300.synth import KVStream, queries
    w = sweep_workload(1, 1024, bits)
    dev = torch.device("cuda")
    cfg = KiviConfig.from_workload(w)
    worst = 0.0
    for layer in range(w.layers):
        cache = KiviCache(cfg, device=dev)
        ref = oracle.Cache(oparams(cfg))
        stream = KVStream(w, layer=layer, device="cpu")
        k, v = stream.next(w.tokens - 1)
        cache.append(k.to(dev), v.to(dev))
        assert ref.append(k.numpy(), v.numpy()) == 0
        k1, v1 = stream.next(1)
        q = queries(w, layer=layer)
        out = cache.append_decode(k1.to(dev), v1.to(dev), q.to(dev)).float().cpu().numpy()
        assert ref.append(k1.numpy(), v1.numpy()) == 0
        torch.cuda.synchronize()
        assert np.array_equal(cache.cache_region().cpu().numpy(), ref.arena()), layer
        err = row_rel_err(out, ref.decode_attn(q.numpy(), threads=8))
        assert err <= TOL, (layer, err)
        worst = max(worst, err)
        assert cache.read_error() == 0
    print(f"32 layers, {bits} bits: worst row error {worst:.2e}")
