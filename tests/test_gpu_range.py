"""The decode over keys, values and queries that span the fp16 range, through
the C ABI against the oracle.

KV-cache quantization guide (pigeon), "How it works", steps 3 and 5: the
quantizer and the attention over the dequantized values hold for any finite
input, and the oracle evaluates them in fp64 for every finite fp16 input.
The tensor-core decode folds the key scales into the query (q_c Δ_c, split
into two fp16 halves) and the value scales into the softmax weights
(p_t Δ_t 2^-k, likewise): with key channels and value tokens near the top of
the fp16 range and queries far above 1, those products leave the fp16 range
unless the kernel rescales them.  These streams reach that regime (the
helpers below assert it from the oracle's own bytes), at 2, 3, 4 and 8 bits,
head dims 64 and 128, MHA and GQA, groups of one and two 32-token chunks,
outlier tables, a window and chunked prefill; and the other end of the range
(values near the fp16 subnormals).  Bytes must be identical and attention
within 2e-3 of the oracle, with every output finite.
"""
import numpy as np
import pytest
import torch

from gpu_util import TOL, Pair, row_rel_err

pytestmark = pytest.mark.gpu

FP16_MAX = 65504.0


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__ as ge
    ge.build()
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def wide_stream(cfg, T, seed, kscale=3.0e3, vscale=2.0e4, tiny=False):
    """Keys N(0,1) with two channels x kscale; values N(0,1) times a per-token
    scale log-uniform in [1, vscale]; everything clipped to the fp16 range.
    tiny: plain N(0,1) keys and values scaled by 2^-8 instead (value steps
    p Δ_t 2^-k among the fp16 subnormals, outputs still normal fp16)."""
    g = torch.Generator().manual_seed(seed)
    shape = (cfg.batch, cfg.h_kv, T, cfg.head_dim)
    k = torch.randn(shape, generator=g)
    v = torch.randn(shape, generator=g)
    if tiny:
        v *= 2.0 ** -8
    else:
        k[..., 1] *= kscale
        k[..., cfg.head_dim - 3] *= -0.7 * kscale
        v *= torch.exp(torch.rand((*shape[:3], 1), generator=g) * float(np.log(vscale)))
    lim = FP16_MAX * 0.999
    return k.clamp(-lim, lim).half(), v.clamp(-lim, lim).half()


def wide_q(cfg, seed, rows=None, big=20.0):
    """N(0,1) queries; every third head x big and head 1 x 3 big (|q| up to a
    few hundred)."""
    g = torch.Generator().manual_seed(seed + 7)
    q = torch.randn((cfg.batch,) + ((rows,) if rows else ()) + (cfg.h_q, cfg.head_dim), generator=g)
    q[..., ::3, :] *= big
    if cfg.h_q > 1:
        q[..., 1, :] *= 3 * big
    return q.clamp(-FP16_MAX, FP16_MAX).half()


def conditioned_err(pair, q, out, exp, rows_q=None):
    """Row error (as row_rel_err) over the rows that fp32 resolves, and the
    share of rows left out.  The kernel evaluates a score as
    Σ_c q_c min_c + Σ_c q_c Δ_c code_c in fp32, whose partial sums reach
    Σ_c |q_c| max_t |k_tc| (the channels' largest keys, min and the code term
    each up to about that); a few fp32 rounding steps of that, δ = 2^-18 of
    it / sqrt(d), is what the score can be off by.  A row's first-order output
    change when every score moves by δ is Σ_t w_t |v_t - o| δ; where that
    exceeds TOL / 2 of the row's largest output (tokens tied within δ whose
    values differ by far more than the output), fp32 scores do not resolve the
    row to TOL, and it is left out."""
    p = pair.ref.p
    rep = p.h_q // p.h_kv
    d = p.head_dim
    T = pair.ref.T
    o = out.reshape(-1, d).astype(np.float64)
    x = exp.reshape(-1, d)
    keep = np.ones(o.shape[0], bool)
    nq = rows_q or 1
    for b in range(p.batch):
        for h in range(p.h_kv):
            K, V, vis = pair.ref.dequant_unit(b, h)
            for j in range(nq):
                P = T - nq + j
                vj = vis & (np.arange(T) <= P)
                for r in range(rep):
                    hq = h * rep + r
                    row = (b * nq + j) * p.h_q + hq
                    qq = (q[b, j, hq] if rows_q else q[b, hq]).double().numpy()
                    s = np.where(vj, K @ qq, -np.inf) / np.sqrt(d)
                    w = np.exp(s - s.max())
                    w /= w.sum()
                    kmax = np.abs(K[vj]).max(axis=0)
                    delta = 2.0 ** -18 * (kmax @ np.abs(qq)) / np.sqrt(d)
                    sens = (w[:, None] * np.abs(V - x[row]) * delta).sum(0).max()
                    keep[row] = sens <= TOL / 2 * np.abs(x[row]).max()
    scale = np.abs(x[keep]).max(1)
    err = float((np.abs(o[keep] - x[keep]).max(1) / np.where(scale == 0, 1, scale)).max()) if keep.any() else 0.0
    return err, 1.0 - keep.mean()


def fp32_floor(pair, q):
    """Row error against the oracle of the same attention evaluated plainly
    in fp32 (fp32 dot products and softmax over the oracle's own dequantized
    values).  Scores far above 2^12 in magnitude lose the 2e-3 bar in any
    fp32 evaluation; the streams here stay well inside what fp32 resolves, so
    that a failure is the kernel's and not fp32's."""
    p = pair.ref.p
    rep = p.h_q // p.h_kv
    exp = pair.ref.decode_attn(q.numpy(), threads=8)
    got = np.zeros_like(exp)
    for b in range(p.batch):
        for h in range(p.h_kv):
            K, V, vis = pair.ref.dequant_unit(b, h)
            K32, V32 = K.astype(np.float32), V.astype(np.float32)
            for r in range(rep):
                s = (K32 @ q[b, h * rep + r].float().numpy()) * np.float32(1.0 / np.sqrt(p.head_dim))
                s = np.where(vis, s, -np.inf).astype(np.float32)
                w = np.exp(s - s.max()).astype(np.float32)
                got[b, h * rep + r] = (w[:, None] * V32).sum(0, dtype=np.float32) / w.sum(dtype=np.float32)
    return row_rel_err(got, exp)


def key_fold_max(pair, q):
    """max over units, heads, frozen groups and channels of |q_c| Δ_c from
    the oracle's bytes: above 65504 the unscaled fp16 fold would overflow."""
    p, L = pair.ref.p, pair.ref.layout
    arena = pair.ref.arena()
    rep = p.h_q // p.h_kv
    d = p.head_dim
    qn = np.abs(q.float().numpy())
    if qn.ndim == 4:   # [B][M][H_q][d]: the largest over the chunk's queries
        qn = qn.max(axis=1)
    best = 0.0
    for b in range(p.batch):
        for h in range(p.h_kv):
            unit = arena[(b * p.h_kv + h) * L["unit_bytes"]:(b * p.h_kv + h + 1) * L["unit_bytes"]]
            for s in range(min(pair.ref.n_groups, L["n_slots"])):
                blk = unit[L["groups"] + s * L["block_bytes"]:]
                delta = blk[L["blk_ks"]:L["blk_ks"] + 2 * d].view(np.float16).astype(np.float64)
                best = max(best, float((qn[b, h * rep:(h + 1) * rep] * delta[:d]).max()))
    return best


def value_delta_max(pair):
    """Largest per-token value Δ of the frozen groups (the fp16 P' = p Δ 2^-k
    overflows once p Δ passes 65504, with p up to 2^8 behind a lazy max)."""
    p, L = pair.ref.p, pair.ref.layout
    arena = pair.ref.arena()
    best = 0.0
    for u in range(p.batch * p.h_kv):
        unit = arena[u * L["unit_bytes"]:(u + 1) * L["unit_bytes"]]
        for s in range(min(pair.ref.n_groups, L["n_slots"])):
            blk = unit[L["groups"] + s * L["block_bytes"]:]
            vs = blk[L["blk_vs"]:L["blk_vs"] + 4 * p.group].view(np.float16).astype(np.float64)
            best = max(best, float(vs[0::2].max()))
    return best


CASES = [
    # 2 bits, MHA, head dim 128: both folds overflow readily
    dict(bits=2, group=32, residual=64, sinks=4, h_q=4, h_kv=4, head_dim=128, batch=2, max_tokens=800),
    # 8 bits, GQA rep 4, head dim 64
    dict(bits=8, group=32, residual=64, sinks=4, h_q=8, h_kv=2, head_dim=64, batch=2, max_tokens=800),
    # 4 bits, GQA rep 8, groups of two 32-token chunks
    dict(bits=4, group=64, residual=64, sinks=2, h_q=16, h_kv=2, head_dim=128, batch=2, max_tokens=800),
    # 2 bits, GQA rep 3 (a head pass of three rows), head dim 64, 16-token chunks
    dict(bits=2, group=16, residual=48, sinks=1, h_q=6, h_kv=2, head_dim=64, batch=2, max_tokens=800),
    # 3 bits (bit stream) at head dim 128, GQA rep 2
    dict(bits=3, group=32, residual=64, sinks=4, h_q=4, h_kv=2, head_dim=128, batch=2, max_tokens=800),
    # 4 bits with 1 % outlier tables
    dict(bits=4, group=32, residual=64, sinks=4, h_q=8, h_kv=2, head_dim=128, batch=2, max_tokens=800,
         outlier_permille=10),
    # 8 bits, sliding window over a wrapping slot ring
    dict(bits=8, group=32, residual=64, sinks=4, h_q=4, h_kv=1, head_dim=128, batch=2, max_tokens=0, window=200),
]


@pytest.mark.parametrize("shape", CASES)
def test_decode_over_fp16_range(shape):
    from kivi_quantized_kv_gb300 import KiviConfig
    cfg = KiviConfig(**shape)
    p = Pair(cfg)
    T = 700
    k, v = wide_stream(cfg, T + 40, seed=cfg.bits * 13 + cfg.head_dim)
    p.append(k[:, :, :T].contiguous(), v[:, :, :T].contiguous())
    assert p.bytes_equal()
    q = wide_q(cfg, seed=cfg.bits)
    # the regime the test is for: the unscaled folds would leave fp16 (the
    # key fold at 2 to 4 bits without outlier tables, where the key steps are
    # wide), and fp32 still resolves the scores
    if cfg.bits <= 4 and cfg.outlier_permille == 0:
        assert key_fold_max(p, q) > FP16_MAX
    assert value_delta_max(p) * 2 ** 8 > FP16_MAX
    assert fp32_floor(p, q) <= TOL / 8
    out = p.gpu.decode(q.cuda()).float().cpu().numpy()
    assert np.isfinite(out).all()
    err, left_out = conditioned_err(p, q, out, p.ref.decode_attn(q.numpy(), threads=8))
    assert err <= TOL and left_out <= 0.25, (err, left_out)
    # fused steps across a group freeze, a fresh query each step
    worst, left = 0.0, []
    for i in range(40):
        kt, vt = k[:, :, T + i:T + i + 1].contiguous(), v[:, :, T + i:T + i + 1].contiguous()
        qi = wide_q(cfg, seed=100 + i)
        out = p.gpu.append_decode(kt.cuda(), vt.cuda(), qi.cuda()).float().cpu().numpy()
        assert p.ref.append(kt.numpy(), vt.numpy()) == 0
        assert np.isfinite(out).all(), i
        err, left_out = conditioned_err(p, qi, out, p.ref.decode_attn(qi.numpy(), threads=8))
        assert err <= TOL, (i, err)
        worst, left = max(worst, err), left + [left_out]
    assert np.mean(left) <= 0.2, np.mean(left)
    assert p.bytes_equal()
    assert p.gpu.read_error() == 0


@pytest.mark.parametrize("shape", [CASES[0], CASES[2]])
def test_prefill_over_fp16_range(shape):
    """Chunked prefill (several query tokens per sequence) over the same
    streams: the multi-query instantiation shares the folds."""
    from kivi_quantized_kv_gb300 import KiviConfig
    cfg = KiviConfig(**shape)
    p = Pair(cfg)
    k, v = wide_stream(cfg, 600, seed=31)
    p.append(k[:, :, :536].contiguous(), v[:, :, :536].contiguous())
    M = 64
    p.append(k[:, :, 536:].contiguous(), v[:, :, 536:].contiguous())
    assert p.bytes_equal()
    q = wide_q(cfg, seed=5, rows=M)
    assert key_fold_max(p, q) > FP16_MAX
    out = p.gpu.prefill(q.cuda()).float().cpu().numpy()
    assert np.isfinite(out).all()
    exp = p.ref.prefill_attn(q.numpy(), threads=8)
    err, left_out = conditioned_err(p, q, out, exp, rows_q=M)
    assert err <= TOL and left_out <= 0.1, (err, left_out)
    assert p.gpu.read_error() == 0


@pytest.mark.parametrize("shape", [CASES[0], CASES[1], CASES[4]])
def test_decode_near_fp16_subnormals(shape):
    """Values scaled by 2^-8: the value steps p Δ_t 2^-k fall among the fp16
    subnormals (unless the kernel scales them up), while the outputs stay
    normal fp16 numbers, so their own rounding is within 2^-11 of the row."""
    from kivi_quantized_kv_gb300 import KiviConfig
    cfg = KiviConfig(**shape)
    p = Pair(cfg)
    k, v = wide_stream(cfg, 700, seed=77, tiny=True)
    p.append(k, v)
    assert p.bytes_equal()
    g = torch.Generator().manual_seed(3)
    q = torch.randn((cfg.batch, cfg.h_q, cfg.head_dim), generator=g).half()
    assert np.abs(p.ref.decode_attn(q.numpy())).max(axis=-1).min() > 2.0 ** -13   # normal fp16 outputs
    assert p.decode_err(q) <= TOL
