"""GPU parity of decode attention (the step before the router) against the
attention oracle, through the C ABI.

The GPU path and the oracle each keep their own fp16 KV caches, fed with the
same token stream; at every step the GPU's attention output (bf16, before
the residual) must lie within 2e-2 x RMS of the oracle's.  Cases cover the
sliding-window ring (wrapping several times), the linear cache of a full
layer with several K/V splits, grouped-query heads, the residual form, and
the full layer step (attention, then the router and experts on the device).
"""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
import synth
from parity import TOL_REL_RMS, bf16_to_f64, check_ids, check_output

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def moe():
    import expert_ffn_streaming_bit_b300 as m
    return m


def _check(y_gpu, y_ref, what):
    g = bf16_to_f64(y_gpu.reshape(-1))
    rms = float(np.sqrt(np.mean(y_ref ** 2)))
    err = float(np.abs(g - y_ref).max())
    # the output is bf16: allow its rounding on top of the tolerance
    tol = TOL_REL_RMS * rms + 2.0 ** -8 * float(np.abs(y_ref).max())
    assert err <= tol, (what, err, tol, rms)
    return err / rms


def _run(moe, shape, layers, T, check_every=1, index=0, residual=False):
    """T tokens through every layer independently (each layer sees the same
    token stream at positions 0..T-1); compared with the oracle."""
    a = moe.moe_attn_create(shape, layers)
    refs = [oracle.AttnState(shape, layers[l],
                             shape.window if shape.sliding[l] else shape.max_seq,
                             shape.window if shape.sliding[l] else 0, shape.theta(l))
            for l in range(len(layers))]
    xs = synth.make_tokens(shape, "tiny", T, index=index)
    xd = xs.cuda()
    worst = 0.0
    flags = moe.MOE_FWD_RESIDUAL if residual else 0
    for p in range(T):
        for l in range(len(layers)):
            y = torch.empty_like(xd[p:p + 1])
            moe.moe_attn_forward(a, l, xd[p:p + 1], p, y, flags=flags)
            yr = refs[l].step(xs[p], p)
            if p % check_every == 0 or p == T - 1:
                torch.cuda.synchronize()
                if residual:
                    x = bf16_to_f64(xs[p])
                    g = bf16_to_f64(y.cpu().reshape(-1)) - x
                    rms = float(np.sqrt(np.mean(yr ** 2)))
                    tol = TOL_REL_RMS * rms + 2.0 ** -8 * np.abs(x + yr)
                    assert np.all(np.abs(g - yr) <= tol), (p, l)
                else:
                    worst = max(worst, _check(y.cpu(), yr, (p, l)))
    return worst


def test_tiny_attention_ring_and_linear_caches(moe):
    """D 256, 4 query heads over 2 kv heads of 64: a sliding layer (window 8,
    its ring wraps five times in 40 tokens) and a full layer."""
    sh = synth.TINY_ATTN
    layers = [synth.make_attn_layer(sh, "tiny", l) for l in range(sh.n_layers)]
    _run(moe, sh, layers, 40)


def test_tiny_attention_with_residual(moe):
    sh = synth.TINY_ATTN
    layers = [synth.make_attn_layer(sh, "tiny", l) for l in range(sh.n_layers)]
    _run(moe, sh, layers, 12, residual=True, index=3)


def test_attention_several_splits(moe):
    """300 tokens: the full layer's last steps use 5 K/V splits, the sliding
    one (window 96) wraps its ring and uses 2."""
    sh = dataclasses.replace(synth.TINY_ATTN, window=96, max_seq=512)
    layers = [synth.make_attn_layer(sh, "tiny", l) for l in range(sh.n_layers)]
    _run(moe, sh, layers, 300, check_every=7, index=4)


def test_attention_positions_must_come_in_order(moe):
    sh = synth.TINY_ATTN
    layers = [synth.make_attn_layer(sh, "tiny", l) for l in range(sh.n_layers)]
    a = moe.moe_attn_create(sh, layers)
    x = synth.make_tokens(sh, "tiny", 1, index=5).cuda()
    y = torch.empty_like(x)
    moe.moe_attn_forward(a, 0, x, 0, y)
    with pytest.raises(moe.MoEError) as ei:
        moe.moe_attn_forward(a, 0, x, 5, y)
    assert ei.value.status == -6
    with pytest.raises(moe.MoEError) as ei:
        moe.moe_attn_forward(a, 1, x, sh.max_seq, y)      # beyond the linear cache
    assert ei.value.status in (-6, -1)
    moe.moe_attn_forward(a, 0, x, 1, y)                    # in order again
    moe.moe_attn_reset(a)
    moe.moe_attn_forward(a, 0, x, 0, y)


def test_gemma_shape_attention(moe):
    """The Gemma-shape reading: D 2816, 16 query heads over 8 kv heads of 256.
    A sliding layer with a 256-token window (it wraps) and a full layer, 400
    tokens, sampled steps checked (the oracle runs every step to build its
    own cache)."""
    sh = dataclasses.replace(synth.GEMMA_ATTN, n_layers=2, window=256, max_seq=1024,
                             sliding=(1, 0))
    layers = []
    for l in range(2):
        L = synth.make_attn_layer(sh, "decode", l, device="cuda")
        layers.append({k: v.to("cpu") for k, v in L.items()})
    oracle.set_threads(0)
    _run(moe, sh, layers, 400, check_every=25, index=6)


def test_decode_step_attention_then_router_and_experts(moe):
    """moe_decode_step: per layer, attention with the residual, then the MoE
    layer on that bf16 output (pre-norm, residual).  It equals running the
    two calls by hand, bit for bit; each stage is checked against its oracle
    on the GPU's own input to that stage (teacher forcing)."""
    ash = synth.TINY_ATTN
    msh = synth.MoEShape("tiny2", 256, 16, 128, 2, 256, 64, 2)
    alayers = [synth.make_attn_layer(ash, "tiny", l) for l in range(2)]
    mlayers = [synth.make_layer(msh, "tiny", l) for l in range(2)]
    a1 = moe.moe_attn_create(ash, alayers)
    a2 = moe.moe_attn_create(ash, alayers)
    h = moe.moe_create(msh, mlayers, max_tokens=1)
    refs = [oracle.AttnState(ash, alayers[l], ash.window if ash.sliding[l] else ash.max_seq,
                             ash.window if ash.sliding[l] else 0, ash.theta(l)) for l in range(2)]
    xs = synth.make_tokens(msh, "tiny", 10, index=7).cuda()
    flags = moe.MOE_FWD_RESIDUAL | moe.MOE_FWD_PRENORM
    for p in range(10):
        y = torch.empty_like(xs[p:p + 1])
        moe.moe_decode_step(a1, h, xs[p:p + 1], p, y, 2)
        cur = xs[p:p + 1]
        for l in range(2):
            xa = torch.empty_like(cur)
            moe.moe_attn_forward(a2, l, cur, p, xa, flags=moe.MOE_FWD_RESIDUAL)
            xm = torch.empty_like(cur)
            st = moe.moe_layer_forward(h, l, xa, xm, flags=flags, want_ids=True)
            torch.cuda.synchronize()
            # attention stage against the oracle, on this stage's GPU input
            yr = refs[l].step(cur.cpu(), p)
            xin = bf16_to_f64(cur.cpu().reshape(-1))
            g = bf16_to_f64(xa.cpu().reshape(-1)) - xin
            tol = TOL_REL_RMS * np.sqrt(np.mean(yr ** 2)) + 2.0 ** -8 * np.abs(xin + yr)
            assert np.all(np.abs(g - yr) <= tol), (p, l)
            # the router and experts on the attention output
            ref = oracle.moe_layer(oracle.LayerView(msh, mlayers[l]), xa.cpu(), prenorm=True)
            assert check_ids(st["ids"], ref, msh.top_k) == 0
            check_output(xm.cpu(), ref["y"], x_bf16=xa.cpu())
            cur = xm
        torch.cuda.synchronize()
        assert torch.equal(y, cur), p
