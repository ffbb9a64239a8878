"""GPU tests of streaming mode: routed experts live in a pinned host pool and
a per-layer set of HBM slots is filled on demand under the LFU policy, the
misses copied on a side stream while the shared expert runs.

Checked: every step's cache plan as the forward call made it (per id: hit,
slot, evicted expert) against the oracle's LFU replay, element by element,
the layer output against the oracle (forced and router-driven ids), and the
injected host->HBM copy failure path (error status, slot left empty, the next
step refetches).  Every call goes through the C ABI."""
import numpy as np
import pytest
import torch

import oracle
import synth
from parity import check_ids, check_output, check_weights

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def moe():
    import expert_ffn_streaming_bit_b300 as m
    return m


def _step(moe, h, x, layer=0, forced=None, flags=0):
    y = torch.empty_like(x)
    st = moe.moe_layer_forward(h, layer, x, y, flags=flags, forced_ids=forced, want_ids=True)
    torch.cuda.synchronize()
    return y, st


def _check_plan(st, hit, slot, ev, where):
    """The forward call's cache step, id by id, equals the oracle's."""
    assert np.array_equal(st["hit"], hit), (where, st["hit"], hit)
    assert np.array_equal(st["slot"], slot), (where, st["slot"], slot)
    assert np.array_equal(st["evicted"], ev), (where, st["evicted"], ev)
    assert st["misses"] == int((hit == 0).sum()), where


def test_tiny_streaming_trace_hits_and_outputs(moe):
    sh = synth.TINY
    L = synth.make_layer(sh, "tiny", 0)
    n_slots = 4
    h = moe.moe_create(sh, [L], n_slots=n_slots, max_tokens=1)
    trace = synth.streaming_trace(sh.n_experts, sh.top_k, 40, 1.1, 1, seed=11)
    lfu = oracle.LFUCache(n_slots, sh.n_experts)
    view = oracle.LayerView(sh, L)
    xs = synth.make_tokens(sh, "tiny", 40, index=11)
    for step in range(40):
        x = xs[step:step + 1]
        y, st = _step(moe, h, x.cuda(), forced=trace[step:step + 1])
        hit, slot, ev = lfu.step(trace[step])
        _check_plan(st, hit, slot, ev, step)
        assert st["hits"] == int(hit.sum()), step
        assert st["bytes_h2d"] == st["misses"] * moe.moe_get_info(h)["expert_blob_bytes"]
        ref = oracle.moe_layer(view, x, trace[step:step + 1])
        assert np.array_equal(st["ids"], trace[step:step + 1])
        check_weights(st["weights"], ref, st["ids"])
        check_output(y.cpu(), ref["y"])


def test_tiny_streaming_router_driven_matches_resident(moe):
    sh = synth.TINY
    L = synth.make_layer(sh, "tiny", 1)
    hs = moe.moe_create(sh, [L], n_slots=3, max_tokens=1)
    view = oracle.LayerView(sh, L)
    xs = synth.make_tokens(sh, "tiny", 12, index=12)
    lfu = oracle.LFUCache(3, sh.n_experts)
    for t in range(12):
        x = xs[t:t + 1]
        y, st = _step(moe, hs, x.cuda(), flags=moe.MOE_FWD_PRENORM | moe.MOE_FWD_RESIDUAL)
        ref = oracle.moe_layer(view, x, prenorm=True)
        assert check_ids(st["ids"], ref, sh.top_k) == 0
        _check_plan(st, *lfu.step(st["ids"][0]), t)
        check_weights(st["weights"], ref, st["ids"])
        check_output(y.cpu(), ref["y"], x_bf16=x)


def test_tiny_streaming_injected_copy_failure(moe):
    sh = synth.TINY
    L = synth.make_layer(sh, "tiny", 2)
    h = moe.moe_create(sh, [L], n_slots=2, max_tokens=1)
    x = synth.make_tokens(sh, "tiny", 1, index=13).cuda()
    forced = np.array([[3, 9]], np.int32)
    moe.moe_debug_inject(h, moe.MOE_INJECT_H2D_FAIL, 1)
    with pytest.raises(moe.MoEError) as ei:
        _step(moe, h, x, forced=forced)
    assert ei.value.status == -5
    torch.cuda.synchronize()
    # the failed expert's slot was left empty: the same step again misses it
    # once more (the other one is now resident) and the output is correct
    y, st = _step(moe, h, x, forced=forced)
    assert st["misses"] == 1 and st["hits"] == 1
    ref = oracle.moe_layer(oracle.LayerView(sh, L), x.cpu(), forced)
    check_output(y.cpu(), ref["y"])
    # slow copies change nothing
    moe.moe_debug_inject(h, moe.MOE_INJECT_SLOW_COPY, 20)
    y2, st2 = _step(moe, h, x, forced=np.array([[5, 9]], np.int32))
    ref2 = oracle.moe_layer(oracle.LayerView(sh, L), x.cpu(), np.array([[5, 9]], np.int32))
    check_output(y2.cpu(), ref2["y"])
    moe.moe_debug_inject(h, moe.MOE_INJECT_NONE, 0)


@pytest.fixture(scope="module")
def gemma_two_layers():
    sh = synth.GEMMA
    out = []
    for l in range(2):
        L = synth.make_layer(sh, "streaming_decode", l, device="cuda")
        out.append(synth.layer_to(L, "cpu"))
        del L
    torch.cuda.empty_cache()
    return out


def test_gemma_streaming_two_layers(moe, gemma_two_layers):
    """Full shape, 16 slots per layer, the Zipf trace with 50% overlap between
    steps; hit/miss counts exact against the oracle's LFU replay; sampled
    steps checked against the oracle."""
    sh = synth.GEMMA
    h = moe.moe_create(sh, gemma_two_layers, n_slots=16, max_tokens=1)
    steps = 24
    traces = [synth.streaming_trace(sh.n_experts, sh.top_k, steps, 1.1, 4, seed=synth.seed_of(3, l, 9))
              for l in range(2)]
    lfus = [oracle.LFUCache(16, sh.n_experts) for _ in range(2)]
    xs = synth.make_tokens(sh, "streaming_decode", steps, index=0)
    flags = moe.MOE_FWD_PRENORM | moe.MOE_FWD_RESIDUAL
    for step in range(steps):
        x = xs[step:step + 1]
        xl = x.cuda()
        for l in range(2):
            y, st = _step(moe, h, xl, layer=l, forced=traces[l][step:step + 1], flags=flags)
            hit, slot, ev = lfus[l].step(traces[l][step])
            _check_plan(st, hit, slot, ev, (step, l))
            if step % 8 == 7:
                ref = oracle.moe_layer(oracle.LayerView(sh, gemma_two_layers[l]), xl.cpu(),
                                       traces[l][step:step + 1], prenorm=True)
                check_weights(st["weights"], ref, st["ids"])
                check_output(y.cpu(), ref["y"], x_bf16=xl.cpu())
            xl = y
