"""GPU tests of streaming mode: routed experts live in a pinned host pool and
a per-layer set of HBM slots is filled on demand under the LFU policy, the
misses copied on a side stream while the shared expert runs.

Checked: every step's cache plan as the forward call made it (per id: hit,
slot, evicted expert) against the oracle's LFU replay, element by element,
the layer output against the oracle (forced and router-driven ids), and the
injected host->HBM copy failure path (error status, slot left empty, the next
step refetches).  Every call goes through the C ABI."""
import os

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


# ------------------------------------------------------- the expert store tier

def test_tiny_streaming_from_the_expert_store(moe, tmp_path):
    """Routed experts read from the expert store file on each miss (bounded
    parallel pread into pinned staging buffers, then the slot copy): every
    step's cache plan equals the oracle's LFU replay, and every output is
    bit-identical to the pinned-pool handle's and within the oracle's
    tolerance."""
    sh = synth.TINY
    L = synth.make_layer(sh, "tiny", 0)
    path = str(tmp_path / "tiny.moestore")
    moe.moe_store_write(sh, [L], path)
    hf = moe.moe_create(sh, [L], n_slots=4, max_tokens=1, expert_store=path, io_threads=4)
    hp = moe.moe_create(sh, [L], n_slots=4, max_tokens=1)
    info = moe.moe_get_info(hf)
    assert info["io_threads"] == 4 and info["pinned_pool_bytes"] == 0
    trace = synth.streaming_trace(sh.n_experts, sh.top_k, 40, 1.1, 1, seed=11)
    lfu = oracle.LFUCache(4, sh.n_experts)
    view = oracle.LayerView(sh, L)
    xs = synth.make_tokens(sh, "tiny", 40, index=11)
    for step in range(40):
        x = xs[step:step + 1].cuda()
        yf, sf = _step(moe, hf, x, forced=trace[step:step + 1])
        yp, sp = _step(moe, hp, x, forced=trace[step:step + 1])
        _check_plan(sf, *lfu.step(trace[step]), step)
        assert torch.equal(yf, yp), step
        check_output(yf.cpu(), oracle.moe_layer(view, x.cpu(), trace[step:step + 1])["y"])
    # router-driven steps read their misses while the shared expert runs
    for t in range(8):
        x = xs[t:t + 1].cuda()
        yf, sf = _step(moe, hf, x, flags=moe.MOE_FWD_PRENORM)
        ref = oracle.moe_layer(view, x.cpu(), prenorm=True)
        assert check_ids(sf["ids"], ref, sh.top_k) == 0
        check_output(yf.cpu(), ref["y"])


def test_tiny_store_read_failure_leaves_the_slot_empty(moe, tmp_path):
    """Host-side fault injection: the first read of the next miss batch fails.
    The call returns MOE_ERR_IO and leaves that expert's slot empty, so the
    same step again misses it once more, reads it and is correct."""
    sh = synth.TINY
    L = synth.make_layer(sh, "tiny", 2)
    path = str(tmp_path / "t2.moestore")
    moe.moe_store_write(sh, [L], path)
    h = moe.moe_create(sh, [L], n_slots=2, max_tokens=1, expert_store=path, io_threads=2)
    x = synth.make_tokens(sh, "tiny", 1, index=13).cuda()
    forced = np.array([[3, 9]], np.int32)
    moe.moe_debug_inject(h, moe.MOE_INJECT_READ_FAIL, 1)
    with pytest.raises(moe.MoEError) as ei:
        _step(moe, h, x, forced=forced)
    assert ei.value.status == -8
    torch.cuda.synchronize()
    y, st = _step(moe, h, x, forced=forced)
    assert st["misses"] == 1 and st["hits"] == 1
    check_output(y.cpu(), oracle.moe_layer(oracle.LayerView(sh, L), x.cpu(), forced)["y"])


def test_store_of_another_shape_is_refused(moe, tmp_path):
    sh = synth.TINY
    L = synth.make_layer(sh, "tiny", 0)
    path = str(tmp_path / "one_layer.moestore")
    moe.moe_store_write(sh, [L], path)
    with pytest.raises(moe.MoEError) as ei:
        moe.moe_create(sh, [L, L], n_slots=4, max_tokens=1, expert_store=path, io_threads=2)
    assert ei.value.status == -1


def test_gemma_streaming_two_layers_from_the_expert_store(moe, gemma_two_layers, tmp_path):
    """Full shape: 16 slots per layer, misses read from the expert store file;
    plans against the oracle's LFU replay every step, outputs bit-identical to
    the pinned-pool handle every step."""
    sh = synth.GEMMA
    path = str(tmp_path / "gemma2.moestore")
    moe.moe_store_write(sh, gemma_two_layers, path)
    hf = moe.moe_create(sh, gemma_two_layers, n_slots=16, max_tokens=1, expert_store=path,
                        io_threads=8)
    hp = moe.moe_create(sh, gemma_two_layers, n_slots=16, max_tokens=1)
    steps = 24
    traces = [synth.streaming_trace(sh.n_experts, sh.top_k, steps, 1.1, 4, seed=synth.seed_of(3, l, 9))
              for l in range(2)]
    lfus = [oracle.LFUCache(16, sh.n_experts) for _ in range(2)]
    xs = synth.make_tokens(sh, "streaming_decode", steps, index=0)
    flags = moe.MOE_FWD_PRENORM | moe.MOE_FWD_RESIDUAL
    for step in range(steps):
        xf = xp = xs[step:step + 1].cuda()
        for l in range(2):
            yf, sf = _step(moe, hf, xf, layer=l, forced=traces[l][step:step + 1], flags=flags)
            yp, _ = _step(moe, hp, xp, layer=l, forced=traces[l][step:step + 1], flags=flags)
            _check_plan(sf, *lfus[l].step(traces[l][step]), (step, l))
            assert torch.equal(yf, yp), (step, l)
            xf, xp = yf, yp
    os.unlink(path)
