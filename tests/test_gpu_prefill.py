"""GPU parity of the multi-token (prefill) path against the oracle.

The path: router GEMM + top-k, token-to-expert bucketing, grouped GEMMs on the
tensor cores (gate/up with the GELU epilogue, then down), gather combine.
Every call goes through the C ABI.  Bucketing is compared bit-exactly with the
oracle's bucketing of the device's own ids; ids follow the near-tie rule of
parity.py; outputs the 2e-2 x RMS tolerance.
"""
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


def _forward(moe, h, x_cpu, flags=0, forced=None):
    x = x_cpu.cuda()
    y = torch.empty_like(x)
    st = moe.moe_layer_forward(h, 0, x, y, flags=flags, forced_ids=forced, want_ids=True)
    torch.cuda.synchronize()
    return y.cpu(), st


def _check_buckets(moe, h, ids, E):
    T = ids.shape[0]
    counts, offsets, perm = moe.moe_last_buckets(h, T)
    rc, ro, rp = oracle.bucket(ids, E)
    assert np.array_equal(counts, rc)
    assert np.array_equal(offsets, ro)
    assert np.array_equal(perm, rp)
    return counts


@pytest.mark.parametrize("T", [2, 5, 64, 333])
def test_tiny_prefill_matches_oracle(moe, T):
    sh = synth.TINY
    L = synth.make_layer(sh, "tiny", 0)
    h = moe.moe_create(sh, [L], max_tokens=T)
    x = synth.make_tokens(sh, "tiny", T, index=30 + T)
    y, st = _forward(moe, h, x)
    ref = oracle.moe_layer(oracle.LayerView(sh, L), x)
    assert check_ids(st["ids"], ref, sh.top_k) <= max(1, T // 200)
    check_weights(st["weights"], ref, st["ids"])
    _check_buckets(moe, h, st["ids"], sh.n_experts)
    check_output(y, ref["y"])


@pytest.mark.parametrize("T", [1024, 1025])
def test_tiny_prefill_bucketing_paths_at_the_boundary(moe, T):
    """T*k = 2048 assignments are bucketed by the one-launch path, 2050 by the
    three-launch one: both must give the oracle's buckets and outputs."""
    sh = synth.TINY
    L = synth.make_layer(sh, "tiny", 4)
    h = moe.moe_create(sh, [L], max_tokens=T)
    x = synth.make_tokens(sh, "tiny", T, index=90 + T)
    y, st = _forward(moe, h, x)
    ref = oracle.moe_layer(oracle.LayerView(sh, L), x)
    assert check_ids(st["ids"], ref, sh.top_k) <= max(1, T // 200)
    check_weights(st["weights"], ref, st["ids"])
    _check_buckets(moe, h, st["ids"], sh.n_experts)
    check_output(y, ref["y"])


@pytest.mark.parametrize("T", [31, 32, 33, 127, 128, 129, 193])
def test_tiny_prefill_gemm_plans_at_their_widths(moe, T):
    """The grouped GEMM runs a narrow plan for batches of at most 32 tokens, a
    medium one up to 128 and a wide one above.  Every token is sent to expert
    0 (and one other), so expert 0's unit is as wide as the batch: the widest
    unit each plan takes (32, 128), one past it (33, 129), and a batch that
    the wide plan cuts into two token tiles (193).  Output, weights and
    buckets are checked against the oracle."""
    sh = synth.TINY
    L = synth.make_layer(sh, "tiny", 5)
    h = moe.moe_create(sh, [L], max_tokens=T)
    x = synth.make_tokens(sh, "tiny", T, index=700 + T)
    forced = np.stack([np.zeros(T, np.int32), 1 + np.arange(T, dtype=np.int32) % (sh.n_experts - 1)],
                      axis=1)
    y, st = _forward(moe, h, x, forced=forced)
    ref = oracle.moe_layer(oracle.LayerView(sh, L), x, forced)
    assert np.array_equal(st["ids"], forced)
    check_weights(st["weights"], ref, st["ids"])
    counts = _check_buckets(moe, h, st["ids"], sh.n_experts)
    assert counts[0] == T
    check_output(y, ref["y"])


def test_tiny_prefill_rejects_bad_forced_ids(moe):
    """Out-of-range or repeated forced ids are refused on the host before any
    launch, and the handle stays usable."""
    sh = synth.TINY
    L = synth.make_layer(sh, "tiny", 2)
    T = 3
    h = moe.moe_create(sh, [L], max_tokens=T)
    x = synth.make_tokens(sh, "tiny", T, index=8)
    for bad in ([[0, 1], [2, 16], [4, 5]], [[0, 1], [-1, 3], [4, 5]], [[0, 1], [7, 7], [4, 5]]):
        with pytest.raises(moe.MoEError) as ei:
            _forward(moe, h, x, forced=np.array(bad, np.int32))
        assert ei.value.status == -1
    good = np.array([[0, 1], [2, 15], [4, 5]], np.int32)
    y, st = _forward(moe, h, x, forced=good)
    assert np.array_equal(st["ids"], good)
    check_output(y, oracle.moe_layer(oracle.LayerView(sh, L), x, good)["y"])


def test_tiny_prefill_multi_tile_experts_prenorm_residual(moe):
    """2600 tokens x top-2 over 16 experts: every expert gets more than 256
    rows, so each is split into several token tiles."""
    sh = synth.TINY
    L = synth.make_layer(sh, "tiny", 1)
    T = 2600
    h = moe.moe_create(sh, [L], max_tokens=T)
    x = synth.make_tokens(sh, "tiny", T, index=77)
    x[::7] = (x[::7].float() * 4096.0).to(torch.bfloat16)  # far outside the unit range
    y, st = _forward(moe, h, x, flags=moe.MOE_FWD_PRENORM | moe.MOE_FWD_RESIDUAL)
    ref = oracle.moe_layer(oracle.LayerView(sh, L), x, prenorm=True)
    assert check_ids(st["ids"], ref, sh.top_k) <= 3
    check_weights(st["weights"], ref, st["ids"])
    counts = _check_buckets(moe, h, st["ids"], sh.n_experts)
    assert counts.min() > 256
    check_output(y, ref["y"], x_bf16=x)


def test_tiny_prefill_forced_ids_and_edge_inputs(moe):
    sh = synth.TINY
    L = synth.make_layer(sh, "tiny", 2)
    T = 6
    h = moe.moe_create(sh, [L], max_tokens=T)
    x = synth.make_tokens(sh, "tiny", T, index=5)
    x[0] = 0
    forced = np.array([[0, 15], [3, 4], [15, 14], [7, 8], [1, 2], [9, 10]], np.int32)
    y, st = _forward(moe, h, x, forced=forced)
    ref = oracle.moe_layer(oracle.LayerView(sh, L), x, forced)
    assert np.array_equal(st["ids"], forced)
    check_weights(st["weights"], ref, st["ids"])
    _check_buckets(moe, h, st["ids"], sh.n_experts)
    assert torch.all(y[0] == 0)
    check_output(y, ref["y"])


def test_tiny_prefill_large_unnormalised_inputs(moe):
    """Without the pre-norm the gated intermediate grows like |x|^2; inputs
    around 3e4 must still match (per-token power-of-two range scaling)."""
    sh = synth.TINY
    L = synth.make_layer(sh, "tiny", 0)
    h = moe.moe_create(sh, [L], max_tokens=4)
    x = synth.make_tokens(sh, "tiny", 4, index=4)
    x[1] = (x[1].float() * 30000.0).to(torch.bfloat16)
    x[3] = (x[3].float() * 1e-4).to(torch.bfloat16)
    y, st = _forward(moe, h, x)
    ref = oracle.moe_layer(oracle.LayerView(sh, L), x)
    # the 1e-4-scaled token has logit gaps below the near-tie margin
    assert check_ids(st["ids"], ref, sh.top_k) <= 1
    for t in range(4):  # each token against its own scale
        check_output(y[t:t + 1], ref["y"][t:t + 1])


def test_tiny_prefill_prenorm_at_extreme_input_scales(moe):
    """With the pre-norm, token rows scaled by 2^-40 or 2^60 (whose per-token
    scalars leave the token prep's fp32 branch for its fp64 one) match the
    oracle like unit-scale rows; each token is held to its own output scale."""
    sh = synth.TINY
    L = synth.make_layer(sh, "tiny", 0)
    T = 6
    h = moe.moe_create(sh, [L], max_tokens=T)
    x = synth.make_tokens(sh, "tiny", T, index=12)
    for t, c in enumerate([1.0, 2.0 ** -40, 2.0 ** 60, 2.0 ** -20, 2.0 ** 30, 1.0]):
        x[t] = (x[t].float() * c).to(torch.bfloat16)
    y, st = _forward(moe, h, x, flags=moe.MOE_FWD_PRENORM)
    ref = oracle.moe_layer(oracle.LayerView(sh, L), x, prenorm=True)
    check_ids(st["ids"], ref, sh.top_k)
    assert np.array_equal(st["ids"], ref["ids"])
    check_weights(st["weights"], ref, st["ids"])
    for t in range(T):
        check_output(y[t:t + 1], ref["y"][t:t + 1])


def test_tiny_prefill_repeated_runs_are_bit_identical(moe):
    sh = synth.TINY
    L = synth.make_layer(sh, "tiny", 3)
    h = moe.moe_create(sh, [L], max_tokens=100)
    x = synth.make_tokens(sh, "tiny", 100, index=6)
    y1, s1 = _forward(moe, h, x)
    y2, s2 = _forward(moe, h, x)
    assert torch.equal(y1, y2) and np.array_equal(s1["ids"], s2["ids"])


def test_tiny_prefill_stack_matches_decode_stack(moe):
    """The multi-token stack (prefill path, layer by layer) against the decode
    stack run token by token: same ids except near-ties, outputs within the
    tolerance of each layer's contribution."""
    sh = synth.MoEShape("tiny4", 256, 16, 128, 2, 256, 64, 4)
    layers = [synth.make_layer(sh, "tiny", l) for l in range(4)]
    T = 24
    h = moe.moe_create(sh, layers, max_tokens=T)
    x = synth.make_tokens(sh, "tiny", T, index=8).cuda()
    yp = torch.empty_like(x)
    moe.moe_forward_stack(h, x, yp, 4)
    torch.cuda.synchronize()
    ids_p, _ = moe.moe_stack_ids(h, 4, T)
    yd = torch.empty_like(x)
    differ = 0
    for t in range(T):
        moe.moe_forward_stack(h, x[t:t + 1], yd[t:t + 1], 4)
        ids_t, _ = moe.moe_stack_ids(h, 4, 1)
        differ += int((ids_t[:, 0] != ids_p[:, t]).any(axis=-1).sum())
    torch.cuda.synchronize()
    # both paths rank fp32 logits summed in different orders: a near-tie may
    # flip one (layer, token), and a flip changes that token's later layers
    assert differ <= 1, differ
    d = (yp.float() - yd.float()).abs()
    scale = (yd.float() - x.float()).pow(2).mean().sqrt()
    assert float(d.max()) <= 4e-2 * float(scale) + 2.0 ** -7 * float(yd.float().abs().max())


def test_tiny_stack_small_batches_run_as_single_token_launches(moe):
    """moe_forward_stack runs fewer than 5 tokens as one single-token decode
    launch each: the batch's outputs, ids and weights are bit-identical to
    running each token alone.  From 5 tokens on the multi-token path runs
    (its buckets exist afterwards)."""
    sh = synth.MoEShape("tiny4", 256, 16, 128, 2, 256, 64, 4)
    layers = [synth.make_layer(sh, "tiny", l) for l in range(4)]
    h = moe.moe_create(sh, layers, max_tokens=5)
    x = synth.make_tokens(sh, "tiny", 5, index=9).cuda()
    yb = torch.empty_like(x[:4])
    moe.moe_forward_stack(h, x[:4], yb, 4)
    ids_b, w_b = moe.moe_stack_ids(h, 4, 4)
    with pytest.raises(moe.MoEError) as ei:
        moe.moe_last_buckets(h, 4)
    assert ei.value.status == -6
    for t in range(4):
        yt = torch.empty_like(x[:1])
        moe.moe_forward_stack(h, x[t:t + 1], yt, 4)
        ids_t, w_t = moe.moe_stack_ids(h, 4, 1)
        assert torch.equal(yt, yb[t:t + 1])
        assert np.array_equal(ids_t[:, 0], ids_b[:, t]) and np.array_equal(w_t[:, 0], w_b[:, t])
    y5 = torch.empty_like(x)
    moe.moe_forward_stack(h, x, y5, 4)
    counts, _, _ = moe.moe_last_buckets(h, 5)
    assert counts.sum() == 5 * sh.top_k


# ---------------------------------------------------------------- full shape

@pytest.fixture(scope="module")
def gemma_zipf_layer():
    sh = synth.GEMMA
    L = synth.make_layer(sh, "chunked_prefill", 0, device="cuda", logit_bias=True)
    out = synth.layer_to(L, "cpu")
    del L
    torch.cuda.empty_cache()
    return out


def _sample_check(moe, sh, L, x, y, st, sample, prenorm=False):
    ref = oracle.moe_layer(oracle.LayerView(sh, L), x[sample], prenorm=prenorm)
    assert check_ids(st["ids"][sample], ref, sh.top_k) <= max(1, len(sample) // 128)
    check_weights(st["weights"][sample], ref, st["ids"][sample])
    check_output(y[sample], ref["y"])


def test_gemma_chunked_prefill_128_zipf(moe, gemma_zipf_layer):
    """One 128-token chunk of the Zipf-biased chunked-prefill workload."""
    sh = synth.GEMMA
    T = 128
    h = moe.moe_create(sh, [gemma_zipf_layer], max_tokens=T)
    x = synth.make_tokens(sh, "chunked_prefill", T, index=0)
    y, st = _forward(moe, h, x)
    counts = _check_buckets(moe, h, st["ids"], sh.n_experts)
    assert counts.max() > 4 * counts.mean()      # uneven, Zipf-like popularity
    _sample_check(moe, sh, gemma_zipf_layer, x, y, st, np.arange(T))   # every token


@pytest.fixture(scope="module")
def gemma_layer():
    sh = synth.GEMMA
    L = synth.make_layer(sh, "prefill", 0, device="cuda")
    out = synth.layer_to(L, "cpu")
    del L
    torch.cuda.empty_cache()
    return out


def test_gemma_large_prefill_4096(moe, gemma_layer):
    """The 4096-token workload in the benchmark's launch configuration;
    bucketing checked in full, outputs on sampled tokens."""
    sh = synth.GEMMA
    T = 4096
    h = moe.moe_create(sh, [gemma_layer], max_tokens=T)
    x = synth.make_tokens(sh, "prefill", T, index=0)
    y, st = _forward(moe, h, x, flags=moe.MOE_FWD_PRENORM)
    counts = _check_buckets(moe, h, st["ids"], sh.n_experts)
    assert counts.sum() == T * sh.top_k
    sample = np.sort(np.random.default_rng(1).choice(T, 256, replace=False))
    _sample_check(moe, sh, gemma_layer, x, y, st, sample, prenorm=True)


def test_gemma_batched_decode_32_tokens(moe, gemma_layer):
    """A batch of 32 decode tokens through one full-size layer with the pre-norm
    and the residual, as the batched-decode benchmark runs them: every token
    checked against the oracle (about 2 rows per expert, so every MMA is the
    narrowest N)."""
    sh = synth.GEMMA
    T = 32
    h = moe.moe_create(sh, [gemma_layer], max_tokens=T)
    x = synth.make_tokens(sh, "decode", T, index=3)
    flags = moe.MOE_FWD_PRENORM | moe.MOE_FWD_RESIDUAL
    y, st = _forward(moe, h, x, flags=flags)
    _check_buckets(moe, h, st["ids"], sh.n_experts)
    ref = oracle.moe_layer(oracle.LayerView(sh, gemma_layer), x, prenorm=True)
    assert check_ids(st["ids"], ref, sh.top_k) <= 1
    check_weights(st["weights"], ref, st["ids"])
    check_output(y, ref["y"], x_bf16=x)


@pytest.fixture(scope="module")
def gemma_decode_layers4():
    sh = synth.GEMMA
    out = []
    for l in range(4):
        L = synth.make_layer(sh, "decode", l, device="cuda")
        out.append(synth.layer_to(L, "cpu"))
        del L
    torch.cuda.empty_cache()
    return out


def test_gemma_multi_token_stack_teacher_forced(moe, gemma_decode_layers4):
    """moe_forward_stack at T = 32 (the multi-token path the batched-decode
    benchmark times) over four full-size layers.  Prefix runs give each
    layer's bf16 input exactly; the oracle is teacher-forced on it, and every
    token's ids, weights and output are checked.  Each layer is also run on
    its captured input without the residual, so the output is held to
    2e-2 x RMS(y) itself rather than to the bf16 rounding of x + y."""
    sh = synth.GEMMA
    layers = gemma_decode_layers4
    T, L = 32, len(layers)
    h = moe.moe_create(sh, layers, max_tokens=T)
    x0 = synth.make_tokens(sh, "decode", T, index=200)
    xd = x0.cuda()
    xs = [x0]
    for n in range(1, L + 1):
        y = torch.empty_like(xd)
        moe.moe_forward_stack(h, xd, y, n)
        torch.cuda.synchronize()
        xs.append(y.cpu())
    ids, w = moe.moe_stack_ids(h, L, T)
    for l in range(L):
        ref = oracle.moe_layer(oracle.LayerView(sh, layers[l]), xs[l], prenorm=True)
        assert check_ids(ids[l], ref, sh.top_k) <= 1
        check_weights(w[l], ref, ids[l])
        check_output(xs[l + 1], ref["y"], x_bf16=xs[l])
        xl = xs[l].cuda()
        yl = torch.empty_like(xl)
        st = moe.moe_layer_forward(h, l, xl, yl, flags=moe.MOE_FWD_PRENORM, want_ids=True)
        assert np.array_equal(st["ids"], ids[l])
        check_output(yl.cpu(), ref["y"])


def test_prefill_gemm_wait_runs_out_and_the_handle_recovers(moe, gemma_layer):
    """Failure detection in the tensor-core GEMM without a fault: the injected
    gate/up launch's MMA issuer waits for an accumulator phase that never
    completes, its 50 ms device-side limit runs out and every role leaves
    through the abort flag.  The status check reports MOE_ERR_TIMEOUT; the
    next multi-token calls on the same handle match the oracle (a tiny layer,
    then the full-size 4096-token layer on sampled tokens)."""
    sh = synth.TINY
    L = synth.make_layer(sh, "tiny", 0)
    T = 333
    h = moe.moe_create(sh, [L], max_tokens=T)
    x = synth.make_tokens(sh, "tiny", T, index=55)
    moe.moe_debug_inject(h, moe.MOE_INJECT_GEMM_STALL, 50)
    with pytest.raises(moe.MoEError) as ei:
        _forward(moe, h, x)
    assert ei.value.status == -4
    y, st = _forward(moe, h, x)
    ref = oracle.moe_layer(oracle.LayerView(sh, L), x)
    assert check_ids(st["ids"], ref, sh.top_k) <= 1
    check_output(y, ref["y"])
    moe.moe_destroy(h)

    gs = synth.GEMMA
    T = 4096
    hg = moe.moe_create(gs, [gemma_layer], max_tokens=T)
    xg = synth.make_tokens(gs, "prefill", T, index=1)
    moe.moe_debug_inject(hg, moe.MOE_INJECT_GEMM_STALL, 50)
    with pytest.raises(moe.MoEError) as ei:
        _forward(moe, hg, xg, flags=moe.MOE_FWD_PRENORM)
    assert ei.value.status == -4
    y, st = _forward(moe, hg, xg, flags=moe.MOE_FWD_PRENORM)
    sample = np.sort(np.random.default_rng(2).choice(T, 32, replace=False))
    _sample_check(moe, gs, gemma_layer, xg, y, st, sample, prenorm=True)
