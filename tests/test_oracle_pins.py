"""Pins of the CPU oracle against facts that do not come from the oracle itself.

Each test names what fixes the expected value: a hand-built lattice, a closed
form, an invariant of the method, a brute-force enumeration, an independent
numpy restatement, or a hand-derived golden file under tests/golden/.
"""
import itertools
import math
import os

import numpy as np
import pytest
import torch

import oracle
import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def f16(x):
    return np.float16(x).view(np.uint16)


# ------------------------------------------------------------ quantiser

@pytest.mark.parametrize("bits", [4, 8])
def test_quantise_lattice_round_trip_is_exact(bits):
    """Groups built on the lattice w = b + s*q with exact fp16 s, b and codes that
    reach 0 and the top level: the quantiser must return s, b, q exactly and the
    dequantised values must equal w exactly."""
    levels = (1 << bits) - 1
    rng = np.random.default_rng(7)
    rows, group = 5, 64
    cols = 2 * group
    s_vals = [2.0 ** -6, 2.0 ** -7, 0.125, 2.0 ** -9, 0.25]
    b_vals = [-0.5, -0.25, 0.125, -1.0, 0.0]
    w = np.empty((rows, cols), np.float32)
    codes = np.empty((rows, cols), np.int64)
    for r in range(rows):
        for g in range(cols // group):
            q = rng.integers(0, levels + 1, group)
            q[rng.integers(group)] = 0
            q[(rng.integers(group - 1) + 1 + np.argmin(q)) % group] = levels
            q[np.argmin(q)] = 0
            codes[r, g * group:(g + 1) * group] = q
            w[r, g * group:(g + 1) * group] = b_vals[r] + s_vals[r] * q
    qb, s, b = oracle.quantise(w, bits, group)
    assert np.all(s == f16(np.array(s_vals)[:, None].repeat(2, 1)))
    assert np.all(b == f16(np.array(b_vals)[:, None].repeat(2, 1)))
    deq = oracle.dequant(qb, s, b, rows, cols, bits, group)
    assert np.array_equal(deq, w.astype(np.float64))
    if bits == 4:
        got = np.empty((rows, cols), np.int64)
        got[:, 0::2] = qb & 15
        got[:, 1::2] = qb >> 4
    else:
        got = qb.astype(np.int64)
    assert np.array_equal(got, codes)


def test_dequant_nibble_order_low_nibble_is_even_column():
    """Byte 0x21 holds column 0 = code 1 (low nibble) and column 1 = code 2."""
    q = np.zeros((1, 32), np.uint8)
    q[0, 0] = 0x21
    q[0, 31] = 0xF0
    s = f16(np.array([[0.5]]))
    b = f16(np.array([[-1.0]]))
    d = oracle.dequant(q, s, b, 1, 64, 4, 64)
    assert d[0, 0] == 0.5 * 1 - 1.0 and d[0, 1] == 0.5 * 2 - 1.0
    assert d[0, 62] == -1.0 and d[0, 63] == 0.5 * 15 - 1.0
    assert np.all(d[0, 2:62] == -1.0)


def test_quantise_constant_group_has_zero_scale():
    w = np.full((2, 64), 0.0371, np.float32)
    q, s, b = oracle.quantise(w, 4, 64)
    assert np.all(s == 0) and np.all(q == 0)
    assert np.all(b == f16(0.0371))
    d = oracle.dequant(q, s, b, 2, 64, 4, 64)
    assert np.all(d == float(np.float16(0.0371)))


@pytest.mark.parametrize("bits", [4, 8])
def test_quantise_error_bound_on_random_groups(bits):
    """|w - deq| <= scale/2 + levels*|scale - (mx-mn)/levels| + |bias - mn| + fp32 slack."""
    levels = (1 << bits) - 1
    rng = np.random.default_rng(3)
    w = (rng.standard_normal((64, 256)) * 0.02).astype(np.float32)
    q, s, b = oracle.quantise(w, bits, 64)
    d = oracle.dequant(q, s, b, 64, 256, bits, 64)
    wg = w.reshape(64, 4, 64).astype(np.float64)
    mn, mx = wg.min(-1), wg.max(-1)
    sf = s.view(np.float16).astype(np.float64)
    bf = b.view(np.float16).astype(np.float64)
    bound = sf / 2 + levels * np.abs(sf - (mx - mn) / levels) + np.abs(bf - mn) + 1e-6 * np.abs(wg).max()
    err = np.abs(d.reshape(64, 4, 64) - wg).max(-1)
    assert np.all(err <= bound)
    # the bound is not vacuous: the error is of the order of half a step
    assert err.mean() < sf.mean()


def test_synth_quantiser_matches_oracle_quantiser_byte_for_byte():
    """The input generator's quantiser (torch) and the oracle's (C) are separate
    code; on random draws they must agree on every byte."""
    for bits in (4, 8):
        w = synth.normal((96, 512), 0.02, 11 + bits)
        qs, ss, bs = synth.quantise_affine(w, bits, 64)
        qo, so, bo = oracle.quantise(w.numpy(), bits, 64)
        assert np.array_equal(qs.numpy(), qo)
        assert np.array_equal(ss.numpy().view(np.uint16), so)
        assert np.array_equal(bs.numpy().view(np.uint16), bo)


# ---------------------------------------------------------------- GELU

def test_gelu_tanh_identities_and_erf_bound():
    # gelu(0) = 0; the tanh form satisfies gelu(x) - gelu(-x) = x exactly in reals
    assert oracle.gelu_tanh(0.0) == 0.0
    for x in np.linspace(-6, 6, 97):
        assert abs(oracle.gelu_tanh(x) - oracle.gelu_tanh(-x) - x) < 1e-12
    # it approximates x*Phi(x) (the exact GELU) to within 1e-3 (Hendrycks & Gimpel);
    # dropping the cubic term would miss this bound by more than 20x at x = 1.5
    for x in np.linspace(-5, 5, 201):
        exact = 0.5 * x * (1 + math.erf(x / math.sqrt(2)))
        assert abs(oracle.gelu_tanh(x) - exact) < 1e-3
    assert abs(oracle.gelu_tanh(10.0) - 10.0) < 1e-12
    assert abs(oracle.gelu_tanh(-10.0)) < 1e-12


# --------------------------------------------------------------- router

def test_topk_equals_brute_force_max_sum_subset():
    rng = np.random.default_rng(5)
    for trial in range(50):
        l = rng.standard_normal(16).astype(np.float32)
        ids = oracle.topk(l, 2)
        best = max(itertools.combinations(range(16), 2), key=lambda c: float(l[list(c)].sum()))
        assert set(ids.tolist()) == set(best)
        assert l[ids[0]] >= l[ids[1]]


def test_topk_ties_go_to_lower_index():
    l = np.array([0.5, 1.0, 1.0, 0.2, 1.0, 1.0], np.float32)
    assert oracle.topk(l, 2).tolist() == [1, 2]
    assert oracle.topk(l, 4).tolist() == [1, 2, 4, 5]
    assert oracle.topk(l, 5).tolist() == [1, 2, 4, 5, 0]


def test_routing_weights_closed_form_and_normalisation():
    rng = np.random.default_rng(9)
    for _ in range(20):
        l = (rng.standard_normal(16) * 3).astype(np.float32)
        ids = oracle.topk(l, 2)
        w = oracle.routing_weights(l, ids)
        d = float(l[ids[1]]) - float(l[ids[0]])
        assert abs(w[0] - 1.0 / (1.0 + math.exp(d))) < 1e-15
        ids8 = oracle.topk(l, 8)
        w8 = oracle.routing_weights(l, ids8)
        assert abs(w8.sum() - 1.0) < 1e-12 and np.all(w8 > 0)
        assert np.all(np.diff(w8) <= 0)


def _numpy_dequant(t, bits, group):
    """Independent numpy restatement of the canonical format (not the oracle's code)."""
    q, s, b = (np.asarray(a) for a in t.numpy())
    if bits == 4:
        codes = np.empty(q.shape[:-1] + (q.shape[-1] * 2,), np.float64)
        codes[..., 0::2] = q & 15
        codes[..., 1::2] = q >> 4
    else:
        codes = q.astype(np.float64)
    sf = np.repeat(s.view(np.float16).astype(np.float64), group, axis=-1)
    bf = np.repeat(b.view(np.float16).astype(np.float64), group, axis=-1)
    return codes * sf + bf


def _bf16_to_f64(x):
    return x.float().numpy().astype(np.float64)


def test_router_logits_match_numpy_restatement():
    sh = synth.TINY
    L = synth.make_layer(sh, "tiny", 0)
    view = oracle.LayerView(sh, L)
    x = synth.make_tokens(sh, "tiny", 3)
    out = oracle.moe_layer(view, x)
    Wr = _numpy_dequant(L["router"], 8, 64)
    ref = (_bf16_to_f64(x) @ Wr.T).astype(np.float32)
    assert np.allclose(out["logits"], ref, rtol=0, atol=1e-6)


def test_router_exact_ties_from_duplicate_rows_pick_lower_index():
    sh = synth.TINY
    L = synth.make_layer(sh, "tiny", 0)
    x = synth.make_tokens(sh, "tiny", 1)
    view = oracle.LayerView(sh, L)
    base = oracle.moe_layer(view, x)
    top = int(base["ids"][0, 0])
    # copy the winning router row into a higher-index row and a lower-index row
    r = L["router"]
    for other in (top + 3) % sh.n_experts, (top + sh.n_experts - 5) % sh.n_experts:
        q, s, b = r.q.clone(), r.scale.clone(), r.bias.clone()
        q[other], s[other], b[other] = q[top], s[top], b[top]
        L2 = dict(L, router=synth.QTensor(q, s, b, 8))
        out = oracle.moe_layer(oracle.LayerView(sh, L2), x)
        assert out["logits"][0, top] == out["logits"][0, other]
        assert out["ids"][0].tolist() == sorted([top, other])
        assert out["w"][0, 0] == out["w"][0, 1] == 0.5


# ---------------------------------------------------------------- layer

def _dense_ffn_numpy(L, e, x, sh):
    g = _numpy_dequant(synth.QTensor(L["gate"].q[e], L["gate"].scale[e], L["gate"].bias[e], 4), 4, 64)
    u = _numpy_dequant(synth.QTensor(L["up"].q[e], L["up"].scale[e], L["up"].bias[e], 4), 4, 64)
    d = _numpy_dequant(synth.QTensor(L["down"].q[e], L["down"].scale[e], L["down"].bias[e], 4), 4, 64)
    a = g @ x
    c = math.sqrt(2 / math.pi)
    h = 0.5 * a * (1 + np.tanh(c * (a + 0.044715 * a ** 3))) * (u @ x)
    return d @ h


def _zero_shared(L, sh):
    z = dict(L)
    for name, rows, cols in (("shared_gate", sh.d_shared, sh.d_model),
                             ("shared_up", sh.d_shared, sh.d_model),
                             ("shared_down", sh.d_model, sh.d_shared)):
        z[name] = synth.qtensor(torch.zeros(rows, cols), 4, sh.group)
    return z


def test_single_expert_layer_is_a_dense_ffn():
    """E = 1, k = 1: the routing weight is exactly 1 and, with the shared branch
    zeroed, the layer equals a dense FFN computed by an independent numpy path."""
    sh = synth.MoEShape("one", d_model=128, n_experts=1, d_expert=192, top_k=1, d_shared=64)
    L = _zero_shared(synth.make_layer(sh, "tiny", 5), sh)
    x = synth.make_tokens(sh, "tiny", 2, index=5)
    out = oracle.moe_layer(oracle.LayerView(sh, L), x)
    assert np.all(out["ids"] == 0) and np.all(out["w"] == 1.0)
    for t in range(2):
        ref = _dense_ffn_numpy(L, 0, _bf16_to_f64(x[t]), sh)
        assert np.allclose(out["y"][t], ref, rtol=1e-12, atol=1e-12)


def test_shared_branch_is_added_unweighted():
    sh = synth.MoEShape("one", d_model=128, n_experts=1, d_expert=64, top_k=1, d_shared=128)
    L = synth.make_layer(sh, "tiny", 6)
    x = synth.make_tokens(sh, "tiny", 1, index=6)
    full = oracle.moe_layer(oracle.LayerView(sh, L), x)["y"][0]
    routed = oracle.moe_layer(oracle.LayerView(sh, _zero_shared(L, sh)), x)["y"][0]
    shared = oracle.ffn(L["shared_gate"].numpy(), L["shared_up"].numpy(), L["shared_down"].numpy(),
                        sh.d_model, sh.d_shared, sh.group, _bf16_to_f64(x[0]))
    assert np.allclose(full, routed + shared, rtol=1e-12, atol=1e-12)


def test_identical_experts_make_routing_irrelevant():
    """If every expert has the same weights, the weights sum to 1 and
    y = FFN(x) + shared(x) whatever the router picks."""
    sh = synth.TINY
    L = synth.make_layer(sh, "tiny", 2)
    for name in ("gate", "up", "down"):
        t = L[name]
        L[name] = synth.QTensor(t.q[:1].expand_as(t.q).contiguous(),
                                t.scale[:1].expand_as(t.scale).contiguous(),
                                t.bias[:1].expand_as(t.bias).contiguous(), 4)
    x = synth.make_tokens(sh, "tiny", 4, index=2)
    out = oracle.moe_layer(oracle.LayerView(sh, L), x)
    z = oracle.moe_layer(oracle.LayerView(sh, _zero_shared(L, sh)), x)
    for t in range(4):
        ref = _dense_ffn_numpy(L, 0, _bf16_to_f64(x[t]), sh)
        assert np.allclose(z["y"][t], ref, rtol=1e-10, atol=1e-12)
        assert len(set(out["ids"][t].tolist())) == sh.top_k


def test_expert_relabelling_permutes_ids_and_keeps_output():
    """Relabelling experts (router rows and expert weights together) maps the
    chosen ids through the relabelling and leaves y bit-identical."""
    sh = synth.TINY
    L = synth.make_layer(sh, "tiny", 3)
    x = synth.make_tokens(sh, "tiny", 4, index=3)
    base = oracle.moe_layer(oracle.LayerView(sh, L), x)
    perm = np.random.default_rng(1).permutation(sh.n_experts)   # new index -> old index
    inv = np.argsort(perm)
    P = dict(L)
    for name in ("router", "gate", "up", "down"):
        t = L[name]
        idx = torch.from_numpy(perm)
        P[name] = synth.QTensor(t.q[idx].contiguous(), t.scale[idx].contiguous(),
                                t.bias[idx].contiguous(), t.bits)
    out = oracle.moe_layer(oracle.LayerView(sh, P), x)
    assert np.array_equal(out["ids"], inv[base["ids"]])
    assert np.array_equal(out["y"], base["y"])
    assert np.array_equal(out["w"], base["w"])


def _numpy_rms(x, eps=1e-6):
    return x / math.sqrt(float(np.mean(x * x)) + eps)


@pytest.mark.parametrize("prenorm", [False, True])
def test_general_layer_is_the_weighted_sum_of_its_experts_plus_shared(prenorm):
    """k = 2 of 16 distinct experts with the shared branch on: for every token,
    y equals sum_i w_i FFN_{id_i}(u) + FFN_shared(u), each FFN computed by the
    independent numpy path from the canonical bytes (u = x, or its RMS
    normalisation).  A dropped term, a weight paired with the wrong expert or
    a shared branch scaled by a routing weight all fail here."""
    sh = synth.TINY
    L = synth.make_layer(sh, "tiny", 7)
    T = 5
    x = synth.make_tokens(sh, "tiny", T, index=17)
    out = oracle.moe_layer(oracle.LayerView(sh, L), x, prenorm=prenorm)
    sg = _numpy_dequant(L["shared_gate"], 4, 64)
    su = _numpy_dequant(L["shared_up"], 4, 64)
    sd = _numpy_dequant(L["shared_down"], 4, 64)
    c = math.sqrt(2 / math.pi)
    for t in range(T):
        u = _bf16_to_f64(x[t])
        if prenorm:
            u = _numpy_rms(u)
        ids = out["ids"][t]
        assert len(set(ids.tolist())) == sh.top_k
        a = sg @ u
        ref = sd @ (0.5 * a * (1 + np.tanh(c * (a + 0.044715 * a ** 3))) * (su @ u))
        for i in range(sh.top_k):
            ref = ref + out["w"][t, i] * _dense_ffn_numpy(L, int(ids[i]), u, sh)
        assert np.allclose(out["y"][t], ref, rtol=1e-10, atol=1e-12)


def test_forced_ids_use_router_softmax_over_the_forced_set():
    sh = synth.TINY
    L = synth.make_layer(sh, "tiny", 4)
    x = synth.make_tokens(sh, "tiny", 2, index=4)
    forced = np.array([[3, 11], [0, 15]], np.int32)
    out = oracle.moe_layer(oracle.LayerView(sh, L), x, forced)
    assert np.array_equal(out["ids"], forced)
    for t in range(2):
        l = out["logits"][t]
        d = float(l[forced[t, 1]]) - float(l[forced[t, 0]])
        assert abs(out["w"][t, 0] - 1 / (1 + math.exp(d))) < 1e-15


def test_prenorm_is_invariant_to_input_scale():
    """The RMS pre-normalisation makes the layer depend on the direction of x
    only: scaling x by a power of two (exact in bf16) changes nothing but the
    eps term, and the expert choice is unchanged."""
    sh = synth.TINY
    L = synth.make_layer(sh, "tiny", 7)
    x = synth.make_tokens(sh, "tiny", 4, index=7)
    view = oracle.LayerView(sh, L)
    base = oracle.moe_layer(view, x, prenorm=True)
    for c in (8.0, 0.125, 64.0):
        out = oracle.moe_layer(view, (x.float() * c).to(torch.bfloat16), prenorm=True)
        assert np.array_equal(out["ids"], base["ids"])
        # eps / c^2 moves the normalised input by at most ~3e-5 relative here
        assert np.abs(out["y"] - base["y"]).max() <= 1e-3 * np.abs(base["y"]).max()
    raw = oracle.moe_layer(view, (x.float() * 64.0).to(torch.bfloat16))
    assert np.abs(raw["y"] - base["y"]).max() > 10 * np.abs(base["y"]).max()


def test_prenorm_leaves_a_unit_rms_input_nearly_unchanged():
    """x with entries +-1 has mean square exactly 1, so the normalised input is
    x / sqrt(1 + 1e-6): the layer output moves by about 5e-7 relative."""
    sh = synth.TINY
    L = synth.make_layer(sh, "tiny", 8)
    rng = np.random.default_rng(8)
    x = torch.from_numpy(rng.choice([-1.0, 1.0], size=(3, sh.d_model)).astype(np.float32))
    x = x.to(torch.bfloat16)
    view = oracle.LayerView(sh, L)
    a = oracle.moe_layer(view, x, prenorm=True)
    b = oracle.moe_layer(view, x)
    assert np.array_equal(a["ids"], b["ids"])
    rel = np.abs(a["y"] - b["y"]).max() / np.abs(b["y"]).max()
    assert 1e-8 < rel < 5e-6, rel


def test_prenorm_of_a_zero_input_is_zero():
    sh = synth.TINY
    L = synth.make_layer(sh, "tiny", 9)
    x = torch.zeros(1, sh.d_model, dtype=torch.bfloat16)
    out = oracle.moe_layer(oracle.LayerView(sh, L), x, prenorm=True)
    assert out["ids"][0].tolist() == list(range(sh.top_k))
    assert np.all(out["y"] == 0.0)


# ------------------------------------------------------------ bucketing

def _read_golden(name):
    rows = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            key, *vals = line.split()
            rows[key] = [int(v) for v in vals]
    return rows


def test_bucket_golden_hand_example():
    g = _read_golden("bucket_3x2.txt")
    ids = np.array(g["ids"], np.int32).reshape(g["T"][0], g["k"][0])
    counts, offsets, perm = oracle.bucket(ids, g["E"][0])
    assert counts.tolist() == g["counts"]
    assert offsets.tolist() == g["offsets"]
    assert perm.tolist() == g["perm"]


def test_bucket_invariants_random():
    rng = np.random.default_rng(2)
    T, k, E = 128, 8, 128
    ids = np.stack([rng.choice(E, k, replace=False) for _ in range(T)]).astype(np.int32)
    counts, offsets, perm = oracle.bucket(ids, E)
    assert counts.sum() == T * k
    assert offsets[0] == 0 and np.array_equal(np.diff(offsets), counts)
    assert np.array_equal(np.sort(perm), np.arange(T * k))
    flat = ids.ravel()
    for e in range(E):
        seg = perm[offsets[e]:offsets[e + 1]]
        assert np.all(flat[seg] == e) and np.all(np.diff(seg) > 0)


# ------------------------------------------------------------ LFU cache

def test_lfu_golden_hand_trace():
    c = oracle.LFUCache(3, 10)
    with open(os.path.join(GOLDEN, "lfu_trace_3slots.txt")) as f:
        lines = [l for l in f if l.strip() and not l.startswith("#")]
    assert len(lines) == 8
    for line in lines:
        step, ids, hits, slots, ev = [p.split() for p in line.split("|")]
        hit, slot, evicted = c.step(np.array([int(v) for v in ids]))
        assert hit.tolist() == [int(v) for v in hits], line
        assert slot.tolist() == [int(v) for v in slots], line
        assert evicted.tolist() == [int(v) for v in ev], line


def test_lfu_invariants_on_zipf_trace():
    trace = synth.streaming_trace(128, 8, 200, 1.1, 4, seed=5)
    c = oracle.LFUCache(16, 128)
    for ids in trace:
        hit, slot, ev = c.step(ids)
        assert len(set(slot.tolist())) == 8
        assert np.array_equal(c.expert[slot], ids)          # every id resident after the step
        res = c.expert[c.expert >= 0]
        assert len(set(res.tolist())) == res.size           # resident ids distinct
        for i in range(8):
            if hit[i]:
                assert ev[i] == -1


def test_lfu_misses_equal_distinct_count_when_everything_fits():
    rng = np.random.default_rng(4)
    pool = rng.choice(128, 16, replace=False)
    c = oracle.LFUCache(16, 128)
    seen, misses = set(), 0
    for _ in range(100):
        ids = rng.choice(pool, 8, replace=False)
        hit, slot, ev = c.step(ids)
        misses += int((hit == 0).sum())
        seen |= set(ids.tolist())
        assert np.all(ev == -1)
    assert misses == len(seen)


def test_lfu_rejects_repeated_ids():
    c = oracle.LFUCache(4, 8)
    with pytest.raises(ValueError):
        c.step(np.array([1, 1]))
