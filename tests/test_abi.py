"""C-ABI checks that need no GPU: the library loads, exports every function
include/moe.h declares, validates configurations before touching CUDA, and its
host-side LFU planner agrees with the oracle's."""
import ctypes
import os
import re
import subprocess

import numpy as np
import pytest

import oracle
import synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def moe():
    from expert_ffn_streaming_bit_b300 import build as b
    b.build()
    import expert_ffn_streaming_bit_b300 as m
    return m


def _declared_functions():
    text = open(os.path.join(ROOT, "include", "moe.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"\b(moe_[a-z_0-9]+)\s*\(", text)
    return sorted(set(names))


def _exported(path):
    out = subprocess.run(["nm", "-D", "--defined-only", path], capture_output=True, text=True,
                         check=True).stdout
    return {l.split()[-1] for l in out.splitlines() if " T " in l}


def test_every_declared_function_is_exported(moe):
    declared = _declared_functions()
    for n in ("moe_create", "moe_layer_forward", "moe_cache_step", "moe_destroy"):
        assert n in declared
    exported = _exported(moe.LIB_PATH)
    missing = [n for n in declared if n not in exported]
    assert not missing, missing
    lib = ctypes.CDLL(moe.LIB_PATH)
    for n in declared:
        assert getattr(lib, n)


def test_only_the_abi_is_exported(moe):
    exported = _exported(moe.LIB_PATH)
    assert all(n.startswith("moe_") for n in exported), sorted(exported)[:10]


def test_status_strings(moe):
    for s in (0, -1, -2, -3, -4, -5, -6, -7):
        assert moe.moe_status_string(s)


@pytest.mark.parametrize("field,value", [("group", 32), ("d_model", 300), ("top_k", 0),
                                         ("top_k", 33), ("n_experts", 100), ("n_slots", 1),
                                         ("max_tokens", 0), ("d_expert", 96)])
def test_create_rejects_bad_configs_without_a_gpu(moe, field, value):
    sh = synth.TINY
    cfg = moe.moe_config(sh.d_model, sh.n_experts, sh.d_expert, sh.top_k, sh.d_shared, sh.group,
                         1, 0, 1)
    setattr(cfg, field, value)
    w = (moe.moe_layer_weights * 1)()
    out = ctypes.c_void_p()
    st = moe._lib.moe_create(ctypes.byref(cfg), w, ctypes.byref(out))
    assert st == -1 and out.value is None
    assert moe.moe_last_error()


def test_create_rejects_missing_weights(moe):
    sh = synth.TINY
    cfg = moe.moe_config(sh.d_model, sh.n_experts, sh.d_expert, sh.top_k, sh.d_shared, sh.group,
                         1, 0, 1)
    w = (moe.moe_layer_weights * 1)()
    out = ctypes.c_void_p()
    assert moe._lib.moe_create(ctypes.byref(cfg), w, ctypes.byref(out)) == -1
    assert "missing" in moe.moe_last_error()


def test_null_handles_are_rejected(moe):
    assert moe._lib.moe_layer_forward(None, 0, None, 1, None, 0, None, None, None) == -1
    assert moe._lib.moe_forward_stack(None, None, 1, None, 1, None) == -1
    assert moe._lib.moe_cache_step(None, 0, None, 1, 0, None) == -1
    moe._lib.moe_destroy(None)


def test_host_planner_matches_oracle_lfu_on_zipf_traces(moe):
    for seed in range(3):
        trace = synth.streaming_trace(128, 8, 300, 1.1, 4, seed=100 + seed)
        a = moe.SlotPlan(16, 128)
        b = oracle.LFUCache(16, 128)
        for ids in trace:
            ha, sa, ea = a.step(ids)
            hb, sb, eb = b.step(ids)
            assert np.array_equal(ha, hb) and np.array_equal(sa, sb) and np.array_equal(ea, eb)


def test_host_planner_golden_trace(moe):
    p = moe.SlotPlan(3, 10)
    path = os.path.join(ROOT, "tests", "golden", "lfu_trace_3slots.txt")
    for line in open(path):
        if line.startswith("#") or not line.strip():
            continue
        _, ids, hits, slots, ev = [x.split() for x in line.split("|")]
        h, s, e = p.step([int(v) for v in ids])
        assert h.tolist() == [int(v) for v in hits]
        assert s.tolist() == [int(v) for v in slots]
        assert e.tolist() == [int(v) for v in ev]


def test_host_planner_rejects_bad_ids_and_keeps_state(moe):
    p = moe.SlotPlan(4, 8)
    p.step([1, 2])
    with pytest.raises(moe.MoEError):
        p.step([3, 3])
    with pytest.raises(moe.MoEError):
        p.step([9])
    with pytest.raises(moe.MoEError):
        p.step([0, 3, 4, 5, 6])
    h, s, e = p.step([1, 2])
    assert h.tolist() == [1, 1]


def test_fault_injection_switches_are_host_side(moe):
    moe.moe_debug_inject(None, moe.MOE_INJECT_PINNED_ALLOC_FAIL)
    moe.moe_debug_inject(None, moe.MOE_INJECT_NONE)
    with pytest.raises(moe.MoEError):
        moe.moe_debug_inject(None, moe.MOE_INJECT_H2D_FAIL, 1)   # needs a handle
    with pytest.raises(moe.MoEError):
        moe.moe_debug_inject(None, moe.MOE_INJECT_DEVICE_STALL, 50)   # needs a handle


def test_binding_constants_match_the_header(moe):
    """Every integer #define and status code of include/moe.h has the same
    value in the Python binding."""
    text = open(os.path.join(ROOT, "include", "moe.h")).read()
    defines = dict((n, int(v)) for n, v in re.findall(r"#define\s+(MOE_[A-Z_0-9]+)\s+(-?\d+)\b", text))
    statuses = dict((n, int(v)) for n, v in re.findall(r"\b(MOE_(?:OK|ERR_[A-Z_]+))\s*=\s*(-?\d+)", text))
    assert "MOE_INJECT_DEVICE_STALL" in defines and "MOE_ERR_DEVICE" in statuses
    for name, value in defines.items():
        assert getattr(moe, name) == value, name
    for name, value in statuses.items():
        assert moe.STATUS[value] == name
