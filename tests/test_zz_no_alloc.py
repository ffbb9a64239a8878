"""moe_forward_stack_noalloc against moe_forward_stack, through the C ABI.

The no-allocation entry point serves callers that may not allocate device
memory while they run (allocator hooks, real-time loops, hosts whose
allocator belongs to another framework).  Its scratch is one fixed device
array inside the library, so two calls in a row reuse the same memory; both
must agree with the ordinary entry point, which uses the handle's own
scratch.  This file is collected last on purpose.
"""
import numpy as np
import pytest
import torch

import synth
from parity import TOL_REL_RMS, bf16_to_f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def moe():
    import expert_ffn_streaming_bit_b300 as m
    return m


def _assert_same(y, y_ref, x0):
    """Both entry points run the same deterministic kernel on the same inputs,
    so the outputs must be bit-identical.  The tolerance of the parity tests
    (2e-2 of the RMS of the stack's contribution plus the bf16 rounding of
    the output) is checked first, so a failure says how far apart they are."""
    g, r, x = bf16_to_f64(y), bf16_to_f64(y_ref), bf16_to_f64(x0)
    rms = float(np.sqrt(np.mean((r - x) ** 2)))
    tol = TOL_REL_RMS * rms + 2.0 ** -8 * np.abs(r)
    assert np.all(np.abs(g - r) <= tol), float(np.abs(g - r).max())
    assert torch.equal(y, y_ref), "within tolerance but not bit-identical"


def _compare(moe, shape, layers, index):
    h = moe.moe_create(shape, layers, max_tokens=1)
    L = len(layers)
    x0 = synth.make_tokens(shape, "tiny", 1, index=index).cuda()
    y_ref = torch.empty_like(x0)
    moe.moe_forward_stack(h, x0, y_ref, L)
    torch.cuda.synchronize()
    outs = []
    for _ in range(2):                      # two calls in a row share the array
        y = torch.full_like(x0, float("nan"))
        assert moe.moe_forward_stack_noalloc(h, x0, y, L, want_status=True) == 0
        torch.cuda.synchronize()
        outs.append(y.cpu())
    for y in outs:
        _assert_same(y, y_ref.cpu(), x0.cpu())
    # a shorter stack on the same handle after the longer one
    y_ref1 = torch.empty_like(x0)
    moe.moe_forward_stack(h, x0, y_ref1, 1)
    y1 = torch.empty_like(x0)
    moe.moe_forward_stack_noalloc(h, x0, y1, 1)
    torch.cuda.synchronize()
    _assert_same(y1.cpu(), y_ref1.cpu(), x0.cpu())
    moe.moe_destroy(h)


def test_noalloc_stack_matches_stack_tiny(moe):
    sh = synth.MoEShape("tiny4", 256, 16, 128, 2, 256, 64, 4)
    layers = [synth.make_layer(sh, "tiny", l) for l in range(4)]
    _compare(moe, sh, layers, index=21)


def test_noalloc_stack_matches_stack_full_shape(moe):
    sh = synth.MoEShape("gemma2", 2816, 128, 704, 8, 2112, 64, 2)
    layers = []
    for l in range(2):
        L = synth.make_layer(sh, "decode", l, device="cuda")
        layers.append(synth.layer_to(L, "cpu"))
        del L
    torch.cuda.empty_cache()
    _compare(moe, sh, layers, index=22)


def test_noalloc_rejects_bad_arguments(moe):
    sh = synth.TINY
    h = moe.moe_create(sh, [synth.make_layer(sh, "tiny", 0)], max_tokens=1)
    x = synth.make_tokens(sh, "tiny", 1, index=23).cuda()
    with pytest.raises(moe.MoEError):
        moe.moe_forward_stack_noalloc(h, x, x, 1)            # y aliases x
    with pytest.raises(moe.MoEError):
        moe.moe_forward_stack_noalloc(h, x, torch.empty_like(x), 2)   # only 1 layer
    moe.moe_destroy(h)


def test_noalloc_reports_a_device_wait_that_ran_out(moe):
    """A device-side failure inside the no-allocation call reaches the caller
    through the status word it asks for, without any allocation: the injected
    launch's first grid barrier waits for arrivals that never come, its 50 ms
    device-side limit runs out and the status reads 1.  The next call on the
    same handle clears the array, reports 0 and matches moe_forward_stack."""
    sh = synth.MoEShape("tiny4", 256, 16, 128, 2, 256, 64, 4)
    layers = [synth.make_layer(sh, "tiny", l) for l in range(4)]
    h = moe.moe_create(sh, layers, max_tokens=1)
    x0 = synth.make_tokens(sh, "tiny", 1, index=24).cuda()
    y_ref = torch.empty_like(x0)
    moe.moe_forward_stack(h, x0, y_ref, 4)
    torch.cuda.synchronize()
    moe.moe_debug_inject(h, moe.MOE_INJECT_DEVICE_STALL, 50)
    y = torch.empty_like(x0)
    assert moe.moe_forward_stack_noalloc(h, x0, y, 4, want_status=True) == 1
    torch.cuda.synchronize()
    y = torch.full_like(x0, float("nan"))
    assert moe.moe_forward_stack_noalloc(h, x0, y, 4, want_status=True) == 0
    torch.cuda.synchronize()
    _assert_same(y.cpu(), y_ref.cpu(), x0.cpu())
    moe.moe_destroy(h)
