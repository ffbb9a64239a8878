"""Seeded synthetic inputs for the MoE layer step.

This module is shared by the tests, the benchmark and the oracle's callers.  It
draws the random numbers (weights, activations, routing traces) and prepares
them in the canonical storage format that the layer step consumes.  It holds
none of the layer step's arithmetic (no router, no top-k, no dequantise, no
FFN, no combine, no cache policy).

Canonical storage of a weight matrix W with ``rows`` outputs and ``cols``
inputs (TurboFieldfare pages, overview table "权重": MLX affine 4-bit with
group 64, 8-bit router):

* ``q``: uint8.  4-bit: ``[rows, cols // 2]``, column ``2i`` in the low
  nibble of byte ``i`` and column ``2i + 1`` in the high nibble.  8-bit:
  ``[rows, cols]``.
* ``scale``, ``bias``: fp16 bit patterns (uint16) ``[rows, cols // group]``;
  groups run along the input dimension.  Element value = scale * q + bias.

Preparing that format from fp32 draws is the pages' install-time repack step
(outside the layer step).  The reading used here: per group, ``mn``/``mx`` in
fp32, ``scale = fp16_rn((mx - mn) / levels)``, ``bias = fp16_rn(mn)``, and
``q = clamp(rint_even((w - f32(bias)) / f32(scale)), 0, levels)`` in fp32, with
``q = 0`` where the fp16 scale is 0.  The oracle carries its own, independent
quantiser for the round-trip checks; a test checks that the two agree
byte for byte.

Draws use torch generators seeded from ``numpy.random.SeedSequence`` with a
spawn key per (workload, layer, tensor), so each tensor is reproducible on its
own.  The stream of numbers depends on the device: the same seed gives one
set of weights on ``cpu`` and another on ``cuda``.  Small cases are drawn on
the CPU; the full 30-layer shapes (22.8 G weights) are drawn on the GPU.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Dict, Optional, Sequence

import numpy as np
import torch

ROOT_SEED = 20261202
WEIGHT_STD = 0.02


@dataclasses.dataclass(frozen=True)
class MoEShape:
    """Dimensions of one MoE layer stack (names follow the pages' model)."""

    name: str
    d_model: int      # D, hidden size
    n_experts: int    # E, routed experts per layer
    d_expert: int     # I, routed expert inner size
    top_k: int        # k, experts chosen per token
    d_shared: int     # S, shared (always-on) expert inner size
    group: int = 64   # quantisation group along the input dimension
    n_layers: int = 1

    def expert_bytes(self) -> int:
        """Canonical bytes of one routed expert (gate + up + down, 4-bit)."""
        return 3 * qbytes(self.d_expert, self.d_model, 4, self.group)

    def shared_bytes(self) -> int:
        return 3 * qbytes(self.d_shared, self.d_model, 4, self.group)

    def router_bytes(self) -> int:
        return qbytes(self.n_experts, self.d_model, 8, self.group)

    def decode_layer_bytes(self) -> int:
        """Weight bytes one token reads in one layer: k experts, shared, router."""
        return self.top_k * self.expert_bytes() + self.shared_bytes() + self.router_bytes()


def qbytes(rows: int, cols: int, bits: int, group: int) -> int:
    """Bytes of a canonical affine-quantised [rows, cols] matrix."""
    return rows * cols * bits // 8 + rows * (cols // group) * 4


# Tiny case (one layer) that the oracle finishes instantly.
TINY = MoEShape("tiny", d_model=256, n_experts=16, d_expert=128, top_k=2, d_shared=256,
                group=64, n_layers=1)
# Gemma 4 26B-A4B MoE block shape: 128 experts, top-8, 30 layers.
GEMMA = MoEShape("gemma4-26b-a4b-moe", d_model=2816, n_experts=128, d_expert=704, top_k=8,
                 d_shared=2112, group=64, n_layers=30)

WORKLOADS = {
    "tiny": dict(shape=TINY, tokens=4, routing="router"),
    "decode": dict(shape=GEMMA, tokens=1, routing="router"),
    "chunked_prefill": dict(shape=GEMMA, tokens=1024, chunk=128, routing="zipf_bias"),
    "streaming_decode": dict(shape=GEMMA, tokens=1, steps=256, n_slots=16, routing="trace"),
    "prefill": dict(shape=GEMMA, tokens=4096, routing="router"),
}
WORKLOAD_IDS = {name: i for i, name in enumerate(WORKLOADS)}
TENSOR_IDS = {name: i for i, name in enumerate(
    ["router", "shared_gate", "shared_up", "shared_down", "gate", "up", "down",
     "x", "logit_bias", "trace"])}


def seed_of(*key: int) -> int:
    """63-bit seed for a spawn key (workload id, layer, tensor id, ...)."""
    ss = np.random.SeedSequence(ROOT_SEED, spawn_key=tuple(int(k) for k in key))
    return int(ss.generate_state(1, dtype=np.uint64)[0] & np.uint64((1 << 63) - 1))


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def normal(shape: Sequence[int], std: float, seed: int, device="cpu") -> torch.Tensor:
    """fp32 N(0, std^2) draws."""
    x = torch.randn(tuple(shape), generator=_gen(seed, device), device=device,
                    dtype=torch.float32)
    return x.mul_(std)


def quantise_affine(w: torch.Tensor, bits: int, group: int):
    """fp32 [..., rows, cols] -> canonical (q, scale, bias); see the module docstring."""
    assert w.dtype == torch.float32 and w.shape[-1] % group == 0
    levels = (1 << bits) - 1
    lead = w.shape[:-1]
    cols = w.shape[-1]
    wg = w.reshape(*lead, cols // group, group)
    mn = wg.amin(dim=-1)
    mx = wg.amax(dim=-1)
    s16 = ((mx - mn) / float(levels)).to(torch.float16)
    b16 = mn.to(torch.float16)
    s32 = s16.to(torch.float32).unsqueeze(-1)
    b32 = b16.to(torch.float32).unsqueeze(-1)
    zero = s32 == 0
    t = (wg - b32) / torch.where(zero, torch.ones_like(s32), s32)
    q = torch.where(zero, torch.zeros_like(t), torch.round(t)).clamp_(0, levels)
    q = q.to(torch.uint8).reshape(*lead, cols)
    if bits == 4:
        q = q[..., 0::2] | (q[..., 1::2] << 4)
    elif bits != 8:
        raise ValueError("bits must be 4 or 8")
    return (q.contiguous(), s16.view(torch.int16).contiguous(),
            b16.view(torch.int16).contiguous())


@dataclasses.dataclass
class QTensor:
    """Canonical affine-quantised matrix (torch tensors; scale/bias as int16 bits)."""

    q: torch.Tensor
    scale: torch.Tensor
    bias: torch.Tensor
    bits: int

    def to(self, device) -> "QTensor":
        return QTensor(self.q.to(device), self.scale.to(device), self.bias.to(device), self.bits)

    def numpy(self):
        return (self.q.cpu().numpy(), self.scale.cpu().numpy().view(np.uint16),
                self.bias.cpu().numpy().view(np.uint16))


def qtensor(w: torch.Tensor, bits: int, group: int) -> QTensor:
    q, s, b = quantise_affine(w, bits, group)
    return QTensor(q, s, b, bits)


def make_layer(shape: MoEShape, workload: str, layer: int, device="cpu",
               std: float = WEIGHT_STD, logit_bias: bool = False) -> Dict[str, object]:
    """All weights of one layer in canonical form.

    Keys: router (8-bit [E, D]); shared_gate/shared_up ([S, D]); shared_down
    ([D, S]); gate/up (stacked [E, I, D]); down ([E, D, I]); logit_bias
    (fp32 [E] or None).
    """
    D, E, I, S, g = shape.d_model, shape.n_experts, shape.d_expert, shape.d_shared, shape.group
    wid = WORKLOAD_IDS[workload]

    def draw(tag, rows, cols, bits, lead=()):
        w = normal((*lead, rows, cols), std, seed_of(wid, layer, TENSOR_IDS[tag]), device)
        out = qtensor(w, bits, g)
        del w
        return out

    out = {
        "router": draw("router", E, D, 8),
        "shared_gate": draw("shared_gate", S, D, 4),
        "shared_up": draw("shared_up", S, D, 4),
        "shared_down": draw("shared_down", D, S, 4),
        "gate": draw("gate", I, D, 4, (E,)),
        "up": draw("up", I, D, 4, (E,)),
        "down": draw("down", D, I, 4, (E,)),
        "logit_bias": None,
    }
    if logit_bias:
        out["logit_bias"] = zipf_logit_bias(E, 1.1, seed_of(wid, layer, TENSOR_IDS["logit_bias"]))
    return out


def make_tokens(shape: MoEShape, workload: str, T: int, index: int = 0, device="cpu",
                std: float = 1.0) -> torch.Tensor:
    """bf16 [T, D] activations: N(0, std^2) fp32 rounded to bf16 (nearest even)."""
    x = normal((T, shape.d_model), std, seed_of(WORKLOAD_IDS[workload], index, TENSOR_IDS["x"]),
               device)
    return x.to(torch.bfloat16)


def zipf_probs(n: int, s: float) -> np.ndarray:
    p = np.arange(1, n + 1, dtype=np.float64) ** (-s)
    return p / p.sum()


def zipf_logit_bias(E: int, s: float, seed: int) -> torch.Tensor:
    """Per-expert fp32 logit bias -s*ln(rank), ranks from a seeded permutation.

    Used to make router-driven expert popularity follow Zipf(s): the expert of
    rank r gets its softmax mass multiplied by r^-s.
    """
    rng = np.random.Generator(np.random.PCG64(seed))
    rank = rng.permutation(E) + 1
    return torch.tensor(-s * np.log(rank.astype(np.float64)), dtype=torch.float32)


def streaming_trace(E: int, k: int, steps: int, s: float, keep: int, seed: int) -> np.ndarray:
    """Forced top-k choices for streaming decode of one layer: int32 [steps, k].

    Step 0 draws k distinct experts from Zipf(s) (ranks mapped to expert ids by
    a seeded permutation), one at a time without replacement.  Each later step
    keeps ``keep`` ids chosen at random from the previous step and draws
    ``k - keep`` new ones from Zipf(s) excluding the kept ones.
    """
    rng = np.random.Generator(np.random.PCG64(seed))
    perm = rng.permutation(E)           # rank r (0-based) -> expert id
    p_rank = zipf_probs(E, s)
    p_exp = np.empty(E)
    p_exp[perm] = p_rank

    def draw(n, exclude):
        chosen = []
        avail = np.ones(E, dtype=bool)
        avail[list(exclude)] = False
        for _ in range(n):
            p = np.where(avail, p_exp, 0.0)
            e = int(rng.choice(E, p=p / p.sum()))
            chosen.append(e)
            avail[e] = False
        return chosen

    out = np.empty((steps, k), dtype=np.int32)
    prev = draw(k, [])
    out[0] = prev
    for t in range(1, steps):
        kept = [int(v) for v in rng.choice(np.array(prev), size=keep, replace=False)]
        new = draw(k - keep, kept)
        prev = kept + new
        out[t] = prev
    return out


def layer_to(layer: Dict[str, object], device) -> Dict[str, object]:
    out = {}
    for key, val in layer.items():
        if isinstance(val, QTensor):
            out[key] = val.to(device)
        elif isinstance(val, torch.Tensor):
            out[key] = val.to(device)
        else:
            out[key] = val
    return out


# ------------------------------------------------------- decode attention

@dataclasses.dataclass(frozen=True)
class AttnShape:
    """Dimensions of the attention blocks in front of the MoE layers.

    The pages give no head shapes; this is the reading used (stated with the
    other readings of the pages): the MoE block's hidden size, grouped-query
    heads, sliding-window layers with a ring cache and full-attention layers
    with a linear cache."""

    name: str
    d_model: int      # D
    n_heads: int      # Hq, query heads
    n_kv_heads: int   # Hkv, key/value heads (Hq % Hkv == 0)
    head_dim: int     # d
    group: int        # quantisation group along the input dimension
    n_layers: int
    window: int       # sliding-window length (the ring cache's capacity)
    max_seq: int      # capacity of a full-attention layer's linear cache
    sliding: tuple    # per layer: 1 sliding window, 0 full attention

    def theta(self, layer: int) -> float:
        return ROPE_THETA_SLIDING if self.sliding[layer] else ROPE_THETA_FULL

    def attn_weight_bytes(self) -> int:
        """Canonical bytes of one layer's 4-bit q, k, v and output projections."""
        qd, kd = self.n_heads * self.head_dim, self.n_kv_heads * self.head_dim
        return (qbytes(qd, self.d_model, 4, self.group) + 2 * qbytes(kd, self.d_model, 4, self.group)
                + qbytes(self.d_model, qd, 4, self.group))


ROPE_THETA_SLIDING = 10000.0
ROPE_THETA_FULL = 1000000.0

TINY_ATTN = AttnShape("tiny-attn", d_model=256, n_heads=4, n_kv_heads=2, head_dim=64, group=64,
                      n_layers=2, window=8, max_seq=64, sliding=(1, 0))
# Gemma 4 26B-A4B reading: 16 query heads and 8 key/value heads of 256, a
# 1024-token window; 25 sliding layers and 5 full-attention layers (every
# sixth layer full).
GEMMA_ATTN = AttnShape("gemma4-26b-a4b-attn", d_model=2816, n_heads=16, n_kv_heads=8,
                       head_dim=256, group=64, n_layers=30, window=1024, max_seq=8192,
                       sliding=tuple(0 if l % 6 == 5 else 1 for l in range(30)))

ATTN_TENSOR_IDS = {name: 16 + i for i, name in enumerate(["wq", "wk", "wv", "wo"])}


def make_attn_layer(shape: AttnShape, workload: str, layer: int, device="cpu",
                    std: float = WEIGHT_STD) -> Dict[str, object]:
    """Canonical 4-bit weights of one attention block: wq [Hq d, D],
    wk / wv [Hkv d, D], wo [D, Hq d] (N(0, std^2) fp32 draws, affine g64)."""
    D, qd, kd = shape.d_model, shape.n_heads * shape.head_dim, shape.n_kv_heads * shape.head_dim
    wid = WORKLOAD_IDS[workload]

    def draw(tag, rows, cols):
        w = normal((rows, cols), std, seed_of(wid, layer, ATTN_TENSOR_IDS[tag]), device)
        out = qtensor(w, 4, shape.group)
        del w
        return out

    return {"wq": draw("wq", qd, D), "wk": draw("wk", kd, D), "wv": draw("wv", kd, D),
            "wo": draw("wo", D, qd)}
