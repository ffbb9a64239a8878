"""The expert store file (the storage tier under the slot cache), host side.

moe_store_write needs no GPU: it repacks every routed expert and writes it at
a page-aligned offset after a header that records the shape.  These tests
read the file back with an independent decoder of the documented qrow layout
(internal.h) and compare every code, scale and bias with the canonical
tensors, so a wrong offset, nibble order or row order fails here."""
import os
import struct

import numpy as np
import pytest

import synth

PAGE = 4096


@pytest.fixture(scope="module")
def moe():
    from expert_ffn_streaming_bit_b300 import build as b
    b.build()
    import expert_ffn_streaming_bit_b300 as m
    return m


def qrow_bytes(K):
    return (K * 9 // 16 + 15) // 16 * 16


def decode_qrow(buf, K):
    """One repacked row of K inputs -> (codes [K], scale bits [K/64], bias bits [K/64]).
    Word w of the codes holds columns 8w..8w+7: byte i has column 8w+i in its
    low nibble and column 8w+4+i in its high nibble."""
    codes = np.frombuffer(buf[:K // 2], np.uint8).reshape(-1, 4)
    out = np.empty((codes.shape[0], 8), np.uint8)
    out[:, 0:4] = codes & 0xF
    out[:, 4:8] = codes >> 4
    sb = np.frombuffer(buf[K // 2:K // 2 + K // 64 * 4], np.uint32)
    return out.reshape(-1), (sb & 0xFFFF).astype(np.uint16), (sb >> 16).astype(np.uint16)


def canonical_codes(q, K):
    """Canonical 4-bit rows [R][K/2] (column 2i in the low nibble) -> [R][K]."""
    q = np.asarray(q)
    out = np.empty(q.shape[:-1] + (K,), np.uint8)
    out[..., 0::2] = q & 0xF
    out[..., 1::2] = q >> 4
    return out


def read_header(path):
    with open(path, "rb") as f:
        raw = f.read(PAGE)
    magic = raw[:8]
    version, D, E, I, K, S, group, L = struct.unpack_from("<8i", raw, 8)
    blob, stride, data = struct.unpack_from("<3q", raw, 48)   # after two reserved words
    return dict(magic=magic, version=version, D=D, E=E, I=I, K=K, S=S, group=group, L=L,
                blob=blob, stride=stride, data=data)


def test_store_file_holds_every_expert_in_the_documented_layout(moe, tmp_path):
    sh = synth.MoEShape("tiny2", 256, 16, 128, 2, 256, 64, 2)
    layers = [synth.make_layer(sh, "tiny", l) for l in range(2)]
    path = str(tmp_path / "experts.moestore")
    moe.moe_store_write(sh, layers, path)
    h = read_header(path)
    D, I = sh.d_model, sh.d_expert
    rbD, rbI = qrow_bytes(D), qrow_bytes(I)
    blob = I * 2 * rbD + D * rbI
    assert h["magic"] == b"MOESTOR1" and h["version"] == 1
    assert (h["D"], h["E"], h["I"], h["K"], h["S"], h["group"], h["L"]) == (D, 16, I, 2, 256, 64, 2)
    assert h["blob"] == blob and h["stride"] % PAGE == 0 and h["stride"] >= blob
    assert h["data"] == PAGE
    assert os.path.getsize(path) == PAGE + 2 * 16 * h["stride"]
    data = open(path, "rb").read()
    for l, L in enumerate(layers):
        g_q, g_s, g_b = L["gate"].numpy()
        u_q, u_s, u_b = L["up"].numpy()
        d_q, d_s, d_b = L["down"].numpy()
        for e in range(sh.n_experts):
            off = h["data"] + (l * sh.n_experts + e) * h["stride"]
            b = data[off:off + h["stride"]]
            assert not any(b[blob:]), "padding after the blob must be zero"
            gate_codes, up_codes = canonical_codes(g_q[e], D), canonical_codes(u_q[e], D)
            for j in range(I):                      # gate row j, then up row j
                for r, (codes, s, bb) in enumerate(((gate_codes, g_s, g_b), (up_codes, u_s, u_b))):
                    c, sc, bi = decode_qrow(b[(2 * j + r) * rbD:(2 * j + r + 1) * rbD], D)
                    assert np.array_equal(c, codes[j]), (l, e, j, r)
                    assert np.array_equal(sc, s[e][j]) and np.array_equal(bi, bb[e][j])
            down_codes = canonical_codes(d_q[e], I)
            base = I * 2 * rbD
            for r in range(D):
                c, sc, bi = decode_qrow(b[base + r * rbI:base + (r + 1) * rbI], I)
                assert np.array_equal(c, down_codes[r]), (l, e, r)
                assert np.array_equal(sc, d_s[e][r]) and np.array_equal(bi, d_b[e][r])


def test_store_write_is_deterministic_and_local(moe, tmp_path):
    """Writing twice gives the same bytes; changing one expert's weights
    changes that expert's region only."""
    sh = synth.MoEShape("tiny1", 256, 16, 128, 2, 256, 64, 1)
    L = synth.make_layer(sh, "tiny", 0)
    a, b, c = (str(tmp_path / n) for n in ("a", "b", "c"))
    moe.moe_store_write(sh, [L], a)
    moe.moe_store_write(sh, [L], b)
    assert open(a, "rb").read() == open(b, "rb").read()
    L2 = dict(L)
    q = L["up"].q.clone()
    q[5] ^= 0x11                                    # expert 5 only
    L2["up"] = synth.QTensor(q, L["up"].scale, L["up"].bias, L["up"].bits)
    moe.moe_store_write(sh, [L2], c)
    h = read_header(a)
    da, dc = open(a, "rb").read(), open(c, "rb").read()
    for e in range(sh.n_experts):
        off = h["data"] + e * h["stride"]
        same = da[off:off + h["stride"]] == dc[off:off + h["stride"]]
        assert same == (e != 5), e


def test_store_write_rejects_bad_arguments(moe, tmp_path):
    sh = synth.TINY
    L = synth.make_layer(sh, "tiny", 0)
    with pytest.raises(moe.MoEError) as ei:
        moe.moe_store_write(sh, [L], "/nonexistent-dir/experts.moestore")
    assert ei.value.status == -8                   # MOE_ERR_IO
    bad = synth.MoEShape("bad", 300, 16, 128, 2, 256, 64, 1)
    with pytest.raises(moe.MoEError) as ei:
        moe.moe_store_write(bad, [L], str(tmp_path / "x"))
    assert ei.value.status == -1
