"""Pins for the oracle's KV-append + RoPE functions (no GPU).

Each test ties the oracle to something other than itself: hand-worked values from
the append page, closed forms (complex multiplication, identity at position 0),
invariants (pair norms, NeoX/interleaved permutation) and the page's layout rules.
"""
import math

import numpy as np
import pytest

from oracle import pagedkv_oracle as orc
from paged_kv_cache_231_gb300 import workloads as wl


def test_past_length_table(golden):
    g = golden("past_length.json")
    for c in g["cases"]:
        got = orc.past_sequence_length(c["total0"], c["key_total"], c["seq_len"])
        assert got == c["expected"], c


def test_rotary_geometry_tables(golden):
    g = golden("rotary_geometry.json")
    R = g["rotary_dim"]
    for layout, inter in (("neox", False), ("interleaved", True)):
        slot, partner, first = orc.rotary_geometry(R, inter)
        assert slot.tolist() == g[layout]["slot"]
        assert partner.tolist() == g[layout]["partner"]
        assert first.tolist() == g[layout]["first"]


@pytest.mark.parametrize("interleaved", [False, True])
def test_rotary_geometry_is_an_involution(interleaved):
    # partner(partner(d)) == d, exactly one member of each pair leads, both use one column
    for R in (2, 4, 8, 64, 128):
        slot, partner, first = orc.rotary_geometry(R, interleaved)
        assert (partner[partner] == np.arange(R)).all()
        assert (first != first[partner]).all()
        assert (slot == slot[partner]).all()
        assert sorted(set(slot.tolist())) == list(range(R // 2))


def test_rotary_worked_example(golden):
    g = golden("rotary_worked.json")
    cos = np.zeros((2, 2))
    sin = np.zeros((2, 2))
    cos[g["position"]] = g["cos_row"]
    sin[g["position"]] = g["sin_row"]
    x = np.array(g["x"])
    neox = orc.rotate_row(x, g["position"], cos, sin, 4, False)
    inter = orc.rotate_row(x, g["position"], cos, sin, 4, True)
    assert neox.tolist() == g["neox_expected"]
    assert inter.tolist() == g["interleaved_expected"]


@pytest.mark.parametrize("interleaved", [False, True])
def test_rotary_dim2_is_complex_multiplication(interleaved):
    # With one pair, the rotation is (x0 + i x1) * (cos + i sin): a library routine.
    rng = np.random.default_rng(0)
    x = rng.standard_normal((50, 6))
    ang = rng.uniform(-3, 3, size=50)
    cos = np.cos(ang)[:, None]
    sin = np.sin(ang)[:, None]
    got = orc.rotate_rows(x, np.arange(50), cos, sin, 2, interleaved)
    z = (x[:, 0] + 1j * x[:, 1]) * np.exp(1j * ang)
    np.testing.assert_allclose(got[:, 0], z.real, rtol=0, atol=1e-12)
    np.testing.assert_allclose(got[:, 1], z.imag, rtol=0, atol=1e-12)
    np.testing.assert_array_equal(got[:, 2:], x[:, 2:])


def test_neox_is_interleaved_under_pair_permutation():
    # NeoX pairs (i, i + half) and interleaved pairs (2i, 2i + 1) use the same column i,
    # so NeoX(x) = P^-1 Interleaved(P x) with P moving i -> 2i and i + half -> 2i + 1.
    rng = np.random.default_rng(1)
    R, D = 16, 20
    half = R // 2
    x = rng.standard_normal((30, D))
    cos, sin = wl.rope_tables(64, R)
    pos = rng.integers(0, 64, size=30)
    perm = np.arange(D)
    perm[:R] = np.array([i // 2 if i % 2 == 0 else half + i // 2 for i in range(R)])
    # perm[k] = NeoX index that goes to interleaved slot k
    inter = orc.rotate_rows(x[:, perm], pos, cos, sin, R, True)
    neox = orc.rotate_rows(x, pos, cos, sin, R, False)
    back = np.empty_like(inter)
    back[:, perm] = inter
    np.testing.assert_allclose(back, neox, rtol=0, atol=1e-12)


@pytest.mark.parametrize("interleaved", [False, True])
def test_rotary_position_zero_is_identity_and_norms_are_kept(interleaved):
    rng = np.random.default_rng(2)
    R = 128
    cos, sin = wl.rope_tables(4096, R)
    assert (cos[0] == 1).all() and (sin[0] == 0).all()
    x = rng.standard_normal((8, 128)).astype(np.float16)
    np.testing.assert_array_equal(orc.rotate_rows(x, [0] * 8, cos, sin, R, interleaved),
                                  x.astype(np.float64))
    pos = rng.integers(0, 4096, size=8)
    y = orc.rotate_rows(x, pos, cos, sin, R, interleaved)
    slot, partner, first = orc.rotary_geometry(R, interleaved)
    lead = np.nonzero(first)[0]
    xn = x.astype(np.float64)[:, lead] ** 2 + x.astype(np.float64)[:, partner[lead]] ** 2
    yn = y[:, lead] ** 2 + y[:, partner[lead]] ** 2
    # fp16 cos/sin satisfy |cos^2 + sin^2 - 1| <= 2 * 2^-11, which bounds the change
    c = cos.astype(np.float64)[pos][:, slot[lead]]
    s = sin.astype(np.float64)[pos][:, slot[lead]]
    np.testing.assert_allclose(yn, xn * (c ** 2 + s ** 2), rtol=1e-12, atol=1e-12)
    assert np.all(np.abs(yn - xn) <= 2.0 ** -9 * xn + 1e-12)


def test_append_layout_worked_example(golden):
    g = golden("append_layout.json")["bnsh"]
    B, H, M, D = g["batch"], g["kv_heads"], g["max_cache_seq"], g["head"]
    src = np.arange(B * H * D, dtype=np.float64).reshape(B, H * D) + 1000
    pk = np.zeros((B, H, M, D))
    pv = np.zeros((B, H, M, D))
    k_out, v_out, written, st = orc.kv_append_rotary(
        src, src + 0.5, packed=False, num_heads=H, kv_num_heads=H, head_size=D, batch=B,
        seq_len=g["seq_len"], total_sequence_length=[g["total0"]],
        key_total_sequence_lengths=g["key_totals"], cos_cache=None, sin_cache=None,
        rotary_dim=0, interleaved=False, present_key=pk, present_value=pv)
    w = g["write"]
    assert np.nonzero(written[w["b"], w["h"]])[0].tolist() == [g["expected_position"]]
    flat = k_out.reshape(-1)
    assert flat[g["expected_flat_index"]] == src[w["b"], w["h"] * D + w["d"]]
    assert v_out.reshape(-1)[g["expected_flat_index"]] == src[w["b"], w["h"] * D + w["d"]] + 0.5
    assert written.sum() == B * H and st == 0


def test_packed_offsets_worked_example(golden):
    g = golden("append_layout.json")["packed"]
    Hq, Hkv, D = g["num_heads"], g["kv_num_heads"], g["head"]
    row = np.array([g["row"]], dtype=np.float64)
    k, v, q = orc.split_new_kv(row, None, None, Hq, Hkv, D)
    assert k.reshape(-1).tolist() == g["expected_key"]
    assert v.reshape(-1).tolist() == g["expected_value"]
    pk = np.zeros((1, Hkv, 4, D))
    k_out, v_out, written, _ = orc.kv_append_rotary(
        row, None, packed=True, num_heads=Hq, kv_num_heads=Hkv, head_size=D, batch=1,
        seq_len=1, total_sequence_length=[3], key_total_sequence_lengths=[3],
        cos_cache=None, sin_cache=None, rotary_dim=0, interleaved=False,
        present_key=pk, present_value=pk.copy())
    assert k_out[0, 0, 2].tolist() == g["expected_key"]
    assert v_out[0, 0, 2].tolist() == g["expected_value"]


@pytest.mark.parametrize("mode", ["decode", "prompt"])
def test_append_leaves_other_rows_untouched(mode):
    c = wl.append_rotary(7, mode=mode, batch=2, num_heads=4, kv_num_heads=2, head_size=16,
                         rotary_dim=8, max_cache_seq=64, prompt_len=5, max_past=50)
    k_out, v_out, written, st = orc.kv_append_rotary(
        c.source, c.value, packed=c.packed, num_heads=4, kv_num_heads=2, head_size=16,
        batch=2, seq_len=c.seq_len, total_sequence_length=c.total_sequence_length,
        key_total_sequence_lengths=c.key_total_sequence_lengths, cos_cache=c.cos_cache,
        sin_cache=c.sin_cache, rotary_dim=8, interleaved=False,
        present_key=c.present_key, present_value=c.present_value)
    assert st == 0
    keep = ~written
    np.testing.assert_array_equal(k_out[keep], c.present_key.astype(np.float64)[keep])
    np.testing.assert_array_equal(v_out[keep], c.present_value.astype(np.float64)[keep])
    assert written.sum() == 2 * 2 * c.seq_len
    if mode == "prompt":
        assert written[:, :, :c.seq_len].all()
    # components at or above rotary_dim are plain copies of the source
    src = c.source.reshape(2 * c.seq_len, -1)
    for b in range(2):
        pos = np.nonzero(written[b, 0])[0]
        for t, p in enumerate(pos):
            krow = src[b * c.seq_len + t, 4 * 16:6 * 16].reshape(2, 16)
            np.testing.assert_array_equal(k_out[b, :, p, 8:], krow[:, 8:].astype(np.float64))


def test_append_position_past_cache_is_skipped():
    pk = np.zeros((1, 1, 4, 2))
    src = np.ones((1, 2))
    k_out, v_out, written, st = orc.kv_append_rotary(
        src, src, packed=False, num_heads=1, kv_num_heads=1, head_size=2, batch=1,
        seq_len=1, total_sequence_length=[9], key_total_sequence_lengths=[9],
        cos_cache=None, sin_cache=None, rotary_dim=0, interleaved=False,
        present_key=pk, present_value=pk.copy())
    assert not written.any() and st == orc.ST_BAD_POSITION
