"""Pins for the oracle's query rotation (no GPU).

The append page rotates keys only; a query rotated at its token's absolute position
with the same rule and tables is the other half of rotary attention. These tests pin
the oracle's query rotation to two facts that do not go through its rotation code:
a rotation pair is a complex number multiplied by cos + i sin of its slot, and with
both query and key rotated the scores depend only on the distance between positions.
"""
import numpy as np
import pytest

from oracle import pagedkv_oracle as orc
from paged_kv_cache_231_gb300 import workloads as wl


def complex_rotate(x, pos, cos, sin, rotary_dim, interleaved):
    """Rotate a head row by complex multiplication: pair (a, b) is a + ib, slot i is
    multiplied by cos[pos, i] + i sin[pos, i]. Interleaved pairs are (2i, 2i+1);
    NeoX pairs are (i, i + rotary_dim/2)."""
    x = np.asarray(x, dtype=np.float64).copy()
    R = rotary_dim
    w = np.asarray(cos[pos], dtype=np.float64) + 1j * np.asarray(sin[pos], dtype=np.float64)
    if interleaved:
        z = (x[0:R:2] + 1j * x[1:R:2]) * w
        x[0:R:2], x[1:R:2] = z.real, z.imag
    else:
        z = (x[:R // 2] + 1j * x[R // 2:R]) * w
        x[:R // 2], x[R // 2:R] = z.real, z.imag
    return x


def run(case, **kw):
    return orc.paged_attention(
        case.query, case.key, case.value, case.key_cache, case.value_cache,
        case.cu_seqlens, case.past_seqlens, case.block_table, case.slot_mapping,
        num_heads=case.num_heads, kv_num_heads=case.kv_num_heads, scale=case.scale,
        cos_cache=case.cos_cache, sin_cache=case.sin_cache, rotary_dim=case.rotary_dim,
        rotary_interleaved=case.rotary_interleaved, **kw)


@pytest.mark.parametrize("interleaved", [False, True])
@pytest.mark.parametrize("rotary_dim", [8, 16])
def test_paged_query_rotation_is_complex_multiplication(interleaved, rotary_dim):
    Hq, Hkv, D, BS = 4, 2, 16, 4
    c = wl.paged_case(41, num_heads=Hq, kv_num_heads=Hkv, head_size=D, block_size=BS,
                      past=[5, 0, 9], new_tokens=[1, 4, 2], rotary_dim=rotary_dim,
                      rotary_interleaved=interleaved)
    out, kc, vc, st = run(c, rotary_query=True)
    assert st == 0
    out = out.reshape(-1, Hq, D)
    smap, _ = orc.sequence_map(c.cu_seqlens, c.past_seqlens)
    G = Hq // Hkv
    for i, (b, t, pos) in enumerate(smap):
        for hq in range(Hq):
            h = hq // G
            q = complex_rotate(c.query[i, hq * D:(hq + 1) * D], pos, c.cos_cache,
                               c.sin_cache, rotary_dim, interleaved)
            keys = range(pos + 1)
            K = np.array([kc[c.block_table[b, j // BS], j % BS, h] for j in keys], np.float64)
            V = np.array([vc[c.block_table[b, j // BS], j % BS, h] for j in keys], np.float64)
            s = c.scale * (K @ q)
            p = np.exp(s - s.max())
            np.testing.assert_allclose(out[i, hq], (p / p.sum()) @ V, rtol=1e-11, atol=1e-13)


def fp64_tables(n, rotary_dim, shift, theta=10000.0):
    half = rotary_dim // 2
    inv = theta ** (-(2.0 * np.arange(half)) / rotary_dim)
    ang = (np.arange(n, dtype=np.float64) + shift)[:, None] * inv[None, :]
    return np.cos(ang), np.sin(ang)


@pytest.mark.parametrize("interleaved", [False, True])
def test_rotated_scores_depend_only_on_relative_position(interleaved):
    # A prompt with no history: every key and query is rotated. Moving every position
    # by the same shift (tables that start `shift` positions later) leaves each
    # query-key angle, hence the attention, unchanged; the only difference left is the
    # fp16 rounding of the stored rotated keys.
    c = wl.paged_case(42, num_heads=4, kv_num_heads=2, head_size=16, block_size=4,
                      past=[0], new_tokens=[12], rotary_dim=16,
                      rotary_interleaved=interleaved)
    outs, key_only = [], []
    for shift in (0, 37):
        c.cos_cache, c.sin_cache = fp64_tables(16, 16, shift)
        outs.append(run(c, rotary_query=True)[0])
        key_only.append(run(c)[0])
    np.testing.assert_allclose(outs[1], outs[0], atol=4e-3)
    # the check has teeth: with the key alone rotated the shift changes the output
    assert np.abs(key_only[1] - key_only[0]).max() > 0.05


def test_query_position_past_table_is_left_unrotated():
    c = wl.paged_case(43, num_heads=2, kv_num_heads=1, head_size=8, block_size=4,
                      past=[5], new_tokens=[3], rotary_dim=8)
    c.cos_cache = c.cos_cache[:7]     # rows for positions 0..6; token 2 sits at 7
    c.sin_cache = c.sin_cache[:7]
    rot, _, _, st = run(c, rotary_query=True)
    plain = run(c)[0]
    assert st == orc.ST_BAD_POSITION
    np.testing.assert_array_equal(rot[2], plain[2])     # position 7: query unrotated
    assert not np.array_equal(rot[0], plain[0])         # position 5: rotated


@pytest.mark.parametrize("interleaved", [False, True])
@pytest.mark.parametrize("packed", [True, False])
@pytest.mark.parametrize("mode", ["decode", "prompt"])
def test_append_query_rotation_is_complex_multiplication(interleaved, packed, mode):
    Hq, Hkv, D, R = 4, 2, 16, 8
    c = wl.append_rotary(44, mode=mode, interleaved=interleaved, batch=3, num_heads=Hq,
                         kv_num_heads=Hkv, head_size=D, rotary_dim=R, max_cache_seq=64,
                         prompt_len=3, max_past=50, packed=packed)
    query = None if packed else wl.normal_f16(wl.rng_for(45), (3 * c.seq_len, Hq * D))
    q_out = orc.append_query_rotary(
        c.source, query, packed=packed, num_heads=Hq, kv_num_heads=Hkv, head_size=D,
        batch=3, seq_len=c.seq_len, total_sequence_length=c.total_sequence_length,
        key_total_sequence_lengths=c.key_total_sequence_lengths, cos_cache=c.cos_cache,
        sin_cache=c.sin_cache, rotary_dim=R, interleaved=interleaved)
    src = c.source if packed else query
    for b in range(3):
        # history: prompt mode when the scalar total equals the new-token count
        total = int(c.total_sequence_length[0])
        past = 0 if total == c.seq_len else int(c.key_total_sequence_lengths[b]) - c.seq_len
        for t in range(c.seq_len):
            row = b * c.seq_len + t
            for hq in range(Hq):
                expect = complex_rotate(src[row, hq * D:(hq + 1) * D], past + t, c.cos_cache,
                                        c.sin_cache, R, interleaved)
                np.testing.assert_allclose(q_out[row, hq * D:(hq + 1) * D], expect,
                                           rtol=1e-15, atol=1e-15)
