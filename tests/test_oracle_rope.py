"""Pins for the rotary-embedding oracle (CPU only).

The formula is pinned by properties any correct rotation has (identity at
position 0, norm preservation, dependence of q.k on the position difference
only, composition of rotations); the float32 path is pinned to the float64
formula and the bf16 rounding to its definition.
"""

import numpy as np
import pytest

from oracle import cache, rope


def _angles_table(max_pos, d, base=10000.0):
    h = d // 2
    inv = base ** (-np.arange(h) * 2.0 / d)
    ang = np.arange(max_pos)[:, None] * inv[None, :]
    return np.cos(ang), np.sin(ang)


def test_position_zero_is_identity():
    rng = np.random.default_rng(0)
    x = rng.standard_normal((5, 64))
    c, s = _angles_table(1, 64)
    assert np.array_equal(rope.rotate_f64(x, c[0], s[0]), x)
    x32 = x.astype(np.float32)
    assert np.array_equal(rope.rotate_f32(x32, np.ones(32), np.zeros(32)), x32)


def test_rotation_preserves_pair_norms():
    rng = np.random.default_rng(1)
    x = rng.standard_normal((7, 128))
    c, s = _angles_table(50, 128)
    y = rope.rotate_f64(x, c[37], s[37])
    n0 = x[:, :64] ** 2 + x[:, 64:] ** 2
    n1 = y[:, :64] ** 2 + y[:, 64:] ** 2
    assert np.max(np.abs(n0 - n1)) < 1e-12


def test_score_depends_only_on_position_difference():
    rng = np.random.default_rng(2)
    q = rng.standard_normal(128)
    k = rng.standard_normal(128)
    c, s = _angles_table(400, 128)
    ref = rope.rotate_f64(q, c[70], s[70]) @ rope.rotate_f64(k, c[20], s[20])
    for t in (1, 13, 250):
        got = rope.rotate_f64(q, c[70 + t], s[70 + t]) @ rope.rotate_f64(k, c[20 + t], s[20 + t])
        assert abs(got - ref) < 1e-9


def test_rotations_compose():
    rng = np.random.default_rng(3)
    x = rng.standard_normal(64)
    c, s = _angles_table(100, 64)
    twice = rope.rotate_f64(rope.rotate_f64(x, c[30], s[30]), c[45], s[45])
    assert np.max(np.abs(twice - rope.rotate_f64(x, c[75], s[75]))) < 1e-12


def test_swapped_halves_or_sign_would_fail_the_pins():
    # a plausible mistake: rotating (x[i], x[i+1]) pairs would not preserve the
    # half-split pair norms checked above
    rng = np.random.default_rng(4)
    x = rng.standard_normal(8)
    c, s = _angles_table(10, 8)
    wrong = x.copy()
    wrong[0::2], wrong[1::2] = (x[0::2] * c[5] - x[1::2] * s[5], x[0::2] * s[5] + x[1::2] * c[5])
    right = rope.rotate_f64(x, c[5], s[5])
    assert np.max(np.abs(wrong - right)) > 1e-3


def test_f32_path_close_to_f64_formula():
    rng = np.random.default_rng(5)
    x = rng.standard_normal((9, 128)).astype(np.float32)
    tab = rope.rope_table(4096, 128)
    for p in (0, 1, 777, 4095):
        got = rope.rotate_f32(x, tab[p, :64], tab[p, 64:]).astype(np.float64)
        ref = rope.rotate_f64(x.astype(np.float64), tab[p, :64].astype(np.float64),
                              tab[p, 64:].astype(np.float64))
        assert np.max(np.abs(got - ref)) <= 4e-7 * np.max(np.abs(ref))


def test_bf16_rounding_is_nearest_even():
    f = np.array([1.0, 1.00390625, 1.01171875, 1.005859375, -2.5, 3.0e-39, 65504.0],
                 dtype=np.float32)
    bits = rope.f32_to_bf16_bits(f)
    # 1 + 2^-8 is a tie between 1 and 1 + 2^-7: rounds to even (1.0)
    assert bits[1] == 0x3F80
    # 1 + 3 * 2^-8 ties between 1 + 2^-7 and 1 + 2^-6: rounds to even (1 + 2^-6)
    assert bits[2] == 0x3F82
    # above the tie rounds up
    assert bits[3] == 0x3F81
    back = rope.bf16_bits_to_f32(bits)
    normal = np.abs(f) >= 2.0 ** -126
    # half an ulp: 2^-8 relative for normals, 2^-134 absolute for subnormals
    assert np.all(np.abs(back - f)[normal] <= np.abs(f)[normal] * 2.0 ** -8)
    assert np.all(np.abs(back - f)[~normal] <= 2.0 ** -134)


def test_append_rope_writes_rotated_k_and_plain_v():
    rng = np.random.default_rng(6)
    t, hq, hkv, d, bs = 5, 4, 2, 16, 4
    k = rng.standard_normal((t, hkv, d)).astype(np.float32)
    v = rng.standard_normal((t, hkv, d)).astype(np.float32)
    q = rng.standard_normal((t, hq, d)).astype(np.float32)
    kc = np.zeros((8, hkv, bs, d), np.float32)
    vc = np.zeros_like(kc)
    tab = rope.rope_table(64, d)
    pos = np.array([0, 3, 9, 33, 63])
    slots = np.array([0, 5, 6, 13, 31])
    qo = rope.append_rope(kc, vc, q, k, v, slots, pos, tab, bs, "f32", cache.append)
    assert np.array_equal(kc[0, :, 0], k[0])                      # position 0: unchanged
    assert np.array_equal(vc[1, :, 1], v[1])                      # V is never rotated
    assert np.array_equal(kc[3, :, 1], rope.rotate_f32(k[3], tab[33, :8], tab[33, 8:]))
    assert np.array_equal(qo[4], rope.rotate_f32(q[4], tab[63, :8], tab[63, 8:]))
    with pytest.raises(IndexError):
        rope.append_rope(kc, vc, q, k, v, slots, pos + 1, tab, bs, "f32", cache.append)
