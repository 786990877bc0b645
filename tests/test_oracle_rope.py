"""Pins of the oracle's table-driven RoPE and its fusion with the cache scatter.

The page ("AI Infra入门干货总结", section "Attention Module") prints no worked
RoPE example, so the oracle is pinned by what the mathematics fixes:
* each rotation pair is a complex number multiplied by e^{i a} (numpy's complex
  exponential, a route that shares nothing with the oracle's rotation matrix);
* closed forms: a unit vector on a pair's first dimension becomes
  (cos a, sin a) on that pair, and angle 0 is the identity;
* invariants: the matrix is orthogonal, norms are kept, dimensions at and
  above rotary_dim pass through bit for bit;
* the relative-position property of angles linear in the position;
* the fused op equals the rotation followed by the pinned scatter.
"""

import numpy as np
import pytest

from oracle import paging, rope


def _angles(max_pos, half, seed):
    rng = np.random.default_rng(seed)
    return rng.uniform(-np.pi, np.pi, size=(max_pos, half))


def _table(angles):
    return np.concatenate([np.cos(angles), np.sin(angles)], axis=1)


def _complex_route(x, positions, angles, rotary_dim, is_neox):
    """Rotation as complex multiplication: z_i = x_a + i x_b, z_i * e^{i a}."""
    out = np.array(x, dtype=np.float64, copy=True)
    half = rotary_dim // 2
    if is_neox:
        re, im = out[..., :half], out[..., half:rotary_dim]
    else:
        re, im = out[..., 0:rotary_dim:2], out[..., 1:rotary_dim:2]
    z = re + 1j * im
    z = z * np.exp(1j * angles[np.asarray(positions)])[:, None, :]
    if is_neox:
        out[..., :half], out[..., half:rotary_dim] = z.real, z.imag
    else:
        out[..., 0:rotary_dim:2], out[..., 1:rotary_dim:2] = z.real, z.imag
    return out


@pytest.mark.parametrize("is_neox", [False, True])
@pytest.mark.parametrize("D,rd", [(128, 128), (64, 64), (128, 64), (80, 32), (16, 2)])
def test_matches_complex_multiplication(is_neox, D, rd):
    T, H, max_pos = 37, 5, 300
    ang = _angles(max_pos, rd // 2, 1 + D + rd)
    rng = np.random.default_rng(7)
    x = rng.standard_normal((T, H, D))
    pos = rng.integers(0, max_pos, size=T)
    got = rope.apply_rope(x, pos, _table(ang), rd, is_neox)
    want = _complex_route(x, pos, ang, rd, is_neox)
    np.testing.assert_allclose(got, want, rtol=0, atol=1e-12)
    # pass-through dimensions are untouched, bit for bit
    assert np.array_equal(got[..., rd:], x[..., rd:])


@pytest.mark.parametrize("is_neox", [False, True])
def test_unit_vector_closed_form(is_neox):
    rd, D, max_pos = 8, 8, 4
    ang = _angles(max_pos, rd // 2, 3)
    for pair in range(rd // 2):
        a = 2 * pair if not is_neox else pair
        b = a + 1 if not is_neox else pair + rd // 2
        x = np.zeros((1, 1, D))
        x[0, 0, a] = 1.0
        out = rope.apply_rope(x, [2], _table(ang), rd, is_neox)[0, 0]
        want = np.zeros(D)
        want[a], want[b] = np.cos(ang[2, pair]), np.sin(ang[2, pair])
        np.testing.assert_allclose(out, want, atol=1e-15)
        # and the second dimension of the pair goes to (-sin a, cos a)
        y = np.zeros((1, 1, D))
        y[0, 0, b] = 1.0
        out = rope.apply_rope(y, [2], _table(ang), rd, is_neox)[0, 0]
        want = np.zeros(D)
        want[a], want[b] = -np.sin(ang[2, pair]), np.cos(ang[2, pair])
        np.testing.assert_allclose(out, want, atol=1e-15)


@pytest.mark.parametrize("is_neox", [False, True])
def test_zero_angle_is_identity_and_matrix_is_orthogonal(is_neox):
    rd = 16
    ang = _angles(10, rd // 2, 5)
    ang[0] = 0.0
    table = _table(ang)
    x = np.random.default_rng(1).standard_normal((4, 3, rd))
    assert np.array_equal(rope.apply_rope(x, [0, 0, 0, 0], table, rd, is_neox), x)
    for p in range(10):
        R = rope.rotation_matrix(table[p], rd, is_neox)
        np.testing.assert_allclose(R.T @ R, np.eye(rd), atol=1e-14)
        assert abs(np.linalg.det(R) - 1.0) < 1e-12  # a rotation, not a reflection
    out = rope.apply_rope(x, [1, 3, 5, 9], table, rd, is_neox)
    np.testing.assert_allclose(np.linalg.norm(out, axis=-1), np.linalg.norm(x, axis=-1), rtol=1e-14)


@pytest.mark.parametrize("is_neox", [False, True])
def test_relative_position_property(is_neox):
    """With angles p * theta_i the score <R_m q, R_n k> depends on n - m only."""
    rd, max_pos = 32, 64
    theta = np.random.default_rng(11).uniform(0.01, 1.5, size=rd // 2)
    table = _table(np.arange(max_pos)[:, None] * theta[None, :])
    rng = np.random.default_rng(12)
    q = rng.standard_normal((1, 1, rd))
    k = rng.standard_normal((1, 1, rd))
    for m, n in [(3, 10), (20, 27), (0, 7), (40, 47), (5, 5), (30, 30), (12, 1), (50, 39)]:
        lhs = np.dot(rope.apply_rope(q, [m], table, rd, is_neox).ravel(),
                     rope.apply_rope(k, [n], table, rd, is_neox).ravel())
        if n >= m:
            rhs = np.dot(q.ravel(), rope.apply_rope(k, [n - m], table, rd, is_neox).ravel())
        else:
            rhs = np.dot(rope.apply_rope(q, [m - n], table, rd, is_neox).ravel(), k.ravel())
        assert abs(lhs - rhs) < 1e-12


def test_pairings_differ_by_a_permutation():
    """The two pairings are the same rotation in permuted coordinates."""
    rd = 12
    table = _table(_angles(3, rd // 2, 9))
    perm = np.concatenate([np.arange(0, rd, 2), np.arange(1, rd, 2)])  # interleaved -> halves
    x = np.random.default_rng(2).standard_normal((1, 2, rd))
    a = rope.apply_rope(x, [1], table, rd, is_neox=False)
    b = rope.apply_rope(x[..., perm], [1], table, rd, is_neox=True)
    np.testing.assert_allclose(a[..., perm], b, atol=1e-14)


def test_position_outside_table_raises():
    table = _table(_angles(4, 2, 1))
    with pytest.raises(IndexError):
        rope.apply_rope(np.zeros((1, 1, 4)), [4], table, 4, False)


@pytest.mark.parametrize("is_neox", [False, True])
def test_fused_op_is_rotation_then_scatter(is_neox):
    T, H, Hkv, D, rd, B, NB, max_pos = 11, 4, 2, 16, 8, 4, 6, 50
    rng = np.random.default_rng(4)
    table = _table(_angles(max_pos, rd // 2, 8))
    q = rng.standard_normal((T, H, D))
    k = rng.standard_normal((T, Hkv, D))
    v = rng.standard_normal((T, Hkv, D))
    pos = rng.integers(0, max_pos, size=T)
    slots = rng.permutation(NB * B)[:T].astype(np.int64)
    slots[3] = -1  # a padding token
    kc = np.full((NB, B, Hkv, D), np.nan)
    vc = np.full((NB, B, Hkv, D), np.nan)
    q_rot, k_rot = rope.rope_reshape_and_cache(pos, q, k, v, kc, vc, slots, table, rd, is_neox)
    np.testing.assert_allclose(q_rot, _complex_route(q, pos, _angles(max_pos, rd // 2, 8), rd, is_neox),
                               atol=1e-12)
    for t in range(T):
        s = int(slots[t])
        if s < 0:
            continue
        assert np.array_equal(kc[s // B, s % B], k_rot[t])
        assert np.array_equal(vc[s // B, s % B], v[t])
    # exactly the T - 1 addressed slots were written
    assert np.isfinite(kc).all(axis=(2, 3)).sum() == T - 1
    kc2 = np.full_like(kc, np.nan)
    vc2 = np.full_like(vc, np.nan)
    paging.write_cache(kc2, vc2, k_rot, v, slots)
    assert np.array_equal(np.nan_to_num(kc, nan=7.0), np.nan_to_num(kc2, nan=7.0))
