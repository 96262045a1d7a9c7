"""Pins of the QKV-projection oracle (``oracle/proj.py``), without a GPU.

Each pin is fixed by mathematics rather than by the oracle's own formula:

* permutation weights: with W's q / k / v blocks permutation matrices (not
  symmetric), the projection at position 0 is a known reordering of x, which
  fixes the orientation of W, the q / k / v block order and the stream order;
* rotation of a basis vector: RoPE of e_j at position p is, by definition of
  a plane rotation, cos(p theta_j) e_j + sin(p theta_j) e_{j+d/2} (and
  -sin(p theta_j) e_{j-d/2} + cos(p theta_j) e_j for the second half), with
  theta_j = 10000^(-2j/d): sign, pairing, base and position;
* orthogonality: RoPE keeps every head's norm, at any position;
* relative position: q(m) . k(n) depends on m - n only;
* v is never rotated;
* a brute-force sum of products on a tiny case.

Every planted mistake of ``oracle.proj.MUTATIONS`` fails at least one pin.
"""
import itertools
import math

import numpy as np
import pytest

from oracle.proj import MUTATIONS, qkv_rope


def _perm_weights(H, d, rng):
    HD = H * d
    perms = [rng.permutation(HD) for _ in range(3)]
    W = np.zeros((3 * HD, HD))
    for part, p in enumerate(perms):
        W[part * HD + np.arange(HD), p] = part + 1.0
    return W, perms


def pin_permutation(mutation=None):
    rng = np.random.default_rng(3)
    B, H, d = 3, 2, 8
    W, perms = _perm_weights(H, d, rng)
    x = rng.normal(size=(B, H * d))
    q, k, v = qkv_rope(x, W, H, d, pos=0, mutation=mutation)
    fails = []
    for part, got in enumerate((q, k, v)):
        want = ((part + 1.0) * x[:, perms[part]]).reshape(B * H, d)
        if got.shape != want.shape or not np.array_equal(got, want):
            fails.append(f"permutation weights, part {part}")
    return fails


def pin_basis_rotation(mutation=None):
    H, d = 1, 16
    half = d // 2
    fails = []
    for j, p in itertools.product((0, 3, half - 1, half, half + 5, d - 1), (1, 7, 300)):
        W = np.zeros((3 * d, d))
        W[np.arange(d), np.arange(d)] = 1.0          # q = x
        W[d + np.arange(d), np.arange(d)] = 1.0      # k = x
        W[2 * d + np.arange(d), np.arange(d)] = 1.0  # v = x
        x = np.zeros((1, d))
        x[0, j] = 1.0
        q, k, v = qkv_rope(x, W, H, d, pos=p, mutation=mutation)
        jj = j % half
        ang = p * 10000.0 ** (-2.0 * jj / d)
        want = np.zeros(d)
        if j < half:
            want[j], want[j + half] = math.cos(ang), math.sin(ang)
        else:
            want[j], want[j - half] = math.cos(ang), -math.sin(ang)
        for name, got in (("q", q[0]), ("k", k[0])):
            if not np.allclose(got, want, rtol=0, atol=1e-15):
                fails.append(f"basis e_{j} at pos {p}: {name}")
        if not np.array_equal(v[0], x[0]):
            fails.append(f"basis e_{j} at pos {p}: v rotated")
    return fails


def pin_norm(mutation=None):
    rng = np.random.default_rng(5)
    B, H, d, hidden = 2, 3, 16, 40
    x = rng.normal(size=(B, hidden))
    W = rng.normal(size=(3 * H * d, hidden))
    q0, k0, _ = qkv_rope(x, W, H, d, pos=0)
    fails = []
    for p in (1, 64, 4095):
        q, k, _ = qkv_rope(x, W, H, d, pos=p, mutation=mutation)
        if not (np.allclose(np.linalg.norm(q, axis=1), np.linalg.norm(q0, axis=1), rtol=1e-13)
                and np.allclose(np.linalg.norm(k, axis=1), np.linalg.norm(k0, axis=1), rtol=1e-13)):
            fails.append(f"norm at pos {p}")
    return fails


def pin_relative_position(mutation=None):
    rng = np.random.default_rng(7)
    B, H, d, hidden = 1, 2, 16, 24
    x = rng.normal(size=(B, hidden))
    W = rng.normal(size=(3 * H * d, hidden))

    def dot(m, n):
        q, _, _ = qkv_rope(x, W, H, d, pos=m, mutation=mutation)
        _, k, _ = qkv_rope(x, W, H, d, pos=n, mutation=mutation)
        return np.sum(q * k, axis=1)

    fails = []
    for m, n, c in ((5, 2, 11), (70, 64, 1000), (3, 9, 57)):
        if not np.allclose(dot(m, n), dot(m + c, n + c), rtol=1e-11, atol=1e-11):
            fails.append(f"relative position m={m} n={n} shift {c}")
    return fails


def pin_v_unrotated(mutation=None):
    rng = np.random.default_rng(9)
    B, H, d, hidden = 2, 2, 8, 16
    x = rng.normal(size=(B, hidden))
    W = rng.normal(size=(3 * H * d, hidden))
    _, _, v0 = qkv_rope(x, W, H, d, pos=0)
    _, _, v = qkv_rope(x, W, H, d, pos=123, mutation=mutation)
    return [] if np.array_equal(v, v0) else ["v depends on the position"]


def pin_brute_force(mutation=None):
    rng = np.random.default_rng(11)
    B, H, d, hidden = 2, 2, 4, 6
    x = rng.integers(-3, 4, size=(B, hidden)).astype(np.float64)
    W = rng.integers(-3, 4, size=(3 * H * d, hidden)).astype(np.float64)
    q, k, v = qkv_rope(x, W, H, d, pos=0, mutation=mutation)
    fails = []
    for b in range(B):
        for h in range(H):
            for i in range(d):
                for part, got in enumerate((q, k, v)):
                    row = part * H * d + h * d + i
                    want = 0.0
                    for c in range(hidden):
                        want += x[b, c] * W[row, c]
                    if got[b * H + h, i] != want:
                        fails.append(f"brute force b={b} h={h} i={i} part={part}")
    return fails[:5]


PINS = [pin_permutation, pin_basis_rotation, pin_norm, pin_relative_position, pin_v_unrotated, pin_brute_force]


@pytest.mark.parametrize("pin", PINS, ids=lambda f: f.__name__)
def test_pin_holds(pin):
    assert pin() == []


@pytest.mark.parametrize("mutation", MUTATIONS)
def test_planted_mistake_is_caught(mutation):
    caught = [p.__name__ for p in PINS if p(mutation)]
    assert caught, f"planted mistake {mutation!r} passes every pin"
