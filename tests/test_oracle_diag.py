"""Pins of the oracle's attention diagnostics (section 3.4: Fig. 8 attention
mass split, Fig. 10 vertical vs diagonal score-vector similarity), without
a GPU.  Closed forms fix each part: uniform attention gives the masses
exactly; logits that depend only on i - j (RoPE-rotated constant vectors)
give a diagonal similarity of exactly 1; logits that depend only on the key
(a constant query) give a vertical similarity of exactly 1.
"""
import math

import numpy as np
import pytest

from oracle.oracle import DIAG_MUTATIONS, diag_set_mutation, diag_stream


def rope(x: np.ndarray, pos: np.ndarray) -> np.ndarray:
    d = x.shape[-1]
    half = d // 2
    inv = 10000.0 ** (-np.arange(half) * 2.0 / d)
    ang = pos[:, None] * inv[None, :]
    x1, x2 = x[..., :half], x[..., half:]
    return np.concatenate([x1 * np.cos(ang) - x2 * np.sin(ang), x2 * np.cos(ang) + x1 * np.sin(ang)], axis=-1)


def pin_uniform():
    L_p, L_dec, d = 7, 45, 16
    mass, v, dg = diag_stream(np.zeros((L_dec, d)), np.ones((L_p, d)), np.ones((L_dec, d)), [1, 3, 10])
    fails = []
    for i in range(L_dec):
        n = L_p + i + 1
        loc = math.ceil(0.1 * (i + 1))
        want = np.array([L_p / n, loc / n, (i + 1 - loc) / n])
        if not np.allclose(mass[i], want, rtol=0, atol=1e-13):
            fails.append(f"uniform mass at i={i}: {mass[i]} != {want}")
    if not (np.allclose(v, 1, atol=1e-13) and np.allclose(dg, 1, atol=1e-13)):
        fails.append(f"uniform similarities {v} {dg}")
    return fails


def pin_relative_position():
    """q_i = RoPE(u, i), k_j = RoPE(w, j): q_i . k_j depends on i - j only, so
    the diagonal score vectors are proportional: diagonal similarity 1."""
    rng = np.random.default_rng(1)
    L_p, L_dec, d = 5, 60, 16
    u, w = rng.normal(0, 2, d), rng.normal(0, 2, d)
    pos = np.arange(L_dec, dtype=np.float64) + L_p
    Q = rope(np.tile(u, (L_dec, 1)), pos)
    Kd = rope(np.tile(w, (L_dec, 1)), pos)
    Kp = rope(rng.normal(0, 2, (L_p, d)), np.arange(L_p, dtype=np.float64))
    _, v, dg = diag_stream(Q, Kp, Kd, [1, 2, 7, 20])
    fails = []
    if not np.allclose(dg, 1, atol=1e-12):
        fails.append(f"relative-position logits: diagonal similarity {dg} != 1")
    if not (v < 1 - 1e-6).all():
        fails.append(f"relative-position logits: vertical similarity {v} should be below 1")
    return fails


def pin_key_only():
    """A constant query: w_i over keys 0..i is proportional to exp(q . k_j),
    the same for every query: vertical similarity 1."""
    rng = np.random.default_rng(2)
    L_p, L_dec, d = 4, 50, 16
    q = rng.normal(0, 1, d)
    Q = np.tile(q, (L_dec, 1))
    Kd = rng.normal(0, 2, (L_dec, d))
    Kp = rng.normal(0, 2, (L_p, d))
    _, v, dg = diag_stream(Q, Kp, Kd, [1, 4, 9])
    fails = []
    if not np.allclose(v, 1, atol=1e-12):
        fails.append(f"key-only logits: vertical similarity {v} != 1")
    if not (dg < 1 - 1e-6).all():
        fails.append(f"key-only logits: diagonal similarity {dg} should be below 1")
    return fails


def pin_masses_sum_to_one():
    rng = np.random.default_rng(3)
    mass, _, _ = diag_stream(rng.normal(size=(30, 8)), rng.normal(size=(6, 8)), rng.normal(size=(30, 8)), [1])
    return [] if np.allclose(mass.sum(1), 1, atol=1e-12) and (mass >= 0).all() else ["masses do not sum to 1"]


PINS = {"uniform": pin_uniform, "relative_position": pin_relative_position, "key_only": pin_key_only,
        "sum": pin_masses_sum_to_one}


@pytest.mark.parametrize("name", list(PINS))
def test_pin_holds(name):
    fails = PINS[name]()
    assert not fails, "\n".join(fails[:10])


@pytest.mark.parametrize("mutation", list(DIAG_MUTATIONS))
def test_planted_mistake_is_caught(mutation):
    diag_set_mutation(mutation)
    try:
        caught = {name: len(fn()) for name, fn in PINS.items()}
    finally:
        diag_set_mutation(None)
    assert any(caught.values()), f"mutation {mutation} passes every pin: {caught}"


def test_bad_distances_are_rejected():
    with pytest.raises(ValueError):
        diag_stream(np.zeros((5, 4)), np.zeros((1, 4)), np.zeros((5, 4)), [5])
