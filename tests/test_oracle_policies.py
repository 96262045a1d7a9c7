"""Pins of the score-based eviction oracle (``oracle/policies.py``: TOVA,
H2O), without a GPU.  Each pin is a case whose answer the definitions fix
in closed form:

* budget never reached: dense attention over the prompt and every decode
  token (fp64 scaled_dot_product_attention);
* N_att = 1: the prompt and the current token only;
* TOVA with every new key scoring highest: the oldest entry always goes,
  i.e. a sliding window of N_att; with every new key scoring lowest: the
  current token always goes, i.e. the first N_att - 1 tokens stay;
* H2O with q = 0 (uniform weights): accumulated weights are harmonic sums
  1 / (L_p + a_s) over the steps an entry was attended, the oldest
  h = N_att - n_recent - 1 tokens stay as heavy hitters and the entry
  leaving the recent window goes;
* all keys equal: TOVA's ties go to the oldest (a sliding window again);
* invariants on random data: cache size, evicted positions never return,
  H2O never evicts from the recent window.

Every planted mistake of ``oracle.policies.MUTATIONS`` fails a pin.
"""
import math

import numpy as np
import pytest
import torch

from oracle.policies import MUTATIONS, POLICIES, PolicyStream


def sdpa(q, K, V):
    q = torch.from_numpy(np.asarray(q, dtype=np.float64))[None, None, None]
    K = torch.from_numpy(np.asarray(K, dtype=np.float64))[None, None]
    V = torch.from_numpy(np.asarray(V, dtype=np.float64))[None, None]
    return torch.nn.functional.scaled_dot_product_attention(q, K, V)[0, 0, 0].numpy()


def run(policy, Kp, Vp, Q, Kd, Vd, N_att, mutation=None):
    st = PolicyStream(Kp.shape[1], Kp.shape[0], N_att, policy, mutation)
    st.prefill(Kp, Vp)
    outs, infos = [], []
    for t in range(len(Q)):
        o, info = st.step(Q[t], Kd[t], Vd[t])
        outs.append(o)
        infos.append(info)
    return st, np.array(outs), infos


def data(seed, L_p=5, L=30, d=8):
    rng = np.random.default_rng(seed)
    return (rng.normal(size=(L_p, d)), rng.normal(size=(L_p, d)), rng.normal(size=(L, d)), rng.normal(size=(L, d)),
            rng.normal(size=(L, d)))


def attended_ok(outs, Kp, Vp, Q, Kd, Vd, sets, what):
    fails = []
    for t, dec in enumerate(sets):
        dec = list(dec)
        want = sdpa(Q[t], np.concatenate([Kp, Kd[dec]]), np.concatenate([Vp, Vd[dec]]))
        if not np.allclose(outs[t], want, rtol=1e-12, atol=1e-12):
            fails.append(f"{what}: step {t}")
    return fails[:3]


def pin_dense(policy, mutation=None):
    Kp, Vp, Q, Kd, Vd = data(1)
    _, outs, _ = run(policy, Kp, Vp, Q, Kd, Vd, N_att=len(Q) + 1, mutation=mutation)
    return attended_ok(outs, Kp, Vp, Q, Kd, Vd, [range(t + 1) for t in range(len(Q))], f"{policy} dense")


def pin_current_only(policy, mutation=None):
    Kp, Vp, Q, Kd, Vd = data(2)
    st, outs, _ = run(policy, Kp, Vp, Q, Kd, Vd, N_att=1, mutation=mutation)
    fails = attended_ok(outs, Kp, Vp, Q, Kd, Vd, [[t] for t in range(len(Q))], f"{policy} N_att=1")
    if st.positions():
        fails.append(f"{policy} N_att=1 keeps {st.positions()}")
    return fails


def _ordered_keys(sign, L=30, d=8, L_p=5):
    rng = np.random.default_rng(3)
    Kp, Vp = rng.normal(size=(L_p, d)), rng.normal(size=(L_p, d))
    Q = np.zeros((L, d))
    Q[:, 0] = 1.0
    Kd = rng.normal(size=(L, d))
    Kd[:, 0] = sign * np.arange(L, dtype=np.float64)  # q_t . k_j grows (or falls) with j
    return Kp, Vp, Q, Kd, rng.normal(size=(L, d))


def pin_tova_sliding(mutation=None):
    Kp, Vp, Q, Kd, Vd = _ordered_keys(+1)
    N = 6
    _, outs, _ = run("tova", Kp, Vp, Q, Kd, Vd, N, mutation)
    return attended_ok(outs, Kp, Vp, Q, Kd, Vd, [range(max(0, t + 1 - N), t + 1) for t in range(len(Q))],
                       "tova newest-highest = sliding window")


def pin_tova_keep_first(mutation=None):
    Kp, Vp, Q, Kd, Vd = _ordered_keys(-1)
    N = 6
    _, outs, _ = run("tova", Kp, Vp, Q, Kd, Vd, N, mutation)
    sets = [range(t + 1) if t < N else list(range(N - 1)) + [t] for t in range(len(Q))]
    return attended_ok(outs, Kp, Vp, Q, Kd, Vd, sets, "tova newest-lowest = first tokens kept")


def pin_tova_ties(mutation=None):
    rng = np.random.default_rng(4)
    L_p, L, d, N = 4, 25, 8, 5
    Kp, Vp, Vd = rng.normal(size=(L_p, d)), rng.normal(size=(L_p, d)), rng.normal(size=(L, d))
    # all decode keys equal, integer q and k (exact dot products in any
    # summation order): every eviction is an exact tie
    Q = rng.integers(-3, 4, size=(L, d)).astype(np.float64)
    Kd = np.tile(rng.integers(-3, 4, size=d).astype(np.float64), (L, 1))
    _, outs, _ = run("tova", Kp, Vp, Q, Kd, Vd, N, mutation)
    return attended_ok(outs, Kp, Vp, Q, Kd, Vd, [range(max(0, t + 1 - N), t + 1) for t in range(len(Q))],
                       "tova ties to the oldest")


def pin_h2o_uniform(mutation=None):
    rng = np.random.default_rng(5)
    L_p, L, d = 3, 28, 8
    fails = []
    for N in (2, 4, 7):
        Kp, Vp, Kd, Vd = (rng.normal(size=(L_p, d)), rng.normal(size=(L_p, d)), rng.normal(size=(L, d)),
                          rng.normal(size=(L, d)))
        Q = np.zeros((L, d))
        st = PolicyStream(d, L_p, N, "h2o", mutation)
        st.prefill(Kp, Vp)
        n_recent = min(math.ceil(N / 2), N - 1)
        h = N - n_recent - 1
        for t in range(L):
            out, _ = st.step(Q[t], Kd[t], Vd[t])
            dec = list(range(t + 1)) if t < N else list(range(h)) + list(range(t - n_recent, t + 1))
            if t == N - 1:
                dec = list(range(N))
            want = np.concatenate([Vp, Vd[dec]]).mean(axis=0)
            if not np.allclose(out, want, rtol=1e-12, atol=1e-12):
                fails.append(f"h2o uniform N={N}: output at step {t}")
                break
            # accumulated weight of the kept entries: sum over attended steps of 1 / (L_p + a_s)
            kept_want = list(range(t + 1)) if t < N - 1 else list(range(h)) + list(range(t - n_recent + 1, t + 1))
            if st.positions() != kept_want:
                fails.append(f"h2o uniform N={N}: kept {st.positions()} != {kept_want} at step {t}")
                break
            for pos, acc in st.accumulated().items():
                want_acc = sum(1.0 / (L_p + min(s + 1, N)) for s in range(pos, t + 1))
                if not math.isclose(acc, want_acc, rel_tol=1e-12):
                    fails.append(f"h2o uniform N={N}: accumulated weight of {pos} at step {t}")
                    break
    return fails[:3]


def pin_invariants(policy, mutation=None):
    Kp, Vp, Q, Kd, Vd = data(6, L=40)
    N = 7
    st = PolicyStream(Kp.shape[1], Kp.shape[0], N, policy, mutation)
    st.prefill(Kp, Vp)
    gone, fails = set(), []
    n_recent = min(math.ceil(N / 2), N - 1)
    for t in range(len(Q)):
        _, info = st.step(Q[t], Kd[t], Vd[t])
        pos = st.positions()
        if len(pos) != min(t + 1, N - 1):
            fails.append(f"{policy}: cache size {len(pos)} at step {t}")
        if info["evicted"] >= 0:
            gone.add(info["evicted"])
            if policy == "h2o" and info["evicted"] > t - n_recent:
                fails.append(f"h2o evicted {info['evicted']} from the recent window at step {t}")
        if gone & set(pos) or any(p > t for p in pos):
            fails.append(f"{policy}: cache {pos} at step {t}")
        if info["attended"] != min(t + 1, N):
            fails.append(f"{policy}: attended {info['attended']} at step {t}")
    return fails[:3]


PINS = ([lambda m=None, p=p: pin_dense(p, m) for p in POLICIES] + [lambda m=None, p=p: pin_current_only(p, m) for p in POLICIES]
        + [pin_tova_sliding, pin_tova_keep_first, pin_tova_ties, pin_h2o_uniform]
        + [lambda m=None, p=p: pin_invariants(p, m) for p in POLICIES])
NAMES = ([f"dense-{p}" for p in POLICIES] + [f"current_only-{p}" for p in POLICIES]
         + ["tova_sliding", "tova_keep_first", "tova_ties", "h2o_uniform"] + [f"invariants-{p}" for p in POLICIES])


@pytest.mark.parametrize("i", range(len(PINS)), ids=NAMES)
def test_pin_holds(i):
    assert PINS[i]() == []


@pytest.mark.parametrize("mutation", MUTATIONS)
def test_planted_mistake_is_caught(mutation):
    caught = [NAMES[i] for i, p in enumerate(PINS) if p(mutation)]
    assert caught, f"planted mistake {mutation!r} passes every pin"
