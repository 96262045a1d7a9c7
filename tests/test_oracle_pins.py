"""The CPU oracle against what the page and mathematics fix (no GPU)."""
import numpy as np
import pytest

from oracle.oracle import MUTATIONS, OracleStream
from tests import pins


@pytest.mark.parametrize("name", list(pins.ALL_PINS))
def test_pin_holds(name):
    fails = pins.ALL_PINS[name]()
    assert not fails, "\n".join(fails[:20])


@pytest.mark.parametrize("mutation", list(MUTATIONS))
def test_planted_mistake_is_caught(mutation):
    """Each planted mistake in the oracle makes at least one pin fail."""
    caught = {name: len(fn(mutation)) for name, fn in pins.ALL_PINS.items()}
    assert any(caught.values()), f"mutation {mutation} passes every pin: {caught}"


def test_worked_example_full_trace():
    """Steps past the page's narration follow from the algorithm on the
    engineered inputs: third pick K1 at t=5, then constant relative offsets."""
    d, L_p, L_dec, Kp, Vp, q, k, v = pins.worked_example_inputs()
    st = OracleStream(d, L_p, 7, 4)
    st.prefill(Kp, Vp)
    seen = []
    for t in range(L_dec):
        _, info = st.step(q[t], k[t], v[t])
        seen.append((info.phase, st.idx(), sorted(st.skip()), info.selected))
    assert [s[0] for s in seen] == [1, 1, 1, 2, 2, 2, 2, 3, 3, 3]
    assert seen[5][3] == 1 and seen[5][2] == [1, 2, 3]
    assert seen[6][1] == [0, 1, 5, 6] and seen[6][3] == -1
    assert seen[7][1] == [1, 2, 6, 7]
    assert seen[8][1] == [2, 3, 7, 8]


def test_near_tie_adoption():
    """A caller pick within 1e-4 relative of the minimum logit is adopted and
    the oracle continues from it; a pick further away is a mismatch."""
    d = 2
    k = np.array([[1.0, 0.0], [-3.0, 0.0], [-3.0 * (1 + 2e-5), 0.0], [5.0, 0.0], [0.5, 0.0], [0.7, 0.0]])
    q = np.tile([1.0, 0.0], (6, 1))
    v = np.eye(6, 2)
    for pick, adopted in ((1, True), (0, False)):
        st = OracleStream(d, 1, 5, 4)
        st.prefill(np.zeros((1, d)), np.zeros((1, d)))
        for t in range(3):
            st.step(q[t], k[t], v[t])
        _, info = st.step(q[3], k[3], v[3], pick=pick)
        assert info.oracle_pick == 2
        assert info.adopted == adopted and info.mismatch == (not adopted)
        assert st.skip() == ([1] if adopted else [2])


def test_rejects_bad_arguments():
    for args in [(4, 2, 5, 6, 0), (4, 2, 5, 0, 0), (4, -1, 5, 3, 0), (4, 2, 5, 4, 4), (0, 2, 5, 3, 0)]:
        with pytest.raises(ValueError):
            OracleStream(*args)
