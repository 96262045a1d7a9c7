"""The launch plan's host logic through the C ABI, without a GPU
(dsa_plan_query touches no device): Algorithm 1's per-step counts against
the fp64 oracle, the sizing of work items and grids on many shapes, the
cost model's choices for the workloads on GB300's occupancy, and argument
checks.

GB300 here: 152 SMs; the decode kernel keeps 3 / 4 / 2 / 2 CTAs per SM
resident under launch pipelines 1-4 (two 8 KB or 6 KB stages per warp, or
three), and the in-CTA merge of split streams fits every pipeline (the
occupancy the library queries on the device at dsa_create).
"""
import numpy as np
import pytest

from ar_image_gen_gb300.synth import WORKLOADS

SMS = 152
CTAS = [3, 4, 2, 2]
XM = [1, 1, 1, 1]
ELEM = {"bf16": 2, "f32": 4, "fp8e4m3": 1}
IO = {"bf16": 2, "f32": 4, "fp8e4m3": 2}
dsa = None  # the binding, once the library is built (fixture below)


@pytest.fixture(scope="module", autouse=True)
def library():
    global dsa
    from __graft_entry__ import build
    build()
    from ar_image_gen_gb300 import dsa as mod
    dsa = mod


def query(heads, d, L_p, N_r, N_att, sink, dtype, t, ctas=CTAS, xm=XM, sms=SMS):
    rc, p = dsa.dsa_plan_query(heads, d, L_p, N_r, N_att, sink, dsa.DTYPES[dtype], t, sms, ctas, xm)
    assert rc == dsa.DSA_OK, dsa.dsa_last_error()
    return p


@pytest.mark.parametrize("L_p,N_r,N_att,sink,steps", [
    (16, 32, 8, 0, 100),     # all three phases
    (20, 64, 12, 4, 150),    # sink fill first (Diagonal+sink4)
    (16, 40, 40, 0, 60),     # dense: never selects
    (8, 20, 1, 0, 50),       # N_att = 1: only the current token among the decode rows
    (0, 30, 5, 0, 70),       # no prompt
    (12, 24, 9, 3, 90),      # sinks with a small window
])
def test_step_counts_follow_the_oracle(L_p, N_r, N_att, sink, steps):
    """Every step's phase, inner step, attended row count and whether it
    selects, as the plan reports them, against the oracle's record of the
    same step (random inputs; the counts do not depend on the values)."""
    from oracle.oracle import OracleStream

    d = 4
    orc = OracleStream(d, L_p, N_r, N_att, sink)
    rng = np.random.default_rng(5)
    orc.prefill(rng.standard_normal((L_p, d)), rng.standard_normal((L_p, d)))
    for t in range(steps):
        _, info = orc.step(*rng.standard_normal((3, d)))
        p = query(3, 64, L_p, N_r, N_att, sink, "bf16", t)
        assert p.phase == info.phase, (t, p.phase, info.phase)
        assert p.t_inner == info.t_inner, t
        # the plan counts the current token of a sink step as a decode row,
        # the oracle as the prefix row it becomes
        assert p.n_prefix + p.n_decode == info.n_prefix + info.n_idx, t
        assert p.select == (1 if info.selected >= 0 else 0), t


def stage_rows(dtype, d, pipeline):
    return (8192 if (pipeline - 1) % 2 == 0 else 6144) // (2 * d * ELEM[dtype])


def test_items_and_grids_cover_every_row():
    """On many random shapes and steps: the pieces of a stream cover its
    rows with none empty, each a whole number of stages and within the item
    list; the grid fits one round of resident CTAs and runs the items in the
    fewest rounds; the bytes are the algorithmic count; the in-CTA merge is
    used exactly for 2 or 4 pieces where it fits."""
    rng = np.random.default_rng(11)
    dtypes = ["bf16", "f32", "fp8e4m3"]
    checked = set()
    for _ in range(600):
        dtype = dtypes[rng.integers(3)]
        d = [64, 128][rng.integers(2)]
        heads = int(rng.choice([1, 7, 64, 512, 1000, 2048, 3072, 9000]))
        L_p = int(rng.integers(0, 1200))
        N_r = int(rng.integers(2, 5000))
        N_att = int(rng.integers(1, N_r + 1))
        sink = int(rng.integers(0, min(5, N_att)))
        if sink and N_att <= sink:
            sink = 0
        t = int(rng.integers(0, 2 * N_r + 10))
        xm = [int(x) for x in rng.integers(0, 2, 4)]
        p = query(heads, d, L_p, N_r, N_att, sink, dtype, t, xm=xm)
        n = p.n_prefix + p.n_decode
        rows = stage_rows(dtype, d, p.pipeline)
        cap = (512 if (p.pipeline - 1) % 2 == 0 else 256) // rows * rows
        assert 1 <= p.pipeline <= 4 and CTAS[p.pipeline - 1] > 0
        assert p.chunk % rows == 0 and p.chunk <= cap
        assert p.nsplit * p.chunk >= n > (p.nsplit - 1) * p.chunk
        assert 1 <= p.grid <= SMS * CTAS[p.pipeline - 1]
        # the fewest rounds of items the resident warps allow, every item in
        # one of them, and no CTA without an item
        items = heads * p.nsplit
        rounds = -(-items // (SMS * CTAS[p.pipeline - 1] * 4))
        assert p.grid * 4 * rounds >= items > (p.grid - 1) * 4 * rounds
        De, Di = d * ELEM[dtype], d * IO[dtype]
        assert p.algo_bytes == heads * (2 * De * (n - 1) + 4 * Di + 2 * De)
        assert p.cta_merge == (1 if p.nsplit in (2, 4) and xm[p.pipeline - 1] else 0)
        checked.add((p.pipeline, min(p.nsplit, 3), p.cta_merge))
    assert len(checked) >= 8  # every pipeline, split and merge form was reached


def test_unavailable_pipelines_are_never_planned():
    for t in (0, 50, 400, 3000):
        for heads in (64, 2048, 8000):
            p = query(heads, 128, 64, 2048, 205, 0, "bf16", t, ctas=[3, 4, 0, 0])
            assert p.pipeline in (1, 2)
            p = query(heads, 128, 64, 2048, 205, 0, "fp8e4m3", t, ctas=[2, 0, 0, 0])
            assert p.pipeline == 1


def plan_of(name, dtype, dense=False):
    wl = WORKLOADS[name]
    if dense:
        wl = wl.dense()
    return query(wl.streams, wl.head_dim, wl.L_p, wl.N_r, wl.N_att, wl.sink, dtype, wl.L_dec - 1)


def test_plan_choices_on_gb300():
    """The cost model's choices on GB300's occupancy for the launches whose
    timings fixed it (the same choices the GPU plan test reads back from
    handles on the device)."""
    p = plan_of("stress-s95", "bf16")
    assert (p.pipeline, p.nsplit) == (3, 1)
    p = plan_of("sweep512-s75", "bf16")
    assert (p.pipeline, p.nsplit) == (3, 1)
    p = plan_of("lumina-s90-b54", "fp8e4m3")
    assert (p.pipeline, p.nsplit) == (1, 1)
    p = plan_of("stress-s95", "fp8e4m3", dense=True)
    assert (p.pipeline, p.nsplit, p.cta_merge) == (3, 17, 0)
    p = plan_of("lumina-s95-b16", "bf16")
    assert (p.pipeline, p.nsplit, p.cta_merge) == (3, 2, 1)
    p = plan_of("lumina-s95-b16", "fp8e4m3")
    assert (p.pipeline, p.nsplit, p.cta_merge) == (2, 4, 1)
    # without the in-CTA merge the same FP8 launch keeps three pieces
    wl = WORKLOADS["lumina-s95-b16"]
    p = query(wl.streams, wl.head_dim, wl.L_p, wl.N_r, wl.N_att, wl.sink, "fp8e4m3", wl.L_dec - 1,
              xm=[0, 0, 0, 0])
    assert (p.nsplit, p.cta_merge) == (3, 0)


def test_plan_query_rejects_bad_arguments():
    ok = dict(heads=8, head_dim=128, L_p=16, N_r=32, N_att=8, sink=0, dtype=dsa.DSA_BF16, t=0, sm_count=SMS)

    def call(ctas=CTAS, **kw):
        a = dict(ok, **kw)
        return dsa.dsa_plan_query(a["heads"], a["head_dim"], a["L_p"], a["N_r"], a["N_att"], a["sink"], a["dtype"],
                                  a["t"], a["sm_count"], ctas, XM)[0]

    assert call() == dsa.DSA_OK
    assert call(ctas=[0, 4, 2, 2]) == dsa.DSA_ERR_ARG
    assert call(sm_count=0) == dsa.DSA_ERR_ARG
    assert call(t=-1) == dsa.DSA_ERR_ARG
    assert call(head_dim=96) == dsa.DSA_ERR_ARG
    assert call(N_att=40) == dsa.DSA_ERR_ARG
    assert call(dtype=7) == dsa.DSA_ERR_ARG
