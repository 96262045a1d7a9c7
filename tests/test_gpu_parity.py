"""Parity of the CUDA decode path (through the C ABI) with the CPU oracle.

Small shapes run every stream through every step; they span several
shared-memory stages, several CTAs per stream, ragged tails and every phase
boundary of Algorithm 1.  Tolerances: max |out - oracle| <= 2e-3 +
1e-2 |oracle|; skip sets bit-exact up to accepted near ties.
"""
from dataclasses import replace

import pytest
import torch

from ar_image_gen_gb300.synth import WORKLOADS, Workload
from tests.parity import run_parity

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    from __graft_entry__ import build
    build()


def small(name, L_p, N_r, N_att, sink=0, grid=10, heads=4, batch=1, d=128, dtype="bf16", seed=7):
    return Workload(name, 1, heads, d, dtype, L_p, grid, N_r, N_att, sink, batch, seed)


def test_tiny_workload_full_trace():
    """Tiny workload (fp32, head_dim 64, L_p 16, 8x8 grid, N_r 32, N_att 8):
    every stream, every one of the 64 steps."""
    rep = run_parity(WORKLOADS["tiny"])
    assert rep.ok, rep.summary()
    assert rep.steps == 64 and rep.selections == 4 * (32 - 8)


CASES = {
    # name: (workload, steps, forced splits)
    "basic": (small("basic", 64, 40, 9, grid=10), 100, 0),
    "ragged-split3": (small("ragged", 37, 71, 13, grid=13, heads=5), 150, 3),
    "sink4": (small("sink4", 20, 64, 12, sink=4, grid=12, heads=6), 130, 0),
    "sink4-split2": (small("sink4s", 20, 64, 12, sink=4, grid=12, heads=6), 130, 2),
    "dense-split3": (small("dense", 16, 80, 80, grid=9), 80, 3),
    "sliding": (small("sliding", 16, 50, 50, grid=11), 120, 0),
    "streaming-sink4": (small("streaming", 16, 30, 30, sink=4, grid=9), 80, 0),
    "n_att-1": (small("natt1", 8, 20, 1, grid=8, heads=3), 50, 0),
    "empty-prompt": (small("noprompt", 0, 30, 5, grid=9, heads=3), 70, 0),
    "long-prompt-split2": (small("longprompt", 100, 40, 8, grid=10), 90, 2),
    "bf16-d64": (small("d64", 16, 40, 8, grid=10, d=64), 90, 0),
    "f32-d128": (small("f32d128", 16, 40, 8, grid=10, dtype="f32"), 90, 0),
    "f32-d64-split4": (small("f32d64", 16, 40, 8, grid=10, d=64, dtype="f32"), 90, 4),
    "many-splits": (small("split7", 16, 40, 8, grid=10), 90, 7),
    "window-wider-than-a-stage-list": (small("wide", 8, 300, 260, grid=18, heads=2), 324, 0),
}


def test_window_wider_than_the_register_mask():
    """A window of 8400 entries: once the window passes 8192 entries (256
    mask words, more than a warp keeps in registers) the kernel reads the
    mask words from global memory while it counts and lists the attended
    offsets.  Every step of a stream pair through the whole selection phase
    (N_att 8200: 200 selections per stream, all past 8192 entries) into
    eviction; masks checked every 400 steps and at the end."""
    wl = small("maskmem", 4, 8400, 8200, grid=92, heads=2, d=64)
    rep = run_parity(wl, steps=8450, mask_every=400)
    assert rep.ok, rep.summary()
    assert rep.steps == 8450 and rep.selections == 2 * (8400 - 8200)


def test_largest_window_is_accepted():
    """N_r - sink = 65536 is the largest window (offsets are 16-bit in the
    kernel's item lists); one entry more is rejected."""
    from ar_image_gen_gb300 import dsa

    code, h = dsa.dsa_create(2, 64, 4, 65536, 8, 0)
    assert code == dsa.DSA_OK
    assert dsa.dsa_destroy(h) == dsa.DSA_OK
    code, h = dsa.dsa_create(2, 64, 4, 65540, 8, 4)
    assert code == dsa.DSA_OK
    assert dsa.dsa_destroy(h) == dsa.DSA_OK
    code, h = dsa.dsa_create(2, 64, 4, 65537, 8, 0)
    assert code == dsa.DSA_ERR_ARG


@pytest.mark.parametrize("name", list(CASES))
def test_small_parity(name):
    wl, steps, splits = CASES[name]
    rep = run_parity(wl, steps=steps, splits=splits)
    assert rep.ok, rep.summary()
    assert rep.steps == steps


# Every launch pipeline forced on cases that reach their limits: ragged
# splits, the sink fill, dense runs, fp32 rows of 1 KB (six-row stages with
# 6 KB stages) and windows longer than one item's row list (256 rows with
# 6 KB stages); pipelines 3 and 4 run three stages per warp.
PIPE_CASES = ["ragged-split3", "sink4", "dense-split3", "f32-d128", "f32-d64-split4", "bf16-d64",
              "window-wider-than-a-stage-list", "long-prompt-split2"]


@pytest.mark.parametrize("pipeline", [1, 2, 3, 4])
@pytest.mark.parametrize("name", PIPE_CASES)
def test_small_parity_each_pipeline(name, pipeline):
    wl, steps, splits = CASES[name]
    rep = run_parity(wl, steps=steps, splits=splits, pipeline=pipeline)
    assert rep.ok, rep.summary()
    assert rep.steps == steps


def test_pipeline_choice_is_reported():
    """The automatic plan, from the launch cost model fitted to measured
    launch times: the steady-state plans of the workloads where the earlier
    rule-based choice was measurably slower, the dense setting of stress-s95,
    small cases where the three-stage pipelines keep streams unsplit, and
    the pipeline knob."""
    from ar_image_gen_gb300.dsa import DSA
    from ar_image_gen_gb300.synth import WORKLOADS

    def steady(name, dtype):
        wl = WORKLOADS[name]
        h = DSA(wl.streams, wl.head_dim, wl.L_p, wl.N_r, wl.N_att, wl.sink, dtype)
        p = h.plan(wl.L_dec - 1)
        h.close()
        return p.pipeline, p.nsplit

    # stress-s95, bf16: unsplit (about 84 us per launch on GB300) rather than
    # shape 1 in two pieces (91 us)
    pipe, ns = steady("stress-s95", "bf16")
    assert ns == 1 and pipe in (1, 3), (pipe, ns)
    # sweep512-s75, bf16: three stages unsplit (54 us) rather than shape 1 in
    # two pieces (61 us)
    assert steady("sweep512-s75", "bf16") == (3, 1)
    # lumina-s90-b54, FP8 rows: two stages of shape 0 unsplit (36 us) rather
    # than three stages (52 us)
    assert steady("lumina-s90-b54", "fp8e4m3") == (1, 1)
    # stress-s95's dense setting (2048 streams of about 8190 rows), FP8 rows:
    # three stages in 16-17 pieces (645 us) rather than two stages of shape 0
    # (806 us)
    wl = WORKLOADS["stress-s95"].dense()
    h = DSA(wl.streams, wl.head_dim, wl.L_p, wl.N_r, wl.N_att, wl.sink, "fp8e4m3")
    p = h.plan(wl.L_dec - 1)
    h.close()
    assert p.pipeline == 3 and p.nsplit == 17, (p.pipeline, p.nsplit)

    sms = torch.cuda.get_device_properties(0).multi_processor_count
    # streams that would be split in two to fill the two-stage grid fit one
    # round of the three-stage grid (8 warps per SM) unsplit: no merge launch
    h = DSA(6 * sms, 128, 64, 288, 29, 0, "bf16")
    p = h.plan(400)
    assert (p.pipeline, p.nsplit) == (3, 1), (p.pipeline, p.nsplit)
    h.set_pipeline(2)
    assert h.plan(400).pipeline == 2
    h.set_pipeline(0)
    assert h.plan(400).pipeline == 3
    h.set_splits(3)
    assert h.plan(400).nsplit == 3
    h.close()
    # a longer stream (164 rows), which the automatic two-stage plans split
    # in two, stays one item with three stages for bf16 rows; FP8 rows, whose
    # warps are bound by their own work, take the two pieces, merged inside
    # the CTA (no merge launch)
    h = DSA(6 * sms, 128, 64, 288, 100, 0, "bf16")
    p = h.plan(400)
    assert (p.pipeline, p.nsplit) == (3, 1), (p.pipeline, p.nsplit)
    h.close()
    h = DSA(6 * sms, 128, 64, 288, 100, 0, "fp8e4m3")
    p = h.plan(400)
    assert p.nsplit == 2 and p.cta_merge == 1, (p.pipeline, p.nsplit, p.cta_merge)
    h.set_merge(1)  # with the merge launch's cost the plan stays unsplit
    assert h.plan(400).nsplit == 1
    h.close()
    # 512 streams of 269 rows: three stages in two pieces (one round) for
    # bf16 rows; FP8 rows, bound by their stage waits, take the two-stage
    # plan's shorter pieces
    h = DSA(512, 128, 64, 2048, 205, 0, "bf16")
    p = h.plan(3000)
    assert p.pipeline in (3, 4) and p.nsplit == 2 and p.cta_merge == 1, (p.pipeline, p.nsplit, p.cta_merge)
    h.close()
    h = DSA(512, 128, 64, 2048, 205, 0, "fp8e4m3")
    p = h.plan(3000)
    assert p.pipeline in (1, 2) and p.nsplit > 1, (p.pipeline, p.nsplit)
    h.close()


@pytest.mark.parametrize("pipeline", [1, 2, 3, 4])
def test_split_count_does_not_change_the_result(pipeline):
    """The argmin is a total order on (logit, offset), and each logit is
    computed by the same lanes whatever the split or the pipeline shape:
    selections are identical across split counts and shapes and outputs
    agree to rounding."""
    from ar_image_gen_gb300.dsa import DSA
    from ar_image_gen_gb300.synth import TraceGen

    wl = small("splits", 48, 64, 10, grid=10, heads=8)
    gen = TraceGen(wl, device="cuda")
    Kp, Vp = gen.prompt()
    results = []
    for ns in (1, 2, 5):
        h = DSA(wl.streams, 128, wl.L_p, wl.N_r, wl.N_att, 0, "bf16")
        h.set_pipeline(pipeline)
        h.set_splits(ns)
        h.prefill(Kp, Vp)
        out = torch.empty((wl.streams, 128), dtype=torch.bfloat16, device="cuda")
        outs = []
        for t in range(100):
            q, k, v = gen.step(t)
            h.decode_step(q, k, v, out)
            outs.append(out.float().clone())
        results.append((torch.stack(outs), h.skip_mask()))
        assert h.sync_status() == 0
        h.close()
    for o, m in results[1:]:
        assert (m == results[0][1]).all()
        assert torch.allclose(o, results[0][0], atol=2e-2, rtol=2e-2)


@pytest.mark.parametrize("splits", [0, 3])
def test_interleaved_handles_on_one_stream(splits):
    """Several handles (layers) stepped round-robin on one stream, as a model
    decodes: each launch may read its own state before it waits for the
    previous launch (another handle), so every layer is checked against its
    own oracle at every step."""
    import numpy as np

    from ar_image_gen_gb300.dsa import DSA
    from ar_image_gen_gb300.synth import TraceGen
    from oracle.oracle import OracleBatch

    wl = small("interleave", 40, 48, 10, grid=9, heads=6)
    S, d = wl.streams, wl.head_dim
    layers = []
    for layer in range(3):
        gen = TraceGen(wl, layer=layer, device="cuda")
        h = DSA(S, d, wl.L_p, wl.N_r, wl.N_att, 0, "bf16")
        if splits:
            h.set_splits(splits)
        K, V = gen.prompt()
        h.prefill(K, V)
        orc = OracleBatch(S, d, wl.L_p, wl.N_r, wl.N_att, 0)
        orc.prefill(K.double().cpu().numpy(), V.double().cpu().numpy())
        layers.append((gen, h, orc, torch.empty((S, d), dtype=torch.bfloat16, device="cuda")))
    for t in range(wl.L_dec):
        steps = [gen.step(t) for gen, _, _, _ in layers]
        for (gen, h, orc, out), (q, k, v) in zip(layers, steps):  # decode launches back to back
            h.decode_step(q, k, v, out)
        torch.cuda.synchronize()
        for (gen, h, orc, out), (q, k, v) in zip(layers, steps):
            sel = h.last_selection()
            picks = np.array([t - r if r >= 0 else -1 for r in sel], dtype=np.int32)
            ref, infos = orc.step(q.double().cpu().numpy(), k.double().cpu().numpy(), v.double().cpu().numpy(),
                                  picks=picks)
            got = out.double().cpu().numpy()
            assert (np.abs(got - ref) <= 2e-3 + 1e-2 * np.abs(ref)).all(), f"t={t}"
            for i, info in enumerate(infos):
                assert not info.mismatch and info.selected == picks[i], f"t={t} stream {i}"
    for gen, h, orc, out in layers:
        assert h.sync_status() == 0
        h.close()


@pytest.mark.parametrize("sink,N_r", [(0, 90), (0, 40), (4, 40)])
def test_step_jump_equals_decoding_zero_rows(sink, N_r):
    """dsa_debug_set_step on a handle that never selects (N_att == N_r): the
    jump to step t0 leaves the state a decode of zero rows up to t0 would
    leave, so later steps match the oracle fed zero k / v rows for steps
    0 .. t0 - 1.  N_r = 90 keeps every entry (dense); N_r = 40 evicts, so
    the zero rows leave the window as real steps replace them; with sinks
    the jumped-over sink rows are zero too."""
    import numpy as np

    from ar_image_gen_gb300.dsa import DSA
    from ar_image_gen_gb300.synth import TraceGen
    from oracle.oracle import OracleBatch

    wl = small("jump", 24, N_r, N_r, sink=sink, grid=9, heads=5)
    S, d, t0 = wl.streams, wl.head_dim, 30
    gen = TraceGen(wl, device="cuda")
    K, V = gen.prompt()
    h = DSA(S, d, wl.L_p, wl.N_r, wl.N_att, sink, "bf16")
    h.prefill(K, V)
    h.debug_set_step(t0)
    assert h.t == t0
    orc = OracleBatch(S, d, wl.L_p, wl.N_r, wl.N_att, sink)
    orc.prefill(K.double().cpu().numpy(), V.double().cpu().numpy())
    zero = np.zeros((S, d))
    for _ in range(t0):
        orc.step(zero, zero, zero)
    out = torch.empty((S, d), dtype=torch.bfloat16, device="cuda")
    for t in range(t0, wl.L_dec):
        q, k, v = gen.step(t)
        h.decode_step(q, k, v, out)
        ref, _ = orc.step(q.double().cpu().numpy(), k.double().cpu().numpy(), v.double().cpu().numpy())
        got = out.double().cpu().numpy()
        assert (np.abs(got - ref) <= 2e-3 + 1e-2 * np.abs(ref)).all(), f"t={t}"
    assert h.sync_status() == 0
    h.close()


def test_step_jump_is_refused_where_it_does_not_apply():
    from ar_image_gen_gb300 import dsa
    from ar_image_gen_gb300.dsa import DSA, DSAError

    wl = small("jumpno", 8, 40, 9, grid=8, heads=2)
    K = torch.zeros((2, 8, 128), dtype=torch.bfloat16, device="cuda")
    h = DSA(2, 128, 8, 40, 9, 0, "bf16")  # selects: N_att < N_r
    h.prefill(K, K)
    with pytest.raises(DSAError) as e:
        h.debug_set_step(10)
    assert e.value.code == dsa.DSA_ERR_ARG
    h.close()
    h = DSA(2, 128, 8, 40, 40, 0, "bf16")
    with pytest.raises(DSAError) as e:  # before prefill
        h.debug_set_step(10)
    assert e.value.code == dsa.DSA_ERR_STATE
    h.prefill(K, K)
    q = torch.zeros((2, 128), dtype=torch.bfloat16, device="cuda")
    out = torch.empty_like(q)
    h.decode_step(q, q, q, out)
    with pytest.raises(DSAError) as e:  # not at step 0
        h.debug_set_step(10)
    assert e.value.code == dsa.DSA_ERR_STATE
    assert h.sync_status() == 0
    h.close()


def test_steady_state_with_a_list_slice_too_long_to_prefetch():
    """1024 rows per stream (a one-row prompt and 1023 attended decode rows)
    in two pieces of 512 (8 KB stages forced): the second piece's decode
    ranks start at 511 (odd), so its slice of the stored offset list,
    counted from the even rank below, is 513 entries, one more than the
    kernel prefetches, and the plan lists those steps' offsets from the
    skip mask as before the steady state.  Every step through selection,
    the step that stores the list and 60 steady-state steps against the
    oracle."""
    wl = small("longslice", 1, 1100, 1023, grid=35, heads=2, d=64)
    rep = run_parity(wl, steps=1160, splits=2, pipeline=1, mask_every=100)
    assert rep.ok, rep.summary()
    assert rep.selections == 2 * (1100 - 1023)


@pytest.mark.parametrize("pipeline", [1, 2, 3, 4])
@pytest.mark.parametrize("dtype,d,splits", [("bf16", 128, 2), ("bf16", 64, 4), ("fp8e4m3", 128, 4), ("f32", 128, 2)])
def test_cta_merge_matches_the_merge_launch(pipeline, dtype, d, splits):
    """Split streams combined inside the decode launch (the pieces on warps
    of one CTA, piece 0 combining them through shared memory) and by the
    merge launch: outputs, selections and skip masks identical bit for bit,
    step after step through the sink fill, selection and eviction; ragged
    pieces (the prompt and the window do not divide evenly)."""
    from ar_image_gen_gb300.dsa import DSA
    from ar_image_gen_gb300.synth import TraceGen

    wl = replace(small("ctamerge", 37, 60, 14, sink=2, grid=10, heads=6, d=d), dtype=dtype)
    gen = TraceGen(wl, device="cuda")
    Kp, Vp = gen.prompt()
    hs = []
    for mode in (0, 1):
        h = DSA(wl.streams, d, wl.L_p, wl.N_r, wl.N_att, wl.sink, dtype)
        h.set_pipeline(pipeline)
        h.set_splits(splits)
        h.set_merge(mode)
        if dtype == "fp8e4m3":
            h.set_kv_scales(*gen.kv_scales())
        h.prefill(Kp, Vp)
        hs.append(h)
    io = torch.float32 if dtype == "f32" else torch.bfloat16
    outs = [torch.empty((wl.streams, d), dtype=io, device="cuda") for _ in hs]
    merged_inside = 0
    for t in range(wl.L_dec):
        q, k, v = gen.step(t)
        pl = hs[0].plan(t)
        merged_inside += pl.cta_merge
        assert hs[1].plan(t).cta_merge == 0
        for h, o in zip(hs, outs):
            h.decode_step(q, k, v, o)
        assert torch.equal(outs[0], outs[1]), f"t={t}: outputs differ"
        if t % 10 == 9 or t == wl.L_dec - 1:
            assert (hs[0].skip_mask() == hs[1].skip_mask()).all(), f"t={t}: skip masks differ"
            assert (hs[0].last_selection() == hs[1].last_selection()).all(), f"t={t}: selections differ"
    for h in hs:
        assert h.sync_status() == 0
        h.close()
    if pipeline == 3:  # three stages per warp (two CTAs per SM) leave room for the exchange area
        assert merged_inside == wl.L_dec
