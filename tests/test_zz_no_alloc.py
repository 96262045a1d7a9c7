"""The allocation-free decode step (dsa_decode_step_noalloc) through the C
ABI, on consecutive calls, against the fp64 oracle and against the
handle-based step.

It is for callers that cannot allocate device memory while decoding (an
engine that reserves all memory for its own KV arena, or a decode loop that
must not call the allocator).  The tests allocate the caller-owned state
with torch, as such a caller would from its own arena, and check step after
step that the outputs are within the parity tolerance of the oracle, that
the selections and skip masks equal the oracle's (near ties adopted as in
the other parity tests) and equal the handle path's, and that the static
status word reads back clean.  This file is collected last so that a
failure here stops a `-x` run only after every other test ran; it also
passes on its own in a fresh process.
"""
import numpy as np
import pytest
import torch

from tests.parity import ATOL, RTOL, mask_offsets

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dsa():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    from __graft_entry__ import build
    build()
    from ar_image_gen_gb300 import dsa as mod
    return mod


CASES = {
    # name: (heads, head_dim, dtype, L_p, grid, N_r, N_att, sink); a prompt of
    # 200 rows splits the few streams over several work items, so the static
    # scratch holds split partials
    "bf16-d128-split": (8, 128, "bf16", 200, 6, 24, 9, 0),
    "bf16-d128-sink4": (8, 128, "bf16", 200, 6, 24, 9, 4),
    "bf16-d64": (6, 64, "bf16", 40, 7, 20, 6, 0),
    "f32-d64": (4, 64, "f32", 16, 8, 32, 8, 0),
    "f32-d128-dense": (5, 128, "f32", 12, 7, 49, 49, 0),
}


@pytest.mark.parametrize("name", list(CASES))
def test_noalloc_steps_match_the_oracle_and_the_handle_path(dsa, name):
    from ar_image_gen_gb300.synth import TraceGen, Workload, torch_dtype
    from oracle.oracle import OracleBatch

    heads, d, dtype, L_p, grid, N_r, N_att, sink = CASES[name]
    wl = Workload("noalloc-" + name, 1, heads, d, dtype, L_p, grid, N_r, N_att, sink, 1, 31)
    S = wl.streams
    tdt = torch_dtype(dtype)
    gen = TraceGen(wl, device="cuda")
    K, V = gen.prompt()
    h = dsa.DSA(S, d, L_p, N_r, N_att, sink, dtype)
    h.prefill(K, V)
    orc = OracleBatch(S, d, L_p, N_r, N_att, sink)
    orc.prefill(K.cpu().double().numpy(), V.cpu().double().numpy())

    # caller-owned state, laid out as dsa_prefill builds it
    Lcap, R = L_p + sink, N_r - sink
    prefix = torch.zeros((S, Lcap, 2, d), dtype=tdt, device="cuda")
    prefix[:, :L_p, 0] = K
    prefix[:, :L_p, 1] = V
    ring = torch.empty((S, R, 2, d), dtype=tdt, device="cuda")
    mask = torch.zeros((S, (R + 31) // 32), dtype=torch.int32, device="cuda")
    last_sel = torch.full((S,), -1, dtype=torch.int32, device="cuda")
    out_h = torch.empty((S, d), dtype=tdt, device="cuda")
    out_n = torch.empty_like(out_h)
    code = dsa.DTYPES[dtype]
    split_steps = selections = 0
    for t in range(wl.L_dec):  # consecutive calls through every phase
        q, k, v = gen.step(t)
        h.decode_step(q, k, v, out_h)
        split_steps += h.plan(t).nsplit > 1
        last_sel.fill_(-1)
        rc = dsa.dsa_decode_step_noalloc(S, d, L_p, N_r, N_att, sink, code, t, prefix, ring, mask, last_sel,
                                         q, k, v, out_n)
        assert rc == dsa.DSA_OK, dsa.dsa_last_error()
        sel = last_sel.cpu().numpy()
        tin = t - sink
        picks = np.array([tin - r if r >= 0 else -1 for r in sel], dtype=np.int32)
        ref, infos = orc.step(q.cpu().double().numpy(), k.cpu().double().numpy(), v.cpu().double().numpy(),
                              picks=picks)
        got = out_n.cpu().double().numpy()
        err = np.abs(got - ref)
        assert (err <= ATOL + RTOL * np.abs(ref)).all(), f"t={t}: max err vs oracle {err.max():.3e}"
        for i, info in enumerate(infos):
            assert not info.mismatch and info.selected == picks[i], f"t={t} stream {i}: selection"
            selections += info.oracle_pick >= 0
        got_mask = mask.cpu().numpy().view("uint32")
        for s in range(S):
            want = set() if tin < 0 else {tin - j for j in orc.streams[s].skip()}
            assert mask_offsets(got_mask[s]) == want, f"t={t} stream {s}: skip set"
        assert (got_mask == h.skip_mask()).all(), f"t={t}: skip masks differ from the handle path"
        assert torch.allclose(out_n.float(), out_h.float(), atol=ATOL, rtol=RTOL), f"t={t}: handle path"
    assert dsa.dsa_decode_step_noalloc_status() == dsa.DSA_OK
    assert h.sync_status() == dsa.DSA_OK
    if N_att < N_r:
        assert selections > 0
    if name.endswith("split"):
        assert split_steps > 0  # the static scratch held split partials
    h.close()


def test_noalloc_refuses_what_does_not_fit_before_reading_pointers(dsa):
    """3000 streams with a 1200-row prompt run in at least three work items
    each (no item holds more than 512 rows): 9000 items of split partials
    need more than the static 4 MiB.  The call is refused on the size before
    any pointer is looked at; the pointers here are all NULL, so a call that
    got past the size check would stop at the pointer check and launch
    nothing."""
    rc = dsa.dsa_decode_step_noalloc(3000, 128, 1200, 64, 8, 0, dsa.DSA_BF16, 0, None, None, None, None,
                                     None, None, None, None)
    assert rc == dsa.DSA_ERR_ARG and "scratch" in dsa.dsa_last_error()
    # without splits only the status word is needed: the same streams with a
    # short prompt pass the size check and stop at the NULL pointers
    rc = dsa.dsa_decode_step_noalloc(3000, 128, 64, 288, 29, 0, dsa.DSA_BF16, 0, None, None, None, None,
                                     None, None, None, None)
    assert rc == dsa.DSA_ERR_ARG and "non-NULL" in dsa.dsa_last_error()
    rc = dsa.dsa_decode_step_noalloc(8, 128, 64, 288, 29, 0, dsa.DSA_BF16, -1, None, None, None, None,
                                     None, None, None, None)
    assert rc == dsa.DSA_ERR_ARG
