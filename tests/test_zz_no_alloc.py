"""The allocation-free decode step (dsa_decode_step_noalloc) against the
handle-based one, through the C ABI, on consecutive calls.

It is for callers that cannot allocate device memory while decoding (an
engine that reserves all memory for its own KV arena, or a decode loop that
must not call the allocator).  The test allocates the caller-owned state
with torch, as such a caller would from its own arena, and checks that both
entry points produce the same outputs and skip masks step after step.  This
file is collected last so that a failure here stops a `-x` run only after
every other test ran; it also passes on its own in a fresh process.
"""
import pytest
import torch

pytestmark = pytest.mark.gpu

ATOL, RTOL = 2e-3, 1e-2


@pytest.fixture(scope="module")
def dsa():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    from __graft_entry__ import build
    build()
    from ar_image_gen_gb300 import dsa as mod
    return mod


@pytest.mark.parametrize("sink", [0, 4])
def test_noalloc_step_matches_handle_step(dsa, sink):
    from ar_image_gen_gb300.synth import TraceGen, Workload

    # long enough prompt that streams split over several work items, so the
    # static scratch (partials, tickets) is used
    wl = Workload("noalloc", 1, 8, 128, "bf16", 200, 6, 24, 9, sink, 1, 31)
    S, d = wl.streams, wl.head_dim
    gen = TraceGen(wl, device="cuda")
    K, V = gen.prompt()
    h = dsa.DSA(S, d, wl.L_p, wl.N_r, wl.N_att, sink, "bf16")
    h.prefill(K, V)
    assert h.plan(0).nsplit > 1

    Lcap, R = wl.L_p + sink, wl.N_r - sink
    prefix = torch.zeros((S, Lcap, 2, d), dtype=torch.bfloat16, device="cuda")
    prefix[:, : wl.L_p, 0] = K
    prefix[:, : wl.L_p, 1] = V
    ring = torch.empty((S, R, 2, d), dtype=torch.bfloat16, device="cuda")
    mask = torch.zeros((S, (R + 31) // 32), dtype=torch.int32, device="cuda")
    last_sel = torch.full((S,), -1, dtype=torch.int32, device="cuda")
    out_h = torch.empty((S, d), dtype=torch.bfloat16, device="cuda")
    out_n = torch.empty_like(out_h)
    for t in range(wl.L_dec):  # consecutive calls through all three phases
        q, k, v = gen.step(t)
        h.decode_step(q, k, v, out_h)
        rc = dsa.dsa_decode_step_noalloc(S, d, wl.L_p, wl.N_r, wl.N_att, sink, dsa.DSA_BF16, t, prefix, ring,
                                         mask, last_sel, q, k, v, out_n)
        assert rc == dsa.DSA_OK, dsa.dsa_last_error()
        ref = out_h.double()
        err = (out_n.double() - ref).abs()
        assert (err <= ATOL + RTOL * ref.abs()).all(), f"t={t}: max err {err.max().item():.3e}"
        got_mask = mask.cpu().numpy().view("uint32")
        assert (got_mask == h.skip_mask()).all(), f"t={t}: skip masks differ"
    assert h.sync_status() == dsa.DSA_OK
    h.close()


def test_noalloc_rejects_what_does_not_fit(dsa):
    # 20000 streams need more split scratch than the static array holds
    dummy = torch.zeros(64, dtype=torch.int32, device="cuda")
    rc = dsa.dsa_decode_step_noalloc(20000, 128, 64, 288, 29, 0, dsa.DSA_BF16, 0, dummy, dummy, dummy, dummy,
                                     dummy, dummy, dummy, dummy)
    assert rc == dsa.DSA_ERR_ARG and "scratch" in dsa.dsa_last_error()
    rc = dsa.dsa_decode_step_noalloc(8, 128, 64, 288, 29, 0, dsa.DSA_BF16, -1, dummy, dummy, dummy, dummy,
                                     dummy, dummy, dummy, dummy)
    assert rc == dsa.DSA_ERR_ARG
