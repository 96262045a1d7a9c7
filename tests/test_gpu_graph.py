"""Graph mode (dsa_set_graph_mode): steady-state decode steps captured once
in a CUDA graph and replayed step after step, against handles stepped on
the host with the same inputs: outputs and skip masks bit for bit, and the
device step counter advances once per replay."""
import numpy as np
import pytest
import torch

from ar_image_gen_gb300.synth import TraceGen, Workload

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    from __graft_entry__ import build
    build()


@pytest.mark.parametrize("sink,splits", [(0, 0), (4, 3), (0, 2)])
def test_graph_replay_matches_host_steps(sink, splits):
    from ar_image_gen_gb300.dsa import DSA, DSA_OK

    wl = Workload("graph", 2, 4, 128, "bf16", 16, 12, 40, 9, sink, 2, 17)
    S, d = wl.streams, wl.head_dim
    gens = [TraceGen(wl, layer=l, device="cuda") for l in range(wl.layers)]
    A = [DSA(S, d, wl.L_p, wl.N_r, wl.N_att, sink) for _ in range(wl.layers)]
    B = [DSA(S, d, wl.L_p, wl.N_r, wl.N_att, sink) for _ in range(wl.layers)]
    for l in range(wl.layers):
        Kp, Vp = gens[l].prompt()
        for h in (A[l], B[l]):
            if splits:
                h.set_splits(splits)
            h.prefill(Kp, Vp)
    outA = [torch.empty((S, d), dtype=torch.bfloat16, device="cuda") for _ in range(wl.layers)]
    outB = [torch.empty_like(outA[0]) for _ in range(wl.layers)]
    t0 = wl.N_r  # steady state from t - sink >= N_r - sink
    for t in range(t0):
        for l in range(wl.layers):
            q, k, v = gens[l].step(t)
            A[l].decode_step(q, k, v, outA[l])
            B[l].decode_step(q, k, v, outB[l])
    bufs = [[torch.empty((S, d), dtype=torch.bfloat16, device="cuda") for _ in range(3)] for _ in range(wl.layers)]
    for h in A:
        h.set_graph_mode(True)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        for l in range(wl.layers):
            A[l].decode_step(*bufs[l], outA[l])
    for h in A:
        h.sync_step()  # capture ran nothing: back to the device's step
        assert h.t == t0
    steps = wl.L_dec - t0
    for i in range(steps):
        t = t0 + i
        for l in range(wl.layers):
            q, k, v = gens[l].step(t)
            for dst, src in zip(bufs[l], (q, k, v)):
                dst.copy_(src)
            B[l].decode_step(q, k, v, outB[l])
        g.replay()
        torch.cuda.synchronize()
        for l in range(wl.layers):
            assert torch.equal(outA[l], outB[l]), f"layer {l}, step {t}"
        if i % 7 == 0 or i == steps - 1:
            for l in range(wl.layers):
                assert np.array_equal(A[l].skip_mask(), B[l].skip_mask())
    for l in range(wl.layers):
        A[l].sync_step()
        assert A[l].t == wl.L_dec and B[l].t == wl.L_dec
        assert A[l].sync_status() == DSA_OK and B[l].sync_status() == DSA_OK
    for h in A + B:
        h.close()


def test_graph_mode_refuses_steps_before_the_steady_state():
    from ar_image_gen_gb300.dsa import DSA, DSAError

    wl = Workload("graph", 1, 2, 128, "bf16", 8, 8, 20, 5, 0, 1, 19)
    gen = TraceGen(wl, device="cuda")
    h = DSA(wl.streams, wl.head_dim, wl.L_p, wl.N_r, wl.N_att)
    Kp, Vp = gen.prompt()
    h.prefill(Kp, Vp)
    h.set_graph_mode(True)
    q, k, v = gen.step(0)
    out = torch.empty_like(q)
    with pytest.raises(DSAError):
        h.decode_step(q, k, v, out)
    h.set_graph_mode(False)
    h.decode_step(q, k, v, out)
    assert h.t == 1
    h.close()
