"""The attention diagnostics (include/dsa_diag.h) on the GPU against the
oracle's fp64 statement of them (section 3.4, Fig. 8 and Fig. 10).

Logits and weights are fp32 on the GPU (bf16 logits on the tensor cores, fp32
ones on FMAs; bf16 products exact, fp32 sums over at most 128 terms), so
masses and cosines agree with fp64 to a few 1e-6; the bound used is 2e-5
absolute.
"""
import numpy as np
import pytest
import torch

from ar_image_gen_gb300.synth import TraceGen, Workload
from oracle.oracle import diag_stream

pytestmark = pytest.mark.gpu
TOL = 2e-5


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    from __graft_entry__ import build
    build()


def trace(wl: Workload, layer: int = 0):
    """Dense trace of one layer: Q, Kd [S, L_dec, d], Kp [S, L_p, d] on the device."""
    gen = TraceGen(wl, layer=layer, device="cuda")
    Kp, _ = gen.prompt()
    qs, ks = [], []
    for t in range(wl.L_dec):
        q, k, _ = gen.step(t)
        qs.append(q)
        ks.append(k)
    return torch.stack(qs, 1).contiguous(), Kp, torch.stack(ks, 1).contiguous()


def oracle_means(Q, Kp, Kd, dists, heads):
    masses, vs, ds = [], [], []
    for s in heads:
        m, v, d = diag_stream(Q[s].double().cpu().numpy(), Kp[s].double().cpu().numpy() if Kp.shape[1] else
                              np.zeros((0, Q.shape[2])), Kd[s].double().cpu().numpy(), dists)
        masses.append(m)
        vs.append(v)
        ds.append(d)
    return np.stack(masses), np.mean(vs, 0), np.mean(ds, 0)


CASES = {
    "bf16-d128": (Workload("dg1", 1, 4, 128, "bf16", 16, 10, 100, 100, 0, 1, 3), [1, 2, 9, 10, 11, 20]),
    "f32-d64": (Workload("dg2", 1, 3, 64, "f32", 9, 8, 64, 64, 0, 1, 4), [1, 7, 8, 9, 30, 63]),
    "no-prompt": (Workload("dg3", 1, 2, 128, "bf16", 0, 7, 49, 49, 0, 1, 5), [1, 7]),
    "janus-layer": (Workload("dg4", 1, 32, 128, "bf16", 64, 24, 576, 576, 0, 1, 6), [1, 23, 24, 25, 48]),
    # bf16 logits run on the tensor cores in 128 x 128 tiles: a prompt longer
    # than one key tile, key tiles that straddle prompt and decoded keys,
    # and a ragged last query tile (289 = 2 x 128 + 33)
    "bf16-d64-long-prompt": (Workload("dg6", 1, 3, 64, "bf16", 200, 17, 289, 289, 0, 1, 8), [1, 16, 17, 18, 100]),
    "bf16-d128-ragged": (Workload("dg7", 1, 2, 128, "bf16", 37, 12, 144, 144, 0, 1, 9), [1, 11, 12, 13, 143]),
}


@pytest.mark.parametrize("name", list(CASES))
def test_parity_with_the_oracle(name):
    from ar_image_gen_gb300.dsa import diag_trace

    wl, dists = CASES[name]
    Q, Kp, Kd = trace(wl)
    S = wl.streams
    step = torch.zeros((S, wl.L_dec, 3), dtype=torch.float32, device="cuda")
    mass, vert, diag = diag_trace(Q, Kp, Kd, dists, step_mass=step)
    heads = range(S) if S <= 8 else [0, 5, 17, 31]
    om, ov, od = oracle_means(Q, Kp, Kd, dists, heads)
    got_step = step.double().cpu().numpy()
    assert np.abs(got_step[list(heads)] - om).max() <= TOL
    assert np.allclose(mass, got_step.reshape(-1, 3).mean(0), atol=1e-9)  # the mean is the mean of the steps
    assert abs(mass.sum() - 1) <= 1e-5
    if S <= 8:  # every head through the oracle: the means themselves
        assert np.abs(mass - om.reshape(-1, 3).mean(0)).max() <= TOL
        assert np.abs(vert - ov).max() <= TOL and np.abs(diag - od).max() <= TOL


def test_relative_position_trace_is_diagonal():
    """q_i = RoPE(u, i), k_j = RoPE(w, j): logits depend on i - j only, so the
    diagonal similarity is 1 (fp32 rounding aside) at every distance."""
    from ar_image_gen_gb300.dsa import diag_trace
    from ar_image_gen_gb300.synth import _rope

    g = torch.Generator(device="cuda").manual_seed(3)
    S, L_p, L_dec, d = 2, 5, 80, 128
    u = torch.randn((S, 1, d), generator=g, device="cuda")
    w = torch.randn((S, 1, d), generator=g, device="cuda")
    pos = torch.arange(L_dec, device="cuda") + L_p
    Q = _rope(u.expand(S, L_dec, d), pos[None, :]).float().contiguous()
    Kd = _rope(w.expand(S, L_dec, d), pos[None, :]).float().contiguous()
    Kp = torch.randn((S, L_p, d), generator=g, device="cuda")
    _, vert, diag = diag_trace(Q, Kp, Kd, [1, 3, 17])
    assert np.abs(diag - 1).max() <= 1e-5
    assert (vert < 1 - 1e-3).all()


def test_heads_split_over_chunks():
    """L_dec 4096 with L_p 64: 68 MB of weights per head, so 16 heads need two
    chunks of the 1 GiB scratch; heads on both sides match the oracle."""
    from ar_image_gen_gb300.dsa import diag_trace

    wl = Workload("dg5", 1, 16, 128, "bf16", 64, 64, 4096, 4096, 0, 1, 7)
    gen = TraceGen(wl, device="cuda")
    Kp, _ = gen.prompt()
    steps = [gen.step(t) for t in range(wl.L_dec)]
    Q = torch.stack([s[0] for s in steps], 1).contiguous()
    Kd = torch.stack([s[1] for s in steps], 1).contiguous()
    del steps
    step = torch.zeros((16, wl.L_dec, 3), dtype=torch.float32, device="cuda")
    mass, _, _ = diag_trace(Q, Kp, Kd, [64], step_mass=step)
    for s in (0, 15):
        om, _, _ = diag_stream(Q[s].double().cpu().numpy(), Kp[s].double().cpu().numpy(), Kd[s].double().cpu().numpy(),
                               [64])
        assert np.abs(step[s].double().cpu().numpy() - om).max() <= TOL
    assert np.allclose(mass, step.double().cpu().numpy().reshape(-1, 3).mean(0), atol=1e-9)
