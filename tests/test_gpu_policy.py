"""The score-based eviction baselines (TOVA, H2O) on the GPU, through the C
ABI, against the fp64 oracle (oracle/policies.py) on the same seeded
grid-structured traces as the diagonal method.

Per step: outputs within max |out - oracle| <= 2e-3 + 1e-2 |oracle|; the
evicted position equal to the oracle's, except at a near tie, where the
oracle adopts the kernel's choice and continues from it; every few steps
the set of positions each stream's cache holds is compared exactly.
"""
from dataclasses import dataclass, field

import numpy as np
import pytest
import torch

from ar_image_gen_gb300.synth import TraceGen, Workload
from oracle.policies import PolicyStream
from tests.parity import ATOL, RTOL

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    from __graft_entry__ import build
    build()


@dataclass
class Report:
    steps: int = 0
    evictions: int = 0
    adopted: int = 0
    max_err: float = 0.0
    failures: list = field(default_factory=list)

    @property
    def ok(self):
        return not self.failures


def run_policy(wl: Workload, policy: str, steps: int, sample=None, check_every: int = 1, shape: int = 0,
               gen_device: str = "cuda") -> Report:
    """Runs `steps` steps of `policy` on the GPU and the sampled streams on
    the oracle.  Inputs are drawn on `gen_device`; the oracle's share is
    taken from host copies."""
    from ar_image_gen_gb300.dsa import DSA_OK, Policy

    gen = TraceGen(wl, device=gen_device)
    S, d = gen.S, wl.head_dim
    sample = list(range(S)) if sample is None else list(sample)
    idx = torch.tensor(sample)
    h = Policy(S, d, wl.L_p, wl.N_att, policy, wl.dtype)
    if shape:
        h.set_shape(shape)
    Kp, Vp = gen.prompt()
    h.prefill(Kp.to("cuda"), Vp.to("cuda"))
    orc = [PolicyStream(d, wl.L_p, wl.N_att, policy) for _ in sample]
    Kh, Vh = Kp.cpu()[idx].double().numpy(), Vp.cpu()[idx].double().numpy()
    for i, o in enumerate(orc):
        o.prefill(Kh[i], Vh[i])
    out = torch.empty((S, d), dtype=Kp.dtype, device="cuda")
    rep = Report()
    for t in range(steps):
        qkv = gen.step(t)
        q, k, v = (x.to("cuda") for x in qkv)
        h.decode_step(q, k, v, out)
        ev = h.last_eviction()  # synchronizes
        qh, kh, vh = (x.cpu()[idx].double().numpy() for x in qkv)
        got = out.cpu()[idx].double().numpy()
        for i, s in enumerate(sample):
            ref, info = orc[i].step(qh[i], kh[i], vh[i], pick=int(ev[s]))
            err = np.abs(got[i] - ref)
            rep.max_err = max(rep.max_err, float(err.max()))
            if (err > ATOL + RTOL * np.abs(ref)).any():
                rep.failures.append(("out", t, s, float(err.max())))
            if info["oracle_pick"] >= 0:
                rep.evictions += 1
            rep.adopted += info["adopted"]
            if info["mismatch"] or info["evicted"] != int(ev[s]):
                rep.failures.append(("evict", t, s, int(ev[s]), info["oracle_pick"], info["min_score"],
                                     info["pick_score"]))
        if t % check_every == check_every - 1 or t == steps - 1:
            pos = h.positions()
            for i, s in enumerate(sample):
                have = sorted(int(x) for x in pos[s] if x >= 0)
                if have != orc[i].positions():
                    rep.failures.append(("cache", t, s, have[:8], orc[i].positions()[:8]))
        rep.steps += 1
        if len(rep.failures) > 10:
            break
    st = h.sync_status()
    if st != DSA_OK:
        rep.failures.append(("status", st))
    h.close()
    return rep


def small(name, L_p, N_att, grid=10, heads=4, batch=1, d=128, dtype="bf16", seed=13):
    return Workload(name, 1, heads, d, dtype, L_p, grid, N_att, N_att, 0, batch, seed)


CASES = {
    # name: (workload, policy, steps)
    "tova-bf16": (small("tova", 16, 9), "tova", 100),
    "tova-f32-d64": (small("tovaf", 12, 7, d=64, dtype="f32"), "tova", 90),
    "tova-n_att-1": (small("tova1", 8, 1, grid=8, heads=3), "tova", 50),
    "tova-empty-prompt": (small("tova0", 0, 6, grid=9, heads=3), "tova", 70),
    "tova-bf16-d64-long-window": (small("tovaw", 20, 40, grid=11, heads=2, d=64), "tova", 121),
    "h2o-bf16": (small("h2o", 16, 9), "h2o", 100),
    "h2o-f32-d64": (small("h2of", 12, 8, d=64, dtype="f32"), "h2o", 90),
    "h2o-n_att-1": (small("h2o1", 8, 1, grid=8, heads=3), "h2o", 50),
    "h2o-n_att-2": (small("h2o2", 8, 2, grid=8, heads=3), "h2o", 50),
    "h2o-empty-prompt": (small("h2o0", 0, 6, grid=9, heads=3), "h2o", 70),
}


# launch shapes: 1 / 2 = 8 KB / 6 KB stages, two per warp; 3 = 8 KB x 3; 6 = 6 KB x 4
@pytest.mark.parametrize("shape", [1, 2, 3, 6])
@pytest.mark.parametrize("name", list(CASES))
def test_policy_parity(name, shape):
    wl, policy, steps = CASES[name]
    rep = run_policy(wl, policy, steps, shape=shape)
    assert rep.ok, (rep.failures[:5], rep.max_err)
    assert rep.steps == steps
    if wl.N_att <= steps:
        assert rep.evictions > 0


@pytest.mark.parametrize("policy", ["tova", "h2o"])
def test_policy_full_size_janus_b96(policy):
    """Janus-Pro-7B-shaped layer at full size (batch 96 x 32 heads = 3072
    streams, more than the grid's warps, so warps carry several streams),
    L_p 64, N_att 29, through 200 steps; 16 sampled streams on the oracle."""
    wl = Workload("janus-b96", 1, 32, 128, "bf16", 64, 24, 29, 29, 0, 96, 20260918)
    rep = run_policy(wl, policy, 200, sample=list(range(0, 3072, 193)), check_every=20)
    assert rep.ok, (rep.failures[:5], rep.max_err)
    assert rep.evictions > 0


def test_policy_timeout_is_reported():
    from ar_image_gen_gb300.dsa import DSA_ERR_TIMEOUT, Policy

    wl = small("tto", 16, 9)
    gen = TraceGen(wl, device="cuda")
    h = Policy(gen.S, wl.head_dim, wl.L_p, wl.N_att, "tova")
    Kp, Vp = gen.prompt()
    h.prefill(Kp, Vp)
    h.set_wait_limit(0)
    q, k, v = gen.step(0)
    out = torch.empty_like(q)
    h.decode_step(q, k, v, out)
    assert h.sync_status() == DSA_ERR_TIMEOUT
    torch.cuda.synchronize()  # the context stays usable
    h.close()


@pytest.mark.parametrize("policy", ["tova", "h2o"])
def test_policy_full_size_lumina_b32(policy):
    """Lumina-mGPT-shaped layer (batch 32 x 32 heads = 1024 streams, L_p 64,
    N_att 205: 269 rows per stream, fewer streams than warps) through 260
    steps, into the eviction phase; 8 sampled streams on the oracle."""
    wl = Workload("lumina-s95-b32", 1, 32, 128, "bf16", 64, 64, 205, 205, 0, 32, 20260920)
    rep = run_policy(wl, policy, 260, sample=list(range(0, 1024, 131)), check_every=26)
    assert rep.ok, (rep.failures[:5], rep.max_err)
    assert rep.evictions > 0


@pytest.mark.parametrize("policy", ["tova", "h2o"])
def test_policy_interleaved_handles_on_one_stream(policy):
    """Three handles (layers) stepped round-robin on one stream, so that
    every launch after the first follows another handle's and issues its
    first stages before the grid dependency wait; each is compared bit for
    bit (outputs, evictions, cache positions) with a twin stepped on a
    stream of its own, whose launches always follow its own."""
    from ar_image_gen_gb300.dsa import DSA_OK, Policy

    wl = small("inter", 16, 9, heads=8, batch=8)
    d, S = wl.head_dim, wl.streams
    gens = [TraceGen(wl, layer=l, device="cuda") for l in range(3)]
    A = [Policy(S, d, wl.L_p, wl.N_att, policy, wl.dtype) for _ in range(3)]
    B = [Policy(S, d, wl.L_p, wl.N_att, policy, wl.dtype) for _ in range(3)]
    own = [torch.cuda.Stream() for _ in range(3)]
    main = torch.cuda.current_stream()
    for l in range(3):
        Kp, Vp = gens[l].prompt()
        A[l].prefill(Kp, Vp)
        B[l].prefill(Kp, Vp)
    torch.cuda.synchronize()
    outA = [torch.empty((S, d), dtype=torch.bfloat16, device="cuda") for _ in range(3)]
    outB = [torch.empty_like(outA[0]) for _ in range(3)]
    for t in range(40):
        qkv = [gens[l].step(t) for l in range(3)]
        torch.cuda.synchronize()
        for l in range(3):
            A[l].decode_step(*qkv[l], outA[l], main)
        for l in range(3):
            with torch.cuda.stream(own[l]):
                B[l].decode_step(*qkv[l], outB[l], own[l])
        torch.cuda.synchronize()
        for l in range(3):
            assert torch.equal(outA[l], outB[l]), (t, l)
            assert np.array_equal(A[l].last_eviction(), B[l].last_eviction()), (t, l)
    for l in range(3):
        assert np.array_equal(A[l].positions(), B[l].positions())
        assert A[l].sync_status() == DSA_OK and B[l].sync_status() == DSA_OK
        A[l].close()
        B[l].close()


def test_policy_shape_knob_accepts_the_six_shapes_only():
    from ar_image_gen_gb300 import dsa

    code, h = dsa.dsa_pol_create(8, 128, 16, 9, dsa.DSA_POLICY_TOVA, dsa.DSA_BF16)
    assert code == dsa.DSA_OK
    for bad in (-1, 7):
        assert dsa.dsa_pol_set_shape(h, bad) == dsa.DSA_ERR_ARG
        assert "shape" in dsa.dsa_last_error()
    for ok in (1, 2, 3, 4, 5, 6, 0):
        assert dsa.dsa_pol_set_shape(h, ok) == dsa.DSA_OK
    assert dsa.dsa_pol_destroy(h) == dsa.DSA_OK
