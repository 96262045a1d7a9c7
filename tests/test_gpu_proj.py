"""The QKV projection with RoPE on the tensor cores (dsa_qkv_rope) and the
fused decode step on it (dsa_decode_step_fused), through the C ABI, against
the fp64 oracle (oracle/proj.py for the projection, the decode oracle for the
attention that follows).

Tolerance of the projection: the kernel multiplies bf16 operands exactly,
sums in fp32 and rounds the rotated result to bf16 once, so an element may
differ from the exact value by half a bf16 step (2^-9 relative) plus the
fp32 summation error; the test allows one bf16 step, 2^-8 |ref|, plus
1e-3 of the outputs' rms.  Any mistake in orientation, block order,
pairing, sign, angle or position moves elements by O(rms).
"""
import numpy as np
import pytest
import torch

from ar_image_gen_gb300.synth import ProjGen, Workload
from oracle.oracle import OracleBatch
from oracle.proj import qkv_rope as oracle_qkv_rope
from tests.parity import ATOL, RTOL, mask_offsets

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    from __graft_entry__ import build
    build()


def wl_for(heads, d, batch, L_p=16, N_r=40, N_att=9, sink=0, grid=10, dtype="bf16", seed=11):
    return Workload("proj", 1, heads, d, dtype, L_p, grid, N_r, N_att, sink, batch, seed)


def project(proj, x, W, pos):
    S = proj.batch * proj.heads
    q, k, v = (torch.empty((S, proj.head_dim), dtype=torch.bfloat16, device="cuda") for _ in range(3))
    proj.qkv_rope(x, W, pos, q, k, v)
    return q, k, v


def check_projection(batch, heads, d, hidden, positions, seed=3):
    from ar_image_gen_gb300.dsa import DSA_OK, Proj

    gen = ProjGen(wl_for(heads, d, batch, seed=seed), device="cuda", hidden=hidden)
    W = gen.weight()
    proj = Proj(batch, heads, d, hidden)
    Wd = W.double().cpu().numpy()
    worst = 0.0
    for i, pos in enumerate(positions):
        x = gen.x(i)
        got = [t.double().cpu().numpy() for t in project(proj, x, W, pos)]
        ref = oracle_qkv_rope(x.double().cpu().numpy(), Wd, heads, d, pos)
        for name, g, r in zip("qkv", got, ref):
            rms = float(np.sqrt(np.mean(r * r)))
            excess = np.abs(g - r) - (2.0 ** -8 * np.abs(r) + 1e-3 * rms)
            worst = max(worst, float(excess.max()))
            assert excess.max() <= 0, (name, pos, float(np.abs(g - r).max()), np.unravel_index(excess.argmax(), g.shape))
    assert proj.sync_status() == DSA_OK
    proj.close()
    return worst


SHAPES = {
    # name: (batch, heads, head_dim, hidden)
    "one-token-one-kblock": (1, 1, 128, 64),
    "d64-pair-of-heads": (3, 2, 64, 128),
    "ragged-batch-17": (17, 4, 128, 320),
    "janus-b32": (32, 32, 128, 4096),
    "lumina-b54": (54, 32, 128, 4096),
    "janus-b96": (96, 32, 128, 4096),
    "batch-256-four-stages": (256, 8, 128, 1024),
    "long-hidden": (5, 2, 128, 8192),
}


@pytest.mark.parametrize("name", list(SHAPES))
def test_projection_matches_oracle(name):
    batch, heads, d, hidden = SHAPES[name]
    check_projection(batch, heads, d, hidden, positions=[0, 1, 63, 8195])


def test_projection_is_deterministic():
    """A split output tile is summed in segment order: repeated calls agree bit for bit."""
    from ar_image_gen_gb300.dsa import Proj

    batch, heads, d, hidden = 96, 32, 128, 4096
    gen = ProjGen(wl_for(heads, d, batch), device="cuda", hidden=hidden)
    W, x = gen.weight(), gen.x(0)
    proj = Proj(batch, heads, d, hidden)
    a = project(proj, x, W, 700)
    for _ in range(3):
        b = project(proj, x, W, 700)
        for u, v in zip(a, b):
            assert torch.equal(u, v)
    proj.close()


def test_timeout_is_reported_and_the_context_recovers():
    """With a wait limit of 0 every bounded wait gives up: the status reports
    DSA_ERR_TIMEOUT, the CUDA context stays usable, and after the limit is
    restored the same context computes correct results again."""
    from ar_image_gen_gb300.dsa import DSA_ERR_TIMEOUT, DSA_OK, Proj

    batch, heads, d, hidden = 8, 4, 128, 512
    gen = ProjGen(wl_for(heads, d, batch), device="cuda", hidden=hidden)
    W, x = gen.weight(), gen.x(0)
    proj = Proj(batch, heads, d, hidden)
    proj.set_wait_limit(0)
    project(proj, x, W, 5)
    assert proj.sync_status() == DSA_ERR_TIMEOUT
    torch.cuda.synchronize()
    proj.set_wait_limit(0xFFFFFFFF)
    got = [t.double().cpu().numpy() for t in project(proj, x, W, 5)]
    assert proj.sync_status() == DSA_OK
    ref = oracle_qkv_rope(x.double().cpu().numpy(), W.double().cpu().numpy(), heads, d, 5)
    for g, r in zip(got, ref):
        assert np.abs(g - r).max() <= 2.0 ** -8 * np.abs(r).max() + 1e-3


def run_fused(wl: Workload, hidden: int, steps: int, sample, kv_scales=None):
    """Steps a fused handle (projection + decode) and a twin handle fed with
    dsa_qkv_rope's outputs; checks the two agree bit for bit (outputs,
    selections, and the stored prefix and ring: with bf16 storage the fused
    step's projection writes the newest token into its slot itself), the
    projection against its oracle, and the sampled streams' attention
    against the decode oracle (outputs within tolerance, selections and skip
    masks exact up to accepted near ties)."""
    from ar_image_gen_gb300.dsa import DSA, DSA_OK, Proj

    gen = ProjGen(wl, device="cuda", hidden=hidden)
    W = gen.weight()
    Wd = W.double().cpu().numpy()
    S, d = wl.streams, wl.head_dim
    fused = DSA(S, d, wl.L_p, wl.N_r, wl.N_att, wl.sink, wl.dtype)
    twin = DSA(S, d, wl.L_p, wl.N_r, wl.N_att, wl.sink, wl.dtype)
    proj_f = Proj(wl.batch, wl.heads, d, hidden)
    proj_t = Proj(wl.batch, wl.heads, d, hidden)
    if kv_scales is not None:
        fused.set_kv_scales(*kv_scales)
        twin.set_kv_scales(*kv_scales)
    torch.manual_seed(5)
    Kp = torch.randn((S, wl.L_p, d), device="cuda").to(torch.bfloat16)
    Vp = torch.randn((S, wl.L_p, d), device="cuda").to(torch.bfloat16)
    fused.prefill(Kp, Vp)
    twin.prefill(Kp, Vp)
    idx = torch.tensor(sample, device="cuda")
    ks = vs = None
    if kv_scales is not None:
        ks, vs = kv_scales[0][sample], kv_scales[1][sample]
    orc = OracleBatch(len(sample), d, wl.L_p, wl.N_r, wl.N_att, wl.sink, k_scales=ks, v_scales=vs)
    orc.prefill(Kp[idx].double().cpu().numpy(), Vp[idx].double().cpu().numpy())
    out_f = torch.empty((S, d), dtype=torch.bfloat16, device="cuda")
    out_t = torch.empty_like(out_f)
    selections = 0
    for t in range(steps):
        x = gen.x(t)
        pos = wl.L_p + t
        fused.decode_step_fused(proj_f, x, W, out_f)
        q, k, v = project(proj_t, x, W, pos)
        twin.decode_step(q, k, v, out_t)
        assert torch.equal(out_f, out_t), f"fused and two-call outputs differ at t={t}"
        sel_f, sel_t = fused.last_selection(), twin.last_selection()
        assert np.array_equal(sel_f, sel_t)
        if (S <= 64 and t % 25 == 24) or t == steps - 1:
            for a, b in zip(fused.copy_state(), twin.copy_state()):
                assert np.array_equal(a, b), f"stored state differs at t={t}"
        if t % 16 == 0 or t == steps - 1:
            ref = oracle_qkv_rope(x.double().cpu().numpy(), Wd, wl.heads, d, pos)
            for g, r in zip((q, k, v), ref):
                g = g.double().cpu().numpy()
                rms = float(np.sqrt(np.mean(r * r)))
                assert (np.abs(g - r) <= 2.0 ** -8 * np.abs(r) + 1e-3 * rms).all(), f"projection at t={t}"
        tin = t - wl.sink
        picks = np.array([tin - sel_f[s] if sel_f[s] >= 0 else -1 for s in sample], dtype=np.int32)
        ref, infos = orc.step(q[idx].double().cpu().numpy(), k[idx].double().cpu().numpy(),
                              v[idx].double().cpu().numpy(), picks=picks)
        got = out_f[idx].double().cpu().numpy()
        assert ((np.abs(got - ref) - (ATOL + RTOL * np.abs(ref))) <= 0).all(), f"attention output at t={t}"
        for i, info in enumerate(infos):
            selections += info.oracle_pick >= 0
            assert not info.mismatch and info.selected == int(picks[i]), f"selection at t={t}, stream {sample[i]}"
    masks_f, masks_t = fused.skip_mask(), twin.skip_mask()
    assert np.array_equal(masks_f, masks_t)
    tin = steps - 1 - wl.sink
    for i, s in enumerate(sample):
        want = {tin - j for j in orc.streams[i].skip()} if tin >= 0 else set()
        assert mask_offsets(masks_f[s]) == want
    assert fused.sync_status() == DSA_OK and twin.sync_status() == DSA_OK
    assert proj_f.sync_status() == DSA_OK and proj_t.sync_status() == DSA_OK
    assert fused.t == steps
    for o in (fused, twin, proj_f, proj_t):
        o.close()
    return selections


def test_fused_step_small():
    wl = wl_for(4, 128, 3, L_p=16, N_r=40, N_att=9, grid=10)
    assert run_fused(wl, hidden=256, steps=100, sample=list(range(12))) > 0


def test_fused_step_sink4_d64():
    wl = wl_for(4, 64, 2, L_p=12, N_r=48, N_att=12, sink=4, grid=10)
    assert run_fused(wl, hidden=192, steps=90, sample=list(range(8))) > 0


def test_fused_step_fp8_storage():
    wl = wl_for(4, 128, 2, L_p=16, N_r=40, N_att=9, grid=9, dtype="fp8e4m3")
    rng = np.random.default_rng(2)
    scales = (np.float32(2.0 ** -5) * (1 + 0.5 * rng.random(8, dtype=np.float32)),
              np.float32(2.0 ** -5) * (1 + 0.5 * rng.random(8, dtype=np.float32)))
    assert run_fused(wl, hidden=128, steps=80, sample=list(range(8)), kv_scales=scales) > 0


def test_fused_step_janus_b96_full_size():
    """Janus-Pro-7B-shaped layer at full size (batch 96, 32 heads of 128,
    hidden 4096, L_p 64, N_r 288, N_att 29) through phase 3."""
    wl = Workload("janus-b96", 1, 32, 128, "bf16", 64, 24, 288, 29, 0, 96, 20260918)
    sample = list(range(0, 3072, 193))
    assert run_fused(wl, hidden=4096, steps=300, sample=sample) > 0


def test_fused_step_lumina_b32_through_phase3():
    """Lumina-mGPT-shaped layer (batch 32, 32 heads of 128, hidden 4096,
    L_p 64, N_r 2048, N_att 205) through the selection phase into eviction
    (2100 steps), fused vs two-call bit-exact and sampled oracle parity."""
    wl = Workload("lumina-s95-b32", 1, 32, 128, "bf16", 64, 64, 2048, 205, 0, 32, 20260920)
    assert run_fused(wl, hidden=4096, steps=2100, sample=list(range(0, 1024, 171))) > 0


def test_fused_step_refuses_graph_mode():
    """The fused step counts steps on the host (the projection's position and
    the newest token's slot come from it), so a handle in graph mode is
    refused before anything is launched."""
    from ar_image_gen_gb300.dsa import DSA, DSA_ERR_STATE, DSAError, Proj

    wl = wl_for(2, 128, 1, L_p=8, N_r=12, N_att=4, grid=5)
    S, d = wl.streams, wl.head_dim
    h = DSA(S, d, wl.L_p, wl.N_r, wl.N_att, 0, "bf16")
    pr = Proj(wl.batch, wl.heads, d, 128)
    K = torch.zeros((S, wl.L_p, d), dtype=torch.bfloat16, device="cuda")
    h.prefill(K, K)
    q = torch.zeros((S, d), dtype=torch.bfloat16, device="cuda")
    out = torch.empty_like(q)
    for _ in range(wl.N_r):
        h.decode_step(q, q, q, out)
    h.set_graph_mode(True)
    x = torch.zeros((wl.batch, 128), dtype=torch.bfloat16, device="cuda")
    W = torch.zeros((3 * wl.heads * d, 128), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(DSAError) as e:
        h.decode_step_fused(pr, x, W, out)
    assert e.value.code == DSA_ERR_STATE
    h.sync_step()
    h.set_graph_mode(False)
    assert h.sync_status() == 0
    h.close()
    pr.close()
