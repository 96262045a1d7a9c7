"""FP8 E4M3 KV storage on the GPU against the oracle's FP8 mode.

The stored codes are compared bit for bit with the oracle's E4M3 encoder;
outputs, selections and skip sets go through the same parity harness as the
bf16 path (same tolerances: the oracle attends over exactly the stored
values, so only fp32 accumulation, the f16 rounding of q and p, and the
bf16 output separate the two).
"""
import numpy as np
import pytest
import torch

from ar_image_gen_gb300.synth import WORKLOADS, TraceGen, Workload
from tests.parity import run_parity
from tests.test_gpu_full import sample_streams

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    from __graft_entry__ import build
    build()


def small(name, L_p, N_r, N_att, sink=0, grid=10, heads=4, batch=1, d=128, seed=7):
    return Workload(name, 1, heads, d, "fp8e4m3", L_p, grid, N_r, N_att, sink, batch, seed)


CASES = {
    # name: (workload, steps, forced splits)
    "basic": (small("basic", 64, 40, 9, grid=10), 100, 0),
    "ragged-split3": (small("ragged", 37, 71, 13, grid=13, heads=5), 150, 3),
    "sink4": (small("sink4", 20, 64, 12, sink=4, grid=12, heads=6), 130, 0),
    "sink4-split2": (small("sink4s", 20, 64, 12, sink=4, grid=12, heads=6), 130, 2),
    "dense-split3": (small("dense", 16, 80, 80, grid=9), 80, 3),
    "n_att-1": (small("natt1", 8, 20, 1, grid=8, heads=3), 50, 0),
    "empty-prompt": (small("noprompt", 0, 30, 5, grid=9, heads=3), 70, 0),
    "d64": (small("d64", 16, 40, 8, grid=10, d=64), 90, 0),
    "d64-split4": (small("d64s", 16, 40, 8, grid=10, d=64), 90, 4),
    "window-wider-than-a-stage-list": (small("wide", 8, 300, 260, grid=18, heads=2), 324, 0),
}


@pytest.mark.parametrize("pipeline", [1, 2, 4])
@pytest.mark.parametrize("name", list(CASES))
def test_small_parity(name, pipeline):
    wl, steps, splits = CASES[name]
    rep = run_parity(wl, steps=steps, splits=splits, pipeline=pipeline)
    assert rep.ok, rep.summary()
    assert rep.steps == steps


@pytest.mark.parametrize("scale", [2.0 ** -9, 64.0])
def test_saturating_and_subnormal_scales(scale):
    """Scale 2^-9: generated magnitudes above 0.875 saturate at 448 * scale;
    scale 64: most elements fall in the subnormal range.  The oracle stores
    the same codes, so parity holds either way."""
    wl = small("extreme", 24, 48, 10, grid=9, heads=4)
    S = wl.streams
    ks = np.full(S, scale, dtype=np.float32)
    vs = np.full(S, scale * 1.5, dtype=np.float32)
    rep = run_parity(wl, steps=81, kv_scales=(ks, vs))
    assert rep.ok, rep.summary()


def test_stored_codes_match_the_oracle_encoder():
    """Prompt rows (prefill kernel), the current token stored from registers
    and tokens stored while themselves skipped: every code of the prefix
    and the ring equals the oracle's E4M3 code of fp32(x) * fp32(1 / scale)."""
    from ar_image_gen_gb300.dsa import DSA
    from oracle.oracle import e4m3_encode

    wl = small("codes", 12, 16, 4, grid=6, heads=3, d=64)
    S, d = wl.streams, wl.head_dim
    gen = TraceGen(wl, device="cuda")
    ks, vs = gen.kv_scales()
    ks[0] = 2.0 ** -9  # one stream saturates
    h = DSA(S, d, wl.L_p, wl.N_r, wl.N_att, 0, "fp8e4m3")
    h.set_kv_scales(ks, vs)
    Kp, Vp = gen.prompt()
    h.prefill(Kp, Vp)
    out = torch.empty((S, d), dtype=torch.bfloat16, device="cuda")
    steps = 22  # past N_r: the ring holds positions 6..21
    ins = []
    for t in range(steps):
        q, k, v = gen.step(t)
        h.decode_step(q, k, v, out)
        ins.append((k.float().cpu().numpy(), v.float().cpu().numpy()))
    pre, ring = h.copy_state()
    assert h.sync_status() == 0
    h.close()
    kinv = (np.float32(1.0) / ks).astype(np.float32)
    vinv = (np.float32(1.0) / vs).astype(np.float32)
    enc = np.vectorize(lambda y: e4m3_encode(float(y)), otypes=[np.uint8])
    Kf, Vf = Kp.float().cpu().numpy(), Vp.float().cpu().numpy()
    want_pre = np.stack([enc(Kf * kinv[:, None, None]), enc(Vf * vinv[:, None, None])], axis=2)
    assert np.array_equal(pre, want_pre)
    for p in range(steps - wl.N_r, steps):
        k, v = ins[p]
        slot = p % wl.N_r
        assert np.array_equal(ring[:, slot, 0], enc(k * kinv[:, None])), p
        assert np.array_equal(ring[:, slot, 1], enc(v * vinv[:, None])), p


def test_scale_knob_errors():
    from ar_image_gen_gb300 import dsa as mod
    from ar_image_gen_gb300.dsa import DSA

    h = DSA(4, 64, 8, 16, 4, 0, "bf16")
    assert mod.dsa_set_kv_scales(h.h, np.ones(4), np.ones(4)) == mod.DSA_ERR_ARG  # not an FP8 handle
    h.close()
    h = DSA(4, 64, 8, 16, 4, 0, "fp8e4m3")
    for bad in ([1, 1, 0, 1], [1, 1, -2, 1], [1, np.inf, 1, 1], [1, np.nan, 1, 1]):
        assert mod.dsa_set_kv_scales(h.h, np.ones(4), np.array(bad, dtype=np.float32)) == mod.DSA_ERR_ARG
    g = torch.Generator(device="cuda").manual_seed(1)
    K = torch.randn((4, 8, 64), generator=g, device="cuda").bfloat16()
    h.prefill(K, K)
    h.set_kv_scales(np.full(4, 0.5, np.float32), np.full(4, 0.25, np.float32))
    q = torch.randn((4, 64), generator=g, device="cuda").bfloat16()
    out = torch.empty_like(q)
    assert mod.dsa_decode_step(h.h, q, q, q, out) == mod.DSA_ERR_STATE  # scales changed: prefill again
    h.prefill(K, K)
    h.decode_step(q, q, q, out)
    assert h.sync_status() == 0
    h.close()


def test_noalloc_rejects_fp8():
    from ar_image_gen_gb300 import dsa as mod

    z = torch.zeros(1 << 16, dtype=torch.uint8, device="cuda")
    rc = mod.dsa_decode_step_noalloc(4, 64, 8, 16, 4, 0, mod.DSA_FP8_E4M3, 0, z, z, z, z, z, z, z, z)
    assert rc == mod.DSA_ERR_ARG and "FP8" in mod.dsa_last_error()


FULL = {"janus-b96": (24, 8), "sweep512-s95": (16, 16), "lumina-s95-b32": (12, 32)}


@pytest.mark.slow
@pytest.mark.parametrize("key", list(FULL))
def test_full_size_parity(key):
    wl = WORKLOADS[key].fp8()
    n, every = FULL[key]
    rep = run_parity(wl, sample=sample_streams(wl.streams, n), mask_every=every, threads=8)
    assert rep.ok, rep.summary()
    assert rep.steps == wl.L_dec


@pytest.mark.parametrize("d", [128, 64])
def test_every_code_reads_back_exactly(d):
    """Every finite E4M3 code (254 of them, both zeros included) as a V
    element of the one prompt row that takes all the attention (its key's
    logit is 57 above the others in log2 units): each output element is
    its code's value times the V scale, exactly (the scale is a power of
    two and E4M3 values fit bf16), which pins the kernel's widening of
    codes, normal and subnormal, of both signs.  Stream s holds codes
    d s .. d s + d - 1, the two NaN codes replaced by zero."""
    from ar_image_gen_gb300.dsa import DSA
    from oracle.oracle import e4m3_decode

    S, L_p, vs = 256 // d, 2, 2.0 ** -3
    codes = np.arange(256).reshape(S, d)
    vals = np.vectorize(lambda c: 0.0 if (c & 0x7F) == 0x7F else e4m3_decode(int(c)))(codes) * vs
    V = torch.zeros((S, L_p, d), dtype=torch.float64)
    V[:, 0, :] = torch.from_numpy(vals)
    K = torch.zeros((S, L_p, d), dtype=torch.float64)
    K[:, 0, 0] = 448.0  # the largest E4M3 value
    h = DSA(S, d, L_p, 8, 4, 0, "fp8e4m3")
    h.set_kv_scales(np.ones(S, np.float32), np.full(S, vs, np.float32))
    h.prefill(K.to(torch.bfloat16).cuda(), V.to(torch.bfloat16).cuda())
    q = torch.zeros((S, d), dtype=torch.bfloat16, device="cuda")
    q[:, 0] = 1.0
    zero = torch.zeros_like(q)
    out = torch.empty_like(q)
    h.decode_step(q, zero, zero, out)
    torch.cuda.synchronize()
    assert torch.equal(out.double().cpu(), torch.from_numpy(vals)), (out.double().cpu() - torch.from_numpy(vals)).abs().max()
    h.close()
