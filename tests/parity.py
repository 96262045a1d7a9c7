"""Parity harness: the CUDA path (through the C ABI) against the CPU oracle.

Both sides see the same seeded inputs: the device draws them, and the
sampled streams' exact values (bf16 or fp32, widened to fp64) are copied to
the oracle.  For FP8 storage both sides get the same per-stream scales and
each quantizes the rows itself.  Per step the harness checks

* outputs: max |out - oracle| <= 2e-3 + 1e-2 |oracle| elementwise;
* selections: the relative offset the kernel appended equals the oracle's
  argmin, except at a near tie (the two logits within 1e-4 relative), where
  the oracle adopts the kernel's choice and continues from it;
* skip sets: the kernel's relative-offset bitmask equals {t' - j : j in the
  oracle's skip_idx} (bit-exact), checked every `mask_every` steps and at
  the end; eviction is covered by the same check and by the outputs.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np
import torch

from ar_image_gen_gb300.synth import TraceGen, Workload
from oracle.oracle import OracleBatch

ATOL, RTOL = 2e-3, 1e-2


@dataclass
class ParityReport:
    steps: int = 0
    streams: int = 0
    max_err: float = 0.0
    worst_excess: float = -1.0      # max of |err| - (ATOL + RTOL |ref|); <= 0 passes
    out_failures: list = field(default_factory=list)
    sel_failures: list = field(default_factory=list)
    mask_failures: list = field(default_factory=list)
    selections: int = 0
    adopted: int = 0
    status: int = 0

    @property
    def ok(self) -> bool:
        return not (self.out_failures or self.sel_failures or self.mask_failures) and self.status == 0

    def summary(self) -> str:
        return (f"steps={self.steps} streams={self.streams} max_err={self.max_err:.3e} "
                f"excess={self.worst_excess:.3e} selections={self.selections} adopted={self.adopted} "
                f"status={self.status} out_fail={self.out_failures[:3]} sel_fail={self.sel_failures[:3]} "
                f"mask_fail={self.mask_failures[:3]}")


def mask_offsets(words: np.ndarray) -> set[int]:
    bits = np.unpackbits(words.astype("<u4").view(np.uint8), bitorder="little")
    return set(int(i) for i in np.nonzero(bits)[0])


def run_parity(wl: Workload, steps: int | None = None, sample: list[int] | None = None,
               splits: int = 0, mask_every: int = 1, layer: int = 0, device: str = "cuda",
               gen_device: str | None = None, threads: int = 1, pipeline: int = 0,
               kv_scales=None) -> ParityReport:
    """Runs `steps` decode steps of one layer of `wl` on the GPU and the
    sampled streams on the oracle; returns the report (does not raise)."""
    from ar_image_gen_gb300.dsa import DSA

    steps = wl.L_dec if steps is None else steps
    gen = TraceGen(wl, layer=layer, device=gen_device or device)
    S, d = gen.S, wl.head_dim
    sample = list(range(S)) if sample is None else list(sample)
    idx = torch.tensor(sample, dtype=torch.long)
    rep = ParityReport(streams=len(sample))

    h = DSA(S, d, wl.L_p, wl.N_r, wl.N_att, wl.sink, wl.dtype)
    if splits:
        h.set_splits(splits)
    if pipeline:
        h.set_pipeline(pipeline)
    ks = vs = None
    if wl.dtype == "fp8e4m3":
        ks, vs = kv_scales if kv_scales is not None else gen.kv_scales()
        h.set_kv_scales(ks, vs)
        ks, vs = ks[sample], vs[sample]
    orc = OracleBatch(len(sample), d, wl.L_p, wl.N_r, wl.N_att, wl.sink, k_scales=ks, v_scales=vs)

    # The sampled streams are taken from host copies (device-to-host copies,
    # no device kernels besides the library's own).
    Kp, Vp = gen.prompt()
    Kp_d, Vp_d = Kp.to(device), Vp.to(device)
    h.prefill(Kp_d, Vp_d)
    orc.prefill(Kp.cpu()[idx].double().numpy(), Vp.cpu()[idx].double().numpy())
    out = torch.empty((S, d), dtype=Kp_d.dtype, device=device)
    for t in range(steps):
        qkv = gen.step(t)
        q, k, v = (x.to(device) for x in qkv)
        h.decode_step(q, k, v, out)
        sel = h.last_selection()  # synchronizes
        tin = t - wl.sink
        picks = np.array([tin - sel[s] if sel[s] >= 0 else -1 for s in sample], dtype=np.int32)
        qh, kh, vh = (x.cpu()[idx].double().numpy() for x in qkv)
        ref, infos = orc.step(qh, kh, vh, picks=picks, threads=threads)
        got = out.cpu()[idx].double().numpy()
        err = np.abs(got - ref)
        excess = err - (ATOL + RTOL * np.abs(ref))
        rep.max_err = max(rep.max_err, float(err.max()))
        rep.worst_excess = max(rep.worst_excess, float(excess.max()))
        if (excess > 0).any():
            bad = np.argwhere(excess > 0)[0]
            rep.out_failures.append((t, sample[bad[0]], int(bad[1]), float(got[tuple(bad)]), float(ref[tuple(bad)])))
        for i, info in enumerate(infos):
            if info.oracle_pick >= 0:
                rep.selections += 1
            rep.adopted += info.adopted
            gpu_sel = int(picks[i])
            if info.mismatch or (info.selected != gpu_sel):
                rep.sel_failures.append((t, sample[i], gpu_sel, info.oracle_pick, info.min_logit, info.pick_logit))
        if (t % mask_every == mask_every - 1) or t == steps - 1:
            masks = h.skip_mask()
            for i, s in enumerate(sample):
                if tin < 0:
                    want = set()
                else:
                    want = {tin - j for j in orc.streams[i].skip()}
                got_set = mask_offsets(masks[s])
                if got_set != want:
                    rep.mask_failures.append((t, s, sorted(got_set)[:8], sorted(want)[:8]))
        rep.steps += 1
        if len(rep.out_failures) + len(rep.sel_failures) + len(rep.mask_failures) > 20:
            break
    rep.status = h.sync_status()
    h.close()
    return rep
