"""The calibrated synthetic traces (Workload.calibrated) split dense
attention as the page's Fig. 8 reports for the models they stand in for
(prompt more than half, middle 6.2 % for Janus-Pro, about 8.5 % for
Lumina-mGPT), measured with the oracle's diagnostics on two heads of layer
0; and the plain recipe is unchanged by the calibration fields."""
from dataclasses import replace

import numpy as np
import pytest
import torch

from ar_image_gen_gb300.synth import WORKLOADS, TraceGen
from oracle.oracle import diag_stream


def mass_split(wl, heads=2):
    wl = replace(wl.with_batch(1), heads=heads)
    gen = TraceGen(wl, device="cpu")
    Kp, _ = gen.prompt()
    steps = [gen.step(t) for t in range(wl.L_dec)]
    Q = torch.stack([x[0] for x in steps], 1).double().numpy()
    Kd = torch.stack([x[1] for x in steps], 1).double().numpy()
    return np.mean([diag_stream(Q[h], Kp[h].double().numpy(), Kd[h], [1])[0].mean(axis=0) for h in range(heads)], axis=0)


@pytest.mark.parametrize("key,middle", [("janus-b32", 0.062), ("sweep512-s95", 0.085)])
def test_calibrated_split_matches_fig8(key, middle):
    prompt, local, mid = mass_split(WORKLOADS[key].calibrated())
    assert prompt > 0.5 and local > mid
    assert abs(mid - middle) < 0.015, (prompt, local, mid)


def test_plain_recipe_is_the_default():
    wl = WORKLOADS["janus-b32"]
    assert wl.qk_gain == 1.0 and wl.prompt_affinity == 0.0
    a = TraceGen(wl).step(3)
    b = TraceGen(replace(wl, qk_gain=1.0, prompt_affinity=0.0)).step(3)
    assert all(torch.equal(x, y) for x, y in zip(a, b))
