"""Seeded synthetic decode traces shaped like the page's image models.

This module draws inputs only.  It holds none of the decode method's
arithmetic, and both the CUDA path and the CPU oracle consume what it draws
(the oracle receives the exact values the device saw, widened to fp64).

Structure (arXiv 2609.19702, section 3, "Diagonal attention sparsity
pattern" and Fig. 11: relevance follows relative spatial position in the
raster-ordered token grid):

* a g x g token grid decoded in raster order, L_dec = g * g; decode token t
  sits at row t // g and column t % g;
* per (layer, head): one pair of Gaussian tables E[g, d], F[g, d] shared by
  q and k (this is what makes neighbouring grid positions score alike), and
  an independent pair for v;
* q_t, k_t = RoPE(E[row] + F[col] + 0.5 * N(0, 1)) at position L_p + t,
  v_t = E_v[row] + F_v[col] + 0.5 * N(0, 1), fresh noise per
  (sequence, head, token, tensor);
* prompt K = RoPE(N(0, 1)) at positions 0 .. L_p - 1, prompt V = N(0, 1);
* RoPE is the rotate-half form with base 10000;
* calibrated variant (Workload.calibrated): q_t = RoPE(g (E[row] + F[col] +
  0.5 N(0, 1)) + a c) and prompt K = RoPE(N(0, 1) + a c), with c the unit
  vector of the lowest-frequency RoPE pair (element d/2 - 1), so every
  query scores every prompt key about a^2 / sqrt(d) higher, decaying slowly
  with distance; g and a^2 per family from CALIBRATION.

Streams of one layer are ordered s = b * heads + h.
"""
from __future__ import annotations

from dataclasses import dataclass, replace

import torch

SEED_BASE = 20260917


def n_att_for(L_dec: int, sparsity_pct: int, N_r: int) -> int:
    """N_att for a sparsity ratio 1 - N_att / L_dec (section 5.1, "Our
    methods"), rounded half up and capped at the window N_r."""
    n = (L_dec * (100 - sparsity_pct) * 2 + 100) // 200
    return max(1, min(n, N_r))


@dataclass(frozen=True)
class Workload:
    name: str
    layers: int
    heads: int
    head_dim: int
    dtype: str          # "f32" / "bf16": element type of q, k, v, out and the KV state;
                        # "fp8e4m3": KV state in FP8 E4M3 with per-stream scales, q, k, v, out bf16
    L_p: int
    grid: int           # L_dec = grid * grid
    N_r: int
    N_att: int
    sink: int
    batch: int
    seed: int
    qk_gain: float = 1.0          # scale of the grid part of q (1: the plain recipe)
    prompt_affinity: float = 0.0  # a*b of the shared q / prompt-key component (0: none)

    @property
    def L_dec(self) -> int:
        return self.grid * self.grid

    @property
    def streams(self) -> int:
        """Independent (sequence, head) streams of one layer."""
        return self.batch * self.heads

    def dense(self) -> "Workload":
        """The 0 % sparsity setting of the same kernel: no eviction, no skip."""
        return replace(self, name=self.name + "-dense", N_r=self.L_dec, N_att=self.L_dec, sink=0)

    def fp8(self) -> "Workload":
        """The same workload with the KV state stored as FP8 E4M3."""
        return replace(self, name=self.name + "-fp8", dtype="fp8e4m3")

    def with_batch(self, batch: int) -> "Workload":
        return replace(self, name=f"{self.name.rsplit('-b', 1)[0]}-b{batch}", batch=batch)

    def calibrated(self) -> "Workload":
        """The same workload with q scaled and a shared query / prompt-key
        component, chosen per model family so that dense attention over the
        trace splits its weight as the page's Fig. 8 reports for the model
        the family stands in for: more than half on the prompt, most of the
        rest on the local tokens (the newest 10 %), and 6.2 % (Janus-Pro) or
        about 8.5 % (Lumina-mGPT) on the middle tokens."""
        g, ab = CALIBRATION[self.seed - SEED_BASE]
        return replace(self, name=self.name + "-cal", qk_gain=g, prompt_affinity=ab)


def _wl(name, cfg, layers, heads, d, dtype, L_p, grid, N_r, pct, batch, sink=0, N_att=None):
    L_dec = grid * grid
    if N_att is None:
        N_att = n_att_for(L_dec, pct, N_r)
    return Workload(name, layers, heads, d, dtype, L_p, grid, N_r, N_att, sink, batch, SEED_BASE + cfg)


# Per workload family (seed offset): q gain and prompt affinity of the
# calibrated traces (Workload.calibrated), fitted on two heads of layer 0 of
# each family's trace with the oracle's attention diagnostics; mass split
# (prompt, local, middle) reached: janus 0.53 / 0.40 / 0.064, sweep512
# 0.64 / 0.28 / 0.083, lumina 0.62 / 0.30 / 0.085, stress 0.61 / 0.31 / 0.084.
CALIBRATION = {1: (0.36, 45.0), 2: (0.34, 50.0), 3: (0.42, 70.0), 4: (0.48, 90.0)}

# The five workload families of the benchmark plan.
WORKLOADS = {
    # tiny oracle check: fp32, head_dim 64, N_att given directly
    "tiny": _wl("tiny", 0, 1, 4, 64, "f32", 16, 8, 32, 0, 1, N_att=8),
    # Janus-Pro-7B-shaped attention stack, 384x384 (576 tokens), 95 %
    "janus-b32": _wl("janus-b32", 1, 30, 32, 128, "bf16", 64, 24, 288, 95, 32),
    "janus-b96": _wl("janus-b96", 1, 30, 32, 128, "bf16", 64, 24, 288, 95, 96),
    # 512x512-shaped sparsity sweep (1024 tokens)
    "sweep512-s0": _wl("sweep512-s0", 2, 32, 32, 128, "bf16", 64, 32, 512, 0, 64),
    "sweep512-s50": _wl("sweep512-s50", 2, 32, 32, 128, "bf16", 64, 32, 512, 50, 64),
    "sweep512-s75": _wl("sweep512-s75", 2, 32, 32, 128, "bf16", 64, 32, 512, 75, 64),
    "sweep512-s90": _wl("sweep512-s90", 2, 32, 32, 128, "bf16", 64, 32, 512, 90, 64),
    "sweep512-s95": _wl("sweep512-s95", 2, 32, 32, 128, "bf16", 64, 32, 512, 95, 64),
    "sweep512-sink4-s95": _wl("sweep512-sink4-s95", 2, 32, 32, 128, "bf16", 64, 32, 512, 95, 64, sink=4),
    # Lumina-mGPT-7B 1024x1024-shaped (4096 tokens)
    "lumina-s90-b16": _wl("lumina-s90-b16", 3, 32, 32, 128, "bf16", 64, 64, 2048, 90, 16),
    "lumina-s90-b32": _wl("lumina-s90-b32", 3, 32, 32, 128, "bf16", 64, 64, 2048, 90, 32),
    "lumina-s90-b54": _wl("lumina-s90-b54", 3, 32, 32, 128, "bf16", 64, 64, 2048, 90, 54),
    "lumina-s95-b16": _wl("lumina-s95-b16", 3, 32, 32, 128, "bf16", 64, 64, 2048, 95, 16),
    "lumina-s95-b32": _wl("lumina-s95-b32", 3, 32, 32, 128, "bf16", 64, 64, 2048, 95, 32),
    "lumina-s95-b54": _wl("lumina-s95-b54", 3, 32, 32, 128, "bf16", 64, 64, 2048, 95, 54),
    # high-resolution stress (8100 tokens)
    "stress-s95": _wl("stress-s95", 4, 32, 32, 128, "bf16", 96, 90, 4050, 95, 64),
}


def torch_dtype(name: str) -> torch.dtype:
    """Element type of the q, k, v, prompt and out tensors of a workload dtype."""
    return {"f32": torch.float32, "bf16": torch.bfloat16, "fp8e4m3": torch.bfloat16}[name]


def _rope(x: torch.Tensor, pos: torch.Tensor) -> torch.Tensor:
    """Rotate-half rotary embedding (base 10000) on the last dim; pos broadcasts
    against x's leading dims."""
    d = x.shape[-1]
    half = d // 2
    inv = 10000.0 ** (-torch.arange(half, dtype=torch.float64, device=x.device) * 2.0 / d)
    ang = pos.to(torch.float64)[..., None] * inv
    cos, sin = torch.cos(ang).to(x.dtype), torch.sin(ang).to(x.dtype)
    x1, x2 = x[..., :half], x[..., half:]
    return torch.cat([x1 * cos - x2 * sin, x2 * cos + x1 * sin], dim=-1)


class TraceGen:
    """Seeded generator of one layer's decode trace (all streams).

    Every draw is keyed by (seed, layer, tensor, step), so a step can be
    regenerated on its own and the device and the host draw the same
    values for the same device type.
    """

    def __init__(self, wl: Workload, layer: int = 0, device: str | torch.device = "cpu",
                 batch: int | None = None, seed: int | None = None):
        self.wl = wl
        self.layer = layer
        self.device = torch.device(device)
        self.batch = wl.batch if batch is None else batch
        self.S = self.batch * wl.heads
        self.seed = wl.seed if seed is None else seed
        self.out_dtype = torch_dtype(wl.dtype)
        g = self._gen(0, 0)
        shape = (wl.heads, wl.grid, wl.head_dim)
        self.E_qk = torch.randn(shape, generator=g, device=self.device, dtype=torch.float32)
        self.F_qk = torch.randn(shape, generator=g, device=self.device, dtype=torch.float32)
        self.E_v = torch.randn(shape, generator=g, device=self.device, dtype=torch.float32)
        self.F_v = torch.randn(shape, generator=g, device=self.device, dtype=torch.float32)

    def _gen(self, kind: int, step: int) -> torch.Generator:
        g = torch.Generator(device=self.device)
        g.manual_seed(((self.seed * 1009 + self.layer) * 7 + kind) * 1_000_003 + step)
        return g

    def kv_scales(self):
        """Per-stream K and V scales of FP8 storage, float32 [S] each: 2^-5
        times a seeded factor in [1, 1.5), so the largest E4M3 value (448)
        maps to 14..21, above the generated magnitudes, and the smallest
        normal one to about 5e-4."""
        g = self._gen(3, 0)
        u = torch.rand((2, self.S), generator=g, device=self.device, dtype=torch.float32)
        sc = (2.0 ** -5) * (1.0 + 0.5 * u)
        return sc[0].cpu().numpy(), sc[1].cpu().numpy()

    def prompt(self):
        """Prompt K, V as [S, L_p, d] in the workload's input dtype."""
        wl = self.wl
        g = self._gen(1, 0)
        shape = (self.S, wl.L_p, wl.head_dim)
        K = torch.randn(shape, generator=g, device=self.device, dtype=torch.float32)
        V = torch.randn(shape, generator=g, device=self.device, dtype=torch.float32)
        pos = torch.arange(wl.L_p, device=self.device)
        if wl.prompt_affinity:
            K[..., wl.head_dim // 2 - 1] += wl.prompt_affinity ** 0.5
        K = _rope(K, pos[None, :])
        return K.to(self.out_dtype).contiguous(), V.to(self.out_dtype).contiguous()

    def step(self, t: int):
        """q, k_new, v_new for decode step t, each [S, d] in the workload dtype."""
        wl = self.wl
        row, col = t // wl.grid, t % wl.grid
        g = self._gen(2, t)
        shape = (self.batch, wl.heads, wl.head_dim)
        nq = torch.randn(shape, generator=g, device=self.device, dtype=torch.float32)
        nk = torch.randn(shape, generator=g, device=self.device, dtype=torch.float32)
        nv = torch.randn(shape, generator=g, device=self.device, dtype=torch.float32)
        base_qk = (self.E_qk[:, row] + self.F_qk[:, col])[None]
        base_v = (self.E_v[:, row] + self.F_v[:, col])[None]
        pos = torch.tensor(wl.L_p + t, device=self.device)
        qx = base_qk + 0.5 * nq
        if wl.qk_gain != 1.0:
            qx = wl.qk_gain * qx
        if wl.prompt_affinity:
            qx[..., wl.head_dim // 2 - 1] += wl.prompt_affinity ** 0.5
        q = _rope(qx, pos)
        k = _rope(base_qk + 0.5 * nk, pos)
        v = base_v + 0.5 * nv
        cast = lambda x: x.reshape(self.S, wl.head_dim).to(self.out_dtype).contiguous()
        return cast(q), cast(k), cast(v)


class ProjGen:
    """Seeded inputs of the QKV projection that feeds a decode step: the
    newest token's hidden state x [batch, hidden] ~ N(0, 1) per step, and one
    weight W [3 * heads * head_dim, hidden] ~ N(0, 1 / hidden) per layer (the
    q rows of all heads, then k, then v), both bf16, so that q, k and v come
    out with unit variance.  hidden defaults to heads * head_dim (4096 for
    the 7B models the workloads stand in for)."""

    def __init__(self, wl: Workload, layer: int = 0, device: str | torch.device = "cpu", batch: int | None = None,
                 hidden: int | None = None, seed: int | None = None):
        self.wl = wl
        self.layer = layer
        self.device = torch.device(device)
        self.batch = wl.batch if batch is None else batch
        self.hidden = wl.heads * wl.head_dim if hidden is None else hidden
        self.seed = wl.seed if seed is None else seed

    def _gen(self, kind: int, step: int) -> torch.Generator:
        g = torch.Generator(device=self.device)
        g.manual_seed(((self.seed * 1009 + self.layer) * 7 + kind) * 1_000_003 + step + 500_000)
        return g

    def weight(self) -> torch.Tensor:
        rows = 3 * self.wl.heads * self.wl.head_dim
        W = torch.randn((rows, self.hidden), generator=self._gen(5, 0), device=self.device, dtype=torch.float32)
        return (W * self.hidden ** -0.5).to(torch.bfloat16).contiguous()

    def x(self, t: int) -> torch.Tensor:
        x = torch.randn((self.batch, self.hidden), generator=self._gen(6, t), device=self.device, dtype=torch.float32)
        return x.to(torch.bfloat16).contiguous()
