"""Pins for the CPU oracle: checks against facts the page and mathematics fix.

Each pin builds oracle streams (optionally with a planted mistake) and
returns a list of failure messages (empty = the pin holds).  The pins are:

* dense      -- N_r = N_att = L_dec reduces to causal attention over the
                prompt and every decode row; checked against torch's
                scaled_dot_product_attention in fp64 (a library routine the
                oracle does not use).
* sliding    -- N_att = N_r: no row is ever selected and the result is
                attention over the prompt plus the last N_r decode rows
                (SlidingWindow, section 5.1 "Sparse KV baselines").
* streaming  -- Diagonal+sink4 with N_att = N_r reduces to StreamingLLM with
                4 decode sinks and a window of N_r - 4 (section 5.1).
* worked     -- the Fig. 12 example (N_r = 7, N_att = 4), facts from
                tests/golden/worked_example.json.
* invariants -- cost analysis and the diagonal premise: KV held <= N_r + L_p,
                attended decode rows = min(t + 1, N_att), one selection per
                step for exactly N_r - N_att steps, relative offsets of the
                skip set never change, skip set inside the live window.
* relative   -- brute force on tiny inputs with an independent formulation
                (skip set kept as relative offsets, argmin taken over the
                softmax weights w exactly as written), compared step by step.
* cost       -- closed forms of the cost analysis: selection steps are
                t = N_att - 1 .. N_r - 2, peak KV is N_r + L_p, steady state
                attends N_att + L_p rows, and the two reduction factors.
* ties       -- exact ties go to the oldest position (the reading taken).
"""
from __future__ import annotations

import json
import os

import numpy as np
import torch

from oracle.oracle import OracleStream

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def sdpa(q: np.ndarray, K: np.ndarray, V: np.ndarray) -> np.ndarray:
    """torch's scaled dot-product attention in fp64 for one query."""
    qt = torch.from_numpy(np.asarray(q, dtype=np.float64))[None, None, None, :]
    Kt = torch.from_numpy(np.asarray(K, dtype=np.float64))[None, None]
    Vt = torch.from_numpy(np.asarray(V, dtype=np.float64))[None, None]
    return torch.nn.functional.scaled_dot_product_attention(qt, Kt, Vt)[0, 0, 0].numpy()


def _trace(rng, d, L_p, L_dec):
    Kp, Vp = rng.standard_normal((L_p, d)), rng.standard_normal((L_p, d))
    q, k, v = (rng.standard_normal((L_dec, d)) for _ in range(3))
    return Kp, Vp, q, k, v


def _close(a, b, tol=1e-10):
    return np.allclose(a, b, rtol=tol, atol=tol)


def pin_dense(mutation=None):
    fails = []
    rng = np.random.default_rng(11)
    d, L_p, L_dec = 8, 5, 12
    Kp, Vp, q, k, v = _trace(rng, d, L_p, L_dec)
    st = OracleStream(d, L_p, L_dec, L_dec, 0, mutation)
    st.prefill(Kp, Vp)
    for t in range(L_dec):
        out, info = st.step(q[t], k[t], v[t])
        ref = sdpa(q[t], np.vstack([Kp, k[: t + 1]]), np.vstack([Vp, v[: t + 1]]))
        if not _close(out, ref):
            fails.append(f"dense t={t}: max err {np.abs(out - ref).max():.3e}")
        if info.selected != -1:
            fails.append(f"dense t={t}: selected {info.selected}")
    return fails


def pin_sliding(mutation=None):
    fails = []
    rng = np.random.default_rng(12)
    d, L_p, L_dec, N = 8, 3, 14, 5
    Kp, Vp, q, k, v = _trace(rng, d, L_p, L_dec)
    st = OracleStream(d, L_p, N, N, 0, mutation)
    st.prefill(Kp, Vp)
    for t in range(L_dec):
        out, info = st.step(q[t], k[t], v[t])
        lo = max(0, t - N + 1)
        ref = sdpa(q[t], np.vstack([Kp, k[lo: t + 1]]), np.vstack([Vp, v[lo: t + 1]]))
        if not _close(out, ref):
            fails.append(f"sliding t={t}: max err {np.abs(out - ref).max():.3e}")
        if info.selected != -1:
            fails.append(f"sliding t={t}: selected {info.selected}")
    return fails


def pin_streaming(mutation=None):
    fails = []
    rng = np.random.default_rng(13)
    d, L_p, L_dec, N, sink = 8, 3, 18, 7, 4
    Kp, Vp, q, k, v = _trace(rng, d, L_p, L_dec)
    st = OracleStream(d, L_p, N, N, sink, mutation)
    st.prefill(Kp, Vp)
    for t in range(L_dec):
        out, _ = st.step(q[t], k[t], v[t])
        keep = list(range(0, min(t, sink - 1) + 1)) + list(range(max(sink, t - (N - sink) + 1), t + 1))
        ref = sdpa(q[t], np.vstack([Kp, k[keep]]), np.vstack([Vp, v[keep]]))
        if not _close(out, ref):
            fails.append(f"streaming t={t}: max err {np.abs(out - ref).max():.3e}")
    return fails


def worked_example_inputs():
    """Engineered inputs for Fig. 12: q_3 = e0 makes K0 the lowest at t=3,
    q_4 = e1 makes K2 the lowest among {K0, K2, K3, K4} at t=4."""
    d, L_p, L_dec = 4, 2, 10
    a = [-2.0, 1.0, 0.5, 0.3, 0.9, 0.7, 0.2, 0.6, 0.8, 0.4]
    b = [0.0, 1.0, -2.0, 0.5, 0.2, 0.4, 0.6, 0.1, 0.3, 0.7]
    c = [0.4, -1.5, 0.0, 0.2, 0.3, 0.1, 0.5, 0.6, 0.7, 0.9]
    k = np.array([[a[j], b[j], c[j], 0.25] for j in range(L_dec)])
    v = np.arange(L_dec * d, dtype=np.float64).reshape(L_dec, d) / 10.0
    q = np.zeros((L_dec, d))
    for t in range(L_dec):
        q[t, 0 if t <= 3 else 1 if t == 4 else 2 if t == 5 else 3] = 1.0
    Kp = np.full((L_p, d), 0.1)
    Vp = np.ones((L_p, d))
    return d, L_p, L_dec, Kp, Vp, q, k, v


def pin_worked(mutation=None):
    with open(os.path.join(GOLDEN, "worked_example.json")) as f:
        g = json.load(f)
    F = {k: v["value"] for k, v in g["facts"].items()}
    N_r, N_att = g["N_r"], g["N_att"]
    d, L_p, L_dec, Kp, Vp, q, k, v = worked_example_inputs()
    st = OracleStream(d, L_p, N_r, N_att, 0, mutation)
    st.prefill(Kp, Vp)
    fails = []
    prev_skip = []
    for t in range(L_dec):
        _, info = st.step(q[t], k[t], v[t])
        skip, idx = st.skip(), st.idx()
        shifted = sorted(set(skip) - ({info.selected} if info.selected >= 0 else set()))
        if t in F["full_attention_steps"] and (info.phase != 1 or prev_skip):
            fails.append(f"worked t={t}: expected full attention, phase {info.phase}")
        if t == 3:
            if idx != F["t3_scored"]:
                fails.append(f"worked t=3: scored {idx}")
            if info.selected != F["t3_pick"] or sorted(skip) != F["t3_skip_after"]:
                fails.append(f"worked t=3: pick {info.selected} skip {skip}")
        if t == 4:
            if shifted != F["t4_skip_after_shift"] or idx != F["t4_idx"]:
                fails.append(f"worked t=4: shifted {shifted} idx {idx}")
            if info.selected != F["t4_pick"] or sorted(skip) != F["t4_skip_after"]:
                fails.append(f"worked t=4: pick {info.selected} skip {skip}")
        if t == 5 and shifted != F["t5_skip_after_shift"]:
            fails.append(f"worked t=5: shifted {shifted}")
        if t >= 3 and info.n_idx != F["attended_in_phase3"]:
            fails.append(f"worked t={t}: |idx| = {info.n_idx}")
        if t == F["first_evict_step"] - 1 and info.phase == 3:
            fails.append("worked: evicted before t=7")
        if t == F["first_evict_step"]:
            if info.phase != 3 or F["t7_evicted"] in idx or info.live_rows != N_r:
                fails.append(f"worked t=7: phase {info.phase} idx {idx} live {info.live_rows}")
        prev_skip = skip
    if len(prev_skip) != F["final_skip_size"]:
        fails.append(f"worked: final |skip| = {len(prev_skip)}")
    return fails


INVARIANT_CASES = [
    # (L_p, N_r, N_att, sink, L_dec, d)
    (3, 7, 4, 0, 20, 6),
    (2, 9, 1, 0, 25, 4),
    (4, 12, 12, 0, 20, 4),
    (3, 10, 6, 4, 26, 5),
    (0, 6, 3, 0, 15, 4),
    (5, 16, 5, 0, 40, 8),
    (2, 8, 5, 4, 22, 4),
]


def pin_invariants(mutation=None):
    fails = []
    rng = np.random.default_rng(14)
    for (L_p, N_r, N_att, sink, L_dec, d) in INVARIANT_CASES:
        tag = f"inv(L_p={L_p},N_r={N_r},N_att={N_att},sink={sink})"
        Kp, Vp, q, k, v = _trace(rng, d, L_p, L_dec)
        st = OracleStream(d, L_p, N_r, N_att, sink, mutation)
        st.prefill(Kp, Vp)
        Nr, Na = N_r - sink, N_att - sink
        offsets = set()
        n_sel = 0
        for t in range(L_dec):
            _, info = st.step(q[t], k[t], v[t])
            skip, idx = st.skip(), st.idx()
            tt = t - sink
            if L_p + info.live_rows > N_r + L_p:
                fails.append(f"{tag} t={t}: KV held {L_p + info.live_rows} > N_r + L_p")
            attended = (info.n_prefix - L_p) + info.n_idx
            if attended != min(t + 1, N_att):
                fails.append(f"{tag} t={t}: attended decode {attended} != {min(t + 1, N_att)}")
            if info.n_prefix != L_p + min(t + 1 if t < sink else sink, sink):
                fails.append(f"{tag} t={t}: prefix rows {info.n_prefix}")
            should_select = tt >= 0 and Na - 1 <= tt <= Nr - 2
            if (info.selected >= 0) != should_select:
                fails.append(f"{tag} t={t}: selected={info.selected}, expected selection={should_select}")
            n_sel += info.selected >= 0
            if info.n_skip != n_sel or info.n_skip > Nr - Na:
                fails.append(f"{tag} t={t}: |skip| {info.n_skip} after {n_sel} selections")
            if tt >= 0:
                new = {tt - j for j in skip}
                added = {tt - info.selected} if info.selected >= 0 else set()
                if new != offsets | added:
                    fails.append(f"{tag} t={t}: relative offsets changed {sorted(offsets)} -> {sorted(new)}")
                offsets = new
                lo = max(0, tt - Nr + 1)
                if any(j < lo or j > tt for j in skip):
                    fails.append(f"{tag} t={t}: skip {skip} outside live window [{lo}, {tt}]")
                if any(j < lo or j > tt for j in idx):
                    fails.append(f"{tag} t={t}: idx {idx} outside live window")
                if set(idx) & (set(skip) - ({info.selected} if info.selected >= 0 else set())):
                    fails.append(f"{tag} t={t}: idx {idx} meets skip {skip}")
    return fails


def _relative_model(Kp, Vp, q, k, v, N_r, N_att, sink):
    """Independent brute force: skipped rows kept as relative offsets r = t - p
    (the diagonal premise, section 4 "Algorithm overview"); argmin of the
    softmax weights w of the attended decode rows."""
    L_dec, d = q.shape
    R: set[int] = set()
    Nr, Na = N_r - sink, N_att - sink
    outs, atts, picks = [], [], []
    for t in range(L_dec):
        if t < sink:
            rows = list(range(t + 1))
            att = []
            outs.append(sdpa(q[t], np.vstack([Kp, k[rows]]), np.vstack([Vp, v[rows]])))
            atts.append(att)
            picks.append(-1)
            continue
        tt = t - sink
        live = range(max(0, tt - Nr + 1), tt + 1)
        att = [p for p in live if (tt - p) not in R]
        rows = list(range(sink)) + [p + sink for p in att]
        outs.append(sdpa(q[t], np.vstack([Kp, k[rows]]), np.vstack([Vp, v[rows]])))
        atts.append(att)
        pick = -1
        if tt >= Na - 1 and len(R) < Nr - Na:
            logits = np.array([q[t] @ k[p + sink] for p in att])
            w = np.exp(logits - logits.max())
            w /= w.sum()
            pick = att[int(np.argmin(w))]
            R.add(tt - pick)
        picks.append(pick)
    return outs, atts, picks


RELATIVE_CASES = [
    (2, 7, 4, 0, 16, 4),
    (1, 5, 2, 0, 14, 3),
    (3, 8, 3, 0, 20, 4),
    (2, 9, 6, 2, 20, 4),
    (0, 4, 1, 0, 10, 2),
]


def pin_relative(mutation=None):
    fails = []
    rng = np.random.default_rng(15)
    for (L_p, N_r, N_att, sink, L_dec, d) in RELATIVE_CASES:
        tag = f"rel(L_p={L_p},N_r={N_r},N_att={N_att},sink={sink})"
        Kp, Vp, q, k, v = _trace(rng, d, L_p, L_dec)
        outs, atts, picks = _relative_model(Kp, Vp, q, k, v, N_r, N_att, sink)
        st = OracleStream(d, L_p, N_r, N_att, sink, mutation)
        st.prefill(Kp, Vp)
        for t in range(L_dec):
            out, info = st.step(q[t], k[t], v[t])
            if st.idx() != atts[t] and t >= sink:
                fails.append(f"{tag} t={t}: idx {st.idx()} vs {atts[t]}")
            if info.selected != picks[t]:
                fails.append(f"{tag} t={t}: pick {info.selected} vs {picks[t]}")
            if not _close(out, outs[t]):
                fails.append(f"{tag} t={t}: out err {np.abs(out - outs[t]).max():.3e}")
    return fails


def pin_cost(mutation=None):
    fails = []
    rng = np.random.default_rng(16)
    d, L_p, L_dec, N_r, N_att = 6, 3, 20, 10, 4
    Kp, Vp, q, k, v = _trace(rng, d, L_p, L_dec)
    sp = OracleStream(d, L_p, N_r, N_att, 0, mutation)
    dn = OracleStream(d, L_p, L_dec, L_dec, 0, mutation)
    sp.prefill(Kp, Vp)
    dn.prefill(Kp, Vp)
    sel_steps, peak_sparse, peak_dense = [], 0, 0
    last_sparse = last_dense = None
    for t in range(L_dec):
        _, i1 = sp.step(q[t], k[t], v[t])
        _, i2 = dn.step(q[t], k[t], v[t])
        if i1.selected >= 0:
            sel_steps.append(t)
        peak_sparse = max(peak_sparse, L_p + i1.live_rows)
        peak_dense = max(peak_dense, L_p + i2.live_rows)
        last_sparse, last_dense = i1.n_prefix + i1.n_idx, i2.n_prefix + i2.n_idx
    if sel_steps != list(range(N_att - 1, N_r - 1)):
        fails.append(f"cost: selection steps {sel_steps}")
    if peak_sparse != N_r + L_p:
        fails.append(f"cost: peak KV {peak_sparse} != N_r + L_p")
    if last_sparse != N_att + L_p:
        fails.append(f"cost: steady attended {last_sparse} != N_att + L_p")
    if abs(peak_dense / peak_sparse - (L_dec + L_p) / (N_r + L_p)) > 1e-12:
        fails.append("cost: memory reduction factor")
    if abs(last_dense / last_sparse - (L_dec + L_p) / (N_att + L_p)) > 1e-12:
        fails.append("cost: compute reduction factor")
    return fails


def pin_ties(mutation=None):
    fails = []
    rng = np.random.default_rng(17)
    d, L_p, L_dec, N_r, N_att = 4, 2, 12, 7, 4
    Kp, Vp, q, _, v = _trace(rng, d, L_p, L_dec)
    k = np.tile(rng.standard_normal(d), (L_dec, 1))  # every decode key alike: exact ties
    st = OracleStream(d, L_p, N_r, N_att, 0, mutation)
    st.prefill(Kp, Vp)
    for t in range(L_dec):
        _, info = st.step(q[t], k[t], v[t])
        idx = st.idx()
        if info.selected >= 0 and info.selected != idx[0]:
            fails.append(f"ties t={t}: picked {info.selected}, oldest attended is {idx[0]}")
    return fails


def _torch_e4m3_store(x: np.ndarray, scale: float) -> np.ndarray:
    """Library model of an FP8 E4M3 stored row: PyTorch's float8_e4m3fn of
    fp32(x) * fp32(1 / scale) (clamped to +-448, the format's largest finite
    value: the library maps beyond 464 to NaN), times scale."""
    inv = np.float32(1.0) / np.float32(scale)
    y = np.clip(x.astype(np.float32) * inv, -448.0, 448.0)
    c = torch.from_numpy(y).to(torch.float8_e4m3fn).to(torch.float64).numpy()
    return c * np.float64(np.float32(scale))


def pin_fp8_store(mutation=None):
    """FP8 KV storage: the oracle with E4M3 storage equals the plain oracle run
    on rows quantized by the library model, bit for bit (outputs and skip
    sets), with sinks, saturating and subnormal elements, and distinct K and
    V scales."""
    fails = []
    for sink in (0, 4):
        rng = np.random.default_rng(5 + sink)
        d, L_p, L_dec, N_r, N_att = 16, 6, 40, 14, 7
        ks, vs = 0.0123, 0.0371
        K = rng.normal(0, 2, (L_p, d)); V = rng.normal(0, 2, (L_p, d))
        q = rng.normal(0, 1, (L_dec, d)); k = rng.normal(0, 2, (L_dec, d)); v = rng.normal(0, 2, (L_dec, d))
        k[3, 0] = 1e3   # saturates
        v[5, 1] = -1e-4  # subnormal range
        a = OracleStream(d, L_p, N_r, N_att, sink, mutation=mutation, kv_scales=(ks, vs))
        b = OracleStream(d, L_p, N_r, N_att, sink)
        a.prefill(K, V)
        b.prefill(_torch_e4m3_store(K, ks), _torch_e4m3_store(V, vs))
        for t in range(L_dec):
            oa, ia = a.step(q[t], k[t], v[t])
            ob, ib = b.step(q[t], _torch_e4m3_store(k[t], ks), _torch_e4m3_store(v[t], vs))
            if not np.array_equal(oa, ob) or ia.selected != ib.selected or a.skip() != b.skip():
                fails.append(f"fp8 store, sink {sink}, t={t}: differs from the library model")
                break
    return fails


ALL_PINS = {
    "dense": pin_dense,
    "sliding": pin_sliding,
    "streaming": pin_streaming,
    "worked": pin_worked,
    "invariants": pin_invariants,
    "relative": pin_relative,
    "cost": pin_cost,
    "ties": pin_ties,
    "fp8_store": pin_fp8_store,
}
