"""Thin ctypes binding over libdsa.so (include/dsa.h).

The module-level functions carry the C names and only marshal arguments:
torch tensors become device pointers, torch streams become cudaStream_t.
Every step of the decode path runs in the library's CUDA kernels; there is
no fallback.  Importing this module raises if libdsa.so has not been built.

Method: "Understanding and Exploiting Diagonal Attention Sparsity in
Autoregressive Image Generation" (arXiv 2609.19702), section 4, Algorithm 1.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

from .build import LIB as _BUILT_LIB

# DSA_LIB may point at another build of the same library (e.g. a variant with
# a different pipeline shape); the default is the in-tree build.
LIB = os.environ.get("DSA_LIB", _BUILT_LIB)

if not os.path.exists(LIB):
    raise ImportError(f"libdsa.so is not built ({LIB}); run ar_image_gen_gb300.build.build()")

_L = ctypes.CDLL(LIB)

DSA_OK = 0
DSA_ERR_ARG = -1
DSA_ERR_STATE = -2
DSA_ERR_OOM = -3
DSA_ERR_CUDA = -4
DSA_ERR_TIMEOUT = -5
DSA_ERR_DEVICE_CHECK = -6
DSA_BF16 = 0
DSA_F32 = 1
DSA_FP8_E4M3 = 2
DTYPES = {"bf16": DSA_BF16, "f32": DSA_F32, "fp8e4m3": DSA_FP8_E4M3}

STATUS_NAMES = {0: "DSA_OK", -1: "DSA_ERR_ARG", -2: "DSA_ERR_STATE", -3: "DSA_ERR_OOM", -4: "DSA_ERR_CUDA",
                -5: "DSA_ERR_TIMEOUT", -6: "DSA_ERR_DEVICE_CHECK"}

EXPORTS = ["dsa_create", "dsa_create_ex", "dsa_prefill", "dsa_decode_step", "dsa_destroy", "dsa_get_step",
           "dsa_get_skip_mask", "dsa_get_last_selection", "dsa_sync_status", "dsa_last_error",
           "dsa_state_bytes", "dsa_plan_step", "dsa_plan_query", "dsa_set_kv_scales", "dsa_set_splits", "dsa_set_pipeline",
           "dsa_set_merge", "dsa_set_wait_limit", "dsa_debug_copy_state", "dsa_debug_set_step",
           "dsa_debug_fail_alloc_after", "dsa_decode_step_noalloc", "dsa_decode_step_noalloc_status", "dsa_diag_trace", "dsa_set_graph_mode",
           "dsa_sync_step",
           "dsa_proj_create", "dsa_proj_destroy", "dsa_qkv_rope", "dsa_decode_step_fused", "dsa_proj_sync_status",
           "dsa_proj_set_wait_limit", "dsa_pol_create", "dsa_pol_destroy", "dsa_pol_prefill", "dsa_pol_decode_step",
           "dsa_pol_get_positions", "dsa_pol_get_last_eviction", "dsa_pol_sync_status", "dsa_pol_set_wait_limit",
           "dsa_pol_set_shape"]


class dsa_step_plan(ctypes.Structure):
    _fields_ = [("phase", ctypes.c_int), ("t_inner", ctypes.c_int), ("n_prefix", ctypes.c_int),
                ("n_decode", ctypes.c_int), ("select", ctypes.c_int), ("nsplit", ctypes.c_int),
                ("chunk", ctypes.c_int), ("grid", ctypes.c_int), ("pipeline", ctypes.c_int),
                ("algo_bytes", ctypes.c_ulonglong), ("cta_merge", ctypes.c_int)]


_P = ctypes.c_void_p
_I = ctypes.c_int
_L.dsa_create.argtypes = [_I] * 6 + [ctypes.POINTER(_P)]
_L.dsa_create_ex.argtypes = [_I] * 7 + [ctypes.POINTER(_P)]
_L.dsa_prefill.argtypes = [_P, _P, _P, _P]
_L.dsa_decode_step.argtypes = [_P, _P, _P, _P, _P, _P]
_L.dsa_destroy.argtypes = [_P]
_L.dsa_get_step.argtypes = [_P, ctypes.POINTER(_I)]
_L.dsa_get_skip_mask.argtypes = [_P, _P, _P]
_L.dsa_get_last_selection.argtypes = [_P, _P, _P]
_L.dsa_sync_status.argtypes = [_P, _P]
_L.dsa_last_error.restype = ctypes.c_char_p
_L.dsa_state_bytes.argtypes = [_I] * 6
_L.dsa_state_bytes.restype = ctypes.c_size_t
_L.dsa_plan_step.argtypes = [_P, _I, ctypes.POINTER(dsa_step_plan)]
_L.dsa_plan_query.argtypes = [_I] * 9 + [_P, _P, ctypes.POINTER(dsa_step_plan)]
_L.dsa_set_splits.argtypes = [_P, _I]
_L.dsa_set_kv_scales.argtypes = [_P, _P, _P]
_L.dsa_debug_copy_state.argtypes = [_P, _P, _P]
_L.dsa_debug_set_step.argtypes = [_P, _I, _P]
_L.dsa_set_pipeline.argtypes = [_P, _I]
_L.dsa_set_merge.argtypes = [_P, _I]
_L.dsa_set_wait_limit.argtypes = [_P, ctypes.c_uint32]
_L.dsa_debug_fail_alloc_after.argtypes = [_I]
_L.dsa_set_graph_mode.argtypes = [_P, _I]
_L.dsa_sync_step.argtypes = [_P, _P]
_L.dsa_decode_step_noalloc.argtypes = [_I] * 8 + [_P] * 9
_L.dsa_decode_step_noalloc_status.argtypes = [_P]
_L.dsa_diag_trace.argtypes = [_I] * 5 + [_P] * 3 + [_I] + [_P] * 6
_L.dsa_proj_create.argtypes = [_I] * 4 + [ctypes.POINTER(_P)]
_L.dsa_proj_destroy.argtypes = [_P]
_L.dsa_qkv_rope.argtypes = [_P, _P, _P, _I, _P, _P, _P, _P]
_L.dsa_decode_step_fused.argtypes = [_P] * 6
_L.dsa_proj_sync_status.argtypes = [_P, _P]
_L.dsa_proj_set_wait_limit.argtypes = [_P, ctypes.c_uint32]
_L.dsa_pol_create.argtypes = [_I] * 6 + [ctypes.POINTER(_P)]
_L.dsa_pol_destroy.argtypes = [_P]
_L.dsa_pol_prefill.argtypes = [_P] * 4
_L.dsa_pol_decode_step.argtypes = [_P] * 6
_L.dsa_pol_get_positions.argtypes = [_P] * 3
_L.dsa_pol_get_last_eviction.argtypes = [_P] * 3
_L.dsa_pol_sync_status.argtypes = [_P] * 2
_L.dsa_pol_set_wait_limit.argtypes = [_P, ctypes.c_uint32]
_L.dsa_pol_set_shape.argtypes = [_P, _I]
DSA_POLICY_TOVA = 1
DSA_POLICY_H2O = 2
POLICIES = {"tova": DSA_POLICY_TOVA, "h2o": DSA_POLICY_H2O}


class DSAError(RuntimeError):
    def __init__(self, code: int, what: str):
        self.code = code
        super().__init__(f"{what}: {STATUS_NAMES.get(code, code)}: {dsa_last_error()}")


def _check(code: int, what: str) -> int:
    if code != DSA_OK:
        raise DSAError(code, what)
    return code


def _ptr(x) -> int | None:
    """Device (or host) address of a tensor / ndarray / int, None for None."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if hasattr(x, "data_ptr"):
        return x.data_ptr()
    if isinstance(x, np.ndarray):
        return x.ctypes.data
    raise TypeError(f"cannot take the address of {type(x)}")


def _stream(stream) -> int | None:
    if stream is None:
        try:
            import torch
            return torch.cuda.current_stream().cuda_stream
        except Exception:
            return None
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def library_path() -> str:
    return LIB


# ---- C names ---------------------------------------------------------------

def dsa_last_error() -> str:
    return (_L.dsa_last_error() or b"").decode()


def dsa_create(heads, head_dim, L_p, N_r, N_att, sink=0):
    h = _P()
    return _L.dsa_create(heads, head_dim, L_p, N_r, N_att, sink, ctypes.byref(h)), h


def dsa_create_ex(heads, head_dim, L_p, N_r, N_att, sink, dtype):
    h = _P()
    return _L.dsa_create_ex(heads, head_dim, L_p, N_r, N_att, sink, dtype, ctypes.byref(h)), h


def dsa_prefill(h, K, V, stream=None) -> int:
    return _L.dsa_prefill(h, _ptr(K), _ptr(V), _stream(stream))


def dsa_decode_step(h, q, k_new, v_new, out, stream=None) -> int:
    return _L.dsa_decode_step(h, _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(out), _stream(stream))


def dsa_destroy(h) -> int:
    return _L.dsa_destroy(h)


def dsa_get_step(h):
    t = _I()
    return _L.dsa_get_step(h, ctypes.byref(t)), t.value


def dsa_get_skip_mask(h, host_dst: np.ndarray, stream=None) -> int:
    assert host_dst.dtype == np.uint32 and host_dst.flags["C_CONTIGUOUS"]
    return _L.dsa_get_skip_mask(h, host_dst.ctypes.data, _stream(stream))


def dsa_get_last_selection(h, host_dst: np.ndarray, stream=None) -> int:
    assert host_dst.dtype == np.int32 and host_dst.flags["C_CONTIGUOUS"]
    return _L.dsa_get_last_selection(h, host_dst.ctypes.data, _stream(stream))


def dsa_sync_status(h, stream=None) -> int:
    return _L.dsa_sync_status(h, _stream(stream))


def dsa_state_bytes(heads, head_dim, L_p, N_r, sink=0, dtype=DSA_BF16) -> int:
    return int(_L.dsa_state_bytes(heads, head_dim, L_p, N_r, sink, dtype))


def dsa_plan_step(h, t):
    p = dsa_step_plan()
    return _L.dsa_plan_step(h, t, ctypes.byref(p)), p


def dsa_plan_query(heads, head_dim, L_p, N_r, N_att, sink, dtype, t, sm_count, ctas_per_sm, cta_merge_ok=None):
    """Host-only plan of step t for a state of these sizes on a device of
    `sm_count` SMs with the given resident CTAs per SM of the 4 launch
    pipelines (and where the in-CTA merge fits); returns (status, plan)."""
    ctas = (ctypes.c_int * 4)(*[int(c) for c in ctas_per_sm])
    ok = None if cta_merge_ok is None else (ctypes.c_int * 4)(*[int(c) for c in cta_merge_ok])
    p = dsa_step_plan()
    code = _L.dsa_plan_query(heads, head_dim, L_p, N_r, N_att, sink, dtype, t, sm_count, ctas, ok, ctypes.byref(p))
    return code, p


def dsa_set_kv_scales(h, k_scale: np.ndarray, v_scale: np.ndarray) -> int:
    k = np.ascontiguousarray(k_scale, dtype=np.float32)
    v = np.ascontiguousarray(v_scale, dtype=np.float32)
    return _L.dsa_set_kv_scales(h, k.ctypes.data, v.ctypes.data)


def dsa_debug_copy_state(h, host_prefix: np.ndarray | None, host_ring: np.ndarray | None) -> int:
    return _L.dsa_debug_copy_state(h, None if host_prefix is None else host_prefix.ctypes.data,
                                   None if host_ring is None else host_ring.ctypes.data)


def dsa_debug_set_step(h, t, stream=None) -> int:
    return _L.dsa_debug_set_step(h, t, _stream(stream))


def dsa_set_splits(h, nsplit) -> int:
    return _L.dsa_set_splits(h, nsplit)


def dsa_set_pipeline(h, pipeline) -> int:
    return _L.dsa_set_pipeline(h, pipeline)


def dsa_set_merge(h, mode) -> int:
    return _L.dsa_set_merge(h, mode)


def dsa_set_wait_limit(h, limit) -> int:
    return _L.dsa_set_wait_limit(h, limit)


def dsa_debug_fail_alloc_after(n) -> int:
    return _L.dsa_debug_fail_alloc_after(n)


def dsa_set_graph_mode(h, on) -> int:
    return _L.dsa_set_graph_mode(h, 1 if on else 0)


def dsa_sync_step(h, stream=None) -> int:
    return _L.dsa_sync_step(h, _stream(stream))


def dsa_decode_step_noalloc(heads, head_dim, L_p, N_r, N_att, sink, dtype, t, prefix, ring, mask, last_sel,
                            q, k_new, v_new, out, stream=None) -> int:
    return _L.dsa_decode_step_noalloc(heads, head_dim, L_p, N_r, N_att, sink, dtype, t, _ptr(prefix), _ptr(ring),
                                      _ptr(mask), _ptr(last_sel), _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(out),
                                      _stream(stream))


def dsa_decode_step_noalloc_status(stream=None) -> int:
    return _L.dsa_decode_step_noalloc_status(_stream(stream))


def dsa_diag_trace(heads, head_dim, L_p, L_dec, dtype, Q, Kp, Kd, dist: np.ndarray, step_mass, mass_mean: np.ndarray,
                   vertical: np.ndarray, diagonal: np.ndarray, stream=None) -> int:
    return _L.dsa_diag_trace(heads, head_dim, L_p, L_dec, dtype, _ptr(Q), _ptr(Kp), _ptr(Kd), len(dist), _ptr(dist),
                             _ptr(step_mass), _ptr(mass_mean), _ptr(vertical), _ptr(diagonal), _stream(stream))


def diag_trace(Q, Kp, Kd, dists, step_mass=None, stream=None):
    """Fig. 8 / Fig. 10 diagnostics of a dense decode trace (include/dsa_diag.h).
    Q, Kd: [heads, L_dec, d], Kp: [heads, L_p, d] device tensors (bf16 or fp32).
    Returns (mass_mean [3], vertical [n], diagonal [n]) as numpy arrays;
    step_mass, if given, is a device float tensor [heads, L_dec, 3] to fill."""
    import torch

    heads, L_dec, d = Q.shape
    L_p = Kp.shape[1] if Kp is not None else 0
    dtype = {torch.bfloat16: DSA_BF16, torch.float32: DSA_F32}[Q.dtype]
    dist = np.ascontiguousarray(dists, dtype=np.int32)
    mass = np.zeros(3)
    vert = np.zeros(len(dist))
    diag = np.zeros(len(dist))
    _check(dsa_diag_trace(heads, d, L_p, L_dec, dtype, Q, Kp if L_p > 0 else None, Kd, dist, step_mass, mass, vert,
                          diag, stream), "dsa_diag_trace")
    return mass, vert, diag


def dsa_proj_create(batch, heads, head_dim, hidden):
    p = _P()
    return _L.dsa_proj_create(batch, heads, head_dim, hidden, ctypes.byref(p)), p


def dsa_proj_destroy(p) -> int:
    return _L.dsa_proj_destroy(p)


def dsa_qkv_rope(p, x, W, pos, q, k, v, stream=None) -> int:
    return _L.dsa_qkv_rope(p, _ptr(x), _ptr(W), pos, _ptr(q), _ptr(k), _ptr(v), _stream(stream))


def dsa_decode_step_fused(h, p, x, W, out, stream=None) -> int:
    return _L.dsa_decode_step_fused(h, p, _ptr(x), _ptr(W), _ptr(out), _stream(stream))


def dsa_proj_sync_status(p, stream=None) -> int:
    return _L.dsa_proj_sync_status(p, _stream(stream))


def dsa_proj_set_wait_limit(p, limit) -> int:
    return _L.dsa_proj_set_wait_limit(p, limit)


def dsa_pol_create(heads, head_dim, L_p, N_att, policy, dtype):
    h = _P()
    return _L.dsa_pol_create(heads, head_dim, L_p, N_att, policy, dtype, ctypes.byref(h)), h


def dsa_pol_destroy(h) -> int:
    return _L.dsa_pol_destroy(h)


def dsa_pol_prefill(h, K, V, stream=None) -> int:
    return _L.dsa_pol_prefill(h, _ptr(K), _ptr(V), _stream(stream))


def dsa_pol_decode_step(h, q, k_new, v_new, out, stream=None) -> int:
    return _L.dsa_pol_decode_step(h, _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(out), _stream(stream))


def dsa_pol_get_positions(h, host_dst: np.ndarray, stream=None) -> int:
    assert host_dst.dtype == np.int32 and host_dst.flags["C_CONTIGUOUS"]
    return _L.dsa_pol_get_positions(h, host_dst.ctypes.data, _stream(stream))


def dsa_pol_get_last_eviction(h, host_dst: np.ndarray, stream=None) -> int:
    assert host_dst.dtype == np.int32 and host_dst.flags["C_CONTIGUOUS"]
    return _L.dsa_pol_get_last_eviction(h, host_dst.ctypes.data, _stream(stream))


def dsa_pol_sync_status(h, stream=None) -> int:
    return _L.dsa_pol_sync_status(h, _stream(stream))


def dsa_pol_set_wait_limit(h, limit) -> int:
    return _L.dsa_pol_set_wait_limit(h, limit)


def dsa_pol_set_shape(h, shape) -> int:
    return _L.dsa_pol_set_shape(h, shape)


# ---- convenience wrappers --------------------------------------------------

class Policy:
    """A score-based eviction baseline handle (include/dsa_policy.h):
    `heads` streams, `policy` "tova" or "h2o", N_att attended decode
    entries, bf16 or f32 rows."""

    def __init__(self, heads, head_dim, L_p, N_att, policy, dtype="bf16"):
        code, h = dsa_pol_create(heads, head_dim, L_p, N_att, POLICIES[policy], DTYPES[dtype])
        _check(code, "dsa_pol_create")
        self.h = h
        self.heads, self.head_dim, self.L_p, self.N_att, self.policy = heads, head_dim, L_p, N_att, policy

    def close(self):
        if getattr(self, "h", None):
            dsa_pol_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def prefill(self, K, V, stream=None):
        _check(dsa_pol_prefill(self.h, K, V, stream), "dsa_pol_prefill")

    def decode_step(self, q, k_new, v_new, out, stream=None):
        _check(dsa_pol_decode_step(self.h, q, k_new, v_new, out, stream), "dsa_pol_decode_step")

    def positions(self, stream=None) -> np.ndarray:
        dst = np.zeros((self.heads, self.N_att), dtype=np.int32)
        _check(dsa_pol_get_positions(self.h, dst, stream), "dsa_pol_get_positions")
        return dst

    def last_eviction(self, stream=None) -> np.ndarray:
        dst = np.zeros(self.heads, dtype=np.int32)
        _check(dsa_pol_get_last_eviction(self.h, dst, stream), "dsa_pol_get_last_eviction")
        return dst

    def sync_status(self, stream=None) -> int:
        return dsa_pol_sync_status(self.h, stream)

    def set_wait_limit(self, limit: int):
        _check(dsa_pol_set_wait_limit(self.h, limit), "dsa_pol_set_wait_limit")

    def set_shape(self, shape: int):
        _check(dsa_pol_set_shape(self.h, shape), "dsa_pol_set_shape")


class Proj:
    """A QKV projection context (include/dsa_proj.h): `batch` tokens, `heads`
    heads of `head_dim`, `hidden` input features."""

    def __init__(self, batch, heads, head_dim, hidden):
        code, p = dsa_proj_create(batch, heads, head_dim, hidden)
        _check(code, "dsa_proj_create")
        self.p = p
        self.batch, self.heads, self.head_dim, self.hidden = batch, heads, head_dim, hidden

    def close(self):
        if getattr(self, "p", None):
            dsa_proj_destroy(self.p)
            self.p = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def qkv_rope(self, x, W, pos, q, k, v, stream=None):
        _check(dsa_qkv_rope(self.p, x, W, pos, q, k, v, stream), "dsa_qkv_rope")

    def sync_status(self, stream=None) -> int:
        return dsa_proj_sync_status(self.p, stream)

    def set_wait_limit(self, limit: int):
        _check(dsa_proj_set_wait_limit(self.p, limit), "dsa_proj_set_wait_limit")


class DSA:
    """One handle: `heads` streams of one layer stepping together."""

    def __init__(self, heads, head_dim, L_p, N_r, N_att, sink=0, dtype="bf16"):
        self.dtype_code = DTYPES[dtype]
        code, h = dsa_create_ex(heads, head_dim, L_p, N_r, N_att, sink, self.dtype_code)
        _check(code, "dsa_create_ex")
        self.h = h
        self.heads, self.head_dim, self.L_p, self.N_r, self.N_att, self.sink = heads, head_dim, L_p, N_r, N_att, sink
        self.mask_words = (N_r - sink + 31) // 32

    def close(self):
        if getattr(self, "h", None):
            dsa_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def prefill(self, K, V, stream=None):
        _check(dsa_prefill(self.h, K, V, stream), "dsa_prefill")

    def decode_step(self, q, k_new, v_new, out, stream=None):
        _check(dsa_decode_step(self.h, q, k_new, v_new, out, stream), "dsa_decode_step")

    def decode_step_fused(self, proj: "Proj", x, W, out, stream=None):
        """Projection of x by W (position L_p + t) and the decode step on it."""
        _check(dsa_decode_step_fused(self.h, proj.p, x, W, out, stream), "dsa_decode_step_fused")

    @property
    def t(self) -> int:
        code, t = dsa_get_step(self.h)
        _check(code, "dsa_get_step")
        return t

    def skip_mask(self, stream=None) -> np.ndarray:
        dst = np.zeros((self.heads, self.mask_words), dtype=np.uint32)
        _check(dsa_get_skip_mask(self.h, dst, stream), "dsa_get_skip_mask")
        return dst

    def last_selection(self, stream=None) -> np.ndarray:
        dst = np.zeros(self.heads, dtype=np.int32)
        _check(dsa_get_last_selection(self.h, dst, stream), "dsa_get_last_selection")
        return dst

    def sync_status(self, stream=None) -> int:
        return dsa_sync_status(self.h, stream)

    def state_bytes(self) -> int:
        """Device bytes of the handle's KV state (prefix, ring, skip mask)."""
        return dsa_state_bytes(self.heads, self.head_dim, self.L_p, self.N_r, self.sink, self.dtype_code)

    def plan(self, t: int | None = None) -> dsa_step_plan:
        code, p = dsa_plan_step(self.h, self.t if t is None else t)
        _check(code, "dsa_plan_step")
        return p

    def set_kv_scales(self, k_scale, v_scale):
        """Per-stream FP8 scales (host arrays of `heads` floats); a prefill must follow."""
        _check(dsa_set_kv_scales(self.h, k_scale, v_scale), "dsa_set_kv_scales")

    def copy_state(self):
        """(prefix, ring) as uint8 arrays [heads, rows, 2, head_dim * element bytes]."""
        eb = {DSA_BF16: 2, DSA_F32: 4, DSA_FP8_E4M3: 1}[self.dtype_code]
        pre = np.zeros((self.heads, self.L_p + self.sink, 2, self.head_dim * eb), dtype=np.uint8)
        ring = np.zeros((self.heads, self.N_r - self.sink, 2, self.head_dim * eb), dtype=np.uint8)
        _check(dsa_debug_copy_state(self.h, pre, ring), "dsa_debug_copy_state")
        return pre, ring

    def set_splits(self, nsplit: int):
        _check(dsa_set_splits(self.h, nsplit), "dsa_set_splits")

    def debug_set_step(self, t: int, stream=None):
        """N_att == N_r handles only, right after prefill: jump to step t
        (the skipped-over decode entries read as zero rows)."""
        _check(dsa_debug_set_step(self.h, t, stream), "dsa_debug_set_step")

    def set_pipeline(self, pipeline: int):
        _check(dsa_set_pipeline(self.h, pipeline), "dsa_set_pipeline")

    def set_merge(self, mode: int):
        """0: split streams merged inside the CTA where possible; 1: always by the merge launch."""
        _check(dsa_set_merge(self.h, mode), "dsa_set_merge")

    def set_wait_limit(self, limit: int):
        _check(dsa_set_wait_limit(self.h, limit), "dsa_set_wait_limit")

    def set_graph_mode(self, on: bool):
        """Steady-state steps replayable from a CUDA graph (the step lives on the device)."""
        _check(dsa_set_graph_mode(self.h, on), "dsa_set_graph_mode")

    def sync_step(self, stream=None):
        _check(dsa_sync_step(self.h, stream), "dsa_sync_step")
