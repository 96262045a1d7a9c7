"""Python wrapper over the C oracle (``dsa_oracle.c``).

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` use this module.  The CUDA library and its
binding never import it.

The oracle is the literal statement of Algorithm 1 ("Diagonal-Aware Sparse
Attention", arXiv 2609.19702 section 4) in fp64; see the header of
``dsa_oracle.c`` for the readings taken where the page is open.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import sysconfig

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "dsa_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")

# Planted mistakes (see dsa_oracle.c); only the pin tests use them.
MUTATIONS = {
    "no_shift": 1,
    "argmax": 2,
    "no_prompt": 3,
    "no_evict": 4,
    "late_phase2": 5,
    "scale": 6,
    "skip_now": 7,
    "budget": 8,
    "newest_tie": 9,
    "fp8_swap": 10,
    "fp8_scale": 11,
    "fp8_trunc": 12,
    "fp8_prompt": 13,
}


class OrcInfo(ctypes.Structure):
    _fields_ = [
        ("phase", ctypes.c_int),
        ("t", ctypes.c_int),
        ("t_inner", ctypes.c_int),
        ("n_prefix", ctypes.c_int),
        ("n_idx", ctypes.c_int),
        ("selected", ctypes.c_int),
        ("oracle_pick", ctypes.c_int),
        ("adopted", ctypes.c_int),
        ("mismatch", ctypes.c_int),
        ("live_rows", ctypes.c_int),
        ("n_skip", ctypes.c_int),
        ("min_logit", ctypes.c_double),
        ("pick_logit", ctypes.c_double),
    ]

    def as_dict(self) -> dict:
        return {name: getattr(self, name) for name, _ in self._fields_}


def build(force: bool = False) -> str:
    """Compiles the oracle with the host C compiler (OpenMP if available)."""
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    cc = os.environ.get("CC", "gcc")
    base = [cc, "-O2", "-std=c11", "-shared", "-fPIC", _SRC, "-o", _LIB + ".tmp", "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True, capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True)
    os.replace(_LIB + ".tmp", _LIB)
    return _LIB


_lib = None


def lib() -> ctypes.CDLL:
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(_LIB)
        P = ctypes.c_void_p
        dp = ctypes.POINTER(ctypes.c_double)
        ip = ctypes.POINTER(ctypes.c_int)
        L.orc_create.restype = P
        L.orc_create.argtypes = [ctypes.c_int] * 5
        L.orc_destroy.argtypes = [P]
        L.orc_set_mutation.argtypes = [P, ctypes.c_int]
        L.orc_prefill.argtypes = [P, dp, dp]
        L.orc_step.argtypes = [P, dp, dp, dp, dp, ctypes.c_int, ctypes.POINTER(OrcInfo)]
        L.orc_get_skip.argtypes = [P, ip, ctypes.c_int]
        L.orc_get_idx.argtypes = [P, ip, ctypes.c_int]
        L.orc_get_step.argtypes = [P]
        L.orc_step_batch.argtypes = [ctypes.POINTER(P), ctypes.c_int, dp, dp, dp, dp, ip,
                                     ctypes.POINTER(OrcInfo), ctypes.c_int]
        L.orc_max_threads.restype = ctypes.c_int
        L.orc_set_kv_fp8.argtypes = [P, ctypes.c_float, ctypes.c_float]
        L.orc_e4m3_encode.argtypes = [ctypes.c_float]
        L.orc_e4m3_encode.restype = ctypes.c_ubyte
        L.orc_e4m3_decode.argtypes = [ctypes.c_ubyte]
        L.orc_e4m3_decode.restype = ctypes.c_double
        L.orc_diag_stream.argtypes = [ctypes.c_int] * 3 + [dp] * 3 + [ctypes.c_int, ip, dp, dp, dp]
        L.orc_diag_set_mutation.argtypes = [ctypes.c_int]
        _lib = L
    return _lib


def _dptr(a: np.ndarray):
    assert a.dtype == np.float64 and a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def e4m3_encode(y: float) -> int:
    """The oracle's E4M3 code of the fp32 value y (nearest, ties to even, satfinite)."""
    return int(lib().orc_e4m3_encode(float(y)))


def e4m3_decode(c: int) -> float:
    """The value of E4M3 code c."""
    return float(lib().orc_e4m3_decode(int(c)))


class OracleStream:
    """One (sequence, layer, head) stream of Algorithm 1.  With `kv_scales`
    = (k_scale, v_scale) the stream stores its K and V rows as FP8 E4M3 codes
    with those scales (see dsa_oracle.c)."""

    def __init__(self, d: int, L_p: int, N_r: int, N_att: int, sink: int = 0, mutation: str | None = None,
                 kv_scales: tuple[float, float] | None = None):
        self._h = lib().orc_create(d, L_p, N_r, N_att, sink)
        if not self._h:
            raise ValueError(f"oracle rejects d={d} L_p={L_p} N_r={N_r} N_att={N_att} sink={sink}")
        self.d, self.L_p, self.N_r, self.N_att, self.sink = d, L_p, N_r, N_att, sink
        if mutation:
            lib().orc_set_mutation(self._h, MUTATIONS[mutation])
        if kv_scales is not None:
            if lib().orc_set_kv_fp8(self._h, float(kv_scales[0]), float(kv_scales[1])) != 0:
                raise ValueError(f"oracle rejects the scales {kv_scales}")

    def __del__(self):
        h, self._h = getattr(self, "_h", None), None
        if h and _lib is not None:
            _lib.orc_destroy(h)

    def prefill(self, Kp: np.ndarray, Vp: np.ndarray) -> None:
        Kp = np.ascontiguousarray(Kp, dtype=np.float64).reshape(self.L_p, self.d)
        Vp = np.ascontiguousarray(Vp, dtype=np.float64).reshape(self.L_p, self.d)
        lib().orc_prefill(self._h, _dptr(Kp), _dptr(Vp))

    def step(self, q, k, v, pick: int = -1):
        q = np.ascontiguousarray(q, dtype=np.float64)
        k = np.ascontiguousarray(k, dtype=np.float64)
        v = np.ascontiguousarray(v, dtype=np.float64)
        out = np.zeros(self.d, dtype=np.float64)
        info = OrcInfo()
        r = lib().orc_step(self._h, _dptr(q), _dptr(k), _dptr(v), _dptr(out), int(pick), ctypes.byref(info))
        if r != 0:
            raise RuntimeError("oracle step failed")
        return out, info

    @property
    def t(self) -> int:
        return lib().orc_get_step(self._h)

    def skip(self) -> list[int]:
        buf = (ctypes.c_int * (self.N_r + 2))()
        n = lib().orc_get_skip(self._h, buf, len(buf))
        return list(buf[:n])

    def idx(self) -> list[int]:
        buf = (ctypes.c_int * (self.N_r + 2))()
        n = lib().orc_get_idx(self._h, buf, len(buf))
        return list(buf[:n])


class OracleBatch:
    """n independent streams stepped together (optionally on host threads)."""

    def __init__(self, n: int, d: int, L_p: int, N_r: int, N_att: int, sink: int = 0,
                 k_scales=None, v_scales=None):
        """k_scales, v_scales: per-stream scales of FP8 E4M3 storage, or None."""
        if (k_scales is None) != (v_scales is None):
            raise ValueError("give both k_scales and v_scales, or neither")
        self.streams = [OracleStream(d, L_p, N_r, N_att, sink,
                                     kv_scales=None if k_scales is None else (k_scales[i], v_scales[i]))
                        for i in range(n)]
        self.n, self.d = n, d
        self._arr = (ctypes.c_void_p * n)(*[s._h for s in self.streams])
        self._infos = (OrcInfo * n)()

    def prefill(self, Kp: np.ndarray, Vp: np.ndarray) -> None:
        for i, s in enumerate(self.streams):
            s.prefill(Kp[i], Vp[i])

    def step(self, q, k, v, picks=None, threads: int = 1):
        q = np.ascontiguousarray(q, dtype=np.float64)
        k = np.ascontiguousarray(k, dtype=np.float64)
        v = np.ascontiguousarray(v, dtype=np.float64)
        out = np.zeros((self.n, self.d), dtype=np.float64)
        pk = None
        if picks is not None:
            pk_arr = np.ascontiguousarray(picks, dtype=np.int32)
            pk = pk_arr.ctypes.data_as(ctypes.POINTER(ctypes.c_int))
        bad = lib().orc_step_batch(self._arr, self.n, _dptr(q), _dptr(k), _dptr(v), _dptr(out),
                                   pk, self._infos, int(threads))
        if bad:
            raise RuntimeError(f"oracle step failed on {bad} streams")
        return out, [self._infos[i] for i in range(self.n)]


def max_threads() -> int:
    return int(lib().orc_max_threads())


DIAG_MUTATIONS = {"local_floor": 1, "shift_query": 2, "with_prompt": 3}


def diag_set_mutation(name: str | None) -> None:
    """Plants a mistake in the diagnostics (pin tests only); None restores."""
    lib().orc_diag_set_mutation(DIAG_MUTATIONS[name] if name else 0)


def diag_stream(Q, Kp, Kd, dists):
    """Fig. 8 / Fig. 10 diagnostics of one stream's dense trace (see
    orc_diag_stream): returns (mass [L_dec, 3], vertical [n], diagonal [n]),
    the similarities averaged over the queries i = 0 .. L_dec - 1 - d."""
    Q = np.ascontiguousarray(Q, dtype=np.float64)
    Kd = np.ascontiguousarray(Kd, dtype=np.float64)
    Kp = np.ascontiguousarray(Kp, dtype=np.float64).reshape(-1, Q.shape[1])
    L_dec, d = Q.shape
    dist = np.ascontiguousarray(dists, dtype=np.int32)
    if (dist < 1).any() or (dist >= L_dec).any():
        raise ValueError("distances must lie in [1, L_dec)")
    mass = np.zeros((L_dec, 3)); vs = np.zeros(len(dist)); ds = np.zeros(len(dist))
    r = lib().orc_diag_stream(d, Kp.shape[0], L_dec, _dptr(Q), _dptr(Kp if Kp.size else np.zeros(1)), _dptr(Kd),
                              len(dist), dist.ctypes.data_as(ctypes.POINTER(ctypes.c_int)), _dptr(mass), _dptr(vs),
                              _dptr(ds))
    if r != 0:
        raise RuntimeError("oracle diagnostics failed")
    cnt = L_dec - dist
    return mass, vs / cnt, ds / cnt
