"""The C-ABI library without a GPU: it builds, loads, exports every symbol
the headers in include/ declare, and rejects bad arguments on the host."""
import ctypes
import os
import re

import pytest

from __graft_entry__ import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def dsa():
    build()
    from ar_image_gen_gb300 import dsa as mod
    return mod


def declared_functions():
    names = set()
    for h in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if h.endswith(".h"):
            text = open(os.path.join(ROOT, "include", h)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names |= set(re.findall(r"\b(dsa_[a-z_]+)\s*\(", text))
    return sorted(names)


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("dsa_create", "dsa_prefill", "dsa_decode_step", "dsa_destroy"):
        assert required in names


def test_library_exports_every_declared_symbol(dsa):
    lib = ctypes.CDLL(dsa.library_path())
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing
    assert set(declared_functions()) == set(dsa.EXPORTS)


@pytest.mark.parametrize("args", [
    (0, 128, 64, 288, 29, 0),      # no streams
    (8, 96, 64, 288, 29, 0),       # unsupported head_dim
    (8, 128, -1, 288, 29, 0),      # negative prompt
    (8, 128, 64, 288, 0, 0),       # N_att < 1
    (8, 128, 64, 288, 289, 0),     # N_att > N_r
    (8, 128, 64, 288, 4, 4),       # N_att <= sink
    (8, 128, 64, 288, 29, -1),     # negative sink
    (8, 128, 64, 70000, 29, 0),    # window beyond the 16-bit offset range
])
def test_create_rejects_bad_arguments(dsa, args):
    code, h = dsa.dsa_create(*args)
    assert code == dsa.DSA_ERR_ARG
    assert not h.value
    assert dsa.dsa_last_error()


def test_create_rejects_bad_dtype(dsa):
    code, h = dsa.dsa_create_ex(8, 128, 64, 288, 29, 0, 7)
    assert code == dsa.DSA_ERR_ARG and "dtype" in dsa.dsa_last_error()


def test_calls_on_a_null_handle_fail_cleanly(dsa):
    null = ctypes.c_void_p()
    assert dsa.dsa_destroy(null) == dsa.DSA_OK
    assert dsa.dsa_prefill(null, None, None) == dsa.DSA_ERR_STATE
    assert dsa.dsa_decode_step(null, 16, 16, 16, 16) == dsa.DSA_ERR_STATE
    assert dsa.dsa_get_step(null)[0] == dsa.DSA_ERR_STATE
    assert dsa.dsa_sync_status(null) == dsa.DSA_ERR_STATE
    assert dsa.dsa_plan_step(null, 0)[0] == dsa.DSA_ERR_STATE
    assert dsa.dsa_debug_set_step(null, 5) == dsa.DSA_ERR_STATE


def test_state_bytes_is_the_kv_bound(dsa):
    # prefix (L_p + sink) + ring (N_r - sink) rows of K and V, plus the mask:
    # the N_r + L_p footprint of the cost analysis.
    S, d, L_p, N_r = 3072, 128, 64, 288
    row = 2 * d * 2
    assert dsa.dsa_state_bytes(S, d, L_p, N_r, 0, dsa.DSA_BF16) == S * ((L_p + N_r) * row + 9 * 4)
    assert dsa.dsa_state_bytes(S, d, L_p, N_r, 4, dsa.DSA_BF16) == S * ((L_p + N_r) * row + 9 * 4)
    assert dsa.dsa_state_bytes(4, 64, 16, 32, 0, dsa.DSA_F32) == 4 * (48 * 2 * 64 * 4 + 4)
    assert dsa.dsa_state_bytes(0, 128, 64, 288, 0, 0) == 0


@pytest.mark.parametrize("kw", [
    dict(heads=0), dict(head_dim=96), dict(L_p=-1), dict(L_dec=0), dict(dtype=2), dict(dist=[0]), dict(dist=[40]),
])
def test_diag_rejects_bad_arguments(dsa, kw):
    import numpy as np

    a = dict(heads=2, head_dim=64, L_p=4, L_dec=40, dtype=dsa.DSA_BF16, dist=[1, 3])
    a.update(kw)
    dist = np.array(a["dist"], dtype=np.int32)
    z = np.zeros(8)
    fake = 1 << 20  # never dereferenced: every case fails validation first
    rc = dsa.dsa_diag_trace(a["heads"], a["head_dim"], a["L_p"], a["L_dec"], a["dtype"], fake, fake, fake, dist, None,
                            z, z, z)
    assert rc == dsa.DSA_ERR_ARG and "dsa_diag_trace" in dsa.dsa_last_error()


@pytest.mark.parametrize("args", [
    (0, 32, 128, 4096),      # no tokens
    (257, 32, 128, 4096),    # batch beyond one tensor-core tile's N
    (8, 32, 96, 4096),       # unsupported head_dim
    (8, 3, 64, 4096),        # heads * head_dim not a multiple of 128
    (8, 32, 128, 4000),      # hidden not a multiple of 64
    (8, 0, 128, 4096),       # no heads
])
def test_proj_create_rejects_bad_arguments(dsa, args):
    code, p = dsa.dsa_proj_create(*args)
    assert code == dsa.DSA_ERR_ARG
    assert not p.value
    assert dsa.dsa_last_error()


def test_proj_calls_on_a_null_context_fail_cleanly(dsa):
    null = ctypes.c_void_p()
    assert dsa.dsa_proj_destroy(null) == dsa.DSA_OK
    assert dsa.dsa_qkv_rope(null, 16, 16, 0, 16, 16, 16) == dsa.DSA_ERR_STATE
    assert dsa.dsa_proj_sync_status(null) == dsa.DSA_ERR_STATE
    assert dsa.dsa_proj_set_wait_limit(null, 0) == dsa.DSA_ERR_STATE
    assert dsa.dsa_decode_step_fused(null, null, 16, 16, 16) == dsa.DSA_ERR_STATE


@pytest.mark.parametrize("args", [
    (0, 128, 16, 9, 1, 0),       # no streams
    (4, 96, 16, 9, 1, 0),        # unsupported head_dim
    (4, 128, -1, 9, 1, 0),       # negative prompt
    (4, 128, 16, 0, 1, 0),       # N_att < 1
    (4, 128, 16, 9, 3, 0),       # unknown policy
    (4, 128, 16, 9, 2, 2),       # FP8 storage not offered for the baselines
])
def test_policy_create_rejects_bad_arguments(dsa, args):
    code, h = dsa.dsa_pol_create(*args)
    assert code == dsa.DSA_ERR_ARG
    assert not h.value
    assert dsa.dsa_last_error()


def test_policy_calls_on_a_null_handle_fail_cleanly(dsa):
    import numpy as np

    null = ctypes.c_void_p()
    assert dsa.dsa_pol_destroy(null) == dsa.DSA_OK
    assert dsa.dsa_pol_prefill(null, None, None) == dsa.DSA_ERR_STATE
    assert dsa.dsa_pol_decode_step(null, 16, 16, 16, 16) == dsa.DSA_ERR_STATE
    assert dsa.dsa_pol_get_positions(null, np.zeros(4, dtype=np.int32)) == dsa.DSA_ERR_STATE
    assert dsa.dsa_pol_sync_status(null) == dsa.DSA_ERR_STATE
