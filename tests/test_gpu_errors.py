"""Error paths of the C ABI on a GPU, none of which faults, traps or hangs
the device: host-side argument and state errors, injected allocation
failures, and the bounded waits of the decode kernel run out on purpose
(wait limit 0), which must come back as DSA_ERR_TIMEOUT with the context
still usable."""
import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dsa():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    from __graft_entry__ import build
    build()
    from ar_image_gen_gb300 import dsa as mod
    return mod


def _inputs(S, d, dtype=torch.bfloat16):
    g = torch.Generator(device="cuda").manual_seed(3)
    return [torch.randn((S, d), generator=g, device="cuda").to(dtype) for _ in range(4)]


def test_decode_before_prefill_is_a_state_error(dsa):
    code, h = dsa.dsa_create(4, 128, 8, 16, 4, 0)
    assert code == dsa.DSA_OK
    q, k, v, out = _inputs(4, 128)
    assert dsa.dsa_decode_step(h, q, k, v, out) == dsa.DSA_ERR_STATE
    assert "prefill" in dsa.dsa_last_error()
    assert dsa.dsa_destroy(h) == dsa.DSA_OK


def test_unaligned_and_null_pointers_are_rejected(dsa):
    code, h = dsa.dsa_create(4, 128, 8, 16, 4, 0)
    K = torch.randn((4, 8, 128), device="cuda").bfloat16()
    assert dsa.dsa_prefill(h, K, K) == dsa.DSA_OK
    q, k, v, out = _inputs(4, 128)
    assert dsa.dsa_decode_step(h, q.data_ptr() + 2, k, v, out) == dsa.DSA_ERR_ARG
    assert dsa.dsa_decode_step(h, q, None, v, out) == dsa.DSA_ERR_ARG
    assert dsa.dsa_prefill(h, None, K) == dsa.DSA_ERR_ARG
    code, t = dsa.dsa_get_step(h)
    assert code == dsa.DSA_OK and t == 0  # rejected calls leave the handle unchanged
    assert dsa.dsa_destroy(h) == dsa.DSA_OK


@pytest.mark.parametrize("n", [1, 2, 3, 4, 5, 6, 7, 8, 9])
def test_injected_allocation_failure(dsa, n):
    before = torch.cuda.mem_get_info()[0]
    dsa.dsa_debug_fail_alloc_after(n)
    code, h = dsa.dsa_create(64, 128, 64, 288, 29, 0)
    dsa.dsa_debug_fail_alloc_after(0)
    if code == dsa.DSA_OK:  # fewer allocations than n: the hook never fired
        assert dsa.dsa_destroy(h) == dsa.DSA_OK
        return
    assert code == dsa.DSA_ERR_OOM and "injected" in dsa.dsa_last_error()
    assert not h.value
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] >= before - (64 << 20)  # nothing large left allocated
    code, h = dsa.dsa_create(64, 128, 64, 288, 29, 0)
    assert code == dsa.DSA_OK
    assert dsa.dsa_destroy(h) == dsa.DSA_OK


@pytest.mark.parametrize("splits", [1, 3])
def test_bounded_wait_timeout_is_reported(dsa, splits):
    from ar_image_gen_gb300.dsa import DSA
    S, d = 6, 128
    h = DSA(S, d, 40, 64, 12, 0, "bf16")
    h.set_splits(splits)
    K = torch.randn((S, 40, d), device="cuda").bfloat16()
    h.prefill(K, K)
    q, k, v, out = _inputs(S, d)
    h.decode_step(q, k, v, out)
    assert h.sync_status() == dsa.DSA_OK
    h.set_wait_limit(0)  # every wait in the kernel gives up at once
    h.decode_step(q, k, v, out)
    assert h.sync_status() == dsa.DSA_ERR_TIMEOUT
    h.close()
    # the context is still usable: a fresh handle decodes normally
    h2 = DSA(S, d, 40, 64, 12, 0, "bf16")
    h2.prefill(K, K)
    for _ in range(5):
        h2.decode_step(q, k, v, out)
    assert h2.sync_status() == dsa.DSA_OK
    assert torch.isfinite(out.float()).all()
    h2.close()


def test_prefill_clears_a_sticky_status(dsa):
    from ar_image_gen_gb300.dsa import DSA
    S, d = 4, 128
    h = DSA(S, d, 8, 16, 4, 0, "bf16")
    K = torch.randn((S, 8, d), device="cuda").bfloat16()
    h.prefill(K, K)
    q, k, v, out = _inputs(S, d)
    h.set_wait_limit(0)
    h.decode_step(q, k, v, out)
    assert h.sync_status() == dsa.DSA_ERR_TIMEOUT
    assert h.sync_status() == dsa.DSA_ERR_TIMEOUT  # sticky
    h.set_wait_limit(0xFFFFFFFF)
    h.prefill(K, K)
    h.decode_step(q, k, v, out)
    assert h.sync_status() == dsa.DSA_OK
    h.close()


def test_pipeline_knob_rejects_unknown_shapes(dsa):
    code, h = dsa.dsa_create(4, 128, 8, 16, 4, 0)
    assert code == dsa.DSA_OK
    for bad in (-1, 5):
        assert dsa.dsa_set_pipeline(h, bad) == dsa.DSA_ERR_ARG
        assert "pipeline" in dsa.dsa_last_error()
    for ok in (1, 2, 3, 4, 0):
        assert dsa.dsa_set_pipeline(h, ok) == dsa.DSA_OK
    assert dsa.dsa_destroy(h) == dsa.DSA_OK
