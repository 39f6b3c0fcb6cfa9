"""Failure detection on the GPU, without a fault (needs a GB300).

The chunk-parallel causal kernel's work items wait for states that other CTAs
publish.  A test hook makes one item never publish (a lost message, made on
purpose) and shortens every bounded wait to 2 ms: the items after it give up,
the launch's abort word stops every CTA, the kernel returns, and
la_get_device_status() reports LA_ERR_TIMEOUT.  The context stays usable: the
next calls, with the hooks off, match the float64 oracle.
"""
import pytest

import workloads
from gpu_util import assert_parity, from_dev, to_dev

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

LA_ERR_TIMEOUT = 5


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from causal_kernelized_attention_gb300 import build
    build.build()
    import causal_kernelized_attention_gb300 as la
    la.load_library()
    return la


def la():
    import causal_kernelized_attention_gb300 as m
    return m


@pytest.mark.parametrize("ticket", [40, 0, 33])
def test_lost_publication_times_out_and_the_next_call_is_clean(orc, ticket):
    """B4 H8 N4096 d64 (32 heads x 32 chunks, the chunk-parallel kernel; ticket t is
    chunk t // 32 of head t % 32): ticket 40 is chunk 1 of head 8, 0 is chunk 0 of
    head 0 (its inclusive prefix is lost), 33 is chunk 1 of head 1."""
    lib = la().load_library()
    q, k, v = workloads.random_inputs(51000 + ticket, 4, 8, 4096, 64, 64, "bf16")
    dq, dk_, dv_ = to_dev(q, "bf16"), to_dev(k, "bf16"), to_dev(v, "bf16")
    assert la().la_get_device_status() == 0
    lib.la_test_set_wait_limit_ns(2_000_000)
    lib.la_test_drop_publication(ticket)
    try:
        la().la_forward_causal(dq, dk_, dv_)
        torch.cuda.synchronize()
        assert la().la_get_device_status() == LA_ERR_TIMEOUT
        assert la().la_get_device_status() == 0  # the status word was read and cleared
    finally:
        lib.la_test_drop_publication(-1)
        lib.la_test_set_wait_limit_ns(0)
    ref = orc.causal_recurrent(q, k, v)
    for _ in range(2):
        o = la().la_forward_causal(dq, dk_, dv_)
        torch.cuda.synchronize()
        assert la().la_get_device_status() == 0
        assert_parity(from_dev(o), ref, "bf16", ("after timeout", ticket))
    # another shape on the same stream's workspaces
    q2, k2, v2 = workloads.random_inputs(52000, 2, 9, 700, 64, 64, "bf16")
    o2 = la().la_forward_causal(to_dev(q2, "bf16"), to_dev(k2, "bf16"), to_dev(v2, "bf16"))
    torch.cuda.synchronize()
    assert la().la_get_device_status() == 0
    assert_parity(from_dev(o2), orc.causal_recurrent(q2, k2, v2), "bf16", "other shape after timeout")


def test_short_wait_limit_alone_does_not_fire(orc):
    """With every publication made, a 50 ms limit never runs out (the chunk-parallel
    kernel at B4 H8 N4096 and the cluster kernel at the headline shape B4 H8 N2048)."""
    lib = la().load_library()
    for N in (4096, 2048):
        q, k, v = workloads.random_inputs(53000 + N, 4, 8, N, 64, 64, "bf16")
        _short_limit_case(lib, orc, q, k, v)


def _short_limit_case(lib, orc, q, k, v):
    dq, dk_, dv_ = to_dev(q, "bf16"), to_dev(k, "bf16"), to_dev(v, "bf16")
    lib.la_test_set_wait_limit_ns(50_000_000)
    try:
        outs = [la().la_forward_causal(dq, dk_, dv_) for _ in range(5)]
        torch.cuda.synchronize()
        assert la().la_get_device_status() == 0
    finally:
        lib.la_test_set_wait_limit_ns(0)
    ref = orc.causal_recurrent(q, k, v)
    for o in outs:
        assert_parity(from_dev(o), ref, "bf16", "short limit")
