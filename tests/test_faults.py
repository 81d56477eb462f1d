"""Failure detection without a GPU fault: host-side refusals before any
launch, and the kernel's bounded waits that end with a status bit."""
import pytest
import torch

from kv_insert_gb300 import qkv_front as qf


@pytest.mark.gpu
def test_bounded_wait_gives_up_and_reports():
    import __graft_entry__
    __graft_entry__.build()
    qf.status()
    qf.selftest_wait(2_000_000)        # 2 ms on a barrier nothing completes
    st = qf.status()
    assert st & qf.STATUS_WAIT_TIMEOUT
    # the context is still usable: a normal call runs and leaves no bit
    from kv_insert_gb300 import workloads as wl
    from _parity import check_workload
    check_workload(wl.WORKLOADS["m1_nkv1_n1152"])
    assert qf.status() == 0


@pytest.mark.gpu
def test_wait_limit_setting_is_checked():
    with pytest.raises(qf.QkvFrontError):
        qf.set_wait_limit(10)
    qf.set_wait_limit(2_000_000_000)
