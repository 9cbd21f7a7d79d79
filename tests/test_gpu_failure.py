"""GPU: the bounded waits of the pipeline kernels give up by themselves and report, with
no fault and no hang (failure detection tested on the device without faulting it)."""
import time

import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ink():
    import relative_position_gqa_gb300 as m
    m._lib.load()
    return m


def _run(ink, mode, ctas):
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    gave_up = torch.zeros(1, dtype=torch.int32, device="cuda")
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    ink.selftest_bounded_wait(mode, ctas, st, gave_up)
    torch.cuda.synchronize()
    return int(st.item()), int(gave_up.item()), time.perf_counter() - t0


def test_wait_with_no_arrival_times_out_and_reports(ink):
    status, gave_up, dt = _run(ink, 0, 8)
    assert status == 4, ink.status_string(status)  # INKLING_ERR_TIMEOUT
    assert gave_up == 8
    assert 0.5 < dt < 30.0
    # the context is still usable: an ordinary kernel runs and syncs
    x = torch.arange(1024, device="cuda", dtype=torch.float32)
    assert float(x.sum().item()) == 1023 * 1024 / 2


def test_wait_gives_up_early_when_another_cta_failed(ink):
    status, gave_up, dt = _run(ink, 1, 8)
    assert status == 6, ink.status_string(status)  # CTA 0's error wins
    assert gave_up == 7
    assert dt < 0.5
