"""The bounded device wait, made to run out on purpose in the safe form: one
CTA waits on an mbarrier that nothing arrives on, with a limit of a few
thousand cycles and nothing else in flight.  The wait must end, record
GLACORE_ERR_TIMEOUT in the device error word and leave the context usable."""
import pytest
import torch

import chunked_gated_linear_chunk_gb300 as glc

pytestmark = pytest.mark.gpu


def test_bounded_wait_runs_out_and_reports_timeout(cuda_ok):
    glc.get_device_error()  # clear
    glc.selftest_wait(20000)
    torch.cuda.synchronize()
    with pytest.raises(glc.GlacoreError) as e:
        glc.get_device_error()
    assert e.value.status == glc.ERR_TIMEOUT
    glc.get_device_error()  # the read cleared it
    # the context still runs work
    x = torch.ones(1024, device="cuda")
    assert float(x.sum().item()) == 1024.0


def test_first_error_is_kept(cuda_ok):
    """Two timeouts in a row leave one TIMEOUT; the word is cleared once read."""
    glc.get_device_error()
    glc.selftest_wait(5000)
    glc.selftest_wait(5000)
    torch.cuda.synchronize()
    with pytest.raises(glc.GlacoreError) as e:
        glc.get_device_error()
    assert e.value.status == glc.ERR_TIMEOUT
    glc.get_device_error()
