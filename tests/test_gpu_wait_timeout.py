"""Failure detection without a GPU fault: every barrier wait in the kernels
is bounded in time, and the first timeout of a CTA makes its later waits
return at once. A self-test kernel waits four times in a row on barriers that
no one arrives on; the first wait must give up after its limit and set bit 1
of the error word, the other three must not wait again, and the kernel (and
the stream) must finish with the context still usable."""
import time

import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("limit_ms", [20, 200])
def test_bounded_wait_gives_up_and_reports(limit_ms):
    from fsdp_buffer_layout_gb300 import vsf as V
    err = torch.zeros(2, dtype=torch.int32, device="cuda")
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    V.vsf_selftest_wait_timeout(err.data_ptr(), limit_ms * 1_000_000,
                                torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    elapsed = time.perf_counter() - t0
    e = err.cpu().tolist()
    assert e[0] & 2, "the wait did not report its timeout"
    assert limit_ms * 1e-3 * 0.9 <= elapsed < limit_ms * 1e-3 + 1.0
    # sticky: four waits take about one limit (four limits if each waited)
    waited_ms = e[1] / 1000.0
    assert limit_ms * 0.9 <= waited_ms < limit_ms * 1.5 + 2.0, waited_ms
    # the context is still usable
    x = torch.arange(1000, device="cuda", dtype=torch.float32)
    assert float(x.sum().item()) == 499500.0
