"""vsf_device_copy, the 128-bit copy kernel behind the benchmark's same-run
copy ceiling: it must copy every byte and nothing else."""
import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("nbytes", [16, 4096 + 48, (1 << 20) + 16 * 7, 64 << 20])
def test_device_copy_copies_every_byte(nbytes):
    from fsdp_buffer_layout_gb300 import vsf as V
    g = torch.Generator(device="cuda").manual_seed(nbytes)
    src = torch.randint(0, 256, (nbytes,), dtype=torch.uint8, device="cuda", generator=g)
    dst = torch.zeros(nbytes + 64, dtype=torch.uint8, device="cuda")
    V.vsf_device_copy(dst.data_ptr(), src.data_ptr(), nbytes,
                      torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    assert torch.equal(dst[:nbytes], src)
    assert not dst[nbytes:].any(), "wrote past the end"
