"""ds4x_copy_async: the kernel-side copy between pinned host memory and the
device (and within the device) is byte-exact for every size, including
tails shorter than its 16-byte words."""

import pytest
import torch

from gpu_path import require_gpu

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("nbytes", [1, 15, 16, 17, 4099, 84736, 67584, 1 << 20])
def test_copy_host_device_round_trip(nbytes):
    B = require_gpu()
    g = torch.Generator().manual_seed(nbytes)
    src_h = torch.randint(0, 256, (nbytes,), dtype=torch.uint8, generator=g).pin_memory()
    dev = torch.full((nbytes,), 7, dtype=torch.uint8, device="cuda")
    B.ds4x_copy_async(dev, src_h)                 # host -> device
    dev2 = torch.zeros_like(dev)
    B.ds4x_copy_async(dev2, dev)                  # device -> device
    back = torch.zeros(nbytes, dtype=torch.uint8).pin_memory()
    B.ds4x_copy_async(back, dev2)                 # device -> host
    torch.cuda.synchronize()
    assert torch.equal(dev.cpu(), src_h)
    assert torch.equal(dev2.cpu(), src_h)
    assert torch.equal(back, src_h)


def test_copy_leaves_neighbours_alone():
    B = require_gpu()
    buf = torch.full((4096,), 0xAB, dtype=torch.uint8, device="cuda")
    src = torch.arange(1000, dtype=torch.int32).to(torch.uint8).pin_memory()
    B.ds4x_copy_async(buf[1024:2024], src)
    torch.cuda.synchronize()
    h = buf.cpu()
    assert torch.equal(h[1024:2024], src)
    assert bool((h[:1024] == 0xAB).all()) and bool((h[2024:] == 0xAB).all())
