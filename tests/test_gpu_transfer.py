"""GPU tests of the step transfers (pkv_copy_to_device / pkv_copy_to_host): byte-exact
copies for any size and alignment, from page-locked host memory (the SM copy kernels)
and from pageable memory (the copy-engine path), in stream order with other work."""
import numpy as np
import pytest

import pagedattention_paged_kv_gb300 as pkv

pytestmark = pytest.mark.gpu

SIZES = [1, 15, 16, 17, 255, 4096 + 3, 2_600_000, 2_600_000 + 9]


@pytest.mark.parametrize("pinned", [True, False])
@pytest.mark.parametrize("offset", [0, 1, 8, 16])
def test_round_trip_is_byte_exact(pinned, offset):
    import torch
    rng = np.random.Generator(np.random.PCG64(17 + offset))
    for n in SIZES:
        host = torch.from_numpy(rng.integers(0, 256, size=n + offset, dtype=np.uint8))
        if pinned:
            host = host.pin_memory()
        src = host[offset:]
        dev = torch.full((n + 32,), 0xAB, dtype=torch.uint8, device="cuda")
        pkv.copy_to_device(dev[16:16 + n], src)
        back_buf = torch.zeros(n + offset, dtype=torch.uint8)
        if pinned:
            back_buf = back_buf.pin_memory()
        back = back_buf[offset:]
        pkv.copy_to_host(back, dev[16:16 + n])
        torch.cuda.synchronize()
        d = dev.cpu().numpy()
        assert np.array_equal(d[16:16 + n], src.numpy()), f"to device, {n} bytes"
        assert np.all(d[:16] == 0xAB) and np.all(d[16 + n:] == 0xAB), f"guard bytes, {n} bytes"
        assert np.array_equal(back.numpy(), src.numpy()), f"to host, {n} bytes"


def test_copies_follow_stream_order():
    """A kernel that writes the device buffer before the copy back, and a copy in before a
    kernel that reads it, see each other's bytes."""
    import torch
    n = 1 << 20
    host = torch.arange(n, dtype=torch.int32).pin_memory()
    dev = torch.empty(n, dtype=torch.int32, device="cuda")
    out = torch.empty(n, dtype=torch.int32).pin_memory()
    for it in range(3):
        pkv.copy_to_device(dev, host)
        dev.add_(it + 1)
        pkv.copy_to_host(out, dev)
        torch.cuda.synchronize()
        assert torch.equal(out, torch.arange(n, dtype=torch.int32) + it + 1)


def test_rejects_a_host_pointer_on_the_device_side():
    import torch
    a = torch.zeros(64, dtype=torch.uint8).pin_memory()
    b = torch.zeros(64, dtype=torch.uint8).pin_memory()
    with pytest.raises(pkv.PagedKVError) as e:
        pkv._check(pkv.lib().pkv_copy_to_device(pkv._ptr(a), pkv._ptr(b), 64, pkv._stream_ptr(None)),
                   "copy_to_device")
    assert e.value.status == -1
    with pytest.raises(ValueError):
        pkv.copy_to_device(torch.zeros(8, dtype=torch.uint8, device="cuda"), torch.zeros(9, dtype=torch.uint8))
