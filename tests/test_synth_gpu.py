"""The device filler of the input generator gives the host filler's bits."""
import numpy as np
import pytest

import synth

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a GPU", allow_module_level=True)


@pytest.mark.parametrize("dtype,sigma", [(synth.F16, 1.0), (synth.BF16, 0.02), (synth.F16, 1 / 128),
                                         (synth.F32, 0.1)])
def test_device_normal_matches_host(dtype, sigma):
    R, C = 777, 1032
    tdt = {synth.F16: torch.float16, synth.BF16: torch.bfloat16, synth.F32: torch.float32}[dtype]
    t = torch.empty((R, C), dtype=tdt, device="cuda")
    synth.dev_normal(t, dtype, 5, synth.TID_B, sigma)
    torch.cuda.synchronize()
    host = synth.normal((R, C), dtype, 5, synth.TID_B, sigma)
    if dtype == synth.F32:
        dev = t.cpu().numpy()
        assert np.array_equal(dev.view(np.uint32), host.view(np.uint32))
    else:
        dev = t.cpu().view(torch.int16).numpy().view(np.uint16)
        assert np.array_equal(dev, host.view(np.uint16))


def test_device_mask_matches_host():
    M, N = 1000, 136
    t = torch.empty(((M + 31) // 32, N), dtype=torch.int32, device="cuda")
    synth.dev_mask_words(t, M, N, 3)
    torch.cuda.synchronize()
    assert np.array_equal(t.cpu().numpy().view(np.uint32), synth.mask_words(M, N, 3))
