"""The Python examples in README.md run as written (forward RELU_AUX_BIAS,
then the DRELU_BGRAD backward that takes its mask), and their outputs agree
with the same arithmetic in torch fp32."""
import os
import re

import pytest

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a GPU", allow_module_level=True)

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_readme_examples_run():
    text = open(os.path.join(ROOT, "README.md")).read()
    blocks = re.findall(r"```python\n(.*?)```", text, flags=re.S)
    assert len(blocks) >= 2
    ns = {}
    torch.manual_seed(0)
    for b in blocks:
        exec(compile(b, "README.md", "exec"), ns)  # noqa: S102
    torch.cuda.synchronize()
    X, W, b, Y = ns["X"], ns["W"], ns["b"], ns["Y"]
    z = X.float() @ W.float() + b.float()
    ref = torch.relu(z)
    err = (Y.float() - ref).abs().max() / ref.abs().max()
    assert err < 2e-2
    # the kernel's mask (bit i % 32 of word [i / 32][j]) matches z > 0 outside
    # the band where accumulation order may flip the sign
    aux = ns["aux"]
    shifts = torch.arange(32, device=aux.device, dtype=torch.int32).view(1, 32, 1)
    bits = ((aux.unsqueeze(1) >> shifts) & 1).reshape(z.shape).bool()
    band = z.abs() < 1e-3 * z.abs().amax(dim=1, keepdim=True)
    assert torch.equal(bits[~band], (z > 0)[~band])
    dY2, W2, dY, db = ns["dY2"], ns["W2"], ns["dY"], ns["db"]
    g = (dY2.float() @ W2.float().t()) * bits.float()
    err = (dY.float() - g).abs().max() / g.abs().max()
    assert err < 2e-2
    col = g.sum(0)
    err = (db - col).abs().max() / col.abs().max()
    assert err < 1e-2
