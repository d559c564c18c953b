"""Shared test helpers: device transfer and the parity criteria.

Criteria (fp16/bf16 outputs): normalised max error max|g - o| / max|o| <= 2e-2
and relative L2 error ||g - o||_2 / ||o||_2 <= 5e-3, the latter being the
relative-norm metric `rel(a, b)` of gemm_swiglu_mlp_fusion.py (``_demo``).
Bias gradients: both forms <= 1e-2. The ReLU mask is compared bit for bit
except where |z_oracle| < 1e-3 * max_j |z_oracle[i, j]| (row i), where the
order of accumulation may legitimately flip the sign.
"""
import numpy as np

OUT_NMAX, OUT_REL = 2e-2, 5e-3
BGRAD_NMAX, BGRAD_REL = 1e-2, 1e-2
BAND = 1e-3


def nmax_err(g, o) -> float:
    g = np.asarray(g, dtype=np.float64)
    o = np.asarray(o, dtype=np.float64)
    den = np.abs(o).max() if o.size else 0.0
    num = np.abs(g - o).max() if o.size else 0.0
    return float(num / den) if den > 0 else float(num)


def rel_l2(g, o) -> float:
    g = np.asarray(g, dtype=np.float64)
    o = np.asarray(o, dtype=np.float64)
    return float(np.linalg.norm(g - o) / max(np.linalg.norm(o), 1e-9))


def assert_close(g, o, nmax=OUT_NMAX, rel=OUT_REL, what="output"):
    e1, e2 = nmax_err(g, o), rel_l2(g, o)
    assert e1 <= nmax and e2 <= rel, f"{what}: normalised max err {e1:.3e}, rel L2 {e2:.3e}"
    return e1, e2


def unpack_words(words: np.ndarray, M: int) -> np.ndarray:
    """column words uint32 [ceil(M/32), N] -> bits uint8 [M, N]"""
    w = np.ascontiguousarray(words).view(np.uint32)
    nw, N = w.shape
    bits = np.unpackbits(w.view(np.uint8), bitorder="little").reshape(nw, N, 32)
    return bits.transpose(0, 2, 1).reshape(nw * 32, N)[:M]


def mask_mismatch(bits_g: np.ndarray, z_o: np.ndarray):
    """(mismatches outside the band, mismatches inside the band)"""
    band = np.abs(z_o) < BAND * np.abs(z_o).max(axis=1, keepdims=True)
    bits_o = (z_o > 0).astype(np.uint8)
    diff = bits_g != bits_o
    return int((diff & ~band).sum()), int((diff & band).sum())


# ------------------------------------------------------------ device helpers
def to_dev(a: np.ndarray, dtype: int):
    """host fp16 (np.float16) / bf16 bits (np.uint16) / uint32 words -> cuda tensor"""
    import torch
    if a.dtype == np.uint32:
        return torch.from_numpy(a.view(np.int32).copy()).cuda()
    t = torch.from_numpy(np.ascontiguousarray(a).view(np.int16).copy()).cuda()
    return t.view(torch.float16 if dtype == 0 else torch.bfloat16)


def to_host_f32(t) -> np.ndarray:
    return t.float().cpu().numpy()


def to_host_words(t) -> np.ndarray:
    return t.cpu().numpy().view(np.uint32)


def torch_dtype(dtype: int):
    import torch
    return torch.float16 if dtype == 0 else torch.bfloat16
