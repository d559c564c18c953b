"""The seeded input generator: its hash is SplitMix64 as published, its normal
draws have the stated mean and spread, and any row regenerates alone."""
import numpy as np
import pytest

import synth

M64 = (1 << 64) - 1
G = 0x9E3779B97F4A7C15


def py_mix(z):
    # SplitMix64 output function (Steele, Lea & Flood 2014), restated
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & M64
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & M64
    return z ^ (z >> 31)


def test_mix_is_splitmix64():
    # the reference generator seeded with 0 starts 0xe220a8397b1dcdaf
    assert synth.mix64(G) == 0xE220A8397B1DCDAF
    for k in [0, 1, 12345, M64, 0xDEADBEEF << 20]:
        assert synth.mix64(k) == py_mix(k)


def test_counter_hash_definition():
    for seed, tid, idx in [(0, 1, 0), (7, 3, 99), (2**40, 100, 2**33 + 5)]:
        key = py_mix((seed + tid * G) & M64)
        assert synth.hash64(seed, tid, idx) == py_mix((key + (idx + 1) * G) & M64)


def test_irwin_hall_definition():
    for e in range(50):
        h1 = synth.hash64(3, 2, 2 * e)
        h2 = synth.hash64(3, 2, 2 * e + 1)
        s = sum((h >> sh) & 0xFFFF for h in (h1, h2) for sh in (0, 16, 32, 48))
        assert synth.irwin_hall(3, 2, e) == 2 * s - 524280


@pytest.mark.parametrize("dtype", [synth.F16, synth.BF16, synth.F32])
def test_normal_moments_and_rounding(dtype):
    x = synth.normal((512, 1024), dtype, 0, synth.TID_A, 0.5)
    xf = synth.bf16_bits_to_f32(x) if dtype == synth.BF16 else x.astype(np.float32)
    assert abs(float(xf.mean())) < 0.005
    assert abs(float(xf.std()) - 0.5) < 0.005
    # value = round(c * scale): recompute three elements by hand
    sc = np.float32(synth.scale(0.5))
    for e in [0, 17, 4095]:
        v = np.float32(synth.irwin_hall(0, synth.TID_A, e)) * sc
        flat = x.reshape(-1)
        if dtype == synth.F16:
            assert flat[e] == np.float16(v)
        elif dtype == synth.F32:
            assert flat[e] == v


def test_rows_regenerate_alone():
    full = synth.normal((300, 40), synth.F16, 9, synth.TID_B, 1.0)
    rows = np.array([0, 5, 299, 123])
    part = synth.normal((300, 40), synth.F16, 9, synth.TID_B, 1.0, rows=rows)
    assert np.array_equal(full[rows].view(np.uint16), part.view(np.uint16))


def test_mask_words_padding_and_rate():
    w = synth.mask_words(70, 33, 1)
    assert w.shape == (3, 33)
    assert np.all(w[2] >> 6 == 0)  # rows 70..95 are padding
    bits = np.unpackbits(w[:2].view(np.uint8)).mean()
    assert abs(bits - 0.5) < 0.05
    part = synth.mask_words(70, 33, 1, word_rows=[2, 0])
    assert np.array_equal(part, w[[2, 0]])


def test_sample_rows():
    r = synth.sample_rows(65536, 64, 0)
    assert r.size > 50 and r.min() >= 0 and r.max() < 65536
    assert np.array_equal(r, synth.sample_rows(65536, 64, 0))


def test_sample_cols():
    c = synth.sample_cols(16384, 64, 0)
    assert c.size > 50 and c.min() >= 0 and c.max() < 16384
    assert np.array_equal(c, synth.sample_cols(16384, 64, 0))
    assert not np.array_equal(c, synth.sample_rows(16384, 64, 0))  # its own stream
