"""Host-side pieces of bench.py that need no GPU: the sampled-row parity
summary (error norms and the ReLU-mask band rule) and the recorded DRAM
traffic lookup."""
import numpy as np

import bench


def _ref(rows, z):
    y = np.maximum(z, 0).astype(np.float32)
    return {"rows_fwd": rows, "rows_bwd": rows, "Y": y, "z": z, "dZ": y.copy()}


def _words_for(rows, bits):
    """aux word rows (r // 32) of each sampled row, holding that row's bits"""
    w = np.zeros((len(rows), bits.shape[1]), dtype=np.uint32)
    for i, r in enumerate(rows):
        w[i] = bits[i].astype(np.uint32) << np.uint32(r % 32)
    return w


def test_sampled_parity_exact_and_band():
    rng = np.random.default_rng(0)
    rows = np.array([3, 40, 77], dtype=np.int64)
    z = rng.standard_normal((3, 64)).astype(np.float32)
    z[0, 5] = 1e-6  # inside the band |z| < 1e-3 max|z| of its row
    ref = _ref(rows, z)
    bits = (z > 0).astype(np.uint8)
    bits[0, 5] ^= 1  # a flip inside the band is allowed
    dev = {"Y": ref["Y"].copy(), "dZ": ref["dZ"].copy(), "aux_rows": _words_for(rows, bits)}
    r = bench.sampled_parity(dev, ref)
    assert r["pass"] and r["Y"]["nmax"] == 0.0 and r["dZ"]["rel_l2"] == 0.0
    assert r["mask_mismatch_in_band"] == 1 and r["mask_mismatch_outside_band"] == 0


def test_sampled_parity_catches_errors():
    rng = np.random.default_rng(1)
    rows = np.array([0, 33], dtype=np.int64)
    z = rng.standard_normal((2, 32)).astype(np.float32) + 3.0  # all well outside the band
    ref = _ref(rows, z)
    bits = (z > 0).astype(np.uint8)
    bits[1, 7] ^= 1
    dev = {"Y": ref["Y"] * 1.05, "dZ": ref["dZ"].copy(), "aux_rows": _words_for(rows, bits)}
    r = bench.sampled_parity(dev, ref)
    assert not r["pass"]
    assert r["mask_mismatch_outside_band"] == 1
    assert abs(r["Y"]["rel_l2"] - 0.05) < 1e-6


def test_recorded_traffic_matches_sources():
    # the committed profile is read back only while its digest matches the sources
    t = bench.recorded_traffic()
    assert t is None or (len(t) == 2 and all(v > 3e9 for v in t))


def test_pick_peak_burst_and_sustained():
    pk = {"bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
    assert bench.pick_peak(pk, "measured", 0.4)[0] == 1900.0   # short loop: burst
    assert bench.pick_peak(pk, "measured", 4.0)[0] == 1700.0   # seconds-long loop: sustained
    assert bench.pick_peak({"bf16_tflops": 1900.0}, "fallback", 9.0)[0] == 1900.0


def test_stats_and_parity_block():
    st = bench.stats_ms([3.0, 1.0, 2.0, 10.0])
    assert st["median"] == 2.5 and st["min"] == 1.0 and st["n"] == 4
    ok = bench._parity_block({"Y": {"nmax": 1e-3, "rel_l2": 1e-4},
                              "bgrad": {"nmax": 5e-3, "rel_l2": 5e-3}}, bgrad_keys=("bgrad",))
    assert ok["pass"]
    # an output error above the output bound fails; the same error on a bias
    # gradient key is held to the bias-gradient bound
    bad = bench._parity_block({"Y": {"nmax": 1e-3, "rel_l2": 6e-3}})
    assert not bad["pass"]
    assert not bench._parity_block({"Y": {"nmax": 0.0, "rel_l2": 0.0}},
                                   mask={"mask_mismatch_outside_band": 1,
                                         "mask_mismatch_in_band": 0})["pass"]


class _Done:
    """Stands in for the finished nvidia-smi process."""

    def terminate(self):
        pass

    def wait(self, timeout=None):
        return 0


def _sample(mhz, power, cap):
    return f"0, {mhz}, 2070, {power}, 0x4, Not Active, Not Active, Not Active, {cap}"


def test_clock_samples_outside_the_timed_region_are_left_out():
    s = bench.ClockSampler(0)
    s.proc = _Done()
    s.lines = [_sample(2070, 160, "Not Active"), _sample(1400, 1370, "Active"),
               _sample(1420, 1375, "Active"), _sample(2070, 170, "Not Active")]
    s.times = [10.0, 10.5, 10.7, 11.2]
    c = s.stop(window=(10.4, 11.0))
    assert c["samples"] == 2 and c["sm_mhz"] == 1410.0 and c["reasons"] == ["sw_power_cap"]
    assert "note" not in c
    c = s.stop(window=(10.55, 10.65))  # no sample inside: say so instead of idle clocks
    assert c["samples"] == 0 and c["sm_mhz"] is None and "200 ms" in c["note"]
    c = s.stop()  # no window: every sample
    assert c["samples"] == 4 and c["sm_mhz"] == 1745.0
    s.keep_from(2)
    assert s.lines[0].startswith("0, 1420") and s.times == [10.7, 11.2]
