"""The seeded input generator (host side): published splitmix64 values,
counter-based slicing, and the workloads' value distributions."""
import numpy as np

from sub_bit_weight_binary_b300 import synth


def test_splitmix64_reference_values():
    # splitmix64 started from state 0 (Vigna's reference generator): the
    # first outputs are splitmix64(0), splitmix64(gamma), ...
    z = synth.splitmix64(np.array([0, 0x9E3779B97F4A7C15], dtype=np.uint64))
    assert int(z[0]) == 0xE220A8397B1DCDAF
    assert int(z[1]) == 0x6E789E6AA1B965F4


def test_counter_slices_agree():
    a = synth.words(7, 3, 0, 1000)
    b = synth.words(7, 3, 250, 500)
    assert np.array_equal(a[250:750], b)
    assert not np.array_equal(synth.words(7, 4, 0, 1000), a)
    assert not np.array_equal(synth.words(8, 3, 0, 1000), a)
    r = synth.gen_ternary_codes(5, 6, 640, row0=0)
    r2 = synth.gen_ternary_codes(5, 3, 640, row0=3)
    assert np.array_equal(r[3:], r2)


def test_distributions():
    t = synth.ternary_codes(1, synth.TID_WTER, 0, 400000)
    frac = [(t == v).mean() for v in (-1, 0, 1)]
    assert abs(frac[0] - 0.3) < 0.005 and abs(frac[1] - 0.4) < 0.005 and abs(frac[2] - 0.3) < 0.005
    b = synth.binary_codes(1, synth.TID_CODES, 0, 200000)
    assert set(np.unique(b)) == {-1, 1} and abs((b == 1).mean() - 0.5) < 0.005
    s = synth.uniform_f16(1, synth.TID_SCALES, 0, 100000, 0.01, 0.05).view(np.float16)
    assert s.min() >= np.float16(0.01) and s.max() <= np.float16(0.05)
    assert abs(float(s.astype(np.float64).mean()) - 0.03) < 0.001
    x = synth.normal_f16(1, synth.TID_X, 0, 200000).view(np.float16).astype(np.float64)
    assert abs(x.mean()) < 0.01 and abs(x.std() - 1.0) < 0.01
    w = synth.bits32(1, synth.TID_WBIN, 0, 100000)
    ones = np.unpackbits(w.view(np.uint8)).mean()
    assert abs(ones - 0.5) < 0.002


def test_config_seeds_distinct():
    seeds = {synth.config_seed(c) for c in range(1, 6)}
    assert len(seeds) == 5
