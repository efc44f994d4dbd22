"""The seeded input generator against its published definitions.

synth draws every input that the oracle and the CUDA library share.  These
tests pin it to the published generator's outputs and to plain properties:
- SplitMix64's reference outputs (Steele, Lea and Flood, OOPSLA 2014; the
  values that the reference C implementation prints for state 1234567);
- each bulk array equals its element-wise draws, whatever the thread split;
- F16 encoding is IEEE round to nearest even, checked with numpy's conversion;
- moments and ranges of the normals, the bounded integers and the Q8_0 blocks
  follow the stated recipe.
"""
import math

import numpy as np

import synth


def test_splitmix64_reference_outputs():
    want = [6457827717110365317, 3203168211198807973, 9817491932198370423, 4593380528125082431,
            16408922859458223821]
    assert [synth.splitmix64_at(1234567, i) for i in range(5)] == want


def test_streams_are_counter_based():
    # element i of a stream is SplitMix64 value i from the stream's key, so
    # consecutive values of one stream continue one sequence; streams and
    # seeds give different sequences
    a = [synth.draw(7, 3, i) for i in range(6)]
    assert len(set(a)) == 6
    assert a != [synth.draw(7, 4, i) for i in range(6)]
    assert a != [synth.draw(8, 3, i) for i in range(6)]
    assert synth.draw(7, 3, 1000003) == synth.draw(7, 3, 1000003)


def test_bulk_arrays_equal_their_element_draws():
    n = 100003
    x = synth.normal_f32(11, 5, n, 0.5, 2.0)
    for i in (0, 1, 2, 777, 50000, n - 1):
        assert x[i] == np.float32(0.5 + 2.0 * synth.normal_at(11, 5, i))
    u = synth.uniform_i32(11, 6, n, -3, 9)
    for i in (0, 1, 999, n - 1):
        assert u[i] == -3 + ((synth.draw(11, 6, i) >> 32) * 13 >> 32)


def test_f16_encoding_is_round_to_nearest_even():
    n = 50000
    h = synth.normal_f16(3, 2, n, 0.0, 3.0)
    f = synth.normal_f32(3, 2, n, 0.0, 3.0)
    assert np.array_equal(h, f.astype(np.float16).view(np.uint16))


def test_normal_moments():
    n = 400000
    x = synth.normal_f32(5, 1, n).astype(np.float64)
    assert abs(x.mean()) < 4 / math.sqrt(n)
    assert abs(x.var() - 1) < 4 * math.sqrt(2 / n)
    # Box-Muller tails: P(|N| > 3) = 0.0027
    frac = np.mean(np.abs(x) > 3)
    assert abs(frac - 0.0026998) < 4 * math.sqrt(0.0027 / n)


def test_bounded_integers_cover_the_range_evenly():
    n = 260000
    u = synth.uniform_i32(5, 2, n, -5, 7)
    assert u.min() == -5 and u.max() == 7
    counts = np.bincount(u + 5, minlength=13)
    expect = n / 13
    chi2 = float(((counts - expect) ** 2 / expect).sum())
    assert chi2 < 40                         # 12 degrees of freedom; p < 1e-4 beyond 40


def test_q8_0_blocks_follow_the_recipe():
    nb = 20000
    q = synth.q8_0_blocks(9, 4, nb * 32, 0.02).reshape(nb, 34)
    d = q[:, :2].copy().view(np.float16).astype(np.float64).ravel()
    qs = q[:, 2:].view(np.int8).astype(np.int64)
    assert qs.min() == -127 and qs.max() == 127          # -128 never drawn
    assert abs(qs.mean()) < 4 * math.sqrt((255 ** 2 - 1) / 12 / qs.size)
    # scale = |N(0, 0.02)| / 127, whose mean is 0.02 * sqrt(2/pi) / 127
    assert np.all(d >= 0)
    assert abs(d.mean() / (0.02 * math.sqrt(2 / math.pi) / 127) - 1) < 0.02
