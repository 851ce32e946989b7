"""The seeded generator: published SplitMix64 outputs, the counter construction, determinism and
the distributions the workloads ask for."""
import numpy as np

import synth


def test_splitmix64_published_outputs_for_seed_1234567():
    # SplitMix64 (Steele, Lea, Flood; Vigna's reference code) from state 1234567
    expect = [6457827717110365317, 3203168211198807973, 9817491932198370423,
              4593380528125082431, 16408922859458223821]
    assert synth.splitmix(1234567, 5).tolist() == expect


def test_words_are_the_splitmix_stream_of_the_tensor_base():
    b = synth.base_state("L3.wq", seed=0)
    assert np.array_equal(synth.words("L3.wq", 100), synth.splitmix(b, 100))
    assert not np.array_equal(synth.words("L3.wq", 10), synth.words("L3.wk", 10))
    assert not np.array_equal(synth.words("L3.wq", 10, seed=1), synth.words("L3.wq", 10, seed=0))


def test_normal_statistics_and_determinism():
    z = synth.normals("stats", 400000)
    assert abs(z.mean()) < 0.01 and abs(z.std() - 1) < 0.01
    assert abs((np.abs(z) < 1).mean() - 0.6827) < 0.005
    w = synth.normal_bf16("w", (1000, 100), 0.0, 0.02)
    assert np.array_equal(w, synth.normal_bf16("w", (1000, 100), 0.0, 0.02))
    f = (w.astype(np.uint32) << 16).view(np.float32)
    assert abs(f.std() - 0.02) < 0.0005


def test_nibbles_uniform_and_scales_positive():
    b = synth.nibbles("n", (200000,))
    lo, hi = b & 15, b >> 4
    for v in (lo, hi):
        counts = np.bincount(v, minlength=16)
        assert counts.min() > 0.9 * len(b) / 16 and counts.max() < 1.1 * len(b) / 16
    s = synth.abs_normal_16("s", (50000,), 0.005, "fp16").view(np.float16).astype(np.float64)
    assert (s >= 0).all() and abs(s.mean() - 0.005 * np.sqrt(2 / np.pi)) < 1e-4


def test_tokens_in_range():
    t = synth.uniform_int("tokens", 10000, 2048)
    assert t.min() >= 0 and t.max() < 2048 and len(np.unique(t)) > 1500
