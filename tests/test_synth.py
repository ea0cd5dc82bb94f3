"""The seeded input generators: determinism, formats and distributions (no GPU)."""
import numpy as np

import synth


def test_layer_is_deterministic_and_shaped():
    a = synth.make_layer(synth.TINY, seed=0)
    b = synth.make_layer(synth.TINY, seed=0)
    c = synth.make_layer(synth.TINY, seed=1)
    E, H, I = 8, 256, 128
    assert a["w13"].shape == (E, 2 * I, H // 8) and a["w13"].dtype == np.int32
    assert a["s13"].shape == (E, 2 * I, H // 32) and a["s13"].dtype == np.uint16
    assert a["w2"].shape == (E, H, I // 8) and a["s2"].shape == (E, H, I // 32)
    for key in a:
        assert np.array_equal(a[key], b[key])
        assert not np.array_equal(a[key], c[key])


def test_chunked_draw_does_not_depend_on_thread_count(monkeypatch):
    shape = (3, synth._CHUNK // 2 + 5)
    a = synth.random_words(shape, 3, 9)
    monkeypatch.setattr(synth, "_threads", lambda: 1)
    b = synth.random_words(shape, 3, 9)
    assert np.array_equal(a, b)


def test_value_distributions():
    w = synth.random_words((64, 1024), 0, 0).view(np.uint32)
    nib = np.stack([(w >> np.uint32(4 * j)) & np.uint32(15) for j in range(8)]).ravel()
    hist = np.bincount(nib, minlength=16) / nib.size
    assert np.abs(hist - 1 / 16).max() < 0.003
    s = synth.uniform_bf16((100000,), 0.005, 0.02, 0, 1)
    sf = (s.astype(np.uint32) << 16).view(np.float32)
    assert sf.min() >= 0.005 * (1 - 2 ** -8) and sf.max() <= 0.02 * (1 + 2 ** -8)
    assert abs(sf.mean() - 0.0125) < 2e-4
    x, logits = synth.make_tokens(64, 512, 384, seed=0)
    xf = (x.astype(np.uint32) << 16).view(np.float32)
    assert abs(xf.std() - 1) < 0.02 and abs(logits.std() - 1) < 0.05


def test_bf16_rounding_ties_to_even():
    vals = np.array([1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -2.5, 3.0e-3], dtype=np.float32)
    bits = synth.f32_to_bf16_bits(vals)
    back = (bits.astype(np.uint32) << 16).view(np.float32)
    assert back[0] == 1.0 and back[1] == 1.0 and back[2] == 1.0 + 2 ** -6 and back[3] == -2.5
    assert abs(back[4] - 3.0e-3) <= 3.0e-3 * 2 ** -8


def test_zipf_targets_capped_and_conserving():
    t = synth.zipf_targets(384, 4096, 8, 1.1)
    assert abs(t.sum() - 4096 * 8) < 1e-6 and t.max() <= 4096 + 1e-9
    assert np.all(np.diff(t) <= 1e-9)


def test_zipf_bias_gives_skewed_popularity():
    E, T, k = 64, 512, 4
    b = synth.zipf_bias(E, T, k, 1.1, 0, 100)
    assert np.array_equal(b, synth.zipf_bias(E, T, k, 1.1, 0, 100))
    _, logits = synth.make_tokens(T, 8, E, seed=0, bias=b)
    top = np.argpartition(-logits, k - 1, axis=1)[:, :k]
    cnt = np.sort(np.bincount(top.ravel(), minlength=E))[::-1].astype(float)
    tgt = synth.zipf_targets(E, T, k, 1.1)
    # the realised load follows the target shape (top experts much busier than the tail)
    assert cnt[0] > 5 * np.median(cnt)
    assert np.corrcoef(np.log(cnt + 1), np.log(tgt + 1))[0, 1] > 0.9
