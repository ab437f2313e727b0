"""The input generator: determinism, stream independence, distribution moments."""
import numpy as np

import synth


def test_streams_are_counter_based_and_deterministic():
    a = synth.tensor(7, synth.TAG_W13, 3, 1001, 1.0, "f32")
    b = np.concatenate([synth.tensor(7, synth.TAG_W13, 1, 1001, 1.0, "f32", major_base=i) for i in range(3)])
    assert np.array_equal(a, b)
    assert np.array_equal(a, synth.tensor(7, synth.TAG_W13, 3, 1001, 1.0, "f32"))
    c = synth.tensor(8, synth.TAG_W13, 3, 1001, 1.0, "f32")
    assert not np.array_equal(a, c)


def test_redraw_changes_only_that_row():
    cfg = synth.config(0)
    att = np.zeros(cfg.T, np.uint32)
    x0 = synth.x_rows(cfg, att)
    att[5] = 1
    x1 = synth.x_rows(cfg, att)
    assert not np.array_equal(x0[5], x1[5])
    assert np.array_equal(np.delete(x0, 5, 0), np.delete(x1, 5, 0))
    assert np.array_equal(synth.x_rows(cfg, att, rows=np.array([5, 2])), x1[[5, 2]])


def test_normal_moments():
    v = synth.tensor(0, synth.TAG_X, 4, 250000, 1.0, "f32").astype(np.float64).ravel()
    assert abs(v.mean()) < 5e-3 and abs(v.std() - 1.0) < 5e-3
    assert abs(np.mean(v ** 4) - 3.0) < 0.05  # Gaussian kurtosis
    assert abs(np.mean(np.abs(v) > 1.96) - 0.05) < 2e-3


def test_ln_matches_libm():
    L = synth.lib()
    for v in [1e-300, 2.0 ** -53, 0.1, 0.5, 0.75, 1.0, 2.0, 129.0]:
        assert abs(L.synth_ln(v) - np.log(v)) <= 4e-16 * max(1.0, abs(np.log(v)))


def test_layer_shapes_and_zipf_bias():
    cfg = synth.config("oss120b_decode")
    rw, rb = synth.router(cfg)
    assert rw.shape == (128, 2880) and rb.shape == (128,)
    rbf = synth.bf16_to_f32(rb)
    assert rbf[0] == 0 and np.all(np.diff(rbf) <= 0)
    assert abs(rbf[127] - 0.5 * np.log(1 / 128)) < 0.02
    b13, b2 = synth.expert_biases(synth.config("qwen235b_prefill"))
    assert b13.shape == (128, 3072) and not b13.any() and not b2.any()
