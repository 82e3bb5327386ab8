"""The offline tuning tool's host logic (weight_only_int4_02_gb300/tune.py), without a
GPU: the sweep plan covers what the dispatcher chooses among, the split cost model's
least-squares fit recovers known constants, and the report picks each shape's fastest
setting."""
import numpy as np

from weight_only_int4_02_gb300 import tune


def test_fit_recovers_the_split_model_constants():
    rng = np.random.default_rng(0)
    truth = [0.15, 0.40, 1.4, 0.006]
    samples = []
    for iters in (16, 43, 64, 172):
        for s in (1, 2, 3, 4, 6, 8):
            for rows in (1, 16, 32):
                us = float(np.dot(tune.split_features(iters, s, 8, rows), truth))
                samples.append((iters, s, rows, us))
    coef, resid = tune.fit_split_model(samples, 8)
    assert np.allclose(coef, truth, rtol=1e-9, atol=1e-12) and resid < 1e-9
    # the model's terms: the longest part's stages, prefetched up to the ring, then streamed
    assert tune.split_features(64, 4, 8, 16) == [8, 8, 1.0, 48]
    assert tune.split_features(10, 1, 8, 16) == [8, 2, 0.0, 0.0]
    noisy = [(it, s, r, us + rng.normal(0, 0.01)) for (it, s, r, us) in samples]
    coef, resid = tune.fit_split_model(noisy, 8)
    assert np.allclose(coef[:2], truth[:2], atol=0.01) and resid < 0.02


def test_sweep_plan_covers_the_dispatchers_choices():
    shapes = [(1, 4096, 4096), (8, 4096, 22016), (16, 4096, 4096), (128, 4096, 12288), (1024, 5120, 15360),
              (4, 4040, 4096)]
    plan = tune.sweep_plan(shapes, sms=152)
    labels = {",".join("%s=%s" % kv for kv in env.items()) or "default": (force, sub) for env, force, sub in plan}
    assert labels["default"] == (0, shapes)
    for cb in (16, 32, 64, 128):
        force, sub = labels["W4A16_DECODE_CB=%d" % cb]
        assert force == 3 and sub == [(1, 4096, 4096), (8, 4096, 22016), (16, 4096, 4096)]   # K % 32, M <= 16
    for cb in (48, 80):
        assert labels["W4A16_DECODE_CB=%d" % cb][1] == [(1, 4096, 4096), (8, 4096, 22016)]   # eight rows only
    assert (1024, 5120, 15360) in labels["W4A16_TILE_M=256"][1]
    assert (1024, 5120, 15360) not in labels["W4A16_TILE_M=16"][1]
    for sp in (1, 2, 4, 8):
        force, sub = labels["W4A16_SPLIT=%d" % sp]
        assert force == 2 and (1024, 5120, 15360) not in sub and (1, 4096, 4096) in sub   # fewer tiles than SMs


def test_best_settings_picks_each_shapes_fastest():
    results = {"default": {"1,4096,4096": 5.0, "128,4096,4096": 14.3},
               "W4A16_TILE_M=32": {"128,4096,4096": 12.2},
               "W4A16_DECODE_CB=32": {"1,4096,4096": 5.8}}
    best = tune.best_settings(results)
    assert best["1,4096,4096"]["best"] == "default" and best["1,4096,4096"]["best_over_default"] == 1.0
    assert best["128,4096,4096"]["best"] == "W4A16_TILE_M=32"
    assert abs(best["128,4096,4096"]["best_over_default"] - 12.2 / 14.3) < 1e-12
