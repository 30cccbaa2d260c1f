"""The seeded input recipe: the distributions the workloads are stated to have (no GPU).

Keys N(0, 1) with outlier channels (4 per kv head of magnitude ~N(40, 5) with a fixed sign, or
1 % of the layer's channels at ~N(50, 5)), values N(0, 1), queries N(0, 1) or "peaked" so that the
top 5 % of tokens hold 0.84 of the softmax mass, all from a counter-based generator, so any slice
equals the same slice of the whole."""
import math

import numpy as np

import synth


def test_deterministic_and_slices_agree():
    w = synth.WORKLOADS[1].scaled(batch=2, kv_heads=3, q_heads=3, prefill_tokens=300, decode_steps=4)
    K = synth.keys(w)
    assert np.array_equal(K, synth.keys(w))
    assert np.array_equal(synth.keys(w, b0=1, nb=1, h0=1, nh=2, t0=100, nt=50), K[1:2, 1:3, 100:150])
    V = synth.values(w)
    assert np.array_equal(synth.values(w, b0=1, nb=1, t0=299, nt=5), V[1:2, :, 299:304])
    assert not np.array_equal(K, V)
    assert not np.array_equal(synth.queries(w, 0), synth.queries(w, 1))


def test_per_head_outlier_channels():
    w = synth.WORKLOADS[1].scaled(batch=1, kv_heads=4, q_heads=4, prefill_tokens=2000, decode_steps=1)
    K = synth.keys(w)[0].astype(np.float64)  # [H][T][D]
    mean, std = K.mean(axis=1), K.std(axis=1)
    for h in range(w.kv_heads):
        big = np.flatnonzero(np.abs(mean[h]) > 20)
        assert len(big) == 4
        assert np.all(np.abs(np.abs(mean[h, big]) - 40) < 1.0)
        assert np.all(np.abs(std[h, big] - 5) < 0.5)
        assert np.all(np.sign(K[h][:, big]) == np.sign(mean[h, big]))  # the sign is fixed per channel
        rest = np.setdiff1d(np.arange(w.head_dim), big)
        assert np.all(np.abs(mean[h, rest]) < 0.15) and np.all(np.abs(std[h, rest] - 1) < 0.1)


def test_layer_one_percent_outliers():
    w = synth.WORKLOADS[2].scaled(batch=1, kv_heads=10, q_heads=10, prefill_tokens=1000, decode_steps=1)
    K = synth.keys(w)[0].astype(np.float64)
    mean = K.mean(axis=1)
    big = np.argwhere(np.abs(mean) > 20)
    assert len(big) == round(0.01 * w.kv_heads * w.head_dim)
    assert np.all(np.abs(np.abs(mean[np.abs(mean) > 20]) - 50) < 1.5)


def test_values_and_normal_queries_are_standard_normal():
    w = synth.WORKLOADS[0].scaled(prefill_tokens=4000)
    V = synth.values(w).astype(np.float64)
    assert abs(V.mean()) < 0.01 and abs(V.std() - 1) < 0.01
    q = np.concatenate([synth.queries(w, s).ravel() for s in range(20)]).astype(np.float64)
    assert abs(q.mean()) < 0.1 and abs(q.std() - 1) < 0.1


def test_peaked_queries_put_84_percent_of_the_mass_on_5_percent_of_tokens():
    w = synth.WORKLOADS[2].scaled(batch=1, kv_heads=2, q_heads=2, prefill_tokens=1500, decode_steps=1)
    T = w.prefill_tokens + 1
    K = synth.keys(w, nt=T)[0].astype(np.float64)
    q = synth.queries(w, 0)[0].astype(np.float64)  # fp16 as the caches get it
    for h in range(w.q_heads):
        s = K[h // w.group_q] @ q[h] / math.sqrt(w.head_dim)
        p = np.exp(s - s.max())
        k = math.ceil(0.05 * T)
        share = np.sort(p)[-k:].sum() / p.sum()
        assert abs(share - 0.84) < 0.02, (h, share)
    # the "normal" recipe is far from peaked
    w0 = w.scaled(queries="normal")
    q0 = synth.queries(w0, 0)[0].astype(np.float64)
    s0 = K[0] @ q0[0] / math.sqrt(w.head_dim)
    p0 = np.exp(s0 - s0.max())
    assert np.sort(p0)[-math.ceil(0.05 * T):].sum() / p0.sum() < 0.84
