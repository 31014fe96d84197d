"""Pins for the oracle's text side (CPU only): BPE ids -> text embedding ->
ResizeMLP (two linear layers with SiLU between them), from
"Qwen3-TTS 移植 ncnn 简明教程" section 1, talker bullet.  Each case is built
so that the result has a closed form that does not go through the oracle."""
import math

import numpy as np
import pytest

import oracle
import synth


def _silu(x):
    return x / (1.0 + math.exp(-x))


def _weights(V, T, H, emb=None, w1=None, b1=None, w2=None, b2=None, seed=0):
    rng = np.random.default_rng(seed)
    return {"text_emb": (rng.standard_normal((V, T)) if emb is None else emb).astype(np.float32),
            "text_fc1_w": (rng.standard_normal((T, T)) * 0.1 if w1 is None else w1).astype(np.float32),
            "text_fc1_b": (rng.standard_normal(T) * 0.1 if b1 is None else b1).astype(np.float32),
            "text_fc2_w": (rng.standard_normal((H, T)) * 0.1 if w2 is None else w2).astype(np.float32),
            "text_fc2_b": (rng.standard_normal(H) * 0.1 if b2 is None else b2).astype(np.float32)}


def test_identity_layers_give_silu_of_the_embedding():
    V, T = 11, 8
    w = _weights(V, T, T, w1=np.eye(T), b1=np.zeros(T), w2=np.eye(T), b2=np.zeros(T))
    ids = [3, 0, 10, 3]
    out = oracle.text_embed(w, synth.F32, ids)
    for r, i in enumerate(ids):
        want = [_silu(float(v)) for v in w["text_emb"][i]]
        assert np.allclose(out[r], want, rtol=0, atol=1e-12)


def test_one_hot_rows_pin_the_gathered_index():
    V, T = 16, 8
    emb = np.zeros((V, T))
    for i in range(V):
        emb[i, i % T] = 3.0 + i    # row i: one entry at column i % T
    w = _weights(V, T, T, emb=emb, w1=np.eye(T), b1=np.zeros(T), w2=np.eye(T), b2=np.zeros(T))
    ids = [13, 2, 7]
    out = oracle.text_embed(w, synth.F32, ids)
    for r, i in enumerate(ids):
        want = np.zeros(T)
        want[i % T] = _silu(3.0 + i)
        assert np.allclose(out[r], want, rtol=0, atol=1e-12)


def test_zero_second_layer_leaves_its_bias():
    V, T, H = 9, 8, 5
    b2 = np.array([0.5, -1.25, 2.0, 0.0, 3.5])
    w = _weights(V, T, H, w2=np.zeros((H, T)), b2=b2)
    out = oracle.text_embed(w, synth.F32, [0, 4, 8])
    assert np.array_equal(out, np.tile(b2, (3, 1)))


def test_silu_sits_between_the_layers():
    """A zero first layer makes the hidden activation SiLU(b1) for every id."""
    V, T, H = 9, 8, 6
    b1 = np.linspace(-2.0, 2.0, T)
    w2 = np.zeros((H, T))
    w2[np.arange(H), np.arange(H)] = 1.0    # output j = hidden j
    b2 = np.arange(H) * 0.25
    w = _weights(V, T, H, w1=np.zeros((T, T)), b1=b1, w2=w2, b2=b2)
    out = oracle.text_embed(w, synth.F32, [1, 5])
    want = [_silu(float(np.float32(b1[j]))) + float(np.float32(b2[j])) for j in range(H)]
    assert np.allclose(out, np.tile(want, (2, 1)), rtol=0, atol=1e-12)


def test_bf16_weights_are_read_exactly():
    """bf16 matrices: the same result as their exact fp32 values."""
    V, T, H = 7, 16, 8
    w32 = _weights(V, T, H, seed=3)
    wb = dict(w32)
    for k in ("text_emb", "text_fc1_w", "text_fc2_w"):
        wb[k] = synth.round_bf16(w32[k])
        w32[k] = synth.bf16_bits_to_f32(wb[k])
    ids = [0, 6, 3]
    assert np.array_equal(oracle.text_embed(wb, synth.BF16, ids), oracle.text_embed(w32, synth.F32, ids))


def test_out_of_range_id_is_refused():
    w = _weights(5, 8, 8)
    with pytest.raises(ValueError):
        oracle.text_embed(w, synth.F32, [0, 5])
    with pytest.raises(ValueError):
        oracle.text_embed(w, synth.F32, [-1])
