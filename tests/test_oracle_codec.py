"""Pins of the codec-decoder oracle against what the pages and mathematics fix:
library routines on special cases (torch CPU convolutions, layer norm, GELU),
closed forms (SnakeBeta, the dequantisation sum, identity configurations),
a full recompute of one transformer layer from its definition, and the
decoder's own invariants (causality, chunk grid, streaming = whole decode)."""
import dataclasses
import json
import os

import numpy as np
import pytest

import oracle
import oracle.codec as oc
import synth
import synth.codec as sc

torch = pytest.importorskip("torch")
F = torch.nn.functional

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "page_facts.json")


def _f(a):
    a = np.asarray(a)
    return synth.bf16_bits_to_f32(a).astype(np.float64) if a.dtype == np.uint16 else a.astype(np.float64)


def _rng(seed):
    return np.random.default_rng(seed)


# ---------------------------------------------------------------- building blocks
@pytest.mark.parametrize("K,d", [(7, 1), (7, 3), (7, 9), (1, 1), (3, 2)])
def test_conv1d_is_causal_torch_conv(K, d):
    r = _rng(K * 10 + d)
    T, Cin, Cout = 40, 5, 6
    x = r.standard_normal((T, Cin))
    W = r.standard_normal((Cout, K, Cin)).astype(np.float32)
    b = r.standard_normal(Cout).astype(np.float32)
    y = oc.conv1d(x, W, b, d)
    xt = torch.from_numpy(x.T[None].copy())
    wt = torch.from_numpy(np.transpose(W.astype(np.float64), (0, 2, 1)).copy())
    ref = F.conv1d(F.pad(xt, ((K - 1) * d, 0)), wt, torch.from_numpy(b.astype(np.float64)), dilation=d)
    np.testing.assert_allclose(y, ref[0].numpy().T, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("s,J", [(2, 1), (3, 2), (8, 2), (5, 2)])
def test_conv_transpose_is_torch_conv_transpose_trimmed(s, J):
    r = _rng(s * 7 + J)
    T, Cin, Cout = 9, 4, 3
    x = r.standard_normal((T, Cin))
    W = r.standard_normal((s, Cout, J, Cin)).astype(np.float32)
    b = r.standard_normal(Cout).astype(np.float32)
    y = oc.conv_transpose(x, W, b, s)
    # torch layout [Cin][Cout][kernel], tap k = r + j s
    Kt = J * s
    wt = np.zeros((Cin, Cout, Kt))
    for k in range(Kt):
        wt[:, :, k] = W[k % s, :, k // s, :].T
    full = F.conv_transpose1d(torch.from_numpy(x.T[None].copy()), torch.from_numpy(wt),
                              torch.from_numpy(b.astype(np.float64)), stride=s)[0].numpy().T
    assert full.shape[0] == (T - 1) * s + Kt
    np.testing.assert_allclose(y, full[:T * s], rtol=1e-12, atol=1e-12)


def test_snake_closed_form():
    r = _rng(3)
    x = r.standard_normal((17, 4)) * 3
    la = np.array([0.0, 0.5, -0.3, 1.0], np.float32)
    lb = np.array([0.0, -0.2, 0.7, 0.1], np.float32)
    y = oc.snake(x, la, lb)
    a, b = np.exp(la.astype(np.float64)), np.exp(lb.astype(np.float64))
    np.testing.assert_allclose(y, x + np.sin(a * x) ** 2 / (b + 1e-9), rtol=1e-13, atol=1e-13)
    # a = b = 1: x + sin^2 x
    y0 = oc.snake(x, np.zeros(4, np.float32), np.zeros(4, np.float32))
    np.testing.assert_allclose(y0, x + np.sin(x) ** 2 / (1 + 1e-9), rtol=1e-13)


def _softmax_attention(q, k, v, H, W):
    T, D = q.shape
    hd = D // H
    out = np.zeros_like(q)
    for h in range(H):
        sl = slice(h * hd, (h + 1) * hd)
        s = q[:, sl] @ k[:, sl].T / np.sqrt(hd)
        for t in range(T):
            m = np.full(T, -np.inf)
            lo = max(0, t - W + 1)
            m[lo:t + 1] = s[t, lo:t + 1]
            p = np.exp(m - m.max())
            out[t, sl] = (p / p.sum()) @ v[:, sl]
    return out


@pytest.mark.parametrize("W", [1, 3, 8, 100])
def test_window_attention_brute_force(W):
    r = _rng(W)
    T, H, hd = 20, 2, 8
    q, k, v = (r.standard_normal((T, H * hd)) for _ in range(3))
    o = oc.window_attention(q, k, v, H, W)
    np.testing.assert_allclose(o, _softmax_attention(q, k, v, H, W), rtol=1e-12, atol=1e-12)
    if W == 1:
        np.testing.assert_allclose(o, v, rtol=1e-13)


# ---------------------------------------------------------------- whole decoder, special cases
def _small(**kw):
    return dataclasses.replace(sc.CODEC_SMALL, **kw)


def test_page_shape_facts():
    facts = json.load(open(GOLDEN))["codec_decoder"]
    d = sc.CODEC_FULL
    assert (d.n_codebooks, d.codebook_size, d.codebook_dim) == (facts["codebooks"], facts["codebook_size"],
                                                                facts["codebook_dim"])
    assert (d.n_layers, d.hidden, d.head_dim, d.window) == (facts["layers"], facts["hidden"], facts["head_dim"],
                                                            facts["window"])
    assert d.rope_theta == facts["rope_theta"] and list(d.strides) == facts["upsample"]
    assert d.samples_per_frame == facts["samples_per_frame"]
    assert facts["samples_per_frame"] * facts["frame_rate_hz"] == facts["sample_rate"]
    st = json.load(open(GOLDEN))["codec_streaming"]
    assert (oc.STREAM_FIRST, oc.STREAM_EVERY, oc.CHUNK_FRAMES, oc.CHUNK_CONTEXT) == (st["first"], st["every"],
                                                                                    st["chunk"], st["context"])


def _identity_weights(d, w):
    """Residual branches off (LayerScale, ConvNeXt gamma, residual-unit output
    convolutions zero) and SnakeBeta ~ identity (exp(b) = e^40): the decoder
    reduces to dequantisation, the final RMSNorm and a chain of plain and
    transposed convolutions."""
    w = dict(w)
    for k in ("ls_attn", "ls_mlp", "gamma"):
        w[k] = np.zeros_like(w[k])
    big = lambda a: np.full_like(a, 40.0)
    blocks = []
    for blk in w["blocks"]:
        blk = dict(blk, snake_b=big(blk["snake_b"]))
        blk["units"] = [dict(u, w2=np.zeros_like(u["w2"]), c2=np.zeros_like(u["c2"])) for u in blk["units"]]
        blocks.append(blk)
    w["blocks"] = blocks
    w["out_b"] = big(w["out_b"])
    return w


def _dequant(d, w, codes):
    E = _f(w["codebooks"])
    zs = E[0][codes[:, 0]]
    za = sum(E[q][codes[:, q]] for q in range(1, d.n_codebooks))
    return zs @ _f(w["proj_sem"]).T + za @ _f(w["proj_ac"]).T


def _rms(x, g, eps):
    return x / np.sqrt((x * x).mean(-1, keepdims=True) + eps) * g


def test_identity_configuration_is_a_convolution_chain():
    d = sc.CODEC_SMALL
    w = _identity_weights(d, sc.make_codec_weights(d, synth.F32, 11))
    codes = sc.make_codes(d, 10, 12)
    wav = oc.Decoder(d, w).decode_window(codes)
    x = _rms(_dequant(d, w, codes), _f(w["final_norm"]), d.rms_eps)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a))

    def tconv(x, W, b, s):   # W [s][Cout][J][Cin]
        Wf = _f(W)
        J = Wf.shape[2]
        wt = np.zeros((Wf.shape[3], Wf.shape[1], J * s))
        for k in range(J * s):
            wt[:, :, k] = Wf[k % s, :, k // s, :].T
        y = F.conv_transpose1d(t(x.T[None]), t(wt), t(_f(b)), stride=s)[0].numpy().T
        return y[:x.shape[0] * s]

    def conv(x, W, b, dil=1):   # W [Cout][K][Cin]
        Wf = np.transpose(_f(W), (0, 2, 1))
        K = Wf.shape[2]
        return F.conv1d(F.pad(t(x.T[None]), ((K - 1) * dil, 0)), t(Wf), t(_f(b)), dilation=dil)[0].numpy().T

    for u in range(d.n_up):
        x = tconv(x, w["up_w"][u], w["up_b"][u], 2)
    x = conv(x, w["in_w"], w["in_b"])
    for i, s in enumerate(d.strides):
        x = x + np.sin(np.exp(_f(w["blocks"][i]["snake_a"])) * x) ** 2 / (np.exp(40.0) + 1e-9)
        x = tconv(x, w["blocks"][i]["tconv_w"], w["blocks"][i]["tconv_b"], s)
    y = conv(x, w["out_w"], w["out_bias"])[:, 0]
    assert wav.shape == (codes.shape[0] * d.samples_per_frame,)
    np.testing.assert_allclose(wav, np.tanh(y), rtol=1e-9, atol=1e-12)


def test_convnext_stage_is_torch_ops():
    """One upsampling stage with its ConvNeXt block on, everything after it an
    identity chain, against torch's depthwise conv, layer_norm and GELU."""
    d = _small(n_layers=0, strides=(2,), dac_channels=2 * 128)
    w = sc.make_codec_weights(d, synth.F32, 21)
    w = _identity_weights(d, w)
    w["gamma"] = sc.make_codec_weights(d, synth.F32, 21)["gamma"]     # ConvNeXt on again
    codes = sc.make_codes(d, 9, 22)
    dec = oc.Decoder(d, w)
    wav = dec.decode_window(codes)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a))
    x = _rms(_dequant(d, w, codes), _f(w["final_norm"]), d.rms_eps)
    for u in range(d.n_up):
        Wf = _f(w["up_w"][u])
        y = np.zeros((x.shape[0] * 2, d.hidden))
        for r in range(2):
            y[r::2] = x @ Wf[r, :, 0, :].T
        x = y + _f(w["up_b"][u])
        xt = t(x.T[None])
        dcv = F.conv1d(F.pad(xt, (6, 0)), t(_f(w["dw_w"][u])[:, None, :]), t(_f(w["dw_b"][u])), groups=d.hidden)
        nrm = F.layer_norm(dcv[0].T, (d.hidden,), t(_f(w["ln_w"][u])), t(_f(w["ln_b"][u])), eps=d.ln_eps)
        h = F.gelu(F.linear(nrm, t(_f(w["fc1_w"][u])), t(_f(w["fc1_b"][u]))))
        h = F.linear(h, t(_f(w["fc2_w"][u])), t(_f(w["fc2_b"][u])))
        x = x + _f(w["gamma"][u]) * h.numpy()
    # identity vocoder tail of one block
    Win = np.transpose(_f(w["in_w"]), (0, 2, 1))
    x = F.conv1d(F.pad(t(x.T[None]), (6, 0)), t(Win), t(_f(w["in_b"])))[0].numpy().T
    blk = w["blocks"][0]
    x = x + np.sin(np.exp(_f(blk["snake_a"])) * x) ** 2 / (np.exp(40.0) + 1e-9)
    Wt = _f(blk["tconv_w"])
    y = np.zeros((x.shape[0] * 2, Wt.shape[1]))
    for r in range(2):
        y[r::2] += x @ Wt[r, :, 0, :].T
        y[r::2][1:] += x[:-1] @ Wt[r, :, 1, :].T
    x = y + _f(blk["tconv_b"])
    Wo = np.transpose(_f(w["out_w"]), (0, 2, 1))
    out = F.conv1d(F.pad(t(x.T[None]), (6, 0)), t(Wo), t(_f(w["out_bias"])))[0, 0].numpy()
    np.testing.assert_allclose(wav, np.tanh(out), rtol=1e-9, atol=1e-11)


def _rope(v, pos, theta):
    hd = v.shape[-1]
    h = hd // 2
    f = theta ** (-2.0 * np.arange(h) / hd)
    a = pos * f
    c, s = np.cos(a), np.sin(a)
    out = v.copy()
    out[..., :h] = v[..., :h] * c - v[..., h:] * s
    out[..., h:] = v[..., h:] * c + v[..., :h] * s
    return out


def test_transformer_layer_recompute():
    """One transformer layer recomputed from its definition: pre-norm RMSNorm,
    q/k/v, rotate-half RoPE (theta 1e4) at the frame index, 8-frame window
    attention, LayerScale, SiLU-gated MLP, final RMSNorm."""
    d = _small(n_layers=1)
    w = sc.make_codec_weights(d, synth.BF16, 31)
    codes = sc.make_codes(d, 14, 32)
    _, lat = oc.Decoder(d, w).decode_window(codes, latent=True)
    x = _dequant(d, w, codes)
    D, H, hd, Fd = d.hidden, d.n_heads, d.head_dim, d.ffn
    h = _rms(x, _f(w["attn_norm"][0]), d.rms_eps)
    qkv = h @ _f(w["wqkv"][0]).T
    q, k, v = qkv[:, :D].copy(), qkv[:, D:2 * D].copy(), qkv[:, 2 * D:]
    for t in range(x.shape[0]):
        for hh in range(H):
            q[t, hh * hd:(hh + 1) * hd] = _rope(q[t, hh * hd:(hh + 1) * hd], t, d.rope_theta)
            k[t, hh * hd:(hh + 1) * hd] = _rope(k[t, hh * hd:(hh + 1) * hd], t, d.rope_theta)
    o = _softmax_attention(q, k, v, H, d.window)
    x = x + _f(w["ls_attn"][0]) * (o @ _f(w["wo"][0]).T)
    h = _rms(x, _f(w["mlp_norm"][0]), d.rms_eps)
    gu = h @ _f(w["wgu"][0]).T
    a = gu[:, :Fd] / (1 + np.exp(-gu[:, :Fd])) * gu[:, Fd:]
    x = x + _f(w["ls_mlp"][0]) * (a @ _f(w["wd"][0]).T)
    np.testing.assert_allclose(lat, _rms(x, _f(w["final_norm"]), d.rms_eps), rtol=1e-10, atol=1e-10)


def test_dequantisation_picks_rows_per_codebook():
    """With one-hot codebook rows and identity projections, the latent before
    the norm is the sum of the selected one-hot rows: any codebook / row
    offset mistake moves a spike."""
    d = _small(n_layers=0, codebook_dim=128)
    w = sc.make_codec_weights(d, synth.F32, 41)
    V, Dc = d.codebook_size, d.codebook_dim
    E = np.zeros((d.n_codebooks, V, Dc), np.float32)
    for q in range(d.n_codebooks):
        for r in range(V):
            E[q, r, (q * 7 + r) % Dc] = 1.0 + q
    w["codebooks"] = E
    w["proj_sem"] = np.eye(d.hidden, Dc, dtype=np.float32)
    w["proj_ac"] = 2 * np.eye(d.hidden, Dc, dtype=np.float32)
    w["final_norm"] = np.ones(d.hidden, np.float32)
    codes = sc.make_codes(d, 6, 42)
    _, lat = oc.Decoder(d, w).decode_window(codes, latent=True)
    for t in range(6):
        x = np.zeros(d.hidden)
        for q in range(d.n_codebooks):
            x[(q * 7 + codes[t, q]) % Dc] += (1.0 + q) * (1.0 if q == 0 else 2.0)
        np.testing.assert_allclose(lat[t], x / np.sqrt((x * x).mean() + d.rms_eps), rtol=1e-12)


# ---------------------------------------------------------------- invariants
def test_causal_prefix():
    d = sc.CODEC_SMALL
    dec = oc.Decoder(d, sc.make_codec_weights(d, synth.BF16, 51))
    codes = sc.make_codes(d, 20, 52)
    full = dec.decode_window(codes)
    for n in (1, 5, 13):
        part = dec.decode_window(codes[:n])
        assert np.array_equal(part, full[:n * d.samples_per_frame])


def test_chunk_grid_and_streaming():
    d = sc.CODEC_SMALL
    dec = oc.Decoder(d, sc.make_codec_weights(d, synth.BF16, 61))
    codes = sc.make_codes(d, 41, 62)
    spf = d.samples_per_frame
    whole = dec.decode(codes, chunk=16, context=5)
    # one chunk = one window
    assert np.array_equal(dec.decode(codes[:16], chunk=16, context=5), dec.decode_window(codes[:16]))
    # chunk 2 = the window from frame 27, its own frames kept
    assert np.array_equal(whole[32 * spf:], dec.decode_window(codes[27:41])[5 * spf:])
    # the left context changes the samples (the window reaches back past it)
    assert not np.array_equal(whole[16 * spf:32 * spf], dec.decode_window(codes[:32])[16 * spf:])
    parts = dec.stream(codes, chunk=16, context=5, first=4, every=3)
    got = np.concatenate([p for _, p in parts])
    assert got.shape == whole.shape
    np.testing.assert_array_equal(got, whole)
    assert parts[0][0] == 4 and len(parts[0][1]) == 4 * spf


def test_bad_code_rejected():
    d = sc.CODEC_SMALL
    dec = oc.Decoder(d, sc.make_codec_weights(d, synth.F32, 71))
    codes = sc.make_codes(d, 3, 72)
    codes[1, 5] = d.codebook_size
    with pytest.raises(ValueError):
        dec.decode_window(codes)
