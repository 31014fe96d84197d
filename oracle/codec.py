"""Oracle for the 12 Hz codec decoder: TEST INFRASTRUCTURE.

Wraps the fp64 CPU decoder in codec.cpp (one window of frames decoded from a
zero state) and composes a whole request from windows the way the Mizuoto
"Qwen3-TTS" page describes it (section "速度"): a grid of 300-frame chunks,
each decoded with the 25 frames before it as left context and only its own
frames' samples kept; streaming output decodes the current chunk from its
regular start after the first 4 frames and then every 12, sending the
samples not sent before.  Only tests/, the smoke check and the benchmark's
CPU-baseline leg may import this module; the product path never does.
"""
from __future__ import annotations

import ctypes

import numpy as np

from . import _L

CHUNK_FRAMES = 300      # frames per chunk of the grid
CHUNK_CONTEXT = 25      # left-context frames decoded before a chunk
STREAM_FIRST = 4        # frames before the first streamed decode
STREAM_EVERY = 12       # frames between later streamed decodes


class OCConfig(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in ("n_codebooks", "codebook_size", "codebook_dim", "hidden", "n_layers",
                                            "n_heads", "head_dim", "ffn", "window")] + \
              [(n, ctypes.c_float) for n in ("rope_theta", "rms_eps", "ln_eps")] + \
              [(n, ctypes.c_int) for n in ("n_up", "up_ffn", "dac_channels", "n_blocks")] + \
              [("strides", ctypes.c_int * 4)]


_P = ctypes.c_void_p


class OCWeights(ctypes.Structure):
    _fields_ = [(n, _P) for n in ("codebooks", "proj_sem", "proj_ac", "attn_norm", "wqkv", "wo", "ls_attn",
                                  "mlp_norm", "wgu", "wd", "ls_mlp", "final_norm", "up_w", "up_b", "dw_w", "dw_b",
                                  "ln_w", "ln_b", "fc1_w", "fc1_b", "fc2_w", "fc2_b", "gamma", "in_w", "in_b")] + \
              [("blk", (_P * 4) * 4), ("unit", ((_P * 8) * 3) * 4)] + \
              [(n, _P) for n in ("out_a", "out_b", "out_w", "out_bias")]


def _f32(a, dtype_bf16: bool):
    a = np.asarray(a)
    if a.dtype == np.uint16:
        return np.ascontiguousarray((a.astype(np.uint32) << 16).view(np.float32))
    return np.ascontiguousarray(a, dtype=np.float32)


def make_config(d) -> OCConfig:
    c = OCConfig(d.n_codebooks, d.codebook_size, d.codebook_dim, d.hidden, d.n_layers, d.n_heads, d.head_dim,
                 d.ffn, d.window, d.rope_theta, d.rms_eps, d.ln_eps, d.n_up, d.up_ffn, d.dac_channels,
                 len(d.strides))
    for i, s in enumerate(d.strides):
        c.strides[i] = s
    return c


class Decoder:
    """fp64 decoder of one set of weights (host arrays from synth.codec)."""

    def __init__(self, dims, weights: dict):
        if len(dims.strides) > 4:
            raise ValueError("at most 4 vocoder blocks")
        self.d = dims
        self.cfg = make_config(dims)
        self.keep = []
        w = OCWeights()

        def p(a):
            a = _f32(a, True)
            self.keep.append(a)
            return a.ctypes.data

        for k in ("codebooks", "proj_sem", "proj_ac", "attn_norm", "wqkv", "wo", "ls_attn", "mlp_norm", "wgu", "wd",
                  "ls_mlp", "final_norm", "up_w", "up_b", "dw_w", "dw_b", "ln_w", "ln_b", "fc1_w", "fc1_b", "fc2_w",
                  "fc2_b", "gamma", "in_w", "in_b", "out_a", "out_b", "out_w", "out_bias"):
            setattr(w, k, p(weights[k]))
        for b, blk in enumerate(weights["blocks"]):
            for i, k in enumerate(("snake_a", "snake_b", "tconv_w", "tconv_b")):
                w.blk[b][i] = p(blk[k])
            for u, unit in enumerate(blk["units"]):
                for i, k in enumerate(("a1", "b1", "w1", "c1", "a2", "b2", "w2", "c2")):
                    w.unit[b][u][i] = p(unit[k])
        self.w = w

    @property
    def spf(self) -> int:
        return self.d.samples_per_frame

    def decode_window(self, codes, latent=False):
        """codes [T, n_codebooks] -> waveform [T * samples_per_frame] (fp64),
        decoded from a zero state (and the transformer output [T, hidden])."""
        codes = np.ascontiguousarray(codes, dtype=np.int32)
        T = codes.shape[0]
        wav = np.zeros(T * self.spf, np.float64)
        lat = np.zeros((T, self.d.hidden), np.float64)
        rc = _L().oracle_codec_decode(ctypes.byref(self.cfg), ctypes.byref(self.w), codes.ctypes.data, T,
                                      lat.ctypes.data, wav.ctypes.data)
        if rc:
            raise ValueError("code outside the codebook")
        return (wav, lat) if latent else wav

    def decode(self, codes, chunk=CHUNK_FRAMES, context=CHUNK_CONTEXT):
        """A whole request on the chunk grid: chunk c covers frames
        [c*chunk, (c+1)*chunk); it is decoded from frame max(0, c*chunk -
        context) and only its own frames' samples are kept."""
        codes = np.asarray(codes)
        T = codes.shape[0]
        out = np.zeros(T * self.spf, np.float64)
        for c0 in range(0, T, chunk):
            s0, e = max(0, c0 - context), min(T, c0 + chunk)
            wav = self.decode_window(codes[s0:e])
            out[c0 * self.spf:e * self.spf] = wav[(c0 - s0) * self.spf:]
        return out

    def stream(self, codes, chunk=CHUNK_FRAMES, context=CHUNK_CONTEXT, first=STREAM_FIRST, every=STREAM_EVERY):
        """Streaming output of a request whose frames arrive one by one: a
        decode after `first` frames, then after every `every` more, and at the
        end; each decodes the current chunk from its regular start up to the
        frames received and sends the samples not sent yet.  Returns the list
        of (frames received, samples sent)."""
        codes = np.asarray(codes)
        T = codes.shape[0]
        sent = 0
        parts = []
        due = first
        for n in range(1, T + 1):
            if n != due and n != T:
                continue
            c0 = ((n - 1) // chunk) * chunk
            # samples of an earlier chunk not yet sent: finish that chunk first
            while sent < c0 * self.spf:
                pc0 = (sent // self.spf // chunk) * chunk
                s0, e = max(0, pc0 - context), pc0 + chunk
                wav = self.decode_window(codes[s0:e])
                piece = wav[sent - s0 * self.spf:]
                parts.append((e, piece))
                sent = e * self.spf
            s0 = max(0, c0 - context)
            wav = self.decode_window(codes[s0:n])
            piece = wav[sent - s0 * self.spf:]
            parts.append((n, piece))
            sent = n * self.spf
            if n == due:
                due += every
        return parts


def conv1d(x, W, b, dilation=1):
    """Causal Conv1d of channels-last x [T, Cin] with W [Cout, K, Cin]."""
    x = np.ascontiguousarray(x, dtype=np.float64)
    W = _f32(W, True)
    T, Cin = x.shape
    Cout, K, _ = W.shape
    bb = None if b is None else _f32(b, True)
    y = np.zeros((T, Cout), np.float64)
    _L().oracle_codec_conv1d(x.ctypes.data, T, Cin, Cout, K, dilation, W.ctypes.data,
                             None if bb is None else bb.ctypes.data, y.ctypes.data)
    return y


def conv_transpose(x, W, b, stride):
    """Causal transposed convolution of x [T, Cin] with W [stride, Cout, J, Cin]
    (kernel J * stride); T * stride output samples."""
    x = np.ascontiguousarray(x, dtype=np.float64)
    W = _f32(W, True)
    T, Cin = x.shape
    s, Cout, J, _ = W.shape
    bb = None if b is None else _f32(b, True)
    y = np.zeros((T * s, Cout), np.float64)
    _L().oracle_codec_conv_transpose(x.ctypes.data, T, Cin, Cout, s, J * s, W.ctypes.data,
                                     None if bb is None else bb.ctypes.data, y.ctypes.data)
    return y


def snake(x, a, b):
    x = np.array(x, dtype=np.float64, order="C")
    T, C = x.shape
    a, b = _f32(a, True), _f32(b, True)
    _L().oracle_codec_snake(x.ctypes.data, T, C, a.ctypes.data, b.ctypes.data)
    return x


def window_attention(q, k, v, n_heads, window):
    """q, k, v [T, H*hd] -> [T, H*hd]: causal attention over the last `window` frames."""
    q, k, v = (np.ascontiguousarray(a, dtype=np.float64) for a in (q, k, v))
    T, D = q.shape
    out = np.zeros((T, D), np.float64)
    _L().oracle_codec_attention(q.ctypes.data, k.ctypes.data, v.ctypes.data, T, n_heads, D // n_heads, window,
                                out.ctypes.data)
    return out
