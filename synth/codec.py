"""Seeded synthetic inputs for the 12 Hz codec decoder: shapes, random-init
weights and code streams.  Holds none of the decoder's arithmetic; both the
oracle and the CUDA path take these arrays as they are.

Shapes follow the Codec Decoder bullet of "Qwen3-TTS 移植 ncnn 简明教程"
(ncnn discussion 6798, section 1): 16 codebooks of 2048 x 256, an 8-layer
transformer of width 512 with head_dim 64 and a 72-frame window, two x2
upsampling stages, and a vocoder with strides 8, 5, 4, 3 (1920 samples per
frame).  Widths the page does not give (transformer MLP 1024, ConvNeXt MLP
2048, vocoder channels 1536 halving per block) are the readings listed with
the design notes.
"""
from __future__ import annotations

import dataclasses

import numpy as np

from . import BF16, F32, normal, randint, _stream


@dataclasses.dataclass(frozen=True)
class CodecDims:
    n_codebooks: int = 16
    codebook_size: int = 2048
    codebook_dim: int = 256
    hidden: int = 512
    n_layers: int = 8
    n_heads: int = 8
    head_dim: int = 64
    ffn: int = 1024
    window: int = 72
    rope_theta: float = 1e4
    rms_eps: float = 1e-5
    ln_eps: float = 1e-6
    n_up: int = 2
    up_ffn: int = 2048
    dac_channels: int = 1536
    strides: tuple = (8, 5, 4, 3)

    @property
    def n_blocks(self) -> int:
        return len(self.strides)

    @property
    def samples_per_frame(self) -> int:
        return (2 ** self.n_up) * int(np.prod(self.strides))


CODEC_FULL = CodecDims()
# a small decoder with every structural feature (several transformer layers,
# a window shorter than the test windows, both upsampling stages, four
# vocoder blocks with odd and even strides)
CODEC_SMALL = CodecDims(codebook_size=64, codebook_dim=32, hidden=128, n_layers=2, n_heads=2, head_dim=64,
                        ffn=256, window=8, up_ffn=256, dac_channels=128, strides=(2, 3, 2, 2))

VEC_KEYS = ("attn_norm", "ls_attn", "mlp_norm", "ls_mlp", "final_norm", "up_b", "dw_w", "dw_b", "ln_w", "ln_b",
            "fc1_b", "fc2_b", "gamma", "in_b", "out_a", "out_b", "out_bias")


def make_codec_weights(d: CodecDims, dtype: int, seed: int) -> dict:
    """Random-init decoder weights (bf16 matrices as uint16 bit patterns; per-
    channel vectors and the depthwise taps fp32), scaled so activations stay
    of order one through the stack.  Layouts: see the keys below; matrices
    are [out][in], convolutions [Cout][K][Cin], transposed convolutions
    [stride][Cout][K/stride][Cin]."""
    D, Dc, V, NQ, F, L = d.hidden, d.codebook_dim, d.codebook_size, d.n_codebooks, d.ffn, d.n_layers
    U, F2, C0 = d.n_up, d.up_ffn, d.dac_channels
    k = iter(range(1, 1 << 20))

    def mat(shape, std):
        return normal(shape, seed, _stream(0x500, next(k)), std, dtype)

    def vec(shape, mean, std):
        return (mean + normal(shape, seed, _stream(0x500, next(k)), std)).astype(np.float32)

    w = {
        "codebooks": mat((NQ, V, Dc), 1.0),
        "proj_sem": mat((D, Dc), 1.0 / np.sqrt(Dc)),
        "proj_ac": mat((D, Dc), 1.0 / np.sqrt(Dc * (NQ - 1))),
        "attn_norm": vec((L, D), 1.0, 0.1),
        "wqkv": mat((L, 3 * D, D), 1.0 / np.sqrt(D)),
        "wo": mat((L, D, D), 1.0 / np.sqrt(D)),
        "ls_attn": vec((L, D), 0.1, 0.02),
        "mlp_norm": vec((L, D), 1.0, 0.1),
        "wgu": mat((L, 2 * F, D), 1.0 / np.sqrt(D)),
        "wd": mat((L, D, F), 1.0 / np.sqrt(F)),
        "ls_mlp": vec((L, D), 0.1, 0.02),
        "final_norm": vec((D,), 1.0, 0.1),
        "up_w": mat((U, 2, D, 1, D), 1.0 / np.sqrt(D)),
        "up_b": vec((U, D), 0.0, 0.02),
        "dw_w": vec((U, D, 7), 0.0, 1.0 / np.sqrt(7)),
        "dw_b": vec((U, D), 0.0, 0.02),
        "ln_w": vec((U, D), 1.0, 0.1),
        "ln_b": vec((U, D), 0.0, 0.1),
        "fc1_w": mat((U, F2, D), 1.0 / np.sqrt(D)),
        "fc1_b": vec((U, F2), 0.0, 0.02),
        "fc2_w": mat((U, D, F2), 1.0 / np.sqrt(F2)),
        "fc2_b": vec((U, D), 0.0, 0.02),
        "gamma": vec((U, D), 0.1, 0.02),
        "in_w": mat((C0, 7, D), 1.0 / np.sqrt(7 * D)),
        "in_b": vec((C0,), 0.0, 0.02),
        "blocks": [],
    }
    C = C0
    for s in d.strides:
        Co = C // 2
        blk = {"snake_a": vec((C,), 0.0, 0.2), "snake_b": vec((C,), 0.0, 0.2),
               "tconv_w": mat((s, Co, 2, C), 1.0 / np.sqrt(2 * C)), "tconv_b": vec((Co,), 0.0, 0.02),
               "units": []}
        for _ in range(3):
            blk["units"].append({"a1": vec((Co,), 0.0, 0.2), "b1": vec((Co,), 0.0, 0.2),
                                 "w1": mat((Co, 7, Co), 0.5 / np.sqrt(7 * Co)), "c1": vec((Co,), 0.0, 0.02),
                                 "a2": vec((Co,), 0.0, 0.2), "b2": vec((Co,), 0.0, 0.2),
                                 "w2": mat((Co, 1, Co), 0.5 / np.sqrt(Co)), "c2": vec((Co,), 0.0, 0.02)})
        w["blocks"].append(blk)
        C = Co
    w["out_a"] = vec((C,), 0.0, 0.2)
    w["out_b"] = vec((C,), 0.0, 0.2)
    w["out_w"] = mat((1, 7, C), 0.15 / np.sqrt(7 * C))
    w["out_bias"] = vec((1,), 0.0, 0.02)
    return w


def make_codes(d: CodecDims, T: int, seed: int) -> np.ndarray:
    """Uniform random codes [T, n_codebooks] int32 (codebook 0 first)."""
    return randint(T * d.n_codebooks, seed, _stream(0x600), 0, d.codebook_size - 1).reshape(T, d.n_codebooks)

