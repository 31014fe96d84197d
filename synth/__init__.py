"""Seeded synthetic inputs for the Qwen3-TTS frame loop.

This module is shared by the oracle and the CUDA path and holds none of the
method's arithmetic: it only produces random-init weights, prompt / trailing
text embeddings and per-row sampling settings, all as host numpy arrays.

Recipe (the configurations of the frame-loop workloads):
  * every matrix and embedding table ~ N(0, 0.02), drawn in fp32 and, for bf16
    models, rounded to bf16 (round-to-nearest-even);
  * RMSNorm weights = 1 (``norm_std`` > 0 gives 1 + N(0, norm_std) instead,
    used by parity cases that must exercise the norm weights);
  * prompt embeddings, trailing text rows and the tts_pad row ~ N(0, 1), fp32;
  * the 1.7B-shaped model adds a 2048->1024 projection (weight N(0, 0.02),
    bias N(0, 0.02)) in front of the code predictor.
"""
from __future__ import annotations

import ctypes
import dataclasses
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SO = os.path.join(_HERE, "_synth.so")
_lock = threading.Lock()
_lib = None

F32 = 0
BF16 = 1


def build(force: bool = False) -> str:
    """Compile gen.c into _synth.so (plain C, OpenMP)."""
    src = os.path.join(_HERE, "gen.c")
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(src):
        tmp = _SO + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", src, "-o", tmp, "-lm"])
        os.replace(tmp, _SO)
    return _SO


def _L():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_SO)
            i64, u64, f32 = ctypes.c_int64, ctypes.c_uint64, ctypes.c_float
            vp = ctypes.c_void_p
            lib.synth_fill_normal_f32.argtypes = [vp, i64, u64, u64, f32]
            lib.synth_fill_normal_bf16.argtypes = [vp, i64, u64, u64, f32]
            lib.synth_round_bf16.argtypes = [vp, vp, i64]
            lib.synth_fill_randint.argtypes = [vp, i64, u64, u64, ctypes.c_int32, ctypes.c_int32]
            lib.synth_fill_u64.argtypes = [vp, i64, u64, u64]
            _lib = lib
    return _lib


def normal(shape, seed: int, stream: int, std: float = 1.0, dtype: int = F32) -> np.ndarray:
    """N(0, std^2) draws; bf16 results are returned as uint16 bit patterns."""
    n = int(np.prod(shape))
    if dtype == BF16:
        out = np.empty(shape, dtype=np.uint16)
        _L().synth_fill_normal_bf16(out.ctypes.data, n, seed, stream, std)
    else:
        out = np.empty(shape, dtype=np.float32)
        _L().synth_fill_normal_f32(out.ctypes.data, n, seed, stream, std)
    return out


def round_bf16(x: np.ndarray) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, dtype=np.uint16)
    _L().synth_round_bf16(x.ctypes.data, out.ctypes.data, x.size)
    return out


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (b.astype(np.uint32) << 16).view(np.float32)


def randint(n: int, seed: int, stream: int, lo: int, hi: int) -> np.ndarray:
    out = np.empty(n, dtype=np.int32)
    _L().synth_fill_randint(out.ctypes.data, n, seed, stream, lo, hi)
    return out


def u64(n: int, seed: int, stream: int) -> np.ndarray:
    out = np.empty(n, dtype=np.uint64)
    _L().synth_fill_u64(out.ctypes.data, n, seed, stream)
    return out


# --------------------------------------------------------------------------
# model shapes and workloads
# --------------------------------------------------------------------------
@dataclasses.dataclass(frozen=True)
class Dims:
    n_layers: int = 28
    hidden: int = 1024
    n_q_heads: int = 16
    n_kv_heads: int = 8
    head_dim: int = 128
    ffn: int = 3072
    codec_vocab: int = 3072
    cp_layers: int = 5
    cp_hidden: int = 1024
    cp_ffn: int = 3072
    cp_vocab: int = 2048
    n_groups: int = 16
    eos_id: int = 2150
    suppress_lo: int = 2048
    suppress_hi: int = 3072
    rms_eps: float = 1e-6
    rope_theta: float = 1e6
    text_vocab: int = 0      # text side (BPE vocabulary; 0 = none)
    text_hidden: int = 0     # text embedding width


DIMS_06B = Dims()
# the text side of the released models: Qwen2 BPE vocabulary, 2048-d embedding
TEXT_VOCAB, TEXT_HIDDEN = 151936, 2048
DIMS_17B = Dims(hidden=2048, ffn=6144)
# Small shapes with the same structure, for fast tests (head_dim stays 128).
DIMS_SMALL = Dims(n_layers=2, hidden=256, ffn=384, codec_vocab=96, cp_layers=2, cp_hidden=256,
                  cp_ffn=320, cp_vocab=64, n_groups=4, eos_id=80, suppress_lo=64, suppress_hi=96)
DIMS_SMALL_PROJ = dataclasses.replace(DIMS_SMALL, hidden=384, ffn=512)
# Small shapes the batch-1 cluster kernel serves (8 clusters x 8 CTAs: widths in
# multiples of 128, FFN in multiples of 512, vocabularies in multiples of 1024).
DIMS_CL = Dims(n_layers=2, hidden=256, ffn=512, codec_vocab=1024, cp_layers=2, cp_hidden=256, cp_ffn=512,
               cp_vocab=1024, n_groups=4, eos_id=1000, suppress_lo=960, suppress_hi=1024)
DIMS_CL_PROJ = dataclasses.replace(DIMS_CL, hidden=512, ffn=1024)


@dataclasses.dataclass
class RowSampling:
    do_sample: int = 0
    temperature: float = 1.0
    top_k: int = 0
    top_p: float = 1.0
    repetition_penalty: float = 1.05
    min_new_tokens: int = 2
    seed: int = 7
    max_frames: int = 4
    force_eos_at_frame: int = -1
    cp_do_sample: int = 0
    cp_temperature: float = 1.0
    cp_top_k: int = 0
    cp_top_p: float = 1.0


@dataclasses.dataclass
class Workload:
    name: str
    dims: Dims
    dtype: int
    weight_seed: int
    batch: int
    prompt_lens: list
    n_text: list
    frames: int
    rows: list            # RowSampling per row
    max_ctx: int
    norm_std: float = 0.0
    input_seed: int = -1  # defaults to weight_seed

    @property
    def iseed(self) -> int:
        return self.weight_seed if self.input_seed < 0 else self.input_seed


def _rows(batch, frames, **kw):
    return [RowSampling(max_frames=frames, **kw) for _ in range(batch)]


def workload(idx: int) -> Workload:
    """The frame-loop workloads (1-based index): the five configurations, then
    the 1.7B shape at batch 32 (6) and batch 256 (7)."""
    if idx == 1:   # tiny oracle check, fp32
        return Workload("0.6B fp32 b1 prompt16 4 frames greedy", DIMS_06B, F32, 0, 1, [16], [0], 4,
                        _rows(1, 4), 20)
    if idx == 2:   # latency path
        return Workload("0.6B bf16 b1 prompt128 100 frames greedy", DIMS_06B, BF16, 1, 1, [128], [64], 100,
                        _rows(1, 100), 228)
    if idx == 3:
        return Workload("1.7B bf16 b1 prompt256 200 frames T0.9 k50", DIMS_17B, BF16, 2, 1, [256], [64], 200,
                        _rows(1, 200, do_sample=1, temperature=0.9, top_k=50, top_p=1.0,
                              cp_do_sample=1, cp_temperature=0.9, cp_top_k=50, cp_top_p=1.0), 456)
    if idx == 4:
        b = 32
        lens = [int(v) for v in randint(b, 3, 0x4C454E, 64, 512)]
        eos = [int(v) for v in randint(b, 3, 0x454F53, 50, 250)]
        rows = _rows(b, 250)
        for r in range(b):
            rows[r].force_eos_at_frame = eos[r]
        return Workload("0.6B bf16 b32 prompt U[64,512] 250 frames greedy forced EOS", DIMS_06B, BF16, 3, b,
                        lens, [64] * b, 250, rows, 768)
    if idx == 5:
        b = 256
        return Workload("0.6B bf16 b256 prompt256 1024 frames T0.9 k50 p0.95", DIMS_06B, BF16, 4, b,
                        [256] * b, [64] * b, 1024,
                        _rows(b, 1024, do_sample=1, temperature=0.9, top_k=50, top_p=0.95,
                              cp_do_sample=1, cp_temperature=0.9, cp_top_k=50, cp_top_p=0.95), 1280)
    # the 1.7B shape at the two batch sizes (variants of the batch-32 and
    # batch-256 workloads above; not among the five configurations)
    if idx == 6:
        b = 32
        lens = [int(v) for v in randint(b, 5, 0x4C454E, 64, 512)]
        eos = [int(v) for v in randint(b, 5, 0x454F53, 50, 250)]
        rows = _rows(b, 250)
        for r in range(b):
            rows[r].force_eos_at_frame = eos[r]
        return Workload("1.7B bf16 b32 prompt U[64,512] 250 frames greedy forced EOS", DIMS_17B, BF16, 5, b,
                        lens, [64] * b, 250, rows, 768)
    if idx == 7:
        b = 256
        return Workload("1.7B bf16 b256 prompt256 1024 frames T0.9 k50 p0.95", DIMS_17B, BF16, 6, b,
                        [256] * b, [64] * b, 1024,
                        _rows(b, 1024, do_sample=1, temperature=0.9, top_k=50, top_p=0.95,
                              cp_do_sample=1, cp_temperature=0.9, cp_top_k=50, cp_top_p=0.95), 1280)
    raise ValueError(idx)


# --------------------------------------------------------------------------
# weights
# --------------------------------------------------------------------------
BLOCK_KEYS = ("attn_norm", "wqkv", "q_norm", "k_norm", "wo", "mlp_norm", "wgu", "wd", "final_norm")


def _stream(kind: int, idx: int = 0) -> int:
    return (kind << 32) | idx


def _block(prefix_kind: int, L: int, H: int, nq: int, nkv: int, hd: int, F: int, dtype: int,
           seed: int, norm_std: float) -> dict:
    def norms(shape, k):
        if norm_std > 0:
            return (1.0 + normal(shape, seed, _stream(prefix_kind + k), norm_std)).astype(np.float32)
        return np.ones(shape, dtype=np.float32)
    qkv = (nq + 2 * nkv) * hd
    return {
        "attn_norm": norms((L, H), 1),
        "wqkv": normal((L, qkv, H), seed, _stream(prefix_kind + 2), 0.02, dtype),
        "q_norm": norms((L, hd), 3),
        "k_norm": norms((L, hd), 4),
        "wo": normal((L, H, nq * hd), seed, _stream(prefix_kind + 5), 0.02, dtype),
        "mlp_norm": norms((L, H), 6),
        "wgu": normal((L, 2 * F, H), seed, _stream(prefix_kind + 7), 0.02, dtype),
        "wd": normal((L, H, F), seed, _stream(prefix_kind + 8), 0.02, dtype),
        "final_norm": norms((H,), 9),
    }


def make_weights(d: Dims, dtype: int, seed: int, norm_std: float = 0.0) -> dict:
    """Random-init weights as host arrays (bf16 as uint16 bit patterns).

    Layout (row-major, output features first):
      talker.*, cp.*  : per-block stacks, see BLOCK_KEYS
          wqkv [L, (nq+2nkv)*hd, H]  rows: q heads, then k heads, then v heads
          wgu  [L, 2F, H]            rows: gate 0..F-1, then up 0..F-1
      codec_emb  [codec_vocab, H]     talker codec embedding
      codec_head [codec_vocab, H]
      cp_emb     [n_groups-1, cp_vocab, H]      predictor tables, talker width
      cp_heads   [n_groups-1, cp_vocab, cp_hidden]
      cp_proj_w  [cp_hidden, H], cp_proj_b [cp_hidden]  (only when H != cp_hidden)
    """
    w = {"talker": _block(0x100, d.n_layers, d.hidden, d.n_q_heads, d.n_kv_heads, d.head_dim, d.ffn,
                          dtype, seed, norm_std),
         "cp": _block(0x200, d.cp_layers, d.cp_hidden, d.n_q_heads, d.n_kv_heads, d.head_dim, d.cp_ffn,
                      dtype, seed, norm_std)}
    w["codec_emb"] = normal((d.codec_vocab, d.hidden), seed, _stream(0x300), 0.02, dtype)
    w["codec_head"] = normal((d.codec_vocab, d.hidden), seed, _stream(0x301), 0.02, dtype)
    w["cp_emb"] = normal((d.n_groups - 1, d.cp_vocab, d.hidden), seed, _stream(0x302), 0.02, dtype)
    w["cp_heads"] = normal((d.n_groups - 1, d.cp_vocab, d.cp_hidden), seed, _stream(0x303), 0.02, dtype)
    if d.hidden != d.cp_hidden:
        w["cp_proj_w"] = normal((d.cp_hidden, d.hidden), seed, _stream(0x304), 0.02, dtype)
        w["cp_proj_b"] = normal((d.cp_hidden,), seed, _stream(0x305), 0.02)
    else:
        w["cp_proj_w"] = None
        w["cp_proj_b"] = None
    return w


def make_text_weights(d: Dims, dtype: int, seed: int) -> dict:
    """Random-init text side: embedding [text_vocab, text_hidden] ~ N(0, 1) (the
    scale of the prompt rows), ResizeMLP layers ~ N(0, 0.02) with biases:
    text_fc1_w [T, T], text_fc1_b [T], text_fc2_w [H, T], text_fc2_b [H]."""
    V, T, H = d.text_vocab, d.text_hidden, d.hidden
    return {"text_emb": normal((V, T), seed, _stream(0x400), 1.0, dtype),
            "text_fc1_w": normal((T, T), seed, _stream(0x401), 0.02, dtype),
            "text_fc1_b": normal((T,), seed, _stream(0x402), 0.02),
            "text_fc2_w": normal((H, T), seed, _stream(0x403), 0.02, dtype),
            "text_fc2_b": normal((H,), seed, _stream(0x404), 0.02)}


def weight_bytes(d: Dims, dtype: int) -> dict:
    """Bytes of each weight group, for roofline accounting."""
    e = 4 if dtype == F32 else 2
    qkv = (d.n_q_heads + 2 * d.n_kv_heads) * d.head_dim

    def layer(H, F):
        mats = qkv * H + H * d.n_q_heads * d.head_dim + 2 * F * H + H * F
        return mats * e + (2 * H + 2 * d.head_dim) * 4
    return {
        "talker_layer": layer(d.hidden, d.ffn),
        "cp_layer": layer(d.cp_hidden, d.cp_ffn),
        "codec_head": d.codec_vocab * d.hidden * e,
        "cp_head": d.cp_vocab * d.cp_hidden * e,
        "cp_proj": (d.cp_hidden * d.hidden * e + d.cp_hidden * 4) if d.hidden != d.cp_hidden else 0,
        "final_norm": d.hidden * 4,
        "cp_final_norm": d.cp_hidden * 4,
    }


# --------------------------------------------------------------------------
# per-workload inputs
# --------------------------------------------------------------------------
def make_inputs(wl: Workload) -> dict:
    """Prompt embeddings [sum(len), H], trailing text [sum(n_text), H], tts_pad [H]."""
    H = wl.dims.hidden
    s = wl.iseed
    lens = list(wl.prompt_lens)
    ntx = list(wl.n_text)
    prompt = normal((sum(lens), H), s, _stream(0x400), 1.0)
    text = normal((max(sum(ntx), 0), H), s, _stream(0x401), 1.0)
    pad = normal((H,), s, _stream(0x402), 1.0)
    return {
        "prompt": prompt,
        "prompt_offsets": np.concatenate([[0], np.cumsum(lens)]).astype(np.int32),
        "text": text,
        "text_offsets": np.concatenate([[0], np.cumsum(ntx)]).astype(np.int32),
        "tts_pad": pad,
    }


def random_logits(n_sets: int, vocab: int, seed: int, scale: float = 2.0, ties: bool = True) -> np.ndarray:
    """Random fp32 logit sets for sampler tests; optionally with exact ties."""
    raw = u64(n_sets * vocab, seed, 0x500).reshape(n_sets, vocab)
    u = ((raw >> np.uint64(11)).astype(np.float64) + 0.5) / float(1 << 53)
    x = (scale * np.log(u / (1 - u))).astype(np.float32)
    if ties:
        # every fourth set: quantise so that many values tie exactly
        x[::4] = (np.round(x[::4] * 4) / 4).astype(np.float32)
    return x
