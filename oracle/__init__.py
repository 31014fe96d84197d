"""Oracle for the Qwen3-TTS frame loop: TEST INFRASTRUCTURE.

A plain fp64 CPU implementation (oracle.cpp) of the talker step, the code
predictor and the logits processors / sampler.  Only tests/, the smoke check
and the benchmark's CPU-baseline leg may import this package; the product
path never does.  It shares no code with the CUDA library.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SO = os.path.join(_HERE, "_oracle.so")
_lock = threading.Lock()
_lib = None

ERR_OK, ERR_ARG, ERR_NAN = 0, 1, 5
REASON_RUNNING, REASON_EOS, REASON_LENGTH = 0, 1, 2


def build(force: bool = False) -> str:
    srcs = [os.path.join(_HERE, f) for f in ("oracle.cpp", "codec.cpp")]
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < max(os.path.getmtime(f) for f in srcs):
        tmp = _SO + f".tmp{os.getpid()}"
        subprocess.check_call(["g++", "-std=c++17", "-O2", "-fopenmp", "-ffp-contract=off", "-fPIC", "-shared",
                               *srcs, "-o", tmp])
        os.replace(tmp, _SO)
    return _SO


class Config(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in ("n_layers", "hidden", "n_q_heads", "n_kv_heads", "head_dim", "ffn",
                                            "codec_vocab", "cp_layers", "cp_hidden", "cp_ffn", "cp_vocab",
                                            "n_groups", "eos_id", "suppress_lo", "suppress_hi")] + \
              [("rms_eps", ctypes.c_float), ("rope_theta", ctypes.c_float), ("dtype", ctypes.c_int)]


class Block(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in ("attn_norm", "wqkv", "q_norm", "k_norm", "wo", "mlp_norm", "wgu",
                                               "wd", "final_norm")]


class Weights(ctypes.Structure):
    _fields_ = [("talker", Block), ("codec_emb", ctypes.c_void_p), ("codec_head", ctypes.c_void_p),
                ("cp", Block), ("cp_emb", ctypes.c_void_p), ("cp_heads", ctypes.c_void_p),
                ("cp_proj_w", ctypes.c_void_p), ("cp_proj_b", ctypes.c_void_p)]


class Sampling(ctypes.Structure):
    _fields_ = [("do_sample", ctypes.c_int), ("temperature", ctypes.c_float), ("top_k", ctypes.c_int),
                ("top_p", ctypes.c_float), ("repetition_penalty", ctypes.c_float), ("min_new_tokens", ctypes.c_int),
                ("seed", ctypes.c_uint64), ("max_frames", ctypes.c_int), ("force_eos_at_frame", ctypes.c_int),
                ("cp_do_sample", ctypes.c_int), ("cp_temperature", ctypes.c_float), ("cp_top_k", ctypes.c_int),
                ("cp_top_p", ctypes.c_float)]


def _L():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_SO)
            vp, i32, f32, f64, u32, u64 = (ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_double,
                                           ctypes.c_uint32, ctypes.c_uint64)
            lib.oracle_create.restype = vp
            lib.oracle_create.argtypes = [ctypes.POINTER(Config), ctypes.POINTER(Weights), i32, i32, i32, i32]
            lib.oracle_destroy.argtypes = [vp]
            lib.oracle_set_threads.restype = i32
            lib.oracle_set_threads.argtypes = [i32]
            lib.oracle_text_embed.restype = i32
            lib.oracle_text_embed.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, vp, i32, vp]
            lib.oracle_prefill.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp]
            lib.oracle_step.argtypes = [vp, i32, vp]
            lib.oracle_get.argtypes = [vp, i32, vp]
            lib.oracle_sample.argtypes = [vp, i32, ctypes.POINTER(Sampling), i32, vp, i32, i32, i32, i32, u32, u32,
                                          u32, vp, vp, vp]
            lib.oracle_philox.argtypes = [vp, vp, vp]
            lib.oracle_spec_expf.restype = f32
            lib.oracle_spec_expf.argtypes = [f32]
            lib.oracle_spec_logf.restype = f32
            lib.oracle_spec_logf.argtypes = [f32]
            lib.oracle_noise_uniform.restype = f32
            lib.oracle_noise_uniform.argtypes = [u64, u32, u32, u32, u32]
            lib.oracle_bf16_round.restype = f64
            lib.oracle_bf16_round.argtypes = [f64]
            lib.oracle_rmsnorm.argtypes = [vp, vp, i32, f64, vp]
            lib.oracle_rope.argtypes = [vp, i32, i32, f32]
            lib.oracle_mrope.argtypes = [vp, i32, vp, vp, i32, f32]
            lib.oracle_attend.argtypes = [vp, vp, vp, i32, i32, i32, i32, i32, vp]
            lib.oracle_codec_decode.restype = i32
            lib.oracle_codec_decode.argtypes = [vp, vp, vp, i32, vp, vp]
            lib.oracle_codec_attention.argtypes = [vp, vp, vp, i32, i32, i32, i32, vp]
            lib.oracle_codec_conv1d.argtypes = [vp, i32, i32, i32, i32, i32, vp, vp, vp]
            lib.oracle_codec_conv_transpose.argtypes = [vp, i32, i32, i32, i32, i32, vp, vp, vp]
            lib.oracle_codec_snake.argtypes = [vp, i32, i32, vp, vp]
            _lib = lib
    return _lib


def lib():
    return _L()


def text_embed(w: dict, dtype: int, ids) -> np.ndarray:
    """Talker-width rows of text ids through the embedding and ResizeMLP (fp64).
    w: text_emb [V][T], text_fc1_w [T][T], text_fc1_b [T] f32, text_fc2_w [H][T],
    text_fc2_b [H] f32 (bf16 matrices as uint16 bit patterns)."""
    emb = np.ascontiguousarray(w["text_emb"])
    w1 = np.ascontiguousarray(w["text_fc1_w"])
    w2 = np.ascontiguousarray(w["text_fc2_w"])
    b1 = np.ascontiguousarray(w["text_fc1_b"], dtype=np.float32)
    b2 = np.ascontiguousarray(w["text_fc2_b"], dtype=np.float32)
    ids = np.ascontiguousarray(ids, dtype=np.int32)
    V, T = emb.shape
    H = w2.shape[0]
    out = np.zeros((len(ids), H), np.float64)
    err = _L().oracle_text_embed(emb.ctypes.data, w1.ctypes.data, b1.ctypes.data, w2.ctypes.data, b2.ctypes.data,
                                 dtype, V, T, H, ids.ctypes.data, len(ids), out.ctypes.data)
    if err:
        raise ValueError("text id out of range")
    return out


def set_threads(n: int) -> int:
    """Worker threads of the oracle's parallel loops (timing only); returns the previous count."""
    return int(_L().oracle_set_threads(int(n)))


def make_config(dims, dtype: int) -> Config:
    c = Config()
    for f, _ in Config._fields_:
        if f == "dtype":
            c.dtype = dtype
        else:
            setattr(c, f, getattr(dims, f))
    return c


def _ptr(a):
    return None if a is None else a.ctypes.data


def make_weights(w: dict) -> Weights:
    ws = Weights()
    for blk in ("talker", "cp"):
        b = getattr(ws, blk)
        for k, _ in Block._fields_:
            setattr(b, k, _ptr(w[blk][k]))
    for k in ("codec_emb", "codec_head", "cp_emb", "cp_heads", "cp_proj_w", "cp_proj_b"):
        setattr(ws, k, _ptr(w[k]))
    return ws


def make_sampling(r) -> Sampling:
    s = Sampling()
    for f, _ in Sampling._fields_:
        setattr(s, f, getattr(r, f))
    return s


class Oracle:
    """Handle over one oracle instance (rows, weights and outputs held alive here)."""

    def __init__(self, dims, dtype, weights: dict, batch: int, max_ctx: int, max_frames: int, capture=True):
        self._w = weights
        self.dims = dims
        self.batch, self.T, self.capture = batch, max_frames, capture
        self._cfg = make_config(dims, dtype)
        self._ws = make_weights(weights)
        self.h = _L().oracle_create(ctypes.byref(self._cfg), ctypes.byref(self._ws), batch, max_ctx, max_frames,
                                    int(capture))
        if not self.h:
            raise ValueError("oracle_create rejected the configuration")

    def __del__(self):
        if getattr(self, "h", None):
            _L().oracle_destroy(self.h)
            self.h = None

    def prefill(self, prompt, prompt_off, text, text_off, pad, rows, row_ids=None, teacher=None):
        B = self.batch
        row_ids = np.arange(B, dtype=np.int32) if row_ids is None else np.asarray(row_ids, dtype=np.int32)
        sp = (Sampling * B)(*[make_sampling(r) for r in rows])
        prompt = np.ascontiguousarray(prompt, dtype=np.float32)
        text = np.ascontiguousarray(text, dtype=np.float32)
        pad = np.ascontiguousarray(pad, dtype=np.float32)
        po = np.ascontiguousarray(prompt_off, dtype=np.int32)
        to = np.ascontiguousarray(text_off, dtype=np.int32)
        self._teacher = None if teacher is None else np.ascontiguousarray(teacher, dtype=np.int32)
        err = _L().oracle_prefill(self.h, prompt.ctypes.data, po.ctypes.data, text.ctypes.data if text.size else None,
                                  to.ctypes.data, pad.ctypes.data, ctypes.cast(sp, ctypes.c_void_p),
                                  row_ids.ctypes.data, _ptr(self._teacher))
        if err:
            raise RuntimeError(f"oracle_prefill error {err}")

    def step(self, n: int):
        err = _L().oracle_step(self.h, n, _ptr(self._teacher))
        if err:
            raise RuntimeError(f"oracle_step error {err}")

    def get(self, what: str) -> np.ndarray:
        B, T, d = self.batch, self.T, self.dims
        G1 = d.n_groups - 1
        spec = {
            "own_sel": (0, (B, T + 1), np.int32), "sel_margin": (1, (B, T + 1), np.float64),
            "codes": (2, (B, T, d.n_groups), np.int32), "own_cp": (3, (B, T, G1), np.int32),
            "cp_margin": (4, (B, T, G1), np.float64), "talker_logits": (5, (B, T + 1, d.codec_vocab), np.float32),
            "cp_logits": (6, (B, T, G1, d.cp_vocab), np.float32), "frames": (7, (B,), np.int32),
            "reason": (8, (B,), np.int32), "selections": (9, (B,), np.int64), "predictor_runs": (10, (B,), np.int64),
        }[what]
        out = np.empty(spec[1], dtype=spec[2])
        err = _L().oracle_get(self.h, spec[0], out.ctypes.data)
        if err:
            raise RuntimeError(f"oracle_get({what}) error {err}")
        return out


def run(wl, weights, inputs, rows=None, teacher=None, capture=True, frames=None, chunks=None):
    """Run a workload (optionally a subset of its rows) through the oracle.

    rows: batch indices to run (default all); their noise row ids stay the
    batch indices.  teacher: [len(rows), T+1, G] codes to force (see
    ``teacher_from_codes``).  chunks: list of step counts (default one call).
    """
    rows = list(range(wl.batch)) if rows is None else list(rows)
    T = wl.frames if frames is None else frames
    lens = [wl.prompt_lens[r] for r in rows]
    ntx = [wl.n_text[r] for r in rows]
    H = wl.dims.hidden
    po_all, to_all = inputs["prompt_offsets"], inputs["text_offsets"]
    prompt = np.concatenate([inputs["prompt"][po_all[r]:po_all[r + 1]] for r in rows]) if rows else None
    text_parts = [inputs["text"][to_all[r]:to_all[r + 1]] for r in rows]
    text = np.concatenate(text_parts) if sum(ntx) else np.zeros((0, H), np.float32)
    po = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    to = np.concatenate([[0], np.cumsum(ntx)]).astype(np.int32)
    o = Oracle(wl.dims, wl.dtype, weights, len(rows), wl.max_ctx, T, capture)
    o.prefill(prompt, po, text, to, inputs["tts_pad"], [wl.rows[r] for r in rows], rows, teacher)
    for n in (chunks or [T]):
        o.step(n)
    return o


def teacher_from_codes(codes, frames, reasons, eos_id, T):
    """Teacher array [B, T+1, G] from a run's outputs: selection k -> [k, 0],
    predictor codes of frame f -> [f, 1..]; the selection that ended a row on
    EOS is EOS; a row that ended on length gets -1 (any non-EOS id)."""
    codes = np.asarray(codes)
    B, _, G = codes.shape
    t = np.full((B, T + 1, G), -1, dtype=np.int32)
    for b in range(B):
        f = int(frames[b])
        t[b, :f] = codes[b, :f]
        if int(reasons[b]) == REASON_EOS:
            t[b, f, 0] = eos_id
    return t


def sample(logits, sp, talker, seen=None, sel_index=0, eos=2150, sup_lo=2048, sup_hi=3072, row=0, frame=0, step=0):
    """One selection through the oracle's processors + draw -> (err, id, margin, processed logits)."""
    logits = np.ascontiguousarray(logits, dtype=np.float32)
    V = logits.shape[0]
    s = make_sampling(sp)
    seen_a = None if seen is None else np.ascontiguousarray(seen, dtype=np.uint8)
    out_id = ctypes.c_int(-1)
    margin = ctypes.c_double(0.0)
    proc = np.empty(V, np.float32)
    err = _L().oracle_sample(logits.ctypes.data, V, ctypes.byref(s), int(talker), _ptr(seen_a), sel_index, eos,
                             sup_lo, sup_hi, row, frame, step, ctypes.byref(out_id), ctypes.byref(margin),
                             proc.ctypes.data)
    return err, out_id.value, margin.value, proc
