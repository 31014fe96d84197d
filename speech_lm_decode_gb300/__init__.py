"""GB300 (sm_103a) Qwen3-TTS 12 Hz frame loop: Python binding of libq3tts.so.

Argument marshalling only: every step of the frame loop runs in the library's
CUDA kernels.  PyTorch provides device memory and the stream.  The library
must have been built (``speech_lm_decode_gb300.build.build()``); importing the
binding without it raises instead of falling back to anything else.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libq3tts.so")

Q3_OK, Q3_ERR_ARG, Q3_ERR_CUDA, Q3_ERR_CAPACITY, Q3_ERR_STATE, Q3_ERR_NAN, Q3_ERR_TIMEOUT, Q3_ERR_BOUNDS = range(8)
Q3_F32, Q3_BF16 = 0, 1
Q3_RUNNING, Q3_FINISHED_EOS, Q3_FINISHED_LENGTH, Q3_FINISHED_ERROR = 0, 1, 2, 3
Q3_PATH_AUTO, Q3_PATH_GRAPH, Q3_PATH_FRAME, Q3_PATH_CLUSTER = 0, 1, 2, 3
PATH_NAMES = {Q3_PATH_GRAPH: "graph", Q3_PATH_FRAME: "frame", Q3_PATH_CLUSTER: "cluster"}

EXPORTS = ("q3tts_workspace_bytes", "q3tts_create", "q3tts_prefill", "q3tts_step_frames", "q3tts_set_capture",
           "q3tts_sample_logits", "q3tts_sample_logits_noalloc", "q3tts_step_kernel_count", "q3tts_step_path",
           "q3tts_text_embed", "q3tts_last_error", "q3tts_destroy")


class Q3Error(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"q3tts error {code}: {msg}")
        self.code = code


class Config(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in ("n_layers", "hidden", "n_q_heads", "n_kv_heads", "head_dim", "ffn",
                                            "codec_vocab", "cp_layers", "cp_hidden", "cp_ffn", "cp_vocab",
                                            "n_groups", "eos_id", "suppress_lo", "suppress_hi")] + \
              [("rms_eps", ctypes.c_float), ("rope_theta", ctypes.c_float)] + \
              [(n, ctypes.c_int) for n in ("dtype", "max_batch", "max_ctx", "max_text", "step_path", "tc_min_tokens",
                                           "debug_sync", "wait_limit_us", "inject_timeout", "text_vocab",
                                           "text_hidden", "separate_projections")]

# execution fields of the config (everything else comes from the model dims)
EXEC_FIELDS = ("step_path", "tc_min_tokens", "debug_sync", "wait_limit_us", "inject_timeout",
               "separate_projections")


class BlockWeights(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in ("attn_norm", "wqkv", "q_norm", "k_norm", "wo", "mlp_norm", "wgu",
                                               "wd", "final_norm")]


class Weights(ctypes.Structure):
    _fields_ = [("talker", BlockWeights), ("codec_emb", ctypes.c_void_p), ("codec_head", ctypes.c_void_p),
                ("cp", BlockWeights), ("cp_emb", ctypes.c_void_p), ("cp_heads", ctypes.c_void_p),
                ("cp_proj_w", ctypes.c_void_p), ("cp_proj_b", ctypes.c_void_p)] + \
              [(n, ctypes.c_void_p) for n in ("text_emb", "text_fc1_w", "text_fc1_b", "text_fc2_w", "text_fc2_b")]

TEXT_KEYS = ("text_emb", "text_fc1_w", "text_fc1_b", "text_fc2_w", "text_fc2_b")


class Sampling(ctypes.Structure):
    _fields_ = [("do_sample", ctypes.c_int), ("temperature", ctypes.c_float), ("top_k", ctypes.c_int),
                ("top_p", ctypes.c_float), ("repetition_penalty", ctypes.c_float), ("min_new_tokens", ctypes.c_int),
                ("seed", ctypes.c_uint64), ("max_frames", ctypes.c_int), ("force_eos_at_frame", ctypes.c_int),
                ("cp_do_sample", ctypes.c_int), ("cp_temperature", ctypes.c_float), ("cp_top_k", ctypes.c_int),
                ("cp_top_p", ctypes.c_float)]


_lib = None


def lib():
    """The loaded libq3tts.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with speech_lm_decode_gb300.build.build()")
        L = ctypes.CDLL(LIB_PATH)
        vp, i32 = ctypes.c_void_p, ctypes.c_int
        L.q3tts_workspace_bytes.restype = ctypes.c_size_t
        L.q3tts_workspace_bytes.argtypes = [ctypes.POINTER(Config)]
        L.q3tts_create.argtypes = [ctypes.POINTER(Config), ctypes.POINTER(Weights), vp, ctypes.c_size_t, vp,
                                   ctypes.POINTER(vp)]
        L.q3tts_prefill.argtypes = [vp, i32, vp, vp, vp, vp, vp, vp, vp]
        L.q3tts_step_frames.argtypes = [vp, i32, vp, vp, vp]
        L.q3tts_set_capture.argtypes = [vp, i32, vp, vp, vp, i32]
        L.q3tts_sample_logits.argtypes = [vp, i32, vp, i32, vp, vp, vp, i32, vp, vp]
        L.q3tts_step_kernel_count.argtypes = [vp, ctypes.POINTER(ctypes.c_int)]
        L.q3tts_step_path.argtypes = [vp, i32, ctypes.POINTER(ctypes.c_int)]
        L.q3tts_text_embed.argtypes = [vp, i32, vp, vp]
        L.q3tts_sample_logits_noalloc.argtypes = [i32, i32, vp, i32, vp, vp, vp, i32, vp, i32, i32, i32, vp, vp]
        L.q3tts_last_error.restype = ctypes.c_char_p
        L.q3tts_last_error.argtypes = [vp]
        L.q3tts_destroy.argtypes = [vp]
        _lib = L
    return _lib


def make_config(dims, dtype: int, max_batch: int, max_ctx: int, max_text: int, **exec_opts) -> Config:
    """exec_opts: step_path, tc_min_tokens, debug_sync, wait_limit_us, inject_timeout,
    separate_projections (default 0)."""
    unknown = set(exec_opts) - set(EXEC_FIELDS)
    if unknown:
        raise ValueError(f"unknown config options {sorted(unknown)}")
    c = Config()
    for f, _ in Config._fields_:
        if f in EXEC_FIELDS:
            setattr(c, f, int(exec_opts.get(f, 0)))
        elif f == "dtype":
            c.dtype = dtype
        elif f == "max_batch":
            c.max_batch = max_batch
        elif f == "max_ctx":
            c.max_ctx = max_ctx
        elif f == "max_text":
            c.max_text = max_text
        else:
            setattr(c, f, getattr(dims, f, 0))
    return c


def make_sampling(r) -> Sampling:
    s = Sampling()
    for f, _ in Sampling._fields_:
        setattr(s, f, getattr(r, f))
    return s


def to_device_weights(w: dict, device="cuda") -> dict:
    """Host weight arrays (bf16 as uint16 bit patterns) -> device tensors of the same layout."""
    import torch

    def dev(a):
        if a is None:
            return None
        t = torch.from_numpy(np.ascontiguousarray(a))
        if a.dtype == np.uint16:
            t = t.view(torch.bfloat16)
        return t.to(device)
    out = {}
    for k, v in w.items():
        out[k] = {kk: dev(vv) for kk, vv in v.items()} if isinstance(v, dict) else dev(v)
    return out


def _ptr(t):
    if t is None:
        return None
    if hasattr(t, "data_ptr"):
        return t.data_ptr()
    return t.ctypes.data


def make_weights(dw: dict) -> Weights:
    ws = Weights()
    for blk in ("talker", "cp"):
        b = getattr(ws, blk)
        for k, _ in BlockWeights._fields_:
            setattr(b, k, _ptr(dw[blk][k]))
    for k in ("codec_emb", "codec_head", "cp_emb", "cp_heads", "cp_proj_w", "cp_proj_b") + TEXT_KEYS:
        setattr(ws, k, _ptr(dw.get(k)))
    return ws


class Q3TTS:
    """One handle: model weights (borrowed device tensors), a workspace and a stream."""

    def __init__(self, dims, dtype: int, device_weights: dict, max_batch: int, max_ctx: int, max_text: int,
                 stream=None, **exec_opts):
        import torch
        self._dw = device_weights
        self.dims, self.dtype = dims, dtype
        self.cfg = make_config(dims, dtype, max_batch, max_ctx, max_text, **exec_opts)
        nbytes = lib().q3tts_workspace_bytes(ctypes.byref(self.cfg))
        if nbytes == 0:
            raise Q3Error(Q3_ERR_ARG, "invalid configuration")
        self.workspace = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
        self.stream = stream if stream is not None else torch.cuda.current_stream()
        self._w = make_weights(device_weights)
        h = ctypes.c_void_p()
        rc = lib().q3tts_create(ctypes.byref(self.cfg), ctypes.byref(self._w), self.workspace.data_ptr(), nbytes,
                                self.stream.cuda_stream, ctypes.byref(h))
        if rc:
            raise Q3Error(rc, "q3tts_create failed")
        self.h = h.value
        self.batch = 0

    def _check(self, rc):
        if rc:
            raise Q3Error(rc, lib().q3tts_last_error(self.h).decode())

    def close(self):
        if getattr(self, "h", None):
            lib().q3tts_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def prefill(self, prompt, prompt_offsets, text, text_offsets, tts_pad, rows, check=True):
        """prompt/text/tts_pad: fp32 numpy arrays or torch tensors (host or cuda)."""
        B = len(rows)
        po = np.ascontiguousarray(prompt_offsets, dtype=np.int32)
        to = np.ascontiguousarray(text_offsets, dtype=np.int32)
        sp = (Sampling * B)(*[make_sampling(r) for r in rows])
        keep = [prompt, text, tts_pad]
        code0 = np.full(B, -1, np.int32)
        rc = lib().q3tts_prefill(self.h, B, _ptr(prompt), po.ctypes.data,
                                 _ptr(text) if text is not None and len(text) else None, to.ctypes.data,
                                 _ptr(tts_pad), ctypes.cast(sp, ctypes.c_void_p), code0.ctypes.data)
        del keep
        if check:
            self._check(rc)
        self.batch = B
        return code0 if check else (rc, code0)

    def step_frames(self, n: int, codes_out=None, check=True):
        """Run n talker steps.  codes_out: None (host numpy returned), or a
        [B, n, G] int32 numpy array / torch tensor to fill."""
        B, G = self.batch, self.dims.n_groups
        out = np.empty((B, n, G), np.int32) if codes_out is None else codes_out
        frames = np.zeros(B, np.int32)
        reasons = np.zeros(B, np.int32)
        rc = lib().q3tts_step_frames(self.h, n, _ptr(out), frames.ctypes.data, reasons.ctypes.data)
        if check:
            self._check(rc)
            return out, frames, reasons
        return rc, out, frames, reasons

    def text_embed(self, ids, out=None, check=True):
        """Talker-width rows of text token ids (gather + ResizeMLP on the GPU).
        ids: int32 numpy array or torch tensor (host or cuda); out: None (host
        numpy returned) or an [n, hidden] float32 array / tensor to fill."""
        n = int(len(ids))
        if isinstance(ids, np.ndarray) or not hasattr(ids, "data_ptr"):
            ids = np.ascontiguousarray(ids, dtype=np.int32)
        rows = np.empty((n, self.dims.hidden), np.float32) if out is None else out
        rc = lib().q3tts_text_embed(self.h, n, _ptr(ids) if n else None, _ptr(rows) if n else None)
        if check:
            self._check(rc)
            return rows
        return rc, rows

    def step_path(self, batch: int) -> int:
        """Q3_PATH_CLUSTER / Q3_PATH_FRAME / Q3_PATH_GRAPH: what runs a step of `batch` rows."""
        p = ctypes.c_int(0)
        self._check(lib().q3tts_step_path(self.h, batch, ctypes.byref(p)))
        return p.value

    def step_kernel_count(self) -> int:
        n = ctypes.c_int(0)
        self._check(lib().q3tts_step_kernel_count(self.h, ctypes.byref(n)))
        return n.value

    def set_capture(self, rows, talker_logits=None, cp_logits=None, max_frames=0):
        r = np.ascontiguousarray(rows, dtype=np.int32)
        self._cap = (r, talker_logits, cp_logits)
        self._check(lib().q3tts_set_capture(self.h, len(r), r.ctypes.data if len(r) else None, _ptr(talker_logits),
                                            _ptr(cp_logits), max_frames))

    def sample_logits(self, logits, talker: bool, params, sel_index, step: int, noise_row, seen=None, check=True):
        """Processors + draw on [n, V] fp32 logits (numpy or torch, host or cuda) -> ids [n]."""
        n = len(params)
        sp = (Sampling * n)(*[make_sampling(r) for r in params])
        sel = np.ascontiguousarray(sel_index, dtype=np.int32)
        nr = np.ascontiguousarray(noise_row, dtype=np.int32)
        if isinstance(logits, np.ndarray):
            logits = np.ascontiguousarray(logits, dtype=np.float32)
        if isinstance(seen, np.ndarray):
            seen = np.ascontiguousarray(seen, dtype=np.uint8)
        ids = np.full(n, -1, np.int32)
        rc = lib().q3tts_sample_logits(self.h, n, _ptr(logits), int(talker), ctypes.cast(sp, ctypes.c_void_p),
                                       _ptr(seen), sel.ctypes.data, step, nr.ctypes.data, ids.ctypes.data)
        if check:
            self._check(rc)
            return ids
        return rc, ids


def sample_logits_noalloc(logits, talker: bool, params, sel_index, step: int, noise_row, eos_id: int,
                          suppress_lo: int, suppress_hi: int, seen=None, stream=None, check=True):
    """Processors + draw without a handle or any device allocation.

    For callers that cannot allocate device memory: logits ([n, V] fp32) and
    seen ([n, V] uint8, optional) must already be CUDA tensors.  Returns the
    ids (host numpy).  Calls that overlap on the GPU race (one shared staging
    area per device)."""
    import torch
    # the library reads n * V * 4 bytes at logits and n * V at seen on the GPU,
    # and n entries of each host array: check all of it before passing pointers
    if not (isinstance(logits, torch.Tensor) and logits.is_cuda and logits.dtype == torch.float32 and
            logits.dim() == 2 and logits.is_contiguous()):
        raise ValueError("logits must be a contiguous 2-D float32 CUDA tensor")
    n, V = int(logits.shape[0]), int(logits.shape[1])
    if seen is not None and not (isinstance(seen, torch.Tensor) and seen.is_cuda and seen.dtype == torch.uint8 and
                                 seen.is_contiguous() and tuple(seen.shape) == (n, V)):
        raise ValueError("seen must be None or a contiguous [n, V] uint8 CUDA tensor")
    sel = np.ascontiguousarray(sel_index, dtype=np.int32)
    nr = np.ascontiguousarray(noise_row, dtype=np.int32)
    if len(params) != n or sel.shape != (n,) or nr.shape != (n,):
        raise ValueError("params, sel_index and noise_row must have one entry per logit set")
    sp = (Sampling * max(n, 1))(*[make_sampling(r) for r in params])
    ids = np.full(max(n, 1), -1, np.int32)
    st = None if stream is None else stream.cuda_stream
    rc = lib().q3tts_sample_logits_noalloc(n, V, _ptr(logits), int(talker), ctypes.cast(sp, ctypes.c_void_p),
                                           _ptr(seen), sel.ctypes.data, step, nr.ctypes.data, eos_id, suppress_lo,
                                           suppress_hi, ids.ctypes.data, st)
    if check and rc:
        raise Q3Error(rc, "q3tts_sample_logits_noalloc failed")
    return ids[:n] if check else (rc, ids[:n])


# ---------------------------------------------------------------- codec decoder (q3codec.h)
CODEC_EXPORTS = ("q3codec_workspace_bytes", "q3codec_create", "q3codec_samples_per_frame", "q3codec_decode_window",
                 "q3codec_decode", "q3codec_stream_reset", "q3codec_stream_push", "q3codec_window_kernel_count",
                 "q3codec_last_error", "q3codec_destroy")
CODEC_MAX_BLOCKS = 4


class CodecConfig(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in ("n_codebooks", "codebook_size", "codebook_dim", "hidden", "n_layers",
                                            "n_heads", "head_dim", "ffn", "window")] + \
              [(n, ctypes.c_float) for n in ("rope_theta", "rms_eps", "ln_eps")] + \
              [(n, ctypes.c_int) for n in ("n_up", "up_ffn", "dac_channels", "n_blocks")] + \
              [("strides", ctypes.c_int * CODEC_MAX_BLOCKS)] + \
              [(n, ctypes.c_int) for n in ("dtype", "max_frames", "tc_min_tokens")]


CODEC_KEYS = ("codebooks", "proj_sem", "proj_ac", "attn_norm", "wqkv", "wo", "ls_attn", "mlp_norm", "wgu", "wd",
              "ls_mlp", "final_norm", "up_w", "up_b", "dw_w", "dw_b", "ln_w", "ln_b", "fc1_w", "fc1_b", "fc2_w",
              "fc2_b", "gamma", "in_w", "in_b")
CODEC_BLOCK_KEYS = ("snake_a", "snake_b", "tconv_w", "tconv_b")
CODEC_UNIT_KEYS = ("a1", "b1", "w1", "c1", "a2", "b2", "w2", "c2")


class CodecWeights(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in CODEC_KEYS] + \
              [("blk", (ctypes.c_void_p * 4) * CODEC_MAX_BLOCKS),
               ("unit", ((ctypes.c_void_p * 8) * 3) * CODEC_MAX_BLOCKS)] + \
              [(n, ctypes.c_void_p) for n in ("out_a", "out_b", "out_w", "out_bias")]


def _codec_lib():
    L = lib()
    if not getattr(L, "_codec_ready", False):
        vp, i32 = ctypes.c_void_p, ctypes.c_int
        L.q3codec_workspace_bytes.restype = ctypes.c_size_t
        L.q3codec_workspace_bytes.argtypes = [ctypes.POINTER(CodecConfig)]
        L.q3codec_create.argtypes = [ctypes.POINTER(CodecConfig), ctypes.POINTER(CodecWeights), vp, ctypes.c_size_t,
                                     vp, ctypes.POINTER(vp)]
        L.q3codec_samples_per_frame.argtypes = [vp]
        L.q3codec_decode_window.argtypes = [vp, vp, i32, i32, vp]
        L.q3codec_decode.argtypes = [vp, vp, i32, vp]
        L.q3codec_stream_reset.argtypes = [vp]
        L.q3codec_stream_push.argtypes = [vp, vp, i32, i32, vp, ctypes.c_long, ctypes.POINTER(ctypes.c_long)]
        L.q3codec_window_kernel_count.argtypes = [vp]
        L.q3codec_last_error.restype = ctypes.c_char_p
        L.q3codec_last_error.argtypes = [vp]
        L.q3codec_destroy.argtypes = [vp]
        L._codec_ready = True
    return L


def make_codec_config(dims, dtype: int, max_frames: int, tc_min_tokens: int = 0) -> CodecConfig:
    c = CodecConfig()
    for f, _ in CodecConfig._fields_:
        if f == "strides":
            for i, s in enumerate(dims.strides):
                c.strides[i] = s
        elif f == "n_blocks":
            c.n_blocks = len(dims.strides)
        elif f == "dtype":
            c.dtype = dtype
        elif f == "max_frames":
            c.max_frames = max_frames
        elif f == "tc_min_tokens":
            c.tc_min_tokens = tc_min_tokens
        else:
            setattr(c, f, getattr(dims, f))
    return c


def codec_to_device(w: dict, device="cuda") -> dict:
    """Host decoder weights (synth layout) -> device tensors of the same layout."""
    import torch

    def dev(a):
        t = torch.from_numpy(np.ascontiguousarray(a))
        if a.dtype == np.uint16:
            t = t.view(torch.bfloat16)
        return t.to(device)
    out = {k: dev(v) for k, v in w.items() if k != "blocks"}
    out["blocks"] = [{k: ([{kk: dev(vv) for kk, vv in u.items()} for u in v] if k == "units" else dev(v))
                      for k, v in b.items()} for b in w["blocks"]]
    return out


class Q3Codec:
    """Codec decoder handle: borrowed device weights, a workspace and a stream."""

    def __init__(self, dims, dtype: int, device_weights: dict, max_frames: int = 325, stream=None,
                 tc_min_tokens: int = 0):
        import torch
        if len(dims.strides) > CODEC_MAX_BLOCKS:
            raise ValueError("at most 4 vocoder blocks")
        self._dw = device_weights
        self.dims, self.dtype = dims, dtype
        self.cfg = make_codec_config(dims, dtype, max_frames, tc_min_tokens)
        L = _codec_lib()
        nbytes = L.q3codec_workspace_bytes(ctypes.byref(self.cfg))
        if nbytes == 0:
            raise Q3Error(Q3_ERR_ARG, "invalid codec configuration")
        self.workspace = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
        self.stream = stream if stream is not None else torch.cuda.current_stream()
        w = CodecWeights()
        for k in CODEC_KEYS + ("out_a", "out_b", "out_w", "out_bias"):
            setattr(w, k, _ptr(device_weights[k]))
        for b, blk in enumerate(device_weights["blocks"]):
            for i, k in enumerate(CODEC_BLOCK_KEYS):
                w.blk[b][i] = _ptr(blk[k])
            for u, unit in enumerate(blk["units"]):
                for i, k in enumerate(CODEC_UNIT_KEYS):
                    w.unit[b][u][i] = _ptr(unit[k])
        self._w = w
        h = ctypes.c_void_p()
        rc = L.q3codec_create(ctypes.byref(self.cfg), ctypes.byref(w), self.workspace.data_ptr(), nbytes,
                              self.stream.cuda_stream, ctypes.byref(h))
        if rc:
            raise Q3Error(rc, "q3codec_create failed")
        self.h = h.value
        self.spf = L.q3codec_samples_per_frame(self.h)

    def _check(self, rc):
        if rc:
            raise Q3Error(rc, _codec_lib().q3codec_last_error(self.h).decode())

    def close(self):
        if getattr(self, "h", None):
            _codec_lib().q3codec_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def _codes(self, codes):
        if hasattr(codes, "data_ptr"):
            return codes
        return np.ascontiguousarray(codes, dtype=np.int32)

    def decode_window(self, codes, keep_from: int = 0, out=None, check=True):
        """codes [T, n_codebooks] int32 (numpy or torch, host or cuda) -> samples of
        frames keep_from..T-1 (numpy float32 unless `out` is given)."""
        codes = self._codes(codes)
        T = int(codes.shape[0])
        wav = np.empty((T - keep_from) * self.spf, np.float32) if out is None else out
        rc = _codec_lib().q3codec_decode_window(self.h, _ptr(codes), T, keep_from, _ptr(wav))
        if check:
            self._check(rc)
            return wav
        return rc, wav

    def decode(self, codes, out=None, check=True):
        """A whole request on the 300/25 chunk grid."""
        codes = self._codes(codes)
        T = int(codes.shape[0])
        wav = np.empty(T * self.spf, np.float32) if out is None else out
        rc = _codec_lib().q3codec_decode(self.h, _ptr(codes), T, _ptr(wav))
        if check:
            self._check(rc)
            return wav
        return rc, wav

    def stream_reset(self):
        self._check(_codec_lib().q3codec_stream_reset(self.h))

    def stream_push(self, codes, final=False, capacity=None, check=True):
        """Append host codes [n, n_codebooks]; returns the samples sent by the
        decodes that became due (numpy float32, possibly empty)."""
        codes = np.ascontiguousarray(codes, dtype=np.int32).reshape(-1, self.dims.n_codebooks)
        n = codes.shape[0]
        cap = capacity if capacity is not None else (n + 2 * 325) * self.spf
        buf = np.empty(max(cap, 1), np.float32)
        got = ctypes.c_long(0)
        rc = _codec_lib().q3codec_stream_push(self.h, codes.ctypes.data if n else None, n, int(final),
                                              buf.ctypes.data, cap, ctypes.byref(got))
        if check:
            self._check(rc)
            return buf[:got.value]
        return rc, buf[:got.value]

    def kernel_count(self) -> int:
        return _codec_lib().q3codec_window_kernel_count(self.h)
