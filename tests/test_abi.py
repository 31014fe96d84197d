"""The C-ABI library loads and exports every entry point include/q3tts.h and
include/q3codec.h declare (CPU only: no compute call is made)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_symbols(header="q3tts.h", prefix="q3tts_"):
    src = open(os.path.join(ROOT, "include", header)).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(" + prefix + r"[a-z_0-9]+)\s*\(", src)))


def test_header_declares_the_boundary():
    names = declared_symbols()
    for n in ("q3tts_create", "q3tts_prefill", "q3tts_step_frames", "q3tts_destroy", "q3tts_sample_logits",
              "q3tts_set_capture", "q3tts_workspace_bytes", "q3tts_last_error"):
        assert n in names


def test_library_exports_every_declared_symbol():
    import speech_lm_decode_gb300 as q3
    from speech_lm_decode_gb300 import build
    build.build()
    lib = ctypes.CDLL(q3.LIB_PATH)
    missing = [n for n in declared_symbols() if not hasattr(lib, n)]
    assert not missing, missing
    assert set(declared_symbols()) >= set(q3.EXPORTS)
    codec = declared_symbols("q3codec.h", "q3codec_")
    assert set(codec) == set(q3.CODEC_EXPORTS), (codec, q3.CODEC_EXPORTS)
    missing = [n for n in codec if not hasattr(lib, n)]
    assert not missing, missing


def test_codec_workspace_and_config_validation():
    """The decoder's configuration is checked before anything is sized: head
    width 64, widths in multiples of 8, vocoder channels that halve evenly."""
    import dataclasses
    import speech_lm_decode_gb300 as q3
    import synth.codec as sc
    L = q3._codec_lib()
    c = q3.make_codec_config(sc.CODEC_FULL, q3.Q3_BF16, 325)
    n = L.q3codec_workspace_bytes(ctypes.byref(c))
    # at least the last vocoder stage's activations: 325 frames x 1920 samples x 96 channels, fp32, twice
    assert n > 2 * 325 * 1920 * 96 * 4
    for bad in (dataclasses.replace(sc.CODEC_FULL, head_dim=128), dataclasses.replace(sc.CODEC_FULL, ffn=1001),
                dataclasses.replace(sc.CODEC_FULL, dac_channels=1000), dataclasses.replace(sc.CODEC_FULL, n_up=3),
                dataclasses.replace(sc.CODEC_FULL, strides=(8, 5, 4, 3, 2))):
        cb = q3.make_codec_config(bad, q3.Q3_BF16, 325) if len(bad.strides) <= 4 else None
        if cb is None:
            continue
        assert L.q3codec_workspace_bytes(ctypes.byref(cb)) == 0, bad
    cb = q3.make_codec_config(sc.CODEC_FULL, q3.Q3_BF16, 0)
    assert L.q3codec_workspace_bytes(ctypes.byref(cb)) == 0
    h = ctypes.c_void_p()
    w = q3.CodecWeights()
    assert L.q3codec_create(ctypes.byref(c), ctypes.byref(w), None, 0, None, ctypes.byref(h)) == q3.Q3_ERR_ARG


def test_workspace_size_and_config_validation():
    import speech_lm_decode_gb300 as q3
    import synth
    L = q3.lib()
    c = q3.make_config(synth.DIMS_06B, q3.Q3_BF16, 1, 228, 64)
    n = L.q3tts_workspace_bytes(ctypes.byref(c))
    # the talker KV cache alone: 2 x 28 layers x 8 heads x 228 positions x 128 x 2 bytes
    assert n > 2 * 28 * 8 * 228 * 128 * 2
    bad = q3.make_config(synth.DIMS_06B, q3.Q3_BF16, 1, 228, 64)
    bad.head_dim = 64
    assert L.q3tts_workspace_bytes(ctypes.byref(bad)) == 0
    bad = q3.make_config(synth.DIMS_06B, 7, 1, 228, 64)
    assert L.q3tts_workspace_bytes(ctypes.byref(bad)) == 0
    h = ctypes.c_void_p()
    w = q3.Weights()
    assert L.q3tts_create(ctypes.byref(c), ctypes.byref(w), None, 0, None, ctypes.byref(h)) == q3.Q3_ERR_ARG


def test_execution_fields_are_validated():
    """The execution choices are explicit config fields: out-of-range values
    make the configuration invalid, and the cluster path (whose packed weight
    image sits in the workspace) grows the workspace only when it is asked for
    and the shape is one it serves."""
    import speech_lm_decode_gb300 as q3
    import synth
    L = q3.lib()

    def size(d=synth.DIMS_06B, **kw):
        c = q3.make_config(d, q3.Q3_BF16, 1, 228, 64, **kw)
        return L.q3tts_workspace_bytes(ctypes.byref(c))
    base = size()
    assert base > 0
    for kw in ({"step_path": 4}, {"step_path": -1}, {"wait_limit_us": -1}, {"inject_timeout": -2},
               {"debug_sync": 2}, {"separate_projections": 2}, {"separate_projections": -1}):
        assert size(**kw) == 0, kw
    # separate q/k/v and gate/up products need no more room in bf16 (the up
    # product reuses the second operand scratch)
    assert size(separate_projections=1) == base
    for p in (q3.Q3_PATH_GRAPH, q3.Q3_PATH_FRAME):
        assert size(step_path=p) == base
    # the packed image holds every matrix once more (about 1.2 GB for the 0.6B shape)
    assert size(step_path=q3.Q3_PATH_CLUSTER) > base + 10 ** 9
    # a shape the cluster kernel does not serve cannot ask for it
    assert size(d=synth.DIMS_SMALL, step_path=q3.Q3_PATH_CLUSTER) == 0
    assert size(d=synth.DIMS_CL, step_path=q3.Q3_PATH_CLUSTER) > 0
    # the text side: both sizes or neither
    import dataclasses
    assert size(d=dataclasses.replace(synth.DIMS_06B, text_vocab=100)) == 0
    assert size(d=dataclasses.replace(synth.DIMS_06B, text_vocab=100, text_hidden=2048)) >= base
    assert size(d=dataclasses.replace(synth.DIMS_06B, text_vocab=100, text_hidden=4096)) > base
