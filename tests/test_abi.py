"""The C-ABI library loads and exports every entry point include/q3tts.h
declares (CPU only: no compute call is made)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_symbols():
    src = open(os.path.join(ROOT, "include", "q3tts.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(q3tts_[a-z_0-9]+)\s*\(", src)))


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
