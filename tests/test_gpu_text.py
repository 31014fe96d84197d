"""GPU parity of the text side (q3tts_text_embed: embedding gather +
ResizeMLP) against the oracle, through the C ABI, and a decode whose trailing
text rows come from text ids on each side."""
import dataclasses

import numpy as np
import pytest

import oracle
import synth
from synth import RowSampling, Workload, F32, BF16
from parity import run_gpu, compare, TOL

pytestmark = pytest.mark.gpu

DIMS_TEXT = dataclasses.replace(synth.DIMS_SMALL, text_vocab=1000, text_hidden=384)


def _handle(q3, d, dtype, dw, max_batch=2, max_ctx=400):
    return q3.Q3TTS(d, dtype, dw, max_batch, max_ctx, 8)


@pytest.mark.parametrize("dtype", [F32, BF16])
def test_text_rows_match_oracle(dtype):
    """Lengths 1, 7 (GEMV), 16, 65 (tensor-core GEMMs for bf16) and 600
    (two 512-row chunks), host and device ids and outputs."""
    import torch
    import speech_lm_decode_gb300 as q3
    d = DIMS_TEXT
    w = synth.make_weights(d, dtype, 31)
    w.update(synth.make_text_weights(d, dtype, 31))
    dw = q3.to_device_weights(w)
    q = _handle(q3, d, dtype, dw)
    rng = np.random.default_rng(5)
    try:
        for n in (1, 7, 16, 65, 600):
            ids = rng.integers(0, d.text_vocab, n).astype(np.int32)
            ids[0] = d.text_vocab - 1
            want = oracle.text_embed(w, dtype, ids)
            got = q.text_embed(ids)
            assert np.max(np.abs(got - want)) <= TOL[dtype], (n, float(np.max(np.abs(got - want))))
            out_dev = torch.empty((n, d.hidden), dtype=torch.float32, device="cuda")
            q.text_embed(torch.from_numpy(ids).cuda(), out=out_dev)
            assert np.array_equal(out_dev.cpu().numpy(), got)
        # bad ids: rejected on the host before anything runs, flagged on the device
        rc, _ = q.text_embed(np.array([0, d.text_vocab], np.int32), check=False)
        assert rc == q3.Q3_ERR_ARG
        rc, _ = q.text_embed(torch.tensor([3, -1], dtype=torch.int32, device="cuda"), check=False)
        assert rc == q3.Q3_ERR_BOUNDS
    finally:
        q.close()


def test_full_size_text_side():
    """The released shapes: 151936-entry BPE vocabulary, 2048-d embedding,
    ResizeMLP 2048 -> 2048 -> 1024 (bf16), 64 trailing ids as in the workloads."""
    import speech_lm_decode_gb300 as q3
    d = dataclasses.replace(synth.DIMS_06B, n_layers=1, cp_layers=1, text_vocab=synth.TEXT_VOCAB,
                            text_hidden=synth.TEXT_HIDDEN)
    w = synth.make_weights(d, BF16, 1)
    w.update(synth.make_text_weights(d, BF16, 1))
    q = _handle(q3, d, BF16, q3.to_device_weights(w), max_batch=1, max_ctx=200)
    try:
        ids = np.random.default_rng(9).integers(0, d.text_vocab, 64).astype(np.int32)
        ids[:2] = [0, d.text_vocab - 1]
        got = q.text_embed(ids)
        want = oracle.text_embed(w, BF16, ids)
        assert np.max(np.abs(got - want)) <= TOL[BF16], float(np.max(np.abs(got - want)))
    finally:
        q.close()


def test_decode_with_text_rows_from_ids():
    """Trailing text given as ids: the GPU turns them into rows with
    q3tts_text_embed and decodes; the oracle builds its own rows from the same
    ids and is compared on the GPU's codes."""
    import speech_lm_decode_gb300 as q3
    d = DIMS_TEXT
    rows = [RowSampling(max_frames=8), RowSampling(max_frames=8, do_sample=1, temperature=0.9, top_k=8,
                                                   cp_do_sample=1, seed=4)]
    wl = Workload("text", d, BF16, 7, 2, [6, 9], [5, 3], 8, rows, 30, norm_std=0.1)
    w = synth.make_weights(d, BF16, wl.weight_seed, norm_std=0.1)
    w.update(synth.make_text_weights(d, BF16, wl.weight_seed))
    dw = q3.to_device_weights(w)
    inp = synth.make_inputs(wl)
    ids = np.random.default_rng(2).integers(0, d.text_vocab, sum(wl.n_text)).astype(np.int32)
    q = _handle(q3, d, BF16, dw)
    try:
        gpu_rows = q.text_embed(ids)
    finally:
        q.close()
    g_inp = dict(inp, text=gpu_rows)
    o_inp = dict(inp, text=oracle.text_embed(w, BF16, ids).astype(np.float32))
    g = run_gpu(wl, dw, g_inp, cap_rows=[0, 1])
    compare(wl, w, o_inp, g)
