"""The codec decoder on the GPU (through the C ABI) against the fp64 oracle.

Tolerance: the waveform is tanh-bounded; products run in fp32 on the CUDA
cores or as bf16 high + low parts of the fp32 operand on the tensor cores
(about 2^-17 relative per operand), accumulated in fp32 through ~40 layers.
The test asks for max |error| <= 2e-4 and a signal-to-error ratio of at
least 60 dB; the pages quote 66 dB between fp32 decodes of different
lengths (Mizuoto "Qwen3-TTS" page, section "速度")."""
import dataclasses

import numpy as np
import pytest

import oracle.codec as oc
import synth
import synth.codec as sc

pytestmark = pytest.mark.gpu

MAX_ABS = 2e-4
MIN_SNR_DB = 60.0


@pytest.fixture(scope="module")
def q3():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    import speech_lm_decode_gb300 as q3
    q3.lib()
    return q3


def snr_db(ref, got):
    err = np.sum((np.asarray(ref, np.float64) - got) ** 2)
    return np.inf if err == 0 else 10 * np.log10(np.sum(np.asarray(ref, np.float64) ** 2) / err)


def check(ref, got, what=""):
    assert got.shape == ref.shape, (what, got.shape, ref.shape)
    assert np.all(np.isfinite(got)), what
    worst = float(np.max(np.abs(got - ref)))
    s = snr_db(ref, got)
    assert worst <= MAX_ABS and s >= MIN_SNR_DB, (what, worst, s)
    return worst, s


def _setup(q3, dims, dtype, seed, max_frames=64, **kw):
    w = sc.make_codec_weights(dims, dtype, seed)
    dec = q3.Q3Codec(dims, dtype, q3.codec_to_device(w), max_frames=max_frames, **kw)
    return w, dec, oc.Decoder(dims, w)


@pytest.mark.parametrize("dtype", [synth.BF16, synth.F32])
@pytest.mark.parametrize("T", [1, 7, 20, 45])
def test_window_small(q3, dtype, T):
    """Windows that put the products on the CUDA-core path (few rows), the
    tensor cores, or both within one decode."""
    w, dec, ora = _setup(q3, sc.CODEC_SMALL, dtype, 100 + T)
    codes = sc.make_codes(sc.CODEC_SMALL, T, 200 + T)
    got = dec.decode_window(codes)
    check(ora.decode_window(codes), got, f"T={T}")


def test_keep_from_and_device_buffers(q3):
    import torch
    w, dec, ora = _setup(q3, sc.CODEC_SMALL, synth.BF16, 7)
    codes = sc.make_codes(sc.CODEC_SMALL, 30, 8)
    full = dec.decode_window(codes)
    tail = dec.decode_window(codes, keep_from=11)
    assert np.array_equal(tail, full[11 * dec.spf:])
    out = torch.empty(30 * dec.spf, dtype=torch.float32, device="cuda")
    dec.decode_window(torch.from_numpy(codes).cuda(), out=out)
    assert np.array_equal(out.cpu().numpy(), full)


def test_whole_request_on_the_chunk_grid(q3):
    """330 frames: two chunks of the 300/25 grid, against the oracle's grid."""
    d = sc.CODEC_SMALL
    w, dec, ora = _setup(q3, d, synth.BF16, 17, max_frames=325)
    codes = sc.make_codes(d, 330, 18)
    got = dec.decode(codes)
    check(ora.decode(codes), got, "grid")


def test_streaming_matches_oracle_schedule(q3):
    d = sc.CODEC_SMALL
    w, dec, ora = _setup(q3, d, synth.BF16, 27, max_frames=325)
    T = 340
    codes = sc.make_codes(d, T, 28)
    ref_parts = ora.stream(codes)
    # the frames arrive in uneven pieces
    rng = np.random.default_rng(5)
    dec.stream_reset()
    got_parts, i = [], 0
    while i < T:
        n = int(min(T - i, rng.integers(1, 20)))
        out = dec.stream_push(codes[i:i + n], final=(i + n == T))
        if out.size:
            got_parts.append(out)
        i += n
    got = np.concatenate(got_parts)
    ref = np.concatenate([p for _, p in ref_parts])
    check(ref, got, "stream")
    # the first decode sends exactly the first 4 frames
    assert got_parts[0].size % dec.spf == 0 and got_parts[0].size >= 4 * dec.spf
    # streaming and the whole request agree up to rounding
    check(ora.decode(codes), got, "stream vs whole")
    with pytest.raises(q3.Q3Error) as e:
        dec.stream_push(codes[:1])
    assert e.value.code == q3.Q3_ERR_STATE


def test_full_size_window(q3):
    """The decoder at the pages' sizes (16 x 2048 x 256 codebooks, 8 layers of
    512, strides 8, 5, 4, 3: 1920 samples per frame): a 12-frame window against
    the oracle, and the first 8 frames of a full 325-frame window (the
    decoder is causal) against the oracle's 8-frame decode."""
    d = sc.CODEC_FULL
    w, dec, ora = _setup(q3, d, synth.BF16, 37, max_frames=325)
    assert dec.spf == 1920
    codes = sc.make_codes(d, 325, 38)
    got = dec.decode_window(codes[:12])
    check(ora.decode_window(codes[:12]), got, "full 12")
    big = dec.decode_window(codes)
    assert big.shape == (325 * 1920,) and np.all(np.isfinite(big)) and np.max(np.abs(big)) <= 1.0
    check(ora.decode_window(codes[:8]), big[:8 * 1920], "full 325 prefix")


def test_errors(q3):
    import torch
    d = sc.CODEC_SMALL
    w, dec, ora = _setup(q3, d, synth.BF16, 47, max_frames=16)
    codes = sc.make_codes(d, 5, 48)
    bad = codes.copy()
    bad[2, 3] = d.codebook_size
    rc, _ = dec.decode_window(bad, check=False)
    assert rc == q3.Q3_ERR_ARG
    rc, _ = dec.decode_window(torch.from_numpy(bad).cuda(), check=False)
    assert rc == q3.Q3_ERR_BOUNDS
    # the handle still works after a device-side error
    check(ora.decode_window(codes), dec.decode_window(codes), "after error")
    rc, _ = dec.decode_window(sc.make_codes(d, 17, 49), check=False)
    assert rc == q3.Q3_ERR_ARG
    # a whole request needs room for a chunk window
    rc, _ = dec.decode(sc.make_codes(d, 40, 50), check=False)
    assert rc == q3.Q3_ERR_ARG
