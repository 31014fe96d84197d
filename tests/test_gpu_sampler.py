"""The GPU logits processors + draw are bit-exact with the oracle's on
identical logits (the frame loop's own sampler, through q3tts_sample_logits)."""
import numpy as np
import pytest

import oracle
import synth
from synth import RowSampling

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def handle():
    import torch
    assert torch.cuda.is_available()
    import speech_lm_decode_gb300 as q3
    d = dataclasses_replace_vocab(synth.DIMS_SMALL)
    w = synth.make_weights(d, synth.F32, 1)
    q = q3.Q3TTS(d, synth.F32, q3.to_device_weights(w), 1, 4, 1)
    yield q
    q.close()


def dataclasses_replace_vocab(d):
    # the handle's vocabularies / specials define the sampler's V, EOS and suppression
    import dataclasses
    return dataclasses.replace(d, codec_vocab=3072, cp_vocab=2048, eos_id=2150, suppress_lo=2048, suppress_hi=3072)


def _param_sets(n, rng):
    ps = []
    for i in range(n):
        kind = i % 6
        r = RowSampling(repetition_penalty=float(rng.choice([1.0, 1.05, 1.3])), min_new_tokens=int(rng.integers(0, 4)),
                        seed=int(rng.integers(0, 2 ** 63)))
        if kind >= 1:
            r.do_sample = r.cp_do_sample = 1
            r.temperature = r.cp_temperature = float(rng.choice([0.5, 0.9, 1.0, 1.7]))
        if kind in (2, 4):
            r.top_k = r.cp_top_k = int(rng.choice([1, 5, 50, 300]))
        if kind in (3, 4, 5):
            r.top_p = r.cp_top_p = float(rng.choice([0.3, 0.8, 0.95, 0.999]))
        ps.append(r)
    return ps


@pytest.mark.parametrize("talker,V", [(True, 3072), (False, 2048)])
def test_sampler_bit_exact(handle, talker, V):
    rng = np.random.default_rng(5 if talker else 6)
    n_total, chunk = 2048, 256
    mism = []
    for c0 in range(0, n_total, chunk):
        lg = synth.random_logits(chunk, V, seed=100 + c0 + int(talker), scale=float(rng.choice([0.5, 2.0, 6.0])))
        ps = _param_sets(chunk, rng)
        sel = rng.integers(0, 6, chunk).astype(np.int32)
        nrow = rng.integers(0, 300, chunk).astype(np.int32)
        seen = (rng.random((chunk, V)) < 0.05).astype(np.uint8)
        step = 0 if talker else int(rng.integers(1, 16))
        ids = handle.sample_logits(lg, talker, ps, sel, step, nrow, seen if talker else None)
        for j in range(chunk):
            err, want, _, _ = oracle.sample(lg[j], ps[j], talker, seen=seen[j] if talker else None,
                                            sel_index=int(sel[j]), eos=2150 if talker else -1,
                                            sup_lo=2048 if talker else 0, sup_hi=3072 if talker else 0,
                                            row=int(nrow[j]), frame=int(sel[j]), step=step)
            assert err == 0
            if want != ids[j]:
                mism.append((c0 + j, want, int(ids[j])))
    assert not mism, mism[:10]


def test_sampler_nan_fails_closed(handle):
    import speech_lm_decode_gb300 as q3
    lg = synth.random_logits(4, 3072, seed=9)
    lg[2, 77] = np.nan
    ps = [RowSampling(do_sample=i % 2) for i in range(4)]
    rc, ids = handle.sample_logits(lg, True, ps, np.zeros(4, np.int32), 0, np.zeros(4, np.int32), check=False)
    assert rc == q3.Q3_ERR_NAN
    assert ids[2] == -1 and ids[0] >= 0 and ids[1] >= 0 and ids[3] >= 0
