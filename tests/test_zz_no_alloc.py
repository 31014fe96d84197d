"""The allocation-free draw entry point (for callers that cannot allocate
device memory) gives the same ids as the handle-based q3tts_sample_logits and
as the oracle's processors + draw, through the C ABI, on two calls in a row.
Collected last on purpose."""
import numpy as np
import pytest

import oracle
import synth
from synth import RowSampling

pytestmark = pytest.mark.gpu


def _params(n, rng, talker):
    ps = []
    for i in range(n):
        r = RowSampling(repetition_penalty=1.05 if talker else 1.0, min_new_tokens=int(rng.integers(0, 3)),
                        seed=int(rng.integers(0, 2 ** 62)))
        if i % 3:
            r.do_sample = r.cp_do_sample = 1
            r.temperature = r.cp_temperature = 0.9
            r.top_k = r.cp_top_k = 50 if i % 2 else 0
            r.top_p = r.cp_top_p = 0.95 if i % 3 == 2 else 1.0
        ps.append(r)
    return ps


@pytest.mark.parametrize("talker,V", [(True, 3072), (False, 2048)])
def test_noalloc_matches_handle_entry_point(talker, V):
    import dataclasses
    import torch
    import speech_lm_decode_gb300 as q3
    d = dataclasses.replace(synth.DIMS_SMALL, codec_vocab=3072, cp_vocab=2048, eos_id=2150, suppress_lo=2048,
                            suppress_hi=3072)
    h = q3.Q3TTS(d, synth.F32, q3.to_device_weights(synth.make_weights(d, synth.F32, 1)), 1, 4, 1)
    rng = np.random.default_rng(17 if talker else 18)
    n = 200
    try:
        for call in range(2):    # two calls in a row: the shared staging area is reused
            lg = synth.random_logits(n, V, seed=300 + call + 10 * int(talker))
            ps = _params(n, rng, talker)
            sel = rng.integers(0, 5, n).astype(np.int32)
            rows = rng.integers(0, 64, n).astype(np.int32)
            seen = (rng.random((n, V)) < 0.05).astype(np.uint8) if talker else None
            step = 0 if talker else 3
            want = h.sample_logits(lg, talker, ps, sel, step, rows, seen)
            lg_dev = torch.from_numpy(lg).cuda()
            seen_dev = torch.from_numpy(seen).cuda() if seen is not None else None
            got = q3.sample_logits_noalloc(lg_dev, talker, ps, sel, step, rows, d.eos_id, d.suppress_lo,
                                           d.suppress_hi, seen=seen_dev)
            assert np.array_equal(got, want), np.nonzero(got != want)[0][:10]
            # and the oracle's own processors + draw on the same logits
            for i in range(n):
                err, oid, _, _ = oracle.sample(lg[i], ps[i], talker, seen=None if seen is None else seen[i],
                                               sel_index=int(sel[i]), eos=d.eos_id, sup_lo=d.suppress_lo,
                                               sup_hi=d.suppress_hi, row=int(rows[i]), frame=int(sel[i]), step=step)
                assert err == 0 and oid == int(got[i]), (i, oid, int(got[i]))
        # a NaN set is reported, and the next call starts clean again
        lg = synth.random_logits(4, V, seed=99)
        lg[1, 5] = np.nan
        ps = _params(4, rng, talker)
        rc, ids = q3.sample_logits_noalloc(torch.from_numpy(lg).cuda(), talker, ps, np.zeros(4, np.int32), 1,
                                           np.zeros(4, np.int32), d.eos_id, d.suppress_lo, d.suppress_hi,
                                           check=False)
        assert rc == q3.Q3_ERR_NAN and ids[1] == -1
        lg[1, 5] = 0.0
        ids = q3.sample_logits_noalloc(torch.from_numpy(lg).cuda(), talker, ps, np.zeros(4, np.int32), 1,
                                       np.zeros(4, np.int32), d.eos_id, d.suppress_lo, d.suppress_hi)
        assert np.all(ids >= 0)
        # beyond the fixed staging size: rejected, nothing run
        big = torch.zeros((1025, V), device="cuda")
        rc, _ = q3.sample_logits_noalloc(big, talker, _params(1025, rng, talker), np.zeros(1025, np.int32), 1,
                                         np.zeros(1025, np.int32), d.eos_id, d.suppress_lo, d.suppress_hi,
                                         check=False)
        assert rc == q3.Q3_ERR_CAPACITY
        # a sampling set with temperature 0 is rejected before anything runs
        bad = _params(4, rng, talker)
        bad[1].do_sample = bad[1].cp_do_sample = 1
        bad[1].temperature = bad[1].cp_temperature = 0.0
        rc, _ = q3.sample_logits_noalloc(torch.from_numpy(lg).cuda(), talker, bad, np.zeros(4, np.int32), 1,
                                         np.zeros(4, np.int32), d.eos_id, d.suppress_lo, d.suppress_hi,
                                         check=False)
        assert rc == q3.Q3_ERR_ARG
        # tensors the library cannot read safely never reach it
        with pytest.raises(ValueError):
            q3.sample_logits_noalloc(torch.from_numpy(lg).cuda().to(torch.bfloat16), talker, ps,
                                     np.zeros(4, np.int32), 1, np.zeros(4, np.int32), d.eos_id, d.suppress_lo,
                                     d.suppress_hi)
        with pytest.raises(ValueError):
            q3.sample_logits_noalloc(torch.from_numpy(lg), talker, ps, np.zeros(4, np.int32), 1,
                                     np.zeros(4, np.int32), d.eos_id, d.suppress_lo, d.suppress_hi)
        with pytest.raises(ValueError):
            q3.sample_logits_noalloc(torch.from_numpy(lg).cuda(), talker, ps[:3], np.zeros(4, np.int32), 1,
                                     np.zeros(4, np.int32), d.eos_id, d.suppress_lo, d.suppress_hi)
    finally:
        h.close()
