"""The shared input generator: determinism and distribution (CPU only)."""
import numpy as np
import torch

import synth


def test_normal_is_deterministic_and_indexed():
    a = synth.normal((1000,), 3, 17, 1.0)
    b = synth.normal((2000,), 3, 17, 1.0)
    assert np.array_equal(a, b[:1000])           # value depends on the index only
    c = synth.normal((1000,), 4, 17, 1.0)
    assert not np.array_equal(a, c)


def test_normal_moments():
    x = synth.normal((400000,), 1, 5, 0.02).astype(np.float64)
    assert abs(x.mean()) < 1e-4
    assert abs(x.std() - 0.02) < 2e-4


def test_bf16_generation_is_rne_of_f32_draws():
    f = synth.normal((50000,), 2, 9, 0.02)
    b = synth.normal((50000,), 2, 9, 0.02, dtype=synth.BF16)
    ref = torch.from_numpy(f).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(b, ref)
    assert np.array_equal(synth.round_bf16(f), ref)


def test_workloads_shapes():
    for i in range(1, 6):
        wl = synth.workload(i)
        assert len(wl.rows) == wl.batch == len(wl.prompt_lens) == len(wl.n_text)
        assert max(wl.prompt_lens) + wl.frames <= wl.max_ctx
    wl4 = synth.workload(4)
    assert all(64 <= n <= 512 for n in wl4.prompt_lens)
    assert all(50 <= r.force_eos_at_frame <= 250 for r in wl4.rows)
    assert synth.workload(5).max_ctx == 256 + 1024
