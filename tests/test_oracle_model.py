"""Pins for the oracle's model arithmetic and generation loop (CPU only)."""
import dataclasses
import math

import numpy as np
import pytest
import torch

import oracle
import synth
from synth import Dims, RowSampling, Workload, F32, BF16

TINY = Dims(n_layers=2, hidden=64, n_q_heads=4, n_kv_heads=2, head_dim=8, ffn=96, codec_vocab=48, cp_layers=2,
            cp_hidden=64, cp_ffn=80, cp_vocab=16, n_groups=4, eos_id=40, suppress_lo=32, suppress_hi=48)


# ------------------------------------------------------------------ pieces
def test_rmsnorm_closed_form():
    L = oracle.lib()
    rng = np.random.default_rng(0)
    x = rng.standard_normal(1024) * 3.0
    w = np.ones(1024, np.float32)
    y = np.empty(1024)
    L.oracle_rmsnorm(x.ctypes.data, w.ctypes.data, 1024, 1e-6, y.ctypes.data)
    # unit weight: output has RMS sqrt(ms/(ms+eps))
    ms = np.mean(x ** 2)
    assert np.sqrt(np.mean(y ** 2)) == pytest.approx(math.sqrt(ms / (ms + 1e-6)), rel=1e-12)
    # scale invariance and the weight multiplies elementwise
    w2 = rng.uniform(0.5, 1.5, 1024).astype(np.float32)
    y2 = np.empty(1024)
    x7 = 7.0 * x     # held: ctypes only borrows the buffer
    L.oracle_rmsnorm(x7.ctypes.data, w2.ctypes.data, 1024, 0.0, y2.ctypes.data)
    y1 = np.empty(1024)
    L.oracle_rmsnorm(x.ctypes.data, w.ctypes.data, 1024, 0.0, y1.ctypes.data)
    np.testing.assert_allclose(y2, y1 * w2.astype(np.float64), rtol=1e-12)


def _rope(x, pos, theta=1e6):
    L = oracle.lib()
    y = np.array(x, np.float64)
    L.oracle_rope(y.ctypes.data, len(y), pos, theta)
    return y


def test_rope_is_rotation_of_half_pairs():
    rng = np.random.default_rng(1)
    x = rng.standard_normal(128)
    assert np.array_equal(_rope(x, 0), x)
    for pos in (1, 7, 300, 1279):
        y = _rope(x, pos)
        # complex form: (x_j + i x_{j+64}) * exp(i * pos * inv_freq_j), angle formed in fp32
        inv = np.array([np.float32(1e6 ** (-2.0 * j / 128)) for j in range(64)], np.float32)
        ang = (np.float32(pos) * inv).astype(np.float64)
        z = (x[:64] + 1j * x[64:]) * np.exp(1j * ang)
        np.testing.assert_allclose(y[:64], z.real, atol=1e-12)
        np.testing.assert_allclose(y[64:], z.imag, atol=1e-12)
        # pairwise norms preserved
        np.testing.assert_allclose(y[:64] ** 2 + y[64:] ** 2, x[:64] ** 2 + x[64:] ** 2, rtol=1e-12)


def test_rope_relative_position():
    rng = np.random.default_rng(2)
    q, k = rng.standard_normal(128), rng.standard_normal(128)
    d1 = _rope(q, 40) @ _rope(k, 10)
    d2 = _rope(q, 130) @ _rope(k, 100)
    assert d1 == pytest.approx(d2, rel=1e-4, abs=1e-4)   # fp32 angles: not exact


@pytest.mark.parametrize("mode,sections", [(0, (16, 24, 24)), (0, (24, 20, 20)), (1, (0, 0, 0))])
def test_mrope_equals_rope_for_equal_positions(mode, sections):
    """mrope with the three position streams equal is plain RoPE, difference
    exactly 0.0 (ncnn discussion 6798, section 1, fact 1)."""
    L = oracle.lib()
    rng = np.random.default_rng(3)
    sec = np.array(sections, np.int32)
    for pos in (0, 5, 129, 1000):
        x = rng.standard_normal(128)
        y = np.array(x)
        p3 = np.array([pos, pos, pos], np.int32)
        L.oracle_mrope(y.ctypes.data, 128, p3.ctypes.data, sec.ctypes.data, mode, 1e6)
        assert np.max(np.abs(y - _rope(x, pos))) == 0.0
        # unequal streams do differ
        p3 = np.array([pos, pos + 3, pos + 9], np.int32)
        z = np.array(x)
        L.oracle_mrope(z.ctypes.data, 128, p3.ctypes.data, sec.ctypes.data, mode, 1e6)
        assert np.max(np.abs(z - _rope(x, pos))) > 0


def test_gqa_attention_brute_force():
    L = oracle.lib()
    rng = np.random.default_rng(4)
    nq, nkv, hd, cap = 4, 2, 8, 10
    for n in (1, 3, 10):
        q = rng.standard_normal((nq, hd))
        K = rng.standard_normal((nkv, cap, hd))
        V = rng.standard_normal((nkv, cap, hd))
        out = np.empty((nq, hd))
        L.oracle_attend(q.ctypes.data, K.ctypes.data, V.ctypes.data, cap, n, nq, nkv, hd, out.ctypes.data)
        Kr = np.repeat(K[:, :n], nq // nkv, axis=0)   # repeat_interleave over heads
        Vr = np.repeat(V[:, :n], nq // nkv, axis=0)
        s = np.einsum("hd,hjd->hj", q, Kr) / math.sqrt(hd)
        p = np.exp(s - s.max(1, keepdims=True))
        p /= p.sum(1, keepdims=True)
        np.testing.assert_allclose(out, np.einsum("hj,hjd->hd", p, Vr), rtol=1e-12, atol=1e-13)


def test_bf16_rounding_matches_torch():
    L = oracle.lib()
    rng = np.random.default_rng(5)
    x = np.concatenate([rng.standard_normal(5000).astype(np.float32),
                        (rng.standard_normal(5000) * 1e-3).astype(np.float32),
                        np.array([1 + 2 ** -8, 1 + 3 * 2 ** -8, -(1 + 2 ** -8), 65504.0], np.float32)])
    ref = torch.from_numpy(x).to(torch.bfloat16).to(torch.float64).numpy()
    got = np.array([L.oracle_bf16_round(float(v)) for v in x])
    assert np.array_equal(got, ref)


# ------------------------------------------------------------------ structured closed form
def _structured(n_text=3, final_w=True, seed=0):
    """Weights whose layers are all identity maps (o and down projections are
    zero), with one-hot embedding tables.  Then every output is a head row
    dotted with the final-norm of a sum of one-hot directions, so the code
    sequence follows from column lookups alone."""
    d = dataclasses.replace(TINY, hidden=64, cp_hidden=64, codec_vocab=16, cp_vocab=8, n_groups=4, eos_id=12,
                            suppress_lo=8, suppress_hi=16)
    rng = np.random.default_rng(seed)
    w = synth.make_weights(d, F32, 11)
    for blk in ("talker", "cp"):
        w[blk]["wo"][:] = 0
        w[blk]["wd"][:] = 0
        w[blk]["wqkv"] *= 20.0
        if final_w:
            w[blk]["final_norm"][:] = rng.uniform(0.5, 1.5, d.hidden).astype(np.float32)
    H, V, cpV, G1 = d.hidden, d.codec_vocab, d.cp_vocab, d.n_groups - 1
    dir_cp = lambda q, c: q * cpV + c            # table q (0-based), code c   -> 0..23
    dir_codec = lambda c: 24 + c                 # codec table row c           -> 24..39
    dir_text = lambda j: 40 + j                  # trailing text row j         -> 40..
    DIR_PAD, DIR_PROMPT = 50, 60
    w["codec_emb"][:] = 0
    w["cp_emb"][:] = 0
    for c in range(V):
        w["codec_emb"][c, dir_codec(c)] = 1
    for q in range(G1):
        for c in range(cpV):
            w["cp_emb"][q, c, dir_cp(q, c)] = 1
    w["cp_heads"][:] = 0
    w["cp_heads"][:, :, :40] = rng.standard_normal((G1, cpV, 40)).astype(np.float32)
    w["codec_head"][:] = rng.standard_normal((V, H)).astype(np.float32)
    w["codec_head"][d.eos_id, DIR_PAD] = 50.0     # the pad row makes EOS win
    prompt = np.zeros((4, H), np.float32)
    prompt[:-1, 61] = rng.standard_normal(3)   # earlier prompt rows: no effect on the last output
    prompt[-1, DIR_PROMPT] = 1.0
    text = np.zeros((n_text, H), np.float32)
    for j in range(n_text):
        text[j, dir_text(j)] = 1.0
    pad = np.zeros(H, np.float32)
    pad[DIR_PAD] = 1.0
    inputs = {"prompt": prompt, "prompt_offsets": np.array([0, 4], np.int32), "text": text,
              "text_offsets": np.array([0, n_text], np.int32), "tts_pad": pad}
    return d, w, inputs, dict(dir_cp=dir_cp, dir_codec=dir_codec, dir_text=dir_text, pad=DIR_PAD,
                              prompt=DIR_PROMPT)


def _expected_structured(d, w, n_text, max_frames, min_new=2):
    """Code sequence implied by identity layers + one-hot tables."""
    fn_t, fn_c = w["talker"]["final_norm"], w["cp"]["final_norm"]
    cpV = d.cp_vocab

    def pick(scores, talker, k):
        s = scores.astype(np.float64).copy()
        if talker:
            if k < min_new:
                s[d.eos_id] = -np.inf
            for i in range(d.suppress_lo, d.suppress_hi):
                if i != d.eos_id:
                    s[i] = -np.inf
        return int(np.argmax(s))      # numpy argmax: first maximal index

    def talker_pick(dirs, k):
        return pick(w["codec_head"][:, dirs] @ fn_t[dirs], True, k)

    sel = [talker_pick([60], 0)]
    frames = []
    k = 0
    while True:
        code0 = sel[-1]
        if code0 == d.eos_id or k >= max_frames:
            break
        k += 1
        codes = [code0]
        tok_dir = 24 + code0
        for s in range(d.n_groups - 1):
            nxt = pick(w["cp_heads"][s][:, tok_dir] * fn_c[tok_dir], False, 0)
            codes.append(nxt)
            tok_dir = s * cpV + nxt        # table s (0-based) holds code s+1
        frames.append(codes)
        dirs = [24 + codes[0]] + [q * cpV + codes[q + 1] for q in range(d.n_groups - 1)]
        dirs.append(40 + (k - 1) if k - 1 < n_text else 50)
        sel.append(talker_pick(dirs, k))
    return frames, sel


@pytest.mark.parametrize("max_frames", [10, 2])
def test_structured_weights_closed_form(max_frames):
    n_text = 3
    d, w, inputs, _ = _structured(n_text)
    row = RowSampling(repetition_penalty=1.0, min_new_tokens=2, max_frames=max_frames)
    wl = Workload("structured", d, F32, 0, 1, [4], [n_text], max_frames, [row], 4 + max_frames)
    o = oracle.run(wl, w, inputs, capture=False)
    frames_exp, sel_exp = _expected_structured(d, w, n_text, max_frames)
    nf = int(o.get("frames")[0])
    assert nf == len(frames_exp)
    assert np.array_equal(o.get("codes")[0, :nf], np.array(frames_exp, np.int32))
    assert list(o.get("own_sel")[0, :nf + 1]) == sel_exp
    # N frames <-> N+1 talker selections, N predictor runs (ncnn discussion 6832, 3.1)
    assert o.get("selections")[0] == nf + 1
    assert o.get("predictor_runs")[0] == nf
    if max_frames == 10:
        # text rows are consumed one per step, then tts_pad, whose row ends the run
        assert nf == n_text + 1 and o.get("reason")[0] == oracle.REASON_EOS
        assert sel_exp[-1] == d.eos_id
    else:
        assert nf == 2 and o.get("reason")[0] == oracle.REASON_LENGTH


def test_structured_weights_detect_offsets():
    """A table/head offset mistake would change the sequence: check that the
    closed form is sensitive to it by shifting the heads by one."""
    d, w, inputs, _ = _structured(3)
    f1, _ = _expected_structured(d, w, 3, 10)
    w2 = dict(w)
    w2["cp_heads"] = np.roll(w["cp_heads"], 1, axis=0)
    f2, _ = _expected_structured(d, w2, 3, 10)
    assert f1 != f2


# ------------------------------------------------------------------ brute force (full recompute)
def _np_block(x, bw, nl, d, H, F):
    """Full-sequence causal Qwen3 block stack in numpy (no cache)."""
    n = x.shape[0]
    hd, nq, nkv = d.head_dim, d.n_q_heads, d.n_kv_heads
    inv = np.array([np.float32(d.rope_theta ** (-2.0 * j / hd)) for j in range(hd // 2)], np.float32)
    ang = (np.arange(n, dtype=np.float32)[:, None] * inv[None, :]).astype(np.float64)
    cos, sin = np.cos(ang), np.sin(ang)

    def rms(v, wt):
        return v / np.sqrt(np.mean(v ** 2, -1, keepdims=True) + d.rms_eps) * wt

    def rot(v):   # v [n, heads, hd]
        a, b = v[..., :hd // 2], v[..., hd // 2:]
        c, s = cos[:, None, :], sin[:, None, :]
        return np.concatenate([a * c - b * s, b * c + a * s], -1)

    mask = np.triu(np.full((n, n), -np.inf), 1)
    for l in range(nl):
        f64 = lambda k: bw[k][l].astype(np.float64)
        h = rms(x, f64("attn_norm"))
        qkv = h @ f64("wqkv").T
        q = qkv[:, :nq * hd].reshape(n, nq, hd)
        k = qkv[:, nq * hd:(nq + nkv) * hd].reshape(n, nkv, hd)
        v = qkv[:, (nq + nkv) * hd:].reshape(n, nkv, hd)
        q = rot(rms(q, f64("q_norm")))
        k = rot(rms(k, f64("k_norm")))
        k = np.repeat(k, nq // nkv, axis=1)
        v = np.repeat(v, nq // nkv, axis=1)
        s = np.einsum("ihd,jhd->hij", q, k) / math.sqrt(hd) + mask
        p = np.exp(s - s.max(-1, keepdims=True))
        p /= p.sum(-1, keepdims=True)
        att = np.einsum("hij,jhd->ihd", p, v).reshape(n, nq * hd)
        x = x + att @ f64("wo").T
        h = rms(x, f64("mlp_norm"))
        gu = h @ f64("wgu").T
        g, u = gu[:, :F], gu[:, F:]
        x = x + (g / (1 + np.exp(-g)) * u) @ f64("wd").T
    return rms(x, bw["final_norm"].astype(np.float64))


@pytest.mark.parametrize("dims", [TINY, dataclasses.replace(TINY, hidden=96, ffn=128)])
def test_incremental_oracle_matches_full_recompute(dims):
    """The oracle's KV-cache path equals a full causal recompute of every
    sequence (talker over prompt + assembled inputs; predictor over its 16
    tokens) on tiny random weights with non-unit norms."""
    wl = Workload("tiny", dims, F32, 5, 1, [6], [2], 3, [RowSampling(max_frames=3, repetition_penalty=1.05)], 9,
                  norm_std=0.2)
    w = synth.make_weights(dims, F32, 5, norm_std=0.2)
    for blk in ("talker", "cp"):
        for k in ("wqkv", "wo", "wgu", "wd"):
            w[blk][k] *= 10.0     # std 0.2: attention and MLP matter
    inp = synth.make_inputs(wl)
    o = oracle.run(wl, w, inp, capture=True)
    codes, sel = o.get("codes")[0], o.get("own_sel")[0]
    tl, cl = o.get("talker_logits")[0], o.get("cp_logits")[0]
    nf = int(o.get("frames")[0])
    assert nf >= 2
    f64 = lambda a: a.astype(np.float64)
    H, Hc, cpV = dims.hidden, dims.cp_hidden, dims.cp_vocab
    proj = (lambda v: v @ f64(w["cp_proj_w"]).T + f64(w["cp_proj_b"])) if H != Hc else (lambda v: v)
    seq = f64(inp["prompt"])
    hs = _np_block(seq, w["talker"], dims.n_layers, dims, H, dims.ffn)
    np.testing.assert_allclose(tl[0], hs[-1] @ f64(w["codec_head"]).T, rtol=1e-9, atol=1e-6)
    h_prev = hs[-1]
    for f in range(nf):
        c = codes[f]
        toks = [h_prev, f64(w["codec_emb"][c[0]])] + [f64(w["cp_emb"][s - 1, c[s]]) for s in range(1, dims.n_groups - 1)]
        hc = _np_block(proj(np.stack(toks)), w["cp"], dims.cp_layers, dims, Hc, dims.cp_ffn)
        for s in range(dims.n_groups - 1):
            np.testing.assert_allclose(cl[f, s], hc[s + 1] @ f64(w["cp_heads"][s]).T, rtol=1e-9, atol=1e-6)
        x = f64(w["codec_emb"][c[0]]) + sum(f64(w["cp_emb"][q - 1, c[q]]) for q in range(1, dims.n_groups))
        x = x + (f64(inp["text"][f]) if f < 2 else f64(inp["tts_pad"]))
        seq = np.vstack([seq, x[None]])
        hs = _np_block(seq, w["talker"], dims.n_layers, dims, H, dims.ffn)
        np.testing.assert_allclose(tl[f + 1], hs[-1] @ f64(w["codec_head"]).T, rtol=1e-9, atol=1e-6)
        h_prev = hs[-1]
        assert sel[f + 1] == (codes[f + 1][0] if f + 1 < nf else sel[f + 1])


# ------------------------------------------------------------------ loop invariants
def _tiny_wl(frames, batch=1, **kw):
    rows = [RowSampling(max_frames=frames, **kw) for _ in range(batch)]
    return Workload("tiny", TINY, F32, 9, batch, [5 + 2 * b for b in range(batch)], [3] * batch, frames, rows,
                    5 + 2 * batch + frames, norm_std=0.1)


@pytest.fixture(scope="module")
def tiny_weights():
    w = synth.make_weights(TINY, F32, 9, norm_std=0.1)
    for blk in ("talker", "cp"):
        for k in ("wqkv", "wo", "wgu", "wd"):
            w[blk][k] *= 10.0
    return w


def test_prefix_property(tiny_weights):
    """A 25-frame run is the exact prefix of a 54-frame run, and chunked
    stepping equals one call (ncnn discussion 6832, section 4)."""
    kw = dict(do_sample=1, temperature=0.9, top_k=8, top_p=0.9, cp_do_sample=1, cp_temperature=0.9, cp_top_k=8,
              cp_top_p=0.9, min_new_tokens=60)
    wl54, wl25 = _tiny_wl(54, **kw), _tiny_wl(25, **kw)
    inp = synth.make_inputs(wl54)
    a = oracle.run(wl54, tiny_weights, inp, capture=False)
    b = oracle.run(wl25, tiny_weights, inp, capture=False)
    c = oracle.run(wl54, tiny_weights, inp, capture=False, chunks=[25, 29])
    assert a.get("frames")[0] == 54 and b.get("frames")[0] == 25
    assert np.array_equal(a.get("codes")[0, :25], b.get("codes")[0])
    assert np.array_equal(a.get("codes"), c.get("codes"))
    assert a.get("selections")[0] == 55 and a.get("predictor_runs")[0] == 54


def test_rows_are_independent_and_forced_eos(tiny_weights):
    kw = dict(do_sample=1, temperature=1.0, top_k=0, top_p=1.0, cp_do_sample=1, min_new_tokens=20)
    wl = _tiny_wl(12, batch=3, **kw)
    wl.rows[1].force_eos_at_frame = 4
    inp = synth.make_inputs(wl)
    full = oracle.run(wl, tiny_weights, inp, capture=False)
    assert full.get("frames")[1] == 4 and full.get("reason")[1] == oracle.REASON_EOS
    assert full.get("selections")[1] == 5 and full.get("predictor_runs")[1] == 4
    assert full.get("reason")[0] == oracle.REASON_LENGTH and full.get("frames")[0] == 12
    for r in (0, 2):
        alone = oracle.run(wl, tiny_weights, inp, rows=[r], capture=False)
        assert np.array_equal(alone.get("codes")[0], full.get("codes")[r])


def test_degenerate_rows(tiny_weights):
    """Rows at the edges of the loop, in one batch: a one-row prompt, EOS
    forced at selection 0 (the row ends with no frame: one selection, no
    predictor run, every code -1), max_frames = 1 (two selections, one
    predictor run, finish reason length) and no trailing text (tts_pad from
    the first step).  Each equals its own single-row run."""
    kw = dict(do_sample=1, temperature=1.0, top_k=0, top_p=1.0, cp_do_sample=1, min_new_tokens=20)
    rows = [RowSampling(max_frames=6, **kw), RowSampling(max_frames=6, force_eos_at_frame=0, **kw),
            RowSampling(max_frames=1, **kw), RowSampling(max_frames=6, **kw)]
    wl = Workload("edges", TINY, F32, 9, 4, [1, 5, 3, 4], [2, 2, 2, 0], 6, rows, 16, norm_std=0.1)
    inp = synth.make_inputs(wl)
    o = oracle.run(wl, tiny_weights, inp, capture=False)
    frames, reason = o.get("frames"), o.get("reason")
    sel, runs, codes = o.get("selections"), o.get("predictor_runs"), o.get("codes")
    assert frames[0] == 6 and reason[0] == oracle.REASON_LENGTH and sel[0] == 7 and runs[0] == 6
    assert frames[1] == 0 and reason[1] == oracle.REASON_EOS and sel[1] == 1 and runs[1] == 0
    assert np.all(codes[1] == -1)
    assert frames[2] == 1 and reason[2] == oracle.REASON_LENGTH and sel[2] == 2 and runs[2] == 1
    assert np.all(codes[2, 1:] == -1) and np.all(codes[2, 0] >= 0)
    assert frames[3] == 6 and reason[3] == oracle.REASON_LENGTH
    for r in range(4):
        alone = oracle.run(wl, tiny_weights, inp, rows=[r], capture=False)
        assert np.array_equal(alone.get("codes")[0], codes[r]), r


def test_teacher_forcing_reproduces_free_run(tiny_weights):
    wl = _tiny_wl(8, min_new_tokens=20)
    inp = synth.make_inputs(wl)
    free = oracle.run(wl, tiny_weights, inp, capture=True)
    t = oracle.teacher_from_codes(free.get("codes"), free.get("frames"), free.get("reason"), TINY.eos_id, 8)
    forced = oracle.run(wl, tiny_weights, inp, capture=True, teacher=t)
    assert np.array_equal(forced.get("codes"), free.get("codes"))
    assert np.array_equal(forced.get("talker_logits"), free.get("talker_logits"))


def test_bf16_mode_rounds_the_cache(tiny_weights):
    """The same (bf16-exact) weights in bf16 and fp32 mode differ only by the
    bf16 rounding of the K/V cache: a small but nonzero difference."""
    wl32 = _tiny_wl(3, min_new_tokens=20)
    inp = synth.make_inputs(wl32)
    wbf = {k: ({kk: (synth.round_bf16(vv) if vv.ndim >= 2 and kk.startswith("w") else vv) for kk, vv in v.items()}
               if isinstance(v, dict) else (synth.round_bf16(v) if v is not None and v.ndim >= 2 else v))
           for k, v in tiny_weights.items()}
    w32 = {k: ({kk: (synth.bf16_bits_to_f32(vv) if vv.dtype == np.uint16 else vv) for kk, vv in v.items()}
               if isinstance(v, dict) else (synth.bf16_bits_to_f32(v) if v is not None and v.dtype == np.uint16 else v))
           for k, v in wbf.items()}
    wlbf = dataclasses.replace(wl32, dtype=BF16)
    a = oracle.run(wl32, w32, inp, capture=True, frames=3)
    t = oracle.teacher_from_codes(a.get("codes"), a.get("frames"), a.get("reason"), TINY.eos_id, 3)
    b = oracle.run(wlbf, wbf, inp, capture=True, teacher=t)
    d = np.abs(a.get("talker_logits") - b.get("talker_logits")).max()
    assert 1e-6 < d < 0.02
