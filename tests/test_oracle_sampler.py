"""Pins for the oracle's logits processors and draw (CPU only).

Each test checks the oracle against something other than itself: published
known-answer vectors, the facts the pages state about the processor chain,
closed forms, or brute force over a tiny vocabulary.
"""
import ctypes
import json
import math
import os

import numpy as np
import pytest

import oracle
import synth
from synth import RowSampling

V = 3072
EOS = 2150


def sp(**kw):
    base = dict(repetition_penalty=1.0, min_new_tokens=0)
    base.update(kw)
    return RowSampling(**base)


def test_page_ids(golden_dir):
    facts = json.load(open(os.path.join(golden_dir, "page_facts.json")))
    d = synth.DIMS_06B
    assert facts["codec_special_ids"]["eos"] == d.eos_id == EOS
    assert facts["codec_special_ids"]["codec_vocab"] == d.codec_vocab
    assert facts["suppress"]["lo"] == d.suppress_lo and facts["suppress"]["hi_inclusive"] + 1 == d.suppress_hi
    assert facts["structure"]["predictor_tables"] == d.n_groups - 1
    assert facts["natural_eos_run"]["talker_selections"] == facts["natural_eos_run"]["frames"] + 1
    assert facts["natural_eos_run"]["predictor_runs"] == facts["natural_eos_run"]["frames"] * 15
    for k in ("natural_eos_run", "prefix_run", "two_frame_run", "ncnn_e2e_run"):
        f = facts[k]
        codes = f.get("codes", f.get("short_codes"))
        frames = f.get("frames", f.get("short_frames"))
        assert codes == 16 * frames


def test_philox_known_answers(golden_dir):
    L = oracle.lib()
    n = 0
    for line in open(os.path.join(golden_dir, "philox4x32_10_kat.txt")):
        if line.startswith("#") or not line.strip():
            continue
        v = [int(x, 16) for x in line.split()]
        ctr = np.array(v[0:4], np.uint32)
        key = np.array(v[4:6], np.uint32)
        out = np.zeros(4, np.uint32)
        L.oracle_philox(ctr.ctypes.data, key.ctypes.data, out.ctypes.data)
        assert list(out) == v[6:10]
        n += 1
    assert n == 3


def test_spec_exp_error_bound():
    L = oracle.lib()
    xs = np.concatenate([np.linspace(-86, 0, 20001), -np.geomspace(1e-8, 86, 5000)]).astype(np.float32)
    got = np.array([L.oracle_spec_expf(float(x)) for x in xs], np.float64)
    ref = np.exp(xs.astype(np.float64))
    assert np.max(np.abs(got - ref) / ref) < 2.5e-7      # about 2 ulp of fp32
    assert L.oracle_spec_expf(0.0) == 1.0
    assert L.oracle_spec_expf(-87.0) == 0.0
    # monotone on a fine grid (the draw relies on w ordering following l ordering)
    grid = np.linspace(-20, 0, 4001).astype(np.float32)
    g = np.array([L.oracle_spec_expf(float(x)) for x in grid])
    assert np.all(np.diff(g) >= 0)


def test_spec_log_error_bound():
    L = oracle.lib()
    us = np.concatenate([np.linspace(2 ** -24, 1 - 2 ** -24, 20001), np.geomspace(2 ** -24, 0.999, 5000)])
    us = us.astype(np.float32)
    got = np.array([L.oracle_spec_logf(float(u)) for u in us], np.float64)
    ref = np.log(us.astype(np.float64))
    assert np.max(np.abs(got - ref) / np.abs(ref)) < 4e-7
    assert L.oracle_spec_logf(0.5) == pytest.approx(-math.log(2), rel=1e-7)


def test_noise_uniform_properties():
    L = oracle.lib()
    us = np.array([L.oracle_noise_uniform(7, 0, 0, 0, t) for t in range(20000)], np.float64)
    assert us.min() > 0 and us.max() < 1
    scaled = us * 2 ** 24
    assert np.all(scaled == np.round(scaled)) and np.all(scaled.astype(np.int64) % 2 == 1)
    assert abs(us.mean() - 0.5) < 0.01
    # each counter component changes the draw
    a = L.oracle_noise_uniform(7, 1, 2, 3, 4)
    for args in [(8, 1, 2, 3, 4), (7, 0, 2, 3, 4), (7, 1, 0, 3, 4), (7, 1, 2, 0, 4), (7, 1, 2, 3, 0)]:
        assert L.oracle_noise_uniform(*args) != a


def test_greedy_ties_go_to_lowest_index():
    lg = np.zeros(V, np.float32)
    lg[[17, 5, 900]] = 3.0
    err, idx, margin, _ = oracle.sample(lg, sp(), talker=True)
    assert err == 0 and idx == 5 and margin == 0.0
    err, idx, _, _ = oracle.sample(lg[:2048], sp(), talker=False, eos=-1, sup_lo=0, sup_hi=0)
    assert idx == 5


@pytest.mark.parametrize("bad", [np.nan, np.inf])
def test_nan_fails_closed(bad):
    lg = np.random.default_rng(0).standard_normal(V).astype(np.float32)
    lg[1234] = bad
    for do_sample in (0, 1):
        err, _, _, _ = oracle.sample(lg, sp(do_sample=do_sample), talker=True)
        assert err == oracle.ERR_NAN
    lg[1234] = -np.inf   # -inf is a legal (masked) logit
    assert oracle.sample(lg, sp(), talker=True)[0] == 0


def test_min_new_tokens_masks_eos_then_next_best():
    lg = np.linspace(-1, 1, V).astype(np.float32)[::-1].copy()  # id 0 is the best code
    lg[EOS] = 5.0
    lg[7] = 4.0
    s = sp(min_new_tokens=2)
    for k, want in ((0, 7), (1, 7), (2, EOS), (3, EOS)):
        err, idx, _, proc = oracle.sample(lg, s, talker=True, sel_index=k)
        assert err == 0 and idx == want
        assert (proc[EOS] == -np.inf) == (k < 2)


def test_suppression_keeps_eos_only():
    lg = np.random.default_rng(1).standard_normal(V).astype(np.float32)
    lg[2500] = 10.0
    err, idx, _, proc = oracle.sample(lg, sp(), talker=True)
    assert idx != 2500 and idx < 2048 or idx == EOS
    sup = np.r_[2048:3072]
    sup = sup[sup != EOS]
    assert np.all(proc[sup] == -np.inf)
    assert proc[EOS] == lg[EOS]
    assert np.array_equal(proc[:2048], lg[:2048])
    # the predictor has no suppression: id 2047 can win there
    lg2 = np.zeros(2048, np.float32)
    lg2[2047] = 1.0
    assert oracle.sample(lg2, sp(), talker=False, eos=-1, sup_lo=0, sup_hi=0)[1] == 2047


def test_repetition_penalty_is_sign_aware():
    rng = np.random.default_rng(2)
    lg = rng.standard_normal(V).astype(np.float32)
    seen = np.zeros(V, np.uint8)
    ids = rng.choice(2048, 200, replace=False)
    seen[ids] = 1
    pen = np.float32(1.05)
    err, _, _, proc = oracle.sample(lg, sp(repetition_penalty=1.05), talker=True, seen=seen)
    want = lg.copy()
    want[ids] = np.where(lg[ids] < 0, lg[ids] * pen, lg[ids] / pen).astype(np.float32)
    sup = np.r_[2048:3072]
    want[sup[sup != EOS]] = -np.inf
    assert np.array_equal(proc, want)
    # a seen id with the top logit loses to a close unseen one
    lg = np.zeros(V, np.float32)
    lg[10], lg[11] = 1.00, 0.97
    seen = np.zeros(V, np.uint8)
    seen[10] = 1
    assert oracle.sample(lg, sp(repetition_penalty=1.05), talker=True, seen=seen)[1] == 11
    assert oracle.sample(lg, sp(repetition_penalty=1.0), talker=True, seen=seen)[1] == 10
    # negative logits move away from zero (become less likely)
    lg = np.full(V, -5.0, np.float32)
    lg[3], lg[4] = -1.00, -1.03
    seen[:] = 0
    seen[3] = 1
    assert oracle.sample(lg, sp(repetition_penalty=1.05), talker=True, seen=seen)[1] == 4


def _brute_kept(lg, T, top_k, top_p):
    """Kept set of temperature -> top-k -> top-p, by sorting in fp64."""
    l = lg.astype(np.float32) / np.float32(T)
    l = l.astype(np.float64)
    n = len(l)
    keep = np.ones(n, bool)
    if 0 < top_k < n:
        kth = np.sort(l)[::-1][top_k - 1]
        keep &= l >= kth
    order = sorted(np.nonzero(keep)[0], key=lambda i: (-l[i], i))
    p = np.exp(l[order] - l[order[0]])
    p /= p.sum()
    if top_p < 1:
        c = np.concatenate([[0.0], np.cumsum(p)[:-1]])
        ok = (c < top_p)
        ok[0] = True
        # avoid sets whose boundary sits within rounding of top_p
        assert np.all(np.abs(c - top_p) > 1e-6)
        order = [i for i, o in zip(order, ok) if o]
    q = np.exp(l[order] - l[order[0]])
    return np.array(order), q / q.sum()


@pytest.mark.parametrize("T,top_k,top_p", [(1.0, 0, 1.0), (0.9, 5, 1.0), (0.7, 0, 0.8), (1.3, 6, 0.9)])
def test_draw_follows_kept_softmax(T, top_k, top_p):
    Vs = 12
    rng = np.random.default_rng(3)
    lg = (rng.standard_normal(Vs) * 0.8).astype(np.float32)
    kept, p = _brute_kept(lg, T, top_k, top_p)
    s = sp(do_sample=1, temperature=T, top_k=top_k, top_p=top_p, cp_do_sample=1, cp_temperature=T, cp_top_k=top_k,
           cp_top_p=top_p)
    n = 40000
    counts = np.zeros(Vs, np.int64)
    for f in range(n):
        err, idx, _, _ = oracle.sample(lg, s, talker=False, eos=-1, sup_lo=0, sup_hi=0, row=1, frame=f, step=3)
        assert err == 0
        counts[idx] += 1
    assert set(np.nonzero(counts)[0]) == set(kept.tolist())
    exp = p * n
    chi2 = float(np.sum((counts[kept] - exp) ** 2 / exp))
    dof = len(kept) - 1
    # 1e-4 upper tail of chi2(dof) is below dof + 8*sqrt(2 dof) + 20 for dof <= 12
    assert chi2 < dof + 8 * math.sqrt(2 * max(dof, 1)) + 20, (chi2, dof)


def test_topk_keeps_ties_at_threshold():
    lg = np.array([3, 2, 2, 2, 1, 0], np.float32)
    s = sp(do_sample=1, top_k=2, cp_do_sample=1, cp_top_k=2)
    seen_ids = set()
    for f in range(3000):
        seen_ids.add(oracle.sample(lg, s, talker=False, eos=-1, sup_lo=0, sup_hi=0, frame=f)[1])
    assert seen_ids == {0, 1, 2, 3}


def test_same_seed_same_draws_and_seed_matters():
    rng = np.random.default_rng(4)
    lg = rng.standard_normal(V).astype(np.float32)
    s1 = sp(do_sample=1, temperature=0.9, top_k=50, top_p=0.95, seed=7)
    s2 = sp(do_sample=1, temperature=0.9, top_k=50, top_p=0.95, seed=8)
    a = [oracle.sample(lg, s1, True, frame=f)[1] for f in range(200)]
    b = [oracle.sample(lg, s1, True, frame=f)[1] for f in range(200)]
    c = [oracle.sample(lg, s2, True, frame=f)[1] for f in range(200)]
    assert a == b and a != c


def _cp_draws(lg, n, **kw):
    s = sp(do_sample=1, cp_do_sample=1, **{k: v for k, v in kw.items()},
           **{"cp_" + k: v for k, v in kw.items()})
    out = []
    for f in range(n):
        err, idx, _, _ = oracle.sample(lg, s, talker=False, eos=-1, sup_lo=0, sup_hi=0, row=2, frame=f, step=5)
        assert err == 0
        out.append(idx)
    return out


def test_degenerate_settings_reduce_to_greedy():
    """top-k 1 on a unique maximum, or a top-p below the largest probability,
    leaves only the argmax: every draw is the greedy choice.  With a tie at the
    top, top-k 1 keeps both tied ids (ties at the k-th value are kept) while a
    tiny top-p keeps only the first in (value desc, index asc) order."""
    rng = np.random.default_rng(11)
    lg = rng.standard_normal(64).astype(np.float32)
    lg[17] = lg.max() + 0.25
    greedy = oracle.sample(lg, sp(), talker=False, eos=-1, sup_lo=0, sup_hi=0)[1]
    assert greedy == 17
    assert set(_cp_draws(lg, 300, temperature=1.3, top_k=1, top_p=1.0)) == {17}
    assert set(_cp_draws(lg, 300, temperature=0.8, top_k=0, top_p=1e-4)) == {17}
    lg[40] = lg[17]                    # tie at the top
    assert oracle.sample(lg, sp(), talker=False, eos=-1, sup_lo=0, sup_hi=0)[1] == 17
    assert set(_cp_draws(lg, 300, temperature=1.3, top_k=1, top_p=1.0)) == {17, 40}
    assert set(_cp_draws(lg, 300, temperature=0.8, top_k=0, top_p=1e-4)) == {17}


def test_unbounded_settings_keep_everything():
    """top-k >= V and top-p = 1 keep the whole vocabulary: over many draws on
    near-flat logits every id shows up, exactly as with both filters off."""
    lg = np.linspace(0.0, 0.05, 16).astype(np.float32)
    a = _cp_draws(lg, 2000, temperature=1.0, top_k=16, top_p=1.0)
    b = _cp_draws(lg, 2000, temperature=1.0, top_k=0, top_p=1.0)
    c = _cp_draws(lg, 2000, temperature=1.0, top_k=1000, top_p=1.0)
    assert set(a) == set(range(16))
    assert a == b == c      # the same noise and the same kept set give the same ids


def test_top_p_keeps_the_smallest_prefix():
    """Softmax mass 0.45 on id 2, 0.44 on id 7, 0.011 on each of the other ten:
    top-p 0.4 keeps only id 2 (the mass before id 7 is 0.45 >= 0.4), top-p 0.5
    keeps ids 2 and 7 (0.45 < 0.5; the mass before the next is 0.89), and the
    rest never appear."""
    p = np.full(12, 0.011)
    p[2], p[7] = 0.45, 0.44
    lg = np.log(p).astype(np.float32)
    assert set(_cp_draws(lg, 400, temperature=1.0, top_k=0, top_p=0.4)) == {2}
    assert set(_cp_draws(lg, 400, temperature=1.0, top_k=0, top_p=0.5)) == {2, 7}


# ---------------------------------------------------------------- decision margin
# Reading of "codes must agree where the top-1 margin exceeds 0.05" for sampled
# draws (a draw whose kept set a 0.05 logit perturbation could change is not
# a decision the tolerance can hold to): the winner's log-score lead over every
# id a small perturbation could keep -- the kept ids and the ids within 0.05 of
# the top-k threshold or of the top-p boundary -- and, when the winner itself
# survives top-k or top-p only narrowly, its distance to that boundary.  Each
# case below is built so that one specific term sets the margin; the noise
# values come from the Philox generator pinned above, and the scores are
# recomputed here with the math library.

def _E(seed, step, i, row=0, frame=0):
    u = oracle.lib().oracle_noise_uniform(seed, row, frame, step, i)
    assert 0.0 < u < 1.0
    return -math.log(u)


def _scores(l, ids, seed, step):
    mx = max(float(l[i]) for i in ids)
    return {i: math.exp(float(l[i]) - mx) / _E(seed, step, i) for i in ids}


def _draw(l, seed, step, top_k=0, top_p=1.0):
    # a predictor draw (no penalty, suppression or min_new): its cp_* settings apply
    s = sp(do_sample=1, temperature=1.0, seed=seed, top_k=top_k, top_p=top_p, cp_do_sample=1, cp_temperature=1.0,
           cp_top_k=top_k, cp_top_p=top_p)
    err, oid, margin, _ = oracle.sample(np.asarray(l, np.float32), s, False, row=0, frame=0, step=step)
    assert err == 0
    return oid, margin


def _seed_where(pred, step, limit=400):
    for seed in range(limit):
        if pred(seed):
            return seed
    raise AssertionError("no seed in range satisfies the case")


def test_margin_score_ratio_without_filters():
    """No top-k / top-p: every id is a competitor; the margin is the winner's
    smallest log-score lead."""
    l = np.array([0.0, 0.3, -0.2, 0.1], np.float32)
    for seed in (1, 2, 3, 11, 40):
        sc = _scores(l, range(4), seed, 5)
        best = max(range(4), key=lambda i: (sc[i], -i))
        want = min(math.log(sc[best] / sc[i]) for i in range(4) if i != best)
        oid, margin = _draw(l, seed, 5)
        assert oid == best
        assert margin >= 0.0 and abs(margin - want) < 1e-5, (seed, margin, want)


def test_margin_counts_an_id_just_outside_top_k():
    """top-k 1 keeps id 0 only; id 1 sits 0.03 below the threshold, so a
    perturbation could keep it: its score counts, and so does the winner's
    distance to the next logit below the threshold."""
    l = np.array([10.0, 9.97, 0.0], np.float32)
    gap = float(np.float32(10.0)) - float(np.float32(9.97))
    # noise where id 1 would have outscored the winner: the score term binds
    seed = _seed_where(lambda s: _E(s, 2, 1) < _E(s, 2, 0), 2)
    sc = _scores(l, [0, 1], seed, 2)
    oid, margin = _draw(l, seed, 2, top_k=1)
    assert oid == 0
    assert abs(margin - math.log(sc[0] / sc[1])) < 1e-5 and margin < gap
    # noise where it would not: the threshold distance binds
    seed = _seed_where(lambda s: _E(s, 2, 1) > _E(s, 2, 0), 2)
    oid, margin = _draw(l, seed, 2, top_k=1)
    assert oid == 0 and abs(margin - gap) < 1e-6


def test_margin_counts_an_id_just_outside_top_p():
    """Three equal logits with top-p 0.665: ids 0 and 1 are kept, id 2 falls
    out with its prefix sum 0.25 % above the boundary, so it stays a
    competitor; chosen noise makes it the closest one."""
    l = np.zeros(3, np.float32)

    def case(s):
        E = [_E(s, 4, i) for i in range(3)]
        best = 0 if E[0] <= E[1] else 1
        other = 1 - best
        return E[2] < E[other] and E[2] > E[best]
    seed = _seed_where(case, 4)
    E = [_E(seed, 4, i) for i in range(3)]
    best = 0 if E[0] <= E[1] else 1
    oid, margin = _draw(l, seed, 4, top_p=0.665)
    assert oid == best
    assert abs(margin - math.log(E[2] / E[best])) < 1e-5
    assert margin < math.log(E[1 - best] / E[best])


def test_margin_of_a_winner_on_the_boundary():
    """The winner survives only narrowly: (a) top-p 0.51 over two equal logits
    keeps id 1 with its prefix sum 2 % under the boundary; (b) top-k 1 keeps id
    0 with a 0.01 lead over the next logit.  The margin is that distance."""
    l = np.zeros(2, np.float32)
    dist = math.log(2.0 * float(np.float32(0.51)))
    seed = _seed_where(lambda s: math.log(_E(s, 6, 0) / _E(s, 6, 1)) > dist, 6)
    oid, margin = _draw(l, seed, 6, top_p=0.51)
    assert oid == 1 and abs(margin - dist) < 1e-9
    l = np.array([1.0, 0.99, -3.0], np.float32)
    gap = float(np.float32(1.0)) - float(np.float32(0.99))
    seed = _seed_where(lambda s: _E(s, 7, 1) > _E(s, 7, 0) * 1.2, 7)
    oid, margin = _draw(l, seed, 7, top_k=1)
    assert oid == 0 and abs(margin - gap) < 1e-9
