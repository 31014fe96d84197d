"""Helpers shared by the GPU parity tests: run a workload through the C ABI
with logit capture, run the oracle teacher-forced on the GPU's codes, and
compare element by element."""
from __future__ import annotations

import dataclasses

import numpy as np

import oracle
import synth

# Logit tolerances of the frame loop: fp32 model and bf16 model.
TOL = {synth.F32: 1e-4, synth.BF16: 3e-2}
MARGIN = 0.05   # codes must agree wherever the oracle's top-1 margin exceeds this


@dataclasses.dataclass
class GpuRun:
    code0: np.ndarray
    codes: np.ndarray
    frames: np.ndarray
    reasons: np.ndarray
    talker_logits: np.ndarray   # [n_cap, T+1, V]
    cp_logits: np.ndarray       # [n_cap, T, G-1, cpV]
    cap_rows: list
    path: int = 0               # step path that ran (Q3_PATH_*)


def run_gpu(wl, dev_weights, inputs, cap_rows, chunks=None, expect_path=None, **exec_opts):
    """exec_opts: config execution fields (step_path, ...); expect_path: the
    batch-1 step path the handle must report (checked when given)."""
    import torch
    import speech_lm_decode_gb300 as q3
    d = wl.dims
    T = wl.frames
    import os
    import sys
    verbose = os.environ.get("Q3TTS_VERBOSE") == "1"

    def log(msg):
        if verbose:
            print(f"[run_gpu] {msg}", file=sys.stderr, flush=True)
    q = q3.Q3TTS(d, wl.dtype, dev_weights, wl.batch, wl.max_ctx, max(max(wl.n_text), 1), **exec_opts)
    log("handle created")
    path = q.step_path(wl.batch)
    if expect_path is not None:
        assert path == expect_path, (q3.PATH_NAMES.get(path), q3.PATH_NAMES.get(expect_path))
    tl = torch.full((len(cap_rows), T + 1, d.codec_vocab), float("nan"), device="cuda")
    cl = torch.full((len(cap_rows), max(T, 1), d.n_groups - 1, d.cp_vocab), float("nan"), device="cuda")
    q.set_capture(cap_rows, tl, cl, T)
    code0 = q.prefill(inputs["prompt"], inputs["prompt_offsets"], inputs["text"], inputs["text_offsets"],
                      inputs["tts_pad"], wl.rows)
    log(f"prefill done: {code0.tolist()[:4]}")
    parts = []
    frames = reasons = None
    for n in (chunks or [T]):
        c, frames, reasons = q.step_frames(n)
        log(f"step_frames({n}) done")
        parts.append(c)
    codes = np.concatenate(parts, axis=1)
    torch.cuda.synchronize()
    out = GpuRun(code0, codes, frames, reasons, tl.cpu().numpy(), cl.cpu().numpy(), list(cap_rows), path)
    q.close()
    return out


def compare(wl, weights, inputs, g: GpuRun, tol=None, margin=MARGIN, report=None, upto=None):
    """Teacher-force the oracle on the GPU's codes for the captured rows and
    check frames, finish reasons, logits (<= tol) and decisions (where the
    oracle's margin > margin).  upto: compare only frames [0, upto) (the
    oracle then stops there).  Returns a summary dict."""
    tol = TOL[wl.dtype] if tol is None else tol
    T = wl.frames if upto is None else min(upto, wl.frames)
    d = wl.dims
    rows = g.cap_rows
    # the GPU run seen through a window of T frames
    gf = np.minimum(g.frames, T)
    gr = np.where((g.frames < T) | ((g.frames == T) & (g.reasons == oracle.REASON_EOS)), g.reasons,
                  oracle.REASON_LENGTH)
    wl_o = dataclasses.replace(wl, frames=T, rows=[dataclasses.replace(r, max_frames=min(r.max_frames, T))
                                                   for r in wl.rows])
    teacher = oracle.teacher_from_codes(g.codes[rows][:, :T], gf[rows], gr[rows], d.eos_id, T)
    o = oracle.run(wl_o, weights, inputs, rows=rows, teacher=teacher, capture=True)
    of, orr = o.get("frames"), o.get("reason")
    otl, ocl = o.get("talker_logits"), o.get("cp_logits")
    own_sel, sel_m = o.get("own_sel"), o.get("sel_margin")
    own_cp, cp_m = o.get("own_cp"), o.get("cp_margin")
    worst_t = worst_c = 0.0
    n_dec = n_checked = n_mismatch = 0
    details = []
    for i, r in enumerate(rows):
        nf = int(gf[r])
        assert int(of[i]) == nf, (r, of[i], nf)
        assert int(orr[i]) == int(gr[r]), (r, orr[i], gr[r])
        forced = wl.rows[r].force_eos_at_frame
        # talker selections 0..nf
        for k in range(nf + 1):
            a, b = g.talker_logits[i, k], otl[i, k]
            fin = np.isfinite(b)
            dt = float(np.max(np.abs(a[fin] - b[fin])))
            worst_t = max(worst_t, dt)
            if k < nf:
                gsel = int(g.codes[r, k, 0])
            elif int(gr[r]) == oracle.REASON_EOS and k != forced:
                gsel = d.eos_id
            else:
                continue
            if k == forced:
                continue
            n_dec += 1
            if sel_m[i, k] > margin:
                n_checked += 1
                if int(own_sel[i, k]) != gsel:
                    n_mismatch += 1
                    o_id = int(own_sel[i, k])
                    details.append(("talker", r, k, gsel, o_id, round(float(sel_m[i, k]), 4),
                                    float(g.talker_logits[i, k, gsel]), float(otl[i, k, gsel]),
                                    float(g.talker_logits[i, k, o_id]), float(otl[i, k, o_id])))
        for f in range(nf):
            for s in range(d.n_groups - 1):
                a, b = g.cp_logits[i, f, s], ocl[i, f, s]
                worst_c = max(worst_c, float(np.max(np.abs(a - b))))
                n_dec += 1
                if cp_m[i, f, s] > margin:
                    n_checked += 1
                    if int(own_cp[i, f, s]) != int(g.codes[r, f, s + 1]):
                        n_mismatch += 1
                        gid, o_id = int(g.codes[r, f, s + 1]), int(own_cp[i, f, s])
                        details.append(("cp", r, f, s, gid, o_id, round(float(cp_m[i, f, s]), 4),
                                        float(g.cp_logits[i, f, s, gid]), float(ocl[i, f, s, gid]),
                                        float(g.cp_logits[i, f, s, o_id]), float(ocl[i, f, s, o_id])))
    # the draws themselves are bit-exact: the oracle's processors + draw on the
    # GPU's own captured logits give the GPU's ids, at every decision
    n_exact, exact_bad = 0, []
    for i, r in enumerate(rows):
        nf = int(gf[r])
        sp = wl.rows[r]
        seen = np.zeros(d.codec_vocab, np.uint8)
        for k in range(nf + 1):
            if k < nf:
                gsel = int(g.codes[r, k, 0])
            elif int(gr[r]) == oracle.REASON_EOS:
                gsel = d.eos_id
            else:
                gsel = None
            if gsel is not None and k != sp.force_eos_at_frame:
                err, oid, _, _ = oracle.sample(g.talker_logits[i, k], sp, True, seen=seen, sel_index=k,
                                               eos=d.eos_id, sup_lo=d.suppress_lo, sup_hi=d.suppress_hi, row=r,
                                               frame=k, step=0)
                n_exact += 1
                if err or oid != gsel:
                    exact_bad.append(("talker", r, k, gsel, oid))
            if gsel is not None and 0 <= gsel < d.codec_vocab:
                seen[gsel] = 1
        for f in range(nf):
            for s in range(d.n_groups - 1):
                err, oid, _, _ = oracle.sample(g.cp_logits[i, f, s], sp, False, eos=-1, sup_lo=0, sup_hi=0, row=r,
                                               frame=f, step=s + 1)
                n_exact += 1
                if err or oid != int(g.codes[r, f, s + 1]):
                    exact_bad.append(("cp", r, f, s, int(g.codes[r, f, s + 1]), oid))
    summary = dict(worst_talker_logit=worst_t, worst_cp_logit=worst_c, decisions=n_dec, checked=n_checked,
                   mismatches=n_mismatch, tol=tol, draws_exact=n_exact, draws_exact_bad=len(exact_bad),
                   details=details[:8] + exact_bad[:8])
    if report is not None:
        report.update(summary)
    assert worst_t <= tol and worst_c <= tol, summary
    assert not exact_bad, summary
    assert n_mismatch == 0, summary
    return summary


def check_run_properties(wl, g: GpuRun):
    """Properties of a whole batch that hold at any size: codes in range for
    emitted frames and -1 after, finish reasons consistent with frame counts."""
    d = wl.dims
    assert np.all(g.reasons != 0), "every row must have finished"
    assert not np.any(g.reasons == 3), "no row may end on NaN logits"
    for r in range(wl.batch):
        nf = int(g.frames[r])
        sp = wl.rows[r]
        c = g.codes[r]
        assert np.all((c[:nf] >= 0) & (c[:nf] < d.cp_vocab)), r
        assert np.all(c[nf:] == -1), r
        if g.reasons[r] == oracle.REASON_LENGTH:
            assert nf == sp.max_frames, r
        else:
            assert nf < sp.max_frames or nf == sp.force_eos_at_frame or nf == sp.max_frames, r
            if sp.force_eos_at_frame >= 0:
                assert nf <= sp.force_eos_at_frame, r
