"""GPU parity of the frame loop against the oracle, through the C ABI."""
import dataclasses

import numpy as np
import pytest

import oracle
import synth
from synth import RowSampling, Workload, F32, BF16
from parity import run_gpu, compare, check_run_properties, TOL

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def q3():
    import torch
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    import speech_lm_decode_gb300 as m
    return m


def small_workload(dims, dtype, frames=12, seed=21):
    rows = [RowSampling(max_frames=frames),
            RowSampling(max_frames=frames, do_sample=1, temperature=0.9, top_k=8, top_p=0.9, cp_do_sample=1,
                        cp_temperature=0.8, cp_top_k=6, cp_top_p=0.95, seed=11),
            RowSampling(max_frames=frames, force_eos_at_frame=5),
            RowSampling(max_frames=frames - 3, do_sample=1, temperature=1.1, top_k=0, top_p=0.8, cp_do_sample=1,
                        min_new_tokens=30)]
    lens = [5, 9, 17, 3]
    return Workload("small", dims, dtype, seed, len(rows), lens, [3, 0, 5, 1], frames, rows,
                    max(lens) + frames + 3, norm_std=0.1)


def small_weights(wl, scale=10.0):
    w = synth.make_weights(wl.dims, wl.dtype, wl.weight_seed, norm_std=wl.norm_std)
    if scale != 1.0:
        # larger projections so that attention and the MLP shape the result
        for blk in ("talker", "cp"):
            for k in ("wqkv", "wo", "wgu", "wd"):
                a = w[blk][k]
                f = synth.bf16_bits_to_f32(a) if a.dtype == np.uint16 else a
                f = (f * scale).astype(np.float32)
                w[blk][k] = synth.round_bf16(f) if a.dtype == np.uint16 else f
    return w


@pytest.mark.parametrize("dims,dtype", [(synth.DIMS_SMALL, F32), (synth.DIMS_SMALL, BF16),
                                        (synth.DIMS_SMALL_PROJ, BF16), (synth.DIMS_SMALL_PROJ, F32)])
def test_small_model_parity(q3, dims, dtype):
    wl = small_workload(dims, dtype)
    w = small_weights(wl)
    inp = synth.make_inputs(wl)
    g = run_gpu(wl, q3.to_device_weights(w), inp, cap_rows=list(range(wl.batch)))
    assert g.frames[2] == 5 and g.reasons[2] == q3.Q3_FINISHED_EOS
    assert g.reasons[1] != q3.Q3_RUNNING and g.reasons[0] != q3.Q3_RUNNING
    s = compare(wl, w, inp, g)
    assert s["checked"] > 0.5 * s["decisions"]


def test_chunked_steps_equal_one_call_and_repeatable(q3):
    wl = small_workload(synth.DIMS_SMALL, BF16, frames=14)
    w = small_weights(wl)
    inp = synth.make_inputs(wl)
    dw = q3.to_device_weights(w)
    a = run_gpu(wl, dw, inp, cap_rows=[0, 1])
    b = run_gpu(wl, dw, inp, cap_rows=[0, 1], chunks=[5, 1, 8])
    assert np.array_equal(a.codes, b.codes)
    assert np.array_equal(a.frames, b.frames) and np.array_equal(a.reasons, b.reasons)
    assert np.array_equal(a.talker_logits, b.talker_logits, equal_nan=True)
    c = run_gpu(wl, dw, inp, cap_rows=[0, 1])
    assert np.array_equal(a.codes, c.codes)


def test_rows_do_not_interact(q3):
    wl = small_workload(synth.DIMS_SMALL, BF16)
    w = small_weights(wl)
    inp = synth.make_inputs(wl)
    dw = q3.to_device_weights(w)
    full = run_gpu(wl, dw, inp, cap_rows=[1])
    # row 1 alone (batch 1) gives the same codes: the noise counter carries the row index 1
    wl1 = dataclasses.replace(wl, batch=2, rows=[wl.rows[0], wl.rows[1]], prompt_lens=wl.prompt_lens[:2],
                              n_text=wl.n_text[:2])
    inp1 = dict(inp)
    po, to = inp["prompt_offsets"], inp["text_offsets"]
    inp1["prompt"] = inp["prompt"][:po[2]]
    inp1["prompt_offsets"] = po[:3]
    inp1["text"] = inp["text"][:to[2]]
    inp1["text_offsets"] = to[:3]
    part = run_gpu(wl1, dw, inp1, cap_rows=[1])
    assert np.array_equal(full.codes[:2], part.codes)


@pytest.mark.parametrize("idx", [1, 2, 3, 4, 5])
def test_full_size_workload(q3, idx):
    """Every workload at its full size, in the launch configuration the
    benchmark times.  The oracle follows the captured rows over the whole run
    (batch 256: the first and last rows over all 1024 frames, so attention is
    compared up to 1280 positions), and properties of every row are checked."""
    wl = synth.workload(idx)
    w = synth.make_weights(wl.dims, wl.dtype, wl.weight_seed)
    inp = synth.make_inputs(wl)
    rows = [0] if wl.batch == 1 else [0, wl.batch - 1]
    # batch 1 runs on the single-launch frame kernel (what the benchmark times)
    expect = q3.Q3_PATH_FRAME if wl.batch == 1 else q3.Q3_PATH_GRAPH
    g = run_gpu(wl, q3.to_device_weights(w), inp, cap_rows=rows, expect_path=expect)
    check_run_properties(wl, g)
    s = compare(wl, w, inp, g)
    s.pop("details", None)
    # most decisions are far from a tie: a margin that collapsed toward zero
    # would leave the codes unchecked
    assert s["checked"] >= 0.5 * s["decisions"], s
    print(f"workload {idx}: frames {g.frames[rows].tolist()} reasons {g.reasons[rows].tolist()} {s}")


@pytest.mark.parametrize("idx,upto", [(6, None), (7, 48)])
def test_full_size_17b_batches(q3, idx, upto):
    """The 1.7B shape (talker hidden 2048, FFN 6144, 2048->1024 predictor
    projection) at batch 32 and batch 256, full size, in the benchmark's
    launch configuration: rows 0 and B-1 against the oracle (batch 256: over
    the first 48 frames), properties of every row."""
    wl = synth.workload(idx)
    w = synth.make_weights(wl.dims, wl.dtype, wl.weight_seed)
    inp = synth.make_inputs(wl)
    rows = [0, wl.batch - 1]
    g = run_gpu(wl, q3.to_device_weights(w), inp, cap_rows=rows, expect_path=q3.Q3_PATH_GRAPH)
    check_run_properties(wl, g)
    s = compare(wl, w, inp, g, upto=upto)
    s.pop("details", None)
    assert s["checked"] >= 0.5 * s["decisions"], s
    print(f"workload {idx}: frames {g.frames[rows].tolist()} reasons {g.reasons[rows].tolist()} {s}")


def test_capacity_and_state_errors(q3):
    wl = small_workload(synth.DIMS_SMALL, BF16)
    w = small_weights(wl, 1.0)
    inp = synth.make_inputs(wl)
    q = q3.Q3TTS(wl.dims, wl.dtype, q3.to_device_weights(w), wl.batch, wl.max_ctx, 8)
    rc, *_ = q.step_frames(1, check=False)
    assert rc == q3.Q3_ERR_STATE
    rows = [dataclasses.replace(r, max_frames=wl.max_ctx) for r in wl.rows]
    rc, _ = q.prefill(inp["prompt"], inp["prompt_offsets"], inp["text"], inp["text_offsets"], inp["tts_pad"], rows,
                      check=False)
    assert rc == q3.Q3_ERR_CAPACITY
    q.close()


def test_nan_logits_fail_closed(q3):
    wl = small_workload(synth.DIMS_SMALL, F32, frames=4)
    w = small_weights(wl, 1.0)
    w["codec_head"][7, 3] = np.nan      # every talker logit row then holds a NaN
    inp = synth.make_inputs(wl)
    q = q3.Q3TTS(wl.dims, wl.dtype, q3.to_device_weights(w), wl.batch, wl.max_ctx, 8)
    rc, code0 = q.prefill(inp["prompt"], inp["prompt_offsets"], inp["text"], inp["text_offsets"], inp["tts_pad"],
                          wl.rows, check=False)
    assert rc == q3.Q3_ERR_NAN
    rc, codes, frames, reasons = q.step_frames(2, check=False)
    assert np.all(reasons == q3.Q3_FINISHED_ERROR) and np.all(frames == 0) and np.all(codes == -1)
    q.close()


def _single_row(wl, r):
    """Row r of a workload as its own batch-1 workload (noise row index 0)."""
    rows = [wl.rows[r]]
    return dataclasses.replace(wl, batch=1, rows=rows, prompt_lens=[wl.prompt_lens[r]], n_text=[wl.n_text[r]])


def _single_inputs(inp, r):
    po, to = inp["prompt_offsets"], inp["text_offsets"]
    return {"prompt": inp["prompt"][po[r]:po[r + 1]], "prompt_offsets": np.array([0, po[r + 1] - po[r]], np.int32),
            "text": inp["text"][to[r]:to[r + 1]], "text_offsets": np.array([0, to[r + 1] - to[r]], np.int32),
            "tts_pad": inp["tts_pad"]}


@pytest.mark.parametrize("path", ["frame", "graph"])
@pytest.mark.parametrize("dims,dtype", [(synth.DIMS_SMALL, BF16), (synth.DIMS_SMALL, F32),
                                        (synth.DIMS_SMALL_PROJ, BF16)])
def test_batch1_paths_parity(q3, dims, dtype, path):
    """Batch 1 on the single-launch frame kernel (epoch-tagged exchange words)
    and on the per-layer kernels, each forced through the config; both match
    the oracle."""
    p = q3.Q3_PATH_FRAME if path == "frame" else q3.Q3_PATH_GRAPH
    wl = small_workload(dims, dtype, frames=10)
    w = small_weights(wl)
    inp = synth.make_inputs(wl)
    dw = q3.to_device_weights(w)
    for r in range(wl.batch):
        wl1, inp1 = _single_row(wl, r), _single_inputs(inp, r)
        g = run_gpu(wl1, dw, inp1, cap_rows=[0], step_path=p, expect_path=p)
        compare(wl1, w, inp1, g)


@pytest.mark.parametrize("dtype", [BF16, F32])
def test_separate_projections(q3, dtype):
    """q/k/v and gate/up as separate products (the unstacked layout): parity
    with the oracle at batch > 1 (tensor-core prefill, GEMV steps), and on the
    per-layer path without tensor cores the same codes and logits bit for bit
    as the stacked products (every output row is the same dot product)."""
    wl = small_workload(synth.DIMS_SMALL, dtype, frames=8)
    w = small_weights(wl)
    inp = synth.make_inputs(wl)
    dw = q3.to_device_weights(w)
    g = run_gpu(wl, dw, inp, cap_rows=[0, wl.batch - 1], separate_projections=1)
    compare(wl, w, inp, g)
    wl1, inp1 = _single_row(wl, 0), _single_inputs(inp, 0)
    a = run_gpu(wl1, dw, inp1, cap_rows=[0], step_path=q3.Q3_PATH_GRAPH, tc_min_tokens=-1)
    b = run_gpu(wl1, dw, inp1, cap_rows=[0], step_path=q3.Q3_PATH_GRAPH, tc_min_tokens=-1, separate_projections=1)
    assert np.array_equal(a.codes, b.codes)
    assert np.array_equal(a.talker_logits, b.talker_logits, equal_nan=True)
    assert np.array_equal(a.cp_logits, b.cp_logits, equal_nan=True)


def test_frame_kernel_chunked_and_repeatable(q3):
    wl = _single_row(small_workload(synth.DIMS_SMALL, BF16, frames=14), 1)
    w = small_weights(wl)
    inp = _single_inputs(synth.make_inputs(small_workload(synth.DIMS_SMALL, BF16, frames=14)), 1)
    dw = q3.to_device_weights(w)
    opts = dict(step_path=q3.Q3_PATH_FRAME, expect_path=q3.Q3_PATH_FRAME)
    a = run_gpu(wl, dw, inp, cap_rows=[0], **opts)
    b = run_gpu(wl, dw, inp, cap_rows=[0], chunks=[3, 4, 7], **opts)
    c = run_gpu(wl, dw, inp, cap_rows=[0], **opts)
    assert np.array_equal(a.codes, b.codes) and np.array_equal(a.codes, c.codes)
    assert np.array_equal(a.talker_logits, c.talker_logits, equal_nan=True)


@pytest.mark.parametrize("dims", [synth.DIMS_CL, synth.DIMS_CL_PROJ], ids=["same-width", "projection"])
def test_cluster_kernel_parity(q3, dims):
    """Batch 1 on the cluster kernel (8 clusters x 8 CTAs, one per KV head),
    every row of the small workload (greedy, sampled with top-k / top-p,
    forced EOS, min_new_tokens) against the oracle."""
    wl = small_workload(dims, BF16, frames=10)
    w = small_weights(wl)
    inp = synth.make_inputs(wl)
    dw = q3.to_device_weights(w)
    checked = decisions = 0
    for r in range(wl.batch):
        wl1, inp1 = _single_row(wl, r), _single_inputs(inp, r)
        g = run_gpu(wl1, dw, inp1, cap_rows=[0], step_path=q3.Q3_PATH_CLUSTER, expect_path=q3.Q3_PATH_CLUSTER)
        s = compare(wl1, w, inp1, g)
        checked += s["checked"]
        decisions += s["decisions"]
    # 1024-way vocabularies leave closer top-2 logits than the 64-way ones of
    # the other small shapes: a lower floor, still far from a collapsed margin
    assert checked >= 0.3 * decisions, (checked, decisions)


def test_cluster_kernel_chunked_and_repeatable(q3):
    """Calls of 3 + 4 + 7 frames give the codes of one 14-frame call, and a
    second run repeats the first bit for bit (fixed reduction orders)."""
    full = small_workload(synth.DIMS_CL, BF16, frames=14)
    wl = _single_row(full, 1)
    w = small_weights(wl)
    inp = _single_inputs(synth.make_inputs(full), 1)
    dw = q3.to_device_weights(w)
    opts = dict(step_path=q3.Q3_PATH_CLUSTER, expect_path=q3.Q3_PATH_CLUSTER)
    a = run_gpu(wl, dw, inp, cap_rows=[0], **opts)
    b = run_gpu(wl, dw, inp, cap_rows=[0], chunks=[3, 4, 7], **opts)
    c = run_gpu(wl, dw, inp, cap_rows=[0], **opts)
    assert np.array_equal(a.codes, b.codes) and np.array_equal(a.codes, c.codes)
    assert np.array_equal(a.talker_logits, c.talker_logits, equal_nan=True)
    assert np.array_equal(a.cp_logits, c.cp_logits, equal_nan=True)


@pytest.mark.parametrize("path", ["frame", "cluster"])
def test_batch1_wait_timeout(q3, path):
    """A device-side wait that runs out, on each single-launch path: the
    readers of one phase (frame kernel) or one cross-cluster exchange (cluster
    kernel) wait for words nobody writes (test-only config field), every wait
    gives up after the configured 2 ms, the step returns Q3_ERR_TIMEOUT and the
    handle can be destroyed; a fresh handle on the same GPU then matches the
    oracle."""
    if path == "frame":
        dims, p, inject = synth.DIMS_SMALL, q3.Q3_PATH_FRAME, 3
    else:
        dims, p, inject = synth.DIMS_CL, q3.Q3_PATH_CLUSTER, 3
    wl = _single_row(small_workload(dims, BF16, frames=6), 0)
    w = small_weights(wl)
    inp = _single_inputs(synth.make_inputs(small_workload(dims, BF16, frames=6)), 0)
    dw = q3.to_device_weights(w)
    q = q3.Q3TTS(wl.dims, wl.dtype, dw, 1, wl.max_ctx, 8, step_path=p, wait_limit_us=2000, inject_timeout=inject)
    assert q.step_path(1) == p
    q.prefill(inp["prompt"], inp["prompt_offsets"], inp["text"], inp["text_offsets"], inp["tts_pad"], wl.rows)
    rc, codes, frames, reasons = q.step_frames(2, check=False)
    assert rc == q3.Q3_ERR_TIMEOUT, rc
    assert frames[0] == 0 and reasons[0] == q3.Q3_RUNNING
    q.close()
    g = run_gpu(wl, dw, inp, cap_rows=[0], step_path=p, expect_path=p)
    compare(wl, w, inp, g)


def test_prefill_attention_tiles(q3):
    """Prompt lengths around the 64-token attention tiles (1, 63, 64, 65, 130,
    200) in one batch: 523 prompt tokens, so one row straddles the 512-token
    prefill chunks.  Every selection's logits depend on the prompt's K / V."""
    lens = [1, 63, 64, 65, 130, 200]
    rows = [RowSampling(max_frames=4) for _ in lens]
    rows[1] = RowSampling(max_frames=4, do_sample=1, temperature=0.9, top_k=8, cp_do_sample=1, seed=5)
    wl = Workload("prefill tiles", synth.DIMS_SMALL, BF16, 23, len(lens), lens, [2] * len(lens), 4, rows,
                  max(lens) + 8, norm_std=0.1)
    w = small_weights(wl)
    inp = synth.make_inputs(wl)
    g = run_gpu(wl, q3.to_device_weights(w), inp, cap_rows=list(range(len(lens))))
    compare(wl, w, inp, g)
