"""Device-side fault reports: a NaN or infinite logit is reported in the
status word and never passes silently (fail-closed errors, "Ollama qwen3_5 MTP
loader and SelfDraft path", Facts; "support the qwen3_5_mtp drafter" issue,
Acceptance criteria).  Covered: spec_verify's greedy, cluster and streaming
paths (16-byte and 4-byte rows), mtp_draft's logits through the handle's word,
clean calls that must leave the word at zero, and the streaming path's bounded
waits made to run out through the test hook: the call reports a timeout,
writes in-range outputs, and the next call is exact again.  The faults are made
on the host (the logits are written with NaN or inf before the call)."""
import numpy as np
import pytest
import torch

import mtp_speculative_decoding_step_gb300 as m
import oracle
import synth
from tests import gpu_common as g

pytestmark = pytest.mark.gpu


def _verify(lg, drafts, params, u, q=None, hist=None, noalloc=False):
    R, dp1, V = lg.shape
    n_acc = torch.full((R,), -7, dtype=torch.int32, device="cuda")
    out = torch.full((R, dp1), -7, dtype=torch.int32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    args = (g.to_dev(lg), g.to_dev(np.ascontiguousarray(drafts, np.int32)), params,
            g.to_dev(np.ascontiguousarray(u, np.float32)), n_acc, out)
    kw = dict(q=None if q is None else g.to_dev(q), hist=None if hist is None else g.to_dev(hist), status=status)
    if noalloc:
        m.spec_verify_noalloc(*args, **kw)
    else:
        ws = torch.zeros(m.spec_verify_workspace_bytes(R, dp1 - 1, V), dtype=torch.uint8, device="cuda")
        m.spec_verify(*args, ws, **kw)
    torch.cuda.synchronize()
    return n_acc.cpu().numpy(), out.cpu().numpy(), int(status.item())


def _in_range(n, out, d, V):
    assert np.all((n >= 0) & (n <= d)), n
    for r in range(len(n)):
        assert np.all((out[r, :n[r] + 1] >= 0) & (out[r, :n[r] + 1] < V)), out[r]


def _greedy_case(R, d, V, seed):
    lg = synth.normal(seed, "st:lg", (R, d + 1, V), std=3.0)
    drafts = lg[:, :d].argmax(-1).astype(np.int32)
    return lg, drafts, np.zeros((R, d + 1), np.float32)


@pytest.mark.parametrize("bad", [np.nan, np.inf, -np.inf])
@pytest.mark.parametrize("noalloc", [False, True])
def test_greedy_verify_reports_nonfinite(bad, noalloc):
    R, d, V = 2, 3, 8192
    lg, drafts, u = _greedy_case(R, d, V, 61)
    n, out, st = _verify(lg, drafts, [dict(temperature=0.0)] * R, u, noalloc=noalloc)
    assert st == 0 and list(n) == [d] * R
    lg[1, 2, 517] = bad
    n, out, st = _verify(lg, drafts, [dict(temperature=0.0)] * R, u, noalloc=noalloc)
    assert st == g.NONFINITE
    _in_range(n, out, d, V)


def test_greedy_verify_all_nan_row_stays_in_range():
    R, d, V = 1, 2, 4096
    lg, drafts, u = _greedy_case(R, d, V, 62)
    lg[0, 0, :] = np.nan
    n, out, st = _verify(lg, drafts, [dict(temperature=0.0)], u)
    assert st == g.NONFINITE
    _in_range(n, out, d, V)


@pytest.mark.parametrize("bad", [np.nan, np.inf])
@pytest.mark.parametrize("noalloc", [False, True])
def test_cluster_verify_reports_nonfinite(bad, noalloc):
    # one sampled row at depth 2: three (row, position) tasks, the cluster path
    R, d, V = 1, 2, 8192
    lg = synth.normal(63, "st:clu", (R, d + 1, V), std=2.0)
    params = [dict(temperature=0.8, top_p=0.9, rep_penalty=1.1)]
    q = np.stack([oracle.transform(lg[0, i], oracle.make_params(0.8, rep_penalty=1.1, top_p=0.9),
                                   np.zeros(0, np.int32))[0] for i in range(d)])[None]
    drafts = q[0].argmax(-1).astype(np.int32)[None]
    u = synth.uniform(63, "st:u", (R, d + 1))
    n, out, st = _verify(lg, drafts, params, u, q=q, noalloc=noalloc)
    assert st == 0
    lg[0, 1, 4000] = bad
    n, out, st = _verify(lg, drafts, params, u, q=q, noalloc=noalloc)
    assert st == g.NONFINITE
    _in_range(n, out, d, V)


def _stream_case(V, seed):
    # 16 rows x depth 3 with top-k 40: more tasks than one wave of 8-CTA
    # clusters, so spec_verify takes the streaming path
    R, d = 16, 3
    lg = synth.normal(seed, "st:str", (R, d + 1, V), std=4.0)
    drafts = lg[:, :d].argmax(-1).astype(np.int32)
    params = [dict(temperature=0.8, top_k=40, top_p=0.95, min_p=0.05, argmax_draft=True)] * R
    u = synth.uniform(seed, "st:stru", (R, d + 1))
    return lg, drafts, params, u


@pytest.mark.parametrize("V", [32768, 32766])
@pytest.mark.parametrize("bad", [np.nan, np.inf])
def test_streaming_verify_reports_nonfinite(V, bad):
    # V = 32768 streams 16-byte rows through the bulk-copy ring; V = 32766
    # takes the 4-byte loads
    lg, drafts, params, u = _stream_case(V, 64)
    n0, out0, st = _verify(lg, drafts, params, u)
    assert st == 0
    lg[5, 3, V - 3] = bad
    n, out, st = _verify(lg, drafts, params, u)
    assert st == g.NONFINITE
    _in_range(n, out, 3, V)
    # rows without the bad logit are untouched
    keep = [r for r in range(16) if r != 5]
    assert np.array_equal(n[keep], n0[keep]) and np.array_equal(out[keep], out0[keep])


def test_streaming_verify_wait_runs_out_and_reports_timeout():
    # the test hook leaves ring stage 1 of every task unfilled and gives each
    # wait 2048 polls: every task gives up, reports a timeout and leaves
    # in-range outputs; the context stays usable and the next call is exact
    V = 152064
    lg, drafts, params, u = _stream_case(V, 65)
    n0, out0, st = _verify(lg, drafts, params, u)
    assert st == 0
    m.mtp_test_verify_stall(1, 2048)
    n, out, st = _verify(lg, drafts, params, u)
    assert st == g.TIMEOUT
    _in_range(n, out, 3, V)
    n1, out1, st = _verify(lg, drafts, params, u)
    assert st == 0 and np.array_equal(n1, n0) and np.array_equal(out1, out0)


def test_draft_reports_nonfinite_logits_in_the_handle_word():
    # a NaN in the target hidden of the newest pair makes every logit of the
    # first head call NaN; the handle's status word reports it
    s = synth.TINY
    rig = g.Rig(s, seed=66, rows=1, capacity=256, prefill=[64], max_depth=2)
    word = g.device_i32(m.mtp_device_status(rig.h))
    word.zero_()
    tok, hid = rig.pairs([[5]], seed_tag="st:draft")
    rig.draft(2, [1], tok, hid, [dict(temperature=0.0)])
    assert int(word.item()) == 0
    m.mtp_set_lengths(rig.h, [64])
    hid[0, 0, 17] = float("nan")
    rig.draft(2, [1], tok, hid, [dict(temperature=0.0)])
    assert int(word.item()) & g.NONFINITE
    rig.close()


def test_batched_draft_nonfinite_row_is_reported_and_others_unchanged():
    # eight rows take the tensor-core head, whose lone-split logits epilogue
    # takes each tile's argmax; a NaN in one row's newest hidden makes that
    # row's logits NaN: the word reports it, its tokens stay in the
    # vocabulary, and the other rows draft what they draft without it
    s = synth.small_shape("bf16", vocab=4096)
    R = 8
    rig = g.Rig(s, seed=67, rows=R, capacity=256, prefill=[64] * R, max_depth=2)
    word = g.device_i32(m.mtp_device_status(rig.h))
    word.zero_()
    tok, hid = rig.pairs([[5 + r] for r in range(R)], seed_tag="st:bdraft")
    greedy = [dict(temperature=0.0)] * R
    clean = np.array(rig.draft(2, [1] * R, tok, hid, greedy)["draft"])
    assert int(word.item()) == 0
    m.mtp_set_lengths(rig.h, [64] * R)
    hid[3, 0, 17] = float("nan")
    bad = np.array(rig.draft(2, [1] * R, tok, hid, greedy)["draft"])
    assert int(word.item()) & g.NONFINITE
    assert bad.min() >= 0 and bad.max() < s.vocab
    keep = [r for r in range(R) if r != 3]
    assert np.array_equal(bad[keep], clean[keep])
    rig.close()
