"""The streaming verify (one CTA per row and position, exact top-k kept in
shared memory) against the oracle. spec_verify takes it for calls with more
row x position tasks than one wave of 8-CTA clusters holds, when every sampled
row cuts to a top-k of at most 256 below the vocabulary; every case here is
such a call. Covered: the sampled parameters of the decoding workload with
argmax drafts at the full vocabulary, dense draft distributions, rows whose
logits tie at the k-th key (quantised) or rise along the vocabulary (every
round overflows the candidate buffer and is offered again), top-k 1 and 256,
greedy rows in the same call, and a vocabulary that is not a multiple of 4.
Decisions must equal the oracle's exactly unless it reports a near-tie."""
import numpy as np
import pytest
import torch

import mtp_speculative_decoding_step_gb300 as m
import oracle
import synth
from tests import gpu_common as g

pytestmark = pytest.mark.gpu


def _verify(lg, drafts, q, params, u, hist):
    R, dp1, V = lg.shape
    ws = torch.zeros(m.spec_verify_workspace_bytes(R, dp1 - 1, V), dtype=torch.uint8, device="cuda")
    n_acc = torch.zeros(R, dtype=torch.int32, device="cuda")
    out = torch.zeros((R, dp1), dtype=torch.int32, device="cuda")
    m.spec_verify(g.to_dev(lg), g.to_dev(np.ascontiguousarray(drafts, np.int32)), params, g.to_dev(u), n_acc, out,
                  ws, q=None if q is None else g.to_dev(q), hist=None if hist is None else g.to_dev(hist))
    torch.cuda.synchronize()
    return n_acc.cpu().numpy(), out.cpu().numpy()


def _check(lg, drafts, q_of, params, u, hist, got_n, got_t, max_near):
    R, dp1, _ = lg.shape
    near = 0
    outcomes = set()
    for r in range(R):
        pr = dict(params[r])
        pr.pop("argmax_draft", None)
        p = oracle.make_params(**pr)
        greedy = oracle.is_greedy(p)
        n, toks, mg = oracle.verify_row(lg[r], drafts[r], None if greedy else q_of(r), p,
                                        np.zeros(0, np.int32) if hist is None else hist[r], u[r])
        if g.verify_near_tie(mg, n, dp1 - 1, greedy):
            near += 1
            continue
        assert got_n[r] == n and np.array_equal(got_t[r], toks), (r, got_n[r], n, got_t[r], toks)
        outcomes.add(n)
    assert near <= max_near
    return outcomes


def _one_hot(drafts, V):
    def q_of(r):
        d = drafts.shape[1]
        q = np.zeros((d, V), np.float32)
        q[np.arange(d), drafts[r]] = 1.0
        return q
    return q_of


def test_decoding_parameters_argmax_drafts_full_vocab():
    R, d, V = 64, 3, 152064
    prm = dict(temperature=0.8, rep_penalty=1.1, top_k=40, top_p=0.95, min_p=0.05, argmax_draft=True)
    lg = synth.normal(71, "vs-lg", (R, d + 1, V), std=4.0)
    hist = synth.randint(71, "vs-hist", (R, 64), V)
    pert = lg[:, :d] + synth.normal(71, "vs-pert", (R, d, V), std=1.0)
    drafts = pert.argmax(2).astype(np.int32)
    u = synth.uniform(71, "vs-u", (R, d + 1))
    params = [prm] * R
    got_n, got_t = _verify(lg, drafts, None, params, u, hist)
    outcomes = _check(lg, drafts, _one_hot(drafts, V), params, u, hist, got_n, got_t, max_near=3)
    assert len(outcomes) >= 2


def test_dense_draft_distributions():
    R, d, V, W = 48, 3, 32768, 32
    prm = dict(temperature=1.0, rep_penalty=1.2, top_k=50, top_p=0.9, min_p=0.0)
    p = oracle.make_params(**prm)
    lg = synth.normal(72, "vd-lg", (R, d + 1, V), std=2.5)
    hist = synth.randint(72, "vd-hist", (R, W), V)
    ql = lg[:, :d] + synth.normal(72, "vd-ql", (R, d, V), std=0.7)
    du = synth.uniform(72, "vd-du", (R, d))
    q = np.zeros((R, d, V), np.float32)
    drafts = np.zeros((R, d), np.int32)
    for r in range(R):
        for i in range(d):
            win = np.concatenate([hist[r], drafts[r, :i]])[-W:].astype(np.int32)
            q[r, i] = oracle.transform(ql[r, i], p, win)[0]
            drafts[r, i] = oracle.draw(q[r, i], float(du[r, i]))[0]
    u = synth.uniform(72, "vd-u", (R, d + 1))
    params = [prm] * R
    got_n, got_t = _verify(lg, drafts, q, params, u, hist)
    outcomes = _check(lg, drafts, lambda r: q[r], params, u, hist, got_n, got_t, max_near=3)
    assert len(outcomes) >= 2


def test_ties_rising_rows_extreme_k_and_greedy_rows():
    R, d, V = 40, 2, 8192
    lg = synth.normal(73, "vt-lg", (R, d + 1, V), std=2.0)
    ramp = np.linspace(-4.0, 4.0, V, dtype=np.float32)
    for r in range(R):
        if r % 4 == 1:
            lg[r] = np.round(lg[r] * 2.0) / 2.0   # many logits tie at the k-th key
        elif r % 4 == 2:
            lg[r] = ramp[None, :] + 0.0            # each round beats every earlier one
    hist = synth.randint(73, "vt-hist", (R, 16), V)
    drafts = np.where(synth.uniform(73, "vt-c", (R, d)) < 0.5, lg[:, :d].argmax(2),
                      synth.randint(73, "vt-x", (R, d), V)).astype(np.int32)
    u = synth.uniform(73, "vt-u", (R, d + 1))
    params = []
    for r in range(R):
        if r % 5 == 4:
            params.append(dict(temperature=0.0, rep_penalty=1.3))   # greedy, penalised
        else:
            params.append(dict(temperature=0.9, rep_penalty=1.15, top_k=(1, 7, 256, 33)[r % 4], top_p=0.85,
                               min_p=0.01, argmax_draft=True))
    got_n, got_t = _verify(lg, drafts, None, params, u, hist)
    _check(lg, drafts, _one_hot(drafts, V), params, u, hist, got_n, got_t, max_near=4)


def test_vocab_not_a_multiple_of_four():
    R, d, V = 64, 2, 1001
    prm = dict(temperature=0.7, top_k=7, top_p=0.95, argmax_draft=True)
    lg = synth.normal(74, "vo-lg", (R, d + 1, V), std=2.0)
    drafts = (lg[:, :d] + synth.normal(74, "vo-p", (R, d, V), std=0.5)).argmax(2).astype(np.int32)
    u = synth.uniform(74, "vo-u", (R, d + 1))
    params = [prm] * R
    got_n, got_t = _verify(lg, drafts, None, params, u, None)
    _check(lg, drafts, _one_hot(drafts, V), params, u, None, got_n, got_t, max_near=3)
