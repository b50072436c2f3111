"""Argmax drafting under a sampled verify (the drafter flag
supports_greedy_draft_argmax, "feat(inference): support the qwen3_5_mtp
drafter" issue, Upstream contract to port).

A sampled row with MTP_SAMPLE_ARGMAX_DRAFT drafts the argmax of its
penalised draft logits, with no sampler, no q and no draft uniforms. The
verify treats that draft as the point mass q = one-hot(x): x is accepted with
probability p(x), and a rejection draws from p with x removed. Both sides are
checked against the oracle on the tiny fp32 head. The drafts must equal the
oracle's greedy drafts under the same penalty. The verify outcome must equal
the oracle's rejection-sampling verify given that one-hot q, exactly, unless
the oracle reports a near-tie."""
import numpy as np
import pytest
import torch

import mtp_speculative_decoding_step_gb300 as m
import oracle
import synth
from tests import gpu_common as g

pytestmark = pytest.mark.gpu
S = synth.TINY
TOL = 1e-5
SAMPLED = dict(temperature=0.8, rep_penalty=1.1, top_k=0, top_p=0.95, min_p=0.02)


def test_argmax_draft_needs_no_sampler_inputs():
    depth = 3
    rig = g.Rig(S, seed=31, rows=1, capacity=512, prefill=[128], max_depth=depth)
    tok, hid = rig.pairs([[9]])
    hist = synth.randint(31, "hist", (1, 64), S.vocab)
    draft = torch.full((1, depth), -1, dtype=torch.int32, device="cuda")
    logits = torch.zeros((1, depth, S.vocab), dtype=torch.float32, device="cuda")
    # no q and no u: the row drafts greedily
    m.mtp_draft(rig.h, depth, [1], tok, hid, [dict(SAMPLED, argmax_draft=True)], draft, hist=g.to_dev(hist),
                logits=logits)
    torch.cuda.synchronize()
    p_draft = oracle.make_params(0.0, rep_penalty=SAMPLED["rep_penalty"])
    ref = rig.oracle_draft(0, depth, [9], g.to_f32(hid)[0, :1], p_draft, hist=hist[0])
    out = draft.cpu().numpy()[0]
    lg = logits.cpu().numpy()[0]
    for k in range(depth):
        assert g.max_rel(lg[k], ref["logits"][k]) < TOL
        if g.draft_near_tie(ref["margins"][k], True, 1e-4):
            return
        assert out[k] == ref["drafts"][k], k
    rig.close()


@pytest.mark.parametrize("params", [SAMPLED, dict(temperature=1.0, top_k=40)])
def test_point_mass_verify(params):
    rows, d, V = 24, 3, S.vocab
    lg = synth.normal(33, "am-lg", (rows, d + 1, V), std=2.0)
    hist = synth.randint(33, "am-hist", (rows, 64), V)
    # drafts: the argmax of a perturbed copy, so some are the target's mode and some not
    pert = lg[:, :d] + synth.normal(33, "am-pert", (rows, d, V), std=1.0)
    drafts = pert.argmax(2).astype(np.int32)
    u = synth.uniform(33, "am-u", (rows, d + 1))
    ws = torch.zeros(m.spec_verify_workspace_bytes(rows, d, V), dtype=torch.uint8, device="cuda")
    n_acc = torch.zeros(rows, dtype=torch.int32, device="cuda")
    out = torch.zeros((rows, d + 1), dtype=torch.int32, device="cuda")
    m.spec_verify(g.to_dev(lg), g.to_dev(drafts), [dict(params, argmax_draft=True)] * rows, g.to_dev(u), n_acc,
                  out, ws, q=None, hist=g.to_dev(hist))
    torch.cuda.synchronize()
    got_n = n_acc.cpu().numpy()
    got_t = out.cpu().numpy()
    p = oracle.make_params(**params)
    near = 0
    outcomes = set()
    for r in range(rows):
        q = np.zeros((d, V), np.float32)
        q[np.arange(d), drafts[r]] = 1.0
        n, toks, mg = oracle.verify_row(lg[r], drafts[r], q, p, hist[r], u[r])
        if g.verify_near_tie(mg, n, d, False):
            near += 1
            continue
        assert got_n[r] == n and np.array_equal(got_t[r], toks), r
        outcomes.add(n)
    assert near <= 2
    assert len(outcomes) >= 2  # both rejections and acceptances were exercised
