"""The top-k cluster transform (rows whose top-k is at most 256, few tasks per
call) on the branches its bound takes: a small k (each CTA's own k-th thread
minimum bounds the top-k), a large k (the k-th of the cluster's 4096 thread
minima), heavily tied logits (the bound admits too many elements and the exact
k-th comes from the cluster radix selection), k = 2 and k = 256, with a
repetition penalty, top-p and min-p on top, and greedy rows with a penalty in
the same call. Verifies against the oracle row by row (exact unless the oracle
reports a near-tie), and one draft step's q and token."""
import numpy as np
import pytest
import torch

import mtp_speculative_decoding_step_gb300 as m
import oracle
import synth
from tests import gpu_common as g

pytestmark = pytest.mark.gpu
V = 152064

CASES = [
    dict(temperature=0.8, top_k=2),
    dict(temperature=0.9, top_k=40, top_p=0.9, rep_penalty=1.2),
    dict(temperature=1.0, top_k=200, min_p=0.01),
    dict(temperature=0.7, top_k=256, top_p=0.95, min_p=0.02),
    dict(temperature=0.0, rep_penalty=1.3),
]


def _case(seed, quantum):
    R, d, W = len(CASES), 2, 32
    lg = synth.normal(seed, "tk:lg", (R, d + 1, V), std=3.0)
    if quantum:
        lg = (np.round(lg / quantum) * quantum).astype(np.float32)
    hist = synth.randint(seed, "tk:hist", (R, W), V)
    ud = synth.uniform(seed, "tk:ud", (R, d))
    u = synth.uniform(seed, "tk:u", (R, d + 1))
    q = np.zeros((R, d, V), np.float32)
    drafts = np.zeros((R, d), np.int32)
    noise = synth.normal(seed, "tk:noise", (R, d, V), std=0.5)
    for r, prm in enumerate(CASES):
        p = oracle.make_params(**prm)
        for i in range(d):
            win = np.concatenate([hist[r], drafts[r, :i]])[-W:].astype(np.int32)
            qi, info = oracle.transform(lg[r, i] + noise[r, i], p, win)
            if oracle.is_greedy(p):
                drafts[r, i] = info.argmax
            else:
                drafts[r, i] = oracle.draw(qi, float(ud[r, i]))[0]
                q[r, i] = qi
    return lg, drafts, q, hist, u


@pytest.mark.parametrize("quantum", [0.0, 0.5])
def test_topk_verify_branches_match_the_oracle(quantum):
    # 5 rows x 3 positions = 15 tasks: the one-cluster-per-task top-k path
    lg, drafts, q, hist, u = _case(95, quantum)
    R, dp1, _ = lg.shape
    ws = torch.zeros(m.spec_verify_workspace_bytes(R, dp1 - 1, V), dtype=torch.uint8, device="cuda")
    n_acc = torch.full((R,), -7, dtype=torch.int32, device="cuda")
    out = torch.full((R, dp1), -7, dtype=torch.int32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    m.spec_verify(g.to_dev(lg), g.to_dev(drafts), CASES, g.to_dev(u), n_acc, out, ws, q=g.to_dev(q),
                  hist=g.to_dev(hist), status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    got_n, got_t = n_acc.cpu().numpy(), out.cpu().numpy()
    near = 0
    for r, prm in enumerate(CASES):
        p = oracle.make_params(**prm)
        n, toks, mg = oracle.verify_row(lg[r], drafts[r], None if oracle.is_greedy(p) else q[r], p, hist[r], u[r])
        if g.verify_near_tie(mg, n, dp1 - 1, oracle.is_greedy(p)):
            near += 1
            continue
        assert got_n[r] == n and np.array_equal(got_t[r], toks), (r, got_n[r], n, got_t[r], toks)
    assert near <= 1


@pytest.mark.parametrize("k", [3, 200])
def test_topk_draft_step_q_and_token(k):
    # one sampled draft step at batch 1 through the top-k kernel: q over the
    # whole vocabulary and the drawn token against the oracle's transform
    S = synth.small_shape("bf16", vocab=32768)
    prm = dict(temperature=0.9, top_k=k, top_p=0.97, rep_penalty=1.1)
    rig = g.Rig(S, seed=96, rows=1, capacity=256, prefill=[77], max_depth=1,
                model=synth.make_model(S, 96, weight_std=0.1))
    hist = synth.randint(96, "tkd:hist", (1, 24), S.vocab)
    tok, hid = rig.pairs([[123]])
    u = np.array([[0.4173]], np.float32)
    out = rig.draft(1, [1], tok, hid, [prm], hist=hist, u=u)
    ref = rig.oracle_draft(0, 1, [123], g.to_f32(hid)[0, :1], oracle.make_params(**prm), hist=hist[0], u=u[0])
    assert g.max_rel(out["logits"][0, 0], ref["logits"][0]) < 1e-2
    assert np.max(np.abs(out["q"][0, 0] - ref["q"][0])) < 1e-3 * ref["q"][0].max()
    assert np.count_nonzero(out["q"][0, 0]) == np.count_nonzero(ref["q"][0])
    if not g.draft_near_tie(ref["margins"][0], False, 1e-3):
        assert out["draft"][0, 0] == ref["drafts"][0]
    rig.close()


def test_greedy_penalty_draft_without_q():
    # greedy rows with a repetition penalty take the top-k sampler as well; with
    # no sampled row the caller may pass no q, which must then stay unwritten
    S = synth.small_shape("bf16", vocab=32768)
    prm = dict(temperature=0.0, rep_penalty=1.3)
    rig = g.Rig(S, seed=97, rows=1, capacity=256, prefill=[77], max_depth=2,
                model=synth.make_model(S, 97, weight_std=0.1))
    hist = synth.randint(97, "tkg:hist", (1, 24), S.vocab)
    tok, hid = rig.pairs([[321]])
    out = rig.draft(2, [1], tok, hid, [prm], hist=hist)
    assert out["q"] is None
    ref = rig.oracle_draft(0, 2, [321], g.to_f32(hid)[0, :1], oracle.make_params(**prm), hist=hist[0])
    for k in range(2):
        assert g.max_rel(out["logits"][0, k], ref["logits"][k]) < 1e-2, k
        if ref["margins"][k] <= 1e-3:
            break
        assert out["draft"][0, k] == ref["drafts"][k], k
    rig.close()
