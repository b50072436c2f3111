"""Edge cases of the verify and draft paths on the GPU, against the oracle:
- the largest verify: 64 rows at depth 16 (block 17) with the longest penalty
  window (128 tokens), greedy and sampled rows mixed;
- a vocabulary that is not a multiple of 4 (1001), so every 16-byte load path
  falls back to its scalar tail;
- drafts outside [0, V): rejected at their position, never read;
- the deepest draft (16 steps) on the tiny head.
Decisions must match the oracle exactly unless it reports a near-tie."""
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


def _case(seed, R, d, V, W, sampled):
    lg = synth.normal(seed, "e-lg", (R, d + 1, V), std=2.5)
    hist = synth.randint(seed, "e-hist", (R, W), V) if W else None
    params = [sampled if r % 2 else dict(temperature=0.0) for r in range(R)]
    q = np.zeros((R, d, V), np.float32)
    drafts = np.zeros((R, d), np.int32)
    du = synth.uniform(seed, "e-du", (R, d))
    ql = synth.normal(seed, "e-ql", (R, d, V), std=2.5)
    for r in range(R):
        p = oracle.make_params(**params[r])
        for i in range(d):
            if oracle.is_greedy(p):
                # greedy drafts: the target's argmax or its neighbour
                drafts[r, i] = lg[r, i].argmax() if (r + i) % 3 else (lg[r, i].argmax() + 1) % V
            else:
                win = np.concatenate([hist[r] if hist is not None else np.zeros(0, np.int32), drafts[r, :i]])
                win = win[len(win) - W:] if W else np.zeros(0, np.int32)
                q[r, i] = oracle.transform(ql[r, i], p, win.astype(np.int32))[0]
                drafts[r, i] = oracle.draw(q[r, i], float(du[r, i]))[0]
    u = synth.uniform(seed, "e-u", (R, d + 1))
    return lg, hist, params, q, drafts, u


def _check(lg, hist, params, q, drafts, u, got_n, got_t, max_near):
    R, dp1, _ = lg.shape
    near = 0
    for r in range(R):
        p = oracle.make_params(**params[r])
        greedy = oracle.is_greedy(p)
        n, toks, mg = oracle.verify_row(lg[r], drafts[r], None if greedy else q[r], p,
                                        np.zeros(0, np.int32) if hist is None else hist[r], u[r])
        if g.verify_near_tie(mg, n, dp1 - 1, greedy):
            near += 1
            continue
        assert got_n[r] == n and np.array_equal(got_t[r], toks), r
    assert near <= max_near


def test_verify_max_rows_depth_and_window():
    sampled = dict(temperature=1.0, rep_penalty=1.2, top_k=20, top_p=0.9, min_p=0.01)
    lg, hist, params, q, drafts, u = _case(51, 64, 16, 2048, 128, sampled)
    got_n, got_t = _verify(lg, drafts, q, params, u, hist)
    _check(lg, hist, params, q, drafts, u, got_n, got_t, max_near=3)
    assert got_n.max() >= 2  # some rows accept deep into the block


@pytest.mark.parametrize("sampled", [dict(temperature=0.9, top_p=0.8),
                                     dict(temperature=1.0, top_k=7, rep_penalty=1.3)])
def test_verify_vocab_not_a_multiple_of_four(sampled):
    lg, hist, params, q, drafts, u = _case(52, 8, 3, 1001, 16, sampled)
    got_n, got_t = _verify(lg, drafts, q, params, u, hist)
    _check(lg, hist, params, q, drafts, u, got_n, got_t, max_near=1)


def test_out_of_range_drafts_are_rejected():
    R, d, V = 6, 3, 2048
    lg = synth.normal(53, "oor-lg", (R, d + 1, V), std=2.0)
    am = lg.argmax(2)
    drafts = am[:, :d].astype(np.int32).copy()
    bad_pos = [0, 1, 2, 0, 1, 2]
    for r in range(R):
        drafts[r, bad_pos[r]] = -1 if r % 2 else V + 5
    u = synth.uniform(53, "oor-u", (R, d + 1))
    got_n, got_t = _verify(lg, drafts, None, [dict(temperature=0.0)] * R, u, None)
    for r in range(R):
        k = bad_pos[r]
        assert got_n[r] == k, r
        assert np.array_equal(got_t[r, :k], drafts[r, :k])
        assert got_t[r, k] == am[r, k]          # the correction: argmax of the stopping row
        assert np.all(got_t[r, k + 1:] == -1)


def test_deepest_draft_on_the_tiny_head():
    depth = 16
    S = synth.TINY
    rig = g.Rig(S, seed=54, rows=1, capacity=512, prefill=[100], max_depth=depth)
    tok, hid = rig.pairs([[3, 4]])
    out = rig.draft(depth, [2], tok, hid, [dict(temperature=0.0)])
    ref = rig.oracle_draft(0, depth, [3, 4], g.to_f32(hid)[0], oracle.make_params(0.0))
    for k in range(depth):
        assert g.max_rel(out["logits"][0, k], ref["logits"][k]) < 1e-5, k
        if ref["margins"][k] <= 1e-4:
            break
        assert out["draft"][0, k] == ref["drafts"][k], k
    assert list(m.mtp_get_lengths(rig.h)) == [100 + 2 + depth - 1]
    rig.close()
