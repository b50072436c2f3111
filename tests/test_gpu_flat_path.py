"""The flat transform: rows without a top-k below the vocabulary (top-p,
min-p, or plain temperature over the whole vocabulary), spread over many CTAs
per (row, position). Drafts and q of sampled draft steps, and the verify's
accepted counts and tokens, against the oracle: at batch 1 and over several
rows, with a repetition penalty, with min-p alone, top-p and min-p together,
plain temperature sampling, argmax drafts beside dense q rows, and greedy
rows with a penalty in the same call. Decisions are exact unless the oracle
reports a near-tie."""
import numpy as np
import pytest
import torch

import mtp_speculative_decoding_step_gb300 as m
import oracle
import synth
from tests import gpu_common as g

pytestmark = pytest.mark.gpu
S = synth.small_shape("bf16", vocab=32768)
TOL = 1e-2

ROWS = [
    dict(temperature=0.9, top_p=0.8, rep_penalty=1.2),
    dict(temperature=0.7, min_p=0.05),
    dict(temperature=1.0, top_p=0.95, min_p=0.02, rep_penalty=0.9),
    dict(temperature=1.1),
]


@pytest.mark.parametrize("R", [1, 4])
def test_flat_draft_steps_match_the_oracle(R):
    depth, W = 3, 16
    # weights N(0, 0.1): logits spread enough that the seeded draws keep clear
    # of every cumulative boundary (smallest oracle margin 2.3e-5 of the mass)
    seed = 93
    model = synth.make_model(S, seed, weight_std=0.1)
    rig = g.Rig(S, seed=seed, rows=R, capacity=512, prefill=[100 + 11 * r for r in range(R)], max_depth=depth,
                model=model)
    params = [ROWS[r % len(ROWS)] for r in range(R)]
    hist = synth.randint(seed, "fl:hist", (R, W), S.vocab)
    toks = [[int(t)] for t in synth.randint(seed, "fl:tok", (R,), S.vocab)]
    tok, hid = rig.pairs(toks)
    u = synth.uniform(seed, "fl:u", (R, depth))
    out = rig.draft(depth, [1] * R, tok, hid, params, hist=hist, u=u)
    hh = g.to_f32(hid)
    near = compared = 0
    for r in range(R):
        p = oracle.make_params(**params[r])
        ref = rig.oracle_draft(r, depth, toks[r], hh[r, :1], p, hist=hist[r], u=u[r])
        for k in range(depth):
            assert g.max_rel(out["logits"][r, k], ref["logits"][k]) < TOL, (r, k)
            assert np.max(np.abs(out["q"][r, k] - ref["q"][k])) < 1e-3 * ref["q"][k].max(), (r, k)
            if g.draft_near_tie(ref["margins"][k], False, 1e-3):
                near += 1
                break
            assert out["draft"][r, k] == ref["drafts"][k], (r, k)
            compared += 1
    assert near == 0 and compared == R * depth, (near, compared)
    rig.close()


def _verify(lg, drafts, q, params, u, hist):
    R, dp1, V = lg.shape
    ws = torch.zeros(m.spec_verify_workspace_bytes(R, dp1 - 1, V), dtype=torch.uint8, device="cuda")
    n_acc = torch.full((R,), -7, dtype=torch.int32, device="cuda")
    out = torch.full((R, dp1), -7, dtype=torch.int32, device="cuda")
    stats = torch.zeros((R, dp1 + 1), dtype=torch.int32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    m.spec_verify(g.to_dev(lg), g.to_dev(np.ascontiguousarray(drafts, np.int32)), params, g.to_dev(u), n_acc, out,
                  ws, q=g.to_dev(q), hist=g.to_dev(hist), stats=stats, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    return n_acc.cpu().numpy(), out.cpu().numpy(), stats.cpu().numpy()


@pytest.mark.parametrize("V", [32768, 152064])
def test_flat_verify_matches_the_oracle(V):
    R, d, W = 8, 3, 24
    params = [dict(temperature=0.0, rep_penalty=1.3) if r % 4 == 3 else dict(ROWS[r % len(ROWS)]) for r in range(R)]
    params[2]["argmax_draft"] = True
    lg = synth.normal(92, f"fv:lg{V}", (R, d + 1, V), std=2.0)
    hist = synth.randint(92, f"fv:hist{V}", (R, W), V)
    noise = synth.normal(92, f"fv:noise{V}", (R, d, V), std=0.7)
    ud = synth.uniform(92, f"fv:ud{V}", (R, d))
    u = synth.uniform(92, f"fv:u{V}", (R, d + 1))
    q = np.zeros((R, d, V), np.float32)
    drafts = np.zeros((R, d), np.int32)
    for r in range(R):
        pr = dict(params[r])
        am = pr.pop("argmax_draft", False)
        p = oracle.make_params(**pr)
        for i in range(d):
            win = np.concatenate([hist[r], drafts[r, :i]])[-W:].astype(np.int32)
            qi, info = oracle.transform(lg[r, i] + noise[r, i], oracle.make_params(**dict(pr, temperature=0.0)) if am
                                        else p, win)
            if am or oracle.is_greedy(p):
                drafts[r, i] = info.argmax
                qi = np.zeros(V, np.float32)
                qi[info.argmax] = 1.0
            else:
                drafts[r, i] = oracle.draw(qi, float(ud[r, i]))[0]
            q[r, i] = qi
    n_got, t_got, st = _verify(lg, drafts, q, params, u, hist)
    near, lengths = 0, set()
    for r in range(R):
        pr = dict(params[r])
        pr.pop("argmax_draft", None)
        p = oracle.make_params(**pr)
        n, toks, mg = oracle.verify_row(lg[r], drafts[r], q[r], p, hist[r], u[r])
        if g.verify_near_tie(mg, n, d, oracle.is_greedy(p)):
            near += 1
            continue
        assert n_got[r] == n and np.array_equal(t_got[r], toks), (r, n_got[r], n, t_got[r], toks)
        assert st[r, 0] == 1 and st[r, 1] == (1 if n < d else 0)
        lengths.add(n)
    assert near <= 1 and len(lengths) >= 2
