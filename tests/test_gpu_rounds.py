"""GPU parity of whole rounds at the 27B shape.

Sampled decoding: temperature 0.8, repetition penalty 1.1 over a 64-token
history, top-k 40, top-p 0.95, min-p 0.05, depth swept 1..6; target rows are
the drafter's logits plus N(0,1) noise (the bonus row N(0,4)), so acceptance is
partial.  Batched decoding: 8 independent rows with draft KV lengths drawn
from U[1024, 16384], depth 3, rows alternating greedy and (T 0.7, top-p 0.9),
one verify over all rows and a per-row rollback.

The verify is fed identical inputs on both sides (the oracle's draft logits
and q); the GPU draft is compared with the oracle's draft.  Decisions must
match exactly unless the oracle reports a near-tie (|p/q - u| < 1e-3 or a draw
within 1e-3 of a cumulative boundary), which is counted."""
import numpy as np
import pytest
import torch

import mtp_speculative_decoding_step_gb300 as m
import oracle
import synth
from tests import gpu_common as g

pytestmark = pytest.mark.gpu
S = synth.QWEN27B
TOL = 1e-2
SAMPLED = dict(temperature=0.8, rep_penalty=1.1, top_k=40, top_p=0.95, min_p=0.05)


def _target_rows(seed, tag, draft_logits, V):
    d = draft_logits.shape[0]
    noise = synth.normal(seed, tag + ":noise", (d, V), std=1.0)
    bonus = synth.normal(seed, tag + ":bonus", (1, V), std=4.0)
    return np.concatenate([draft_logits + noise, bonus]).astype(np.float32)


def _compare_draft(out, ref, r, depth):
    """Compare the GPU draft of row r with the oracle's, up to the first near-tie."""
    for k in range(depth):
        assert g.max_rel(out["logits"][r, k], ref["logits"][k]) < TOL, (r, k)
        if ref["q"] is not None:
            assert np.max(np.abs(out["q"][r, k] - ref["q"][k])) < 1e-3 * max(ref["q"][k].max(), 1e-6)
        if g.draft_near_tie(ref["margins"][k], ref["q"] is None, 1e-3):
            return k, True
        assert out["draft"][r, k] == ref["drafts"][k], (r, k)
    return depth, False


@pytest.mark.parametrize("depth", [1, 2, 3, 4, 5, 6])
def test_sampled_round_depth(model27, depth):
    seed = 10 + depth
    rig = g.Rig(S, seed=seed, rows=1, capacity=4096 + 128, prefill=[4096], max_depth=6, model=model27)
    hist = synth.randint(seed, "hist", (1, 64), S.vocab)
    p = oracle.make_params(**SAMPLED)
    toks = [int(synth.randint(seed, "tok0", (1,), S.vocab)[0])]
    near = 0
    for rnd in range(2):
        tok, hid = rig.pairs([toks], seed_tag=f"r{rnd}")
        u_d = synth.uniform(seed, f"ud{rnd}", (1, depth))
        out = rig.draft(depth, [len(toks)], tok, hid, [SAMPLED], hist=hist, u=u_d)
        ref = rig.oracle_draft(0, depth, toks, g.to_f32(hid)[0], p, hist=hist[0], u=u_d[0])
        upto, tie = _compare_draft(out, ref, 0, depth)
        near += tie
        lg = _target_rows(seed, f"t{rnd}", ref["logits"], S.vocab)
        u_v = synth.uniform(seed, f"uv{rnd}", (1, depth + 1))
        got = rig.verify(lg[None], ref["drafts"][None], ref["q"][None], [SAMPLED], u_v, hist=hist)
        n, out_tok, mg = oracle.verify_row(lg, ref["drafts"], ref["q"], p, hist[0], u_v[0])
        if g.verify_near_tie(mg, n, depth, False):
            near += 1
        else:
            assert got["n_acc"][0] == n and np.array_equal(got["out_tok"][0], out_tok)
        if tie:
            break
        # roll back both sides and chain: the n+1 committed tokens become pending pairs
        m.kv_rollback(rig.h, 1, depth)
        rig.olen[0] -= depth - 1
        assert list(m.mtp_get_lengths(rig.h)) == [rig.olen[0]]
        committed = [int(t) for t in out_tok[: n + 1]]
        hist = np.concatenate([hist[:, n + 1:], np.array([committed], np.int32)], axis=1)
        toks = committed
    assert near <= 1
    rig.close()


def test_batched_rows_ragged(model27):
    seed = 40
    R, depth = 8, 3
    lens = [int(x) for x in (1024 + synth.randint(seed, "lens", (R,), 16384 - 1024 + 1))]
    cap = (max(lens) + 64 + 63) // 64 * 64
    rig = g.Rig(S, seed=seed, rows=R, capacity=cap, prefill=lens, max_depth=depth, model=model27)
    params = [dict(temperature=0.0) if r % 2 == 0 else dict(temperature=0.7, top_p=0.9) for r in range(R)]
    hist = synth.randint(seed, "hist", (R, 64), S.vocab)
    toks = [[int(t)] for t in synth.randint(seed, "tok0", (R,), S.vocab)]
    tok, hid = rig.pairs(toks)
    u_d = synth.uniform(seed, "ud", (R, depth))
    out = rig.draft(depth, [1] * R, tok, hid, params, hist=hist, u=u_d)
    hh = g.to_f32(hid)
    refs = []
    for r in range(R):
        p = oracle.make_params(**params[r])
        ref = rig.oracle_draft(r, depth, toks[r], hh[r], p, hist=hist[r], u=u_d[r])
        _compare_draft(out, ref, r, depth)
        refs.append(ref)
    lg = np.stack([_target_rows(seed, f"t{r}", refs[r]["logits"], S.vocab) for r in range(R)])
    drafts = np.stack([x["drafts"] for x in refs])
    q = np.zeros((R, depth, S.vocab), np.float32)
    for r in range(R):
        if refs[r]["q"] is not None:
            q[r] = refs[r]["q"]
    u_v = synth.uniform(seed, "uv", (R, depth + 1))
    stats = torch.zeros((R, depth + 2), dtype=torch.int32, device="cuda")
    got = rig.verify(lg, drafts, q, params, u_v, hist=hist, stats=stats)
    near = 0
    n_ref = []
    for r in range(R):
        p = oracle.make_params(**params[r])
        n, out_tok, mg = oracle.verify_row(lg[r], drafts[r], refs[r]["q"], p, hist[r], u_v[r])
        n_ref.append(n)
        if g.verify_near_tie(mg, n, depth, params[r].get("temperature", 0.0) == 0.0):
            near += 1
            continue
        assert got["n_acc"][r] == n and np.array_equal(got["out_tok"][r], out_tok), r
    assert near <= 1
    st = stats.cpu().numpy()
    assert np.all(st[:, 0] == 1)
    np.testing.assert_array_equal(st[:, 1], (got["n_acc"] < depth).astype(np.int32))
    # per-row rollback: draft KV keeps the first call's slot; target lengths trim by block - (n+1)
    tlen = torch.tensor([x + depth + 1 for x in lens], dtype=torch.int32, device="cuda")
    n_acc = torch.tensor(got["n_acc"], dtype=torch.int32, device="cuda")
    m.kv_rollback(rig.h, R, depth, n_acc=n_acc, target_len=tlen)
    torch.cuda.synchronize()
    assert list(m.mtp_get_lengths(rig.h)) == [x + 1 for x in lens]
    assert list(tlen.cpu().numpy()) == [lens[r] + got["n_acc"][r] + 1 for r in range(R)]
    rig.close()
