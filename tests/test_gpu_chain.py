"""Chain equals block on the GPU ("support the qwen3_5_mtp drafter" issue,
Reproduction instructions, Test 3: verifying a block of T tokens must give what
the single-token chain gives).  d calls of spec_verify at depth 1, chained
through the accepted drafts and the penalty window, must commit exactly the
tokens one depth-d call commits, for every row; the block call is also checked
against the oracle.  Greedy rows (plain, and with a repetition penalty, which
takes the transform path) and sampled rows with the decoding workload's
parameters (temperature 0.8, penalty 1.1 over the window, top-k 40, top-p 0.95,
min-p 0.05)."""
import numpy as np
import pytest
import torch

import mtp_speculative_decoding_step_gb300 as m
import oracle
import synth
from tests import gpu_common as g

pytestmark = pytest.mark.gpu

R, D, V, W = 8, 4, 32768, 8


def _window(hist, drafts, i):
    seq = list(hist) + list(drafts[:i])
    return np.array(seq[-W:], np.int32)


def _call(lg, drafts, q, params, u, hist):
    rows, dp1, _ = lg.shape
    ws = torch.zeros(m.spec_verify_workspace_bytes(rows, dp1 - 1, V), dtype=torch.uint8, device="cuda")
    n_acc = torch.full((rows,), -7, dtype=torch.int32, device="cuda")
    out = torch.full((rows, dp1), -7, dtype=torch.int32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    m.spec_verify(g.to_dev(np.ascontiguousarray(lg)), g.to_dev(np.ascontiguousarray(drafts, np.int32)), params,
                  g.to_dev(np.ascontiguousarray(u, np.float32)), n_acc, out, ws,
                  q=None if q is None else g.to_dev(np.ascontiguousarray(q)), hist=g.to_dev(hist), status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    return n_acc.cpu().numpy(), out.cpu().numpy()


def _case(kind, seed):
    lg = synth.normal(seed, f"chain:{kind}:lg", (R, D + 1, V), std=4.0)
    hist = synth.randint(seed, f"chain:{kind}:hist", (R, W), V).astype(np.int32)
    u = synth.uniform(seed, f"chain:{kind}:u", (R, D + 1))
    if kind == "sampled":
        prm = dict(temperature=0.8, rep_penalty=1.1, top_k=40, top_p=0.95, min_p=0.05)
        op = oracle.make_params(**prm)
        noise = synth.normal(seed, f"chain:{kind}:noise", (R, D, V), std=1.0)
        ud = synth.uniform(seed, f"chain:{kind}:ud", (R, D))
        q = np.zeros((R, D, V), np.float32)
        drafts = np.zeros((R, D), np.int32)
        for r in range(R):
            for i in range(D):
                q[r, i], _ = oracle.transform(lg[r, i] + noise[r, i], op, _window(hist[r], drafts[r], i))
                drafts[r, i] = oracle.draw(q[r, i], float(ud[r, i]))[0]
        return lg, drafts, q, [prm] * R, op, u, hist
    prm = dict(temperature=0.0, rep_penalty=1.1 if kind == "greedy_pen" else 1.0)
    op = oracle.make_params(**prm)
    # drafts: the (penalised) argmax of each row with probability 0.7, else the runner-up
    coin = synth.uniform(seed, f"chain:{kind}:coin", (R, D)) < 0.7
    drafts = np.zeros((R, D), np.int32)
    for r in range(R):
        for i in range(D):
            _, info = oracle.transform(lg[r, i], op, _window(hist[r], drafts[r], i))
            alt = int(np.argsort(-lg[r, i])[1])
            drafts[r, i] = info.argmax if coin[r, i] or alt == info.argmax else alt
    return lg, drafts, None, [prm] * R, op, u, hist


@pytest.mark.parametrize("kind", ["greedy", "greedy_pen", "sampled"])
def test_chain_of_depth_one_verifies_equals_one_block_verify(kind):
    lg, drafts, q, params, op, u, hist = _case(kind, 70 + ["greedy", "greedy_pen", "sampled"].index(kind))
    n_blk, out_blk = _call(lg, drafts, q, params, u, hist)
    # the chain: call j (all rows at once) verifies x_j against rows j-1 and j
    # with the window advanced by x_1..x_{j-1} and the uniforms (u[j-1], u[D])
    calls = []
    for j in range(1, D + 1):
        hj = np.stack([_window(hist[r], drafts[r], j - 1) for r in range(R)])
        uj = np.stack([u[:, j - 1], u[:, D]], axis=1)
        calls.append(_call(lg[:, j - 1:j + 1], drafts[:, j - 1:j], None if q is None else q[:, j - 1:j], params,
                           uj, hj))
    lengths = set()
    for r in range(R):
        toks = []
        for j in range(1, D + 1):
            n, out = calls[j - 1][0][r], calls[j - 1][1][r]
            if n == 0:
                toks.append(int(out[0]))
                break
            toks.append(int(drafts[r, j - 1]))
            if j == D:
                toks.append(int(out[1]))
        assert n_blk[r] == len(toks) - 1 and list(out_blk[r, :n_blk[r] + 1]) == toks, (r, n_blk[r], out_blk[r], toks)
        assert all(out_blk[r, n_blk[r] + 1:] == -1)
        lengths.add(int(n_blk[r]))
        # and the block call against the oracle (unless it reports a near-tie)
        n_o, t_o, mg = oracle.verify_row(lg[r], drafts[r], None if q is None else q[r], op, hist[r], u[r])
        if not g.verify_near_tie(mg, n_o, D, oracle.is_greedy(op)):
            assert n_o == n_blk[r] and np.array_equal(t_o, out_blk[r]), (r, n_o, t_o, out_blk[r])
    assert len(lengths) >= 2  # the rows stop at different positions
