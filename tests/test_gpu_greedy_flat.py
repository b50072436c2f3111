"""The greedy verify over many rows as one balanced stream (equal ranges of
the flattened [rows][depth+1][V] logits per CTA, one key per touched segment,
a per-row finish): exact argmax matches against the oracle where ranges cross
many segments (small vocabularies, every thread's consecutive loads landing
in different segments), at the deepest block, with exact ties split across
ranges (the lower id wins), and with -0.0 / +0.0 maxima (equal values: the
lower id wins, as in the oracle's comparison). Vocabularies that are not a
multiple of 4 take the one-launch cluster kernel instead, checked the same way."""
import numpy as np
import pytest
import torch

import mtp_speculative_decoding_step_gb300 as m
import oracle
import synth
from tests import gpu_common as g

pytestmark = pytest.mark.gpu


def _verify(lg, drafts):
    R, dp1, V = lg.shape
    ws = torch.zeros(m.spec_verify_workspace_bytes(R, dp1 - 1, V), dtype=torch.uint8, device="cuda")
    n_acc = torch.full((R,), -7, dtype=torch.int32, device="cuda")
    out = torch.full((R, dp1), -7, dtype=torch.int32, device="cuda")
    stats = torch.zeros((R, dp1 + 1), dtype=torch.int32, device="cuda")
    u = torch.full((R, dp1), 0.5, dtype=torch.float32, device="cuda")
    m.spec_verify(g.to_dev(np.ascontiguousarray(lg)), g.to_dev(np.ascontiguousarray(drafts, np.int32)),
                  [dict(temperature=0.0)] * R, u, n_acc, out, ws, stats=stats)
    torch.cuda.synchronize()
    return n_acc.cpu().numpy(), out.cpu().numpy(), stats.cpu().numpy()


def _check(lg, drafts):
    got_n, got_t, st = _verify(lg, drafts)
    p = oracle.make_params(0.0)
    d = drafts.shape[1]
    lengths = set()
    for r in range(lg.shape[0]):
        n, toks, _ = oracle.verify_row(lg[r], drafts[r], None, p, np.zeros(0, np.int32),
                                       np.full(d + 1, 0.5, np.float32))
        assert got_n[r] == n and np.array_equal(got_t[r], toks), (r, got_n[r], n, got_t[r], toks)
        assert st[r, 0] == 1 and st[r, 1] == (1 if n < d else 0) and list(st[r, 2:]) == [1] * n + [0] * (d - n)
        lengths.add(n)
    return lengths


def _drafts(lg, seed):
    R, dp1, V = lg.shape
    d = dp1 - 1
    am = lg[:, :d].argmax(-1)
    miss = synth.uniform(seed, "gf:miss", (R, d)) < 0.25
    return np.where(miss, (am + 1 + synth.randint(seed, "gf:off", (R, d), V - 1)) % V, am).astype(np.int32)


@pytest.mark.parametrize("R,d,V", [(64, 16, 64), (64, 16, 1024), (48, 7, 4100 - 4), (64, 3, 152064), (1, 2, 152064),
                                   (8, 3, 32766), (40, 3, 152062)])
def test_flat_greedy_matches_oracle(R, d, V):
    # (the last two vocabularies are not multiples of 4: one cluster per row
    # in a single launch takes them)
    lg = synth.normal(80 + d, f"gf:lg{V}", (R, d + 1, V), std=3.0)
    lengths = _check(lg, _drafts(lg, 80 + d))
    assert R < 8 or len(lengths) >= 2


def test_flat_greedy_ties_across_ranges_and_signed_zeros():
    R, d, V = 64, 3, 152064
    lg = synth.normal(90, "gf:ties", (R, d + 1, V), std=1.0)
    # an exact tie of the maximum at both ends of a segment: far apart, so in
    # different ranges; the lower id wins
    lg[3, 1, 10] = 50.0
    lg[3, 1, V - 5] = 50.0
    lg[17, 0, V - 3] = 40.0
    lg[17, 0, 2] = 40.0
    # a segment whose maximum is zero: -0.0 at a lower id than +0.0
    lg[30, 2, :] = -np.abs(lg[30, 2, :]) - 1.0
    lg[30, 2, 100] = -0.0
    lg[30, 2, 120000] = 0.0
    drafts = lg[:, :d].argmax(-1).astype(np.int32)
    drafts[3, 1] = 10
    drafts[17, 0] = 2
    drafts[30, 2] = 100
    _check(lg, drafts)
    got_n, got_t, _ = _verify(lg, drafts)
    assert got_n[3] >= 2 and got_t[3, 1] == 10
    assert got_t[17, 0] == 2
