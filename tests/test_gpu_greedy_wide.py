"""The greedy verify at wide shapes: many rows at the full vocabulary, and a
vocabulary of 2^20 with maxima deep inside it and an exact tie. Greedy
decisions are argmax matches (value desc, id asc), so they are compared
exactly with the oracle."""
import numpy as np
import pytest
import torch

import mtp_speculative_decoding_step_gb300 as m
import oracle
import synth
from tests import gpu_common as g

pytestmark = pytest.mark.gpu


def _verify_greedy(lg, drafts):
    R, dp1, V = lg.shape
    ws = torch.zeros(m.spec_verify_workspace_bytes(R, dp1 - 1, V), dtype=torch.uint8, device="cuda")
    n_acc = torch.zeros(R, dtype=torch.int32, device="cuda")
    out = torch.zeros((R, dp1), dtype=torch.int32, device="cuda")
    u = torch.full((R, dp1), 0.5, dtype=torch.float32, device="cuda")
    m.spec_verify(g.to_dev(lg), g.to_dev(np.ascontiguousarray(drafts, np.int32)), [dict(temperature=0.0)] * R,
                  u, n_acc, out, ws)
    torch.cuda.synchronize()
    return n_acc.cpu().numpy(), out.cpu().numpy()


def _expect(lg, drafts):
    p = oracle.make_params(0.0)
    res = []
    for r in range(lg.shape[0]):
        n, toks, _ = oracle.verify_row(lg[r], drafts[r], None, p, np.zeros(0, np.int32),
                                       np.full(lg.shape[1], 0.5, np.float32))
        res.append((n, toks))
    return res


@pytest.mark.parametrize("R", [40, 64])
def test_many_greedy_rows_full_vocab(R):
    d, V = 3, 152064
    lg = synth.normal(61, f"gw-lg{R}", (R, d + 1, V), std=4.0)
    am = lg.argmax(2)
    drafts = np.where((np.arange(R)[:, None] + np.arange(d)[None, :]) % 4 == 3, (am[:, :d] + 1) % V, am[:, :d])
    got_n, got_t = _verify_greedy(lg, drafts.astype(np.int32))
    for r, (n, toks) in enumerate(_expect(lg, drafts.astype(np.int32))):
        assert got_n[r] == n and np.array_equal(got_t[r], toks), r


def test_greedy_vocab_2_pow_20():
    d, V = 2, 1 << 20
    lg = synth.normal(62, "gw-big", (1, d + 1, V), std=1.0)
    # each row's maximum sits deep inside a 65536-wide slice, past its first
    # 32768 logits, and row 1 carries an exact tie resolved by the lower id
    lg[0, 0, 5 * 65536 + 60001] = 9.0
    lg[0, 1, 11 * 65536 + 40000] = 9.5
    lg[0, 1, 12 * 65536 + 50000] = 9.5
    lg[0, 2, 15 * 65536 + 65535] = 8.0
    drafts = np.array([[5 * 65536 + 60001, 11 * 65536 + 40000]], np.int32)
    got_n, got_t = _verify_greedy(lg, drafts)
    n, toks = _expect(lg, drafts)[0]
    assert n == 2 and toks[2] == 15 * 65536 + 65535
    assert got_n[0] == n and np.array_equal(got_t[0], toks)
