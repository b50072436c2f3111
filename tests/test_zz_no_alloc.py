"""spec_verify_noalloc: the verify for callers that cannot allocate device
memory (hosts whose own pool owns the device, or code where cudaMalloc would
stall or is not allowed). Called through the C ABI twice in a row on the same
inputs, it must give exactly the results of spec_verify with a workspace
(token and acceptance decisions are bit-exact in every parity test), and
the oracle's decisions row by row. This file is collected last on purpose."""
import ctypes

import numpy as np
import pytest
import torch

import mtp_speculative_decoding_step_gb300 as m
import oracle
import synth
from tests import gpu_common as g

pytestmark = pytest.mark.gpu


def _inputs(seed, rows, depth, V):
    lg = synth.normal(seed, "na:lg", (rows, depth + 1, V), std=3.0)
    ql = synth.normal(seed, "na:q", (rows, depth, V), std=3.0)
    q = np.exp(ql - ql.max(-1, keepdims=True))
    q = (q / q.sum(-1, keepdims=True)).astype(np.float32)
    drafts = np.stack([[int(np.searchsorted(np.cumsum(q[r, i].astype(np.float64)),
                                            synth.uniform(seed, f"na:d{r}:{i}", (1,))[0] * q[r, i].sum(),
                                            side="right")) for i in range(depth)] for r in range(rows)])
    drafts = np.minimum(drafts, V - 1).astype(np.int32)
    u = synth.uniform(seed, "na:u", (rows, depth + 1))
    hist = synth.randint(seed, "na:h", (rows, 16), V)
    params = [dict(temperature=0.0) if r % 3 == 0 else
              dict(temperature=0.9, rep_penalty=1.1, top_k=50, top_p=0.9, min_p=0.02) for r in range(rows)]
    return lg, q, drafts, u, hist, params


def test_noalloc_matches_workspace_verify_twice():
    rows, depth, V = 12, 3, 2048
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    for call in range(2):
        lg, q, drafts, u, hist, params = _inputs(60 + call, rows, depth, V)
        args = (dev(lg), dev(drafts), params, dev(u))
        ws = torch.zeros(m.spec_verify_workspace_bytes(rows, depth, V), dtype=torch.uint8, device="cuda")
        n_ref = torch.zeros(rows, dtype=torch.int32, device="cuda")
        o_ref = torch.zeros((rows, depth + 1), dtype=torch.int32, device="cuda")
        m.spec_verify(*args, n_ref, o_ref, ws, q=dev(q), hist=dev(hist))
        n_na = torch.full((rows,), -7, dtype=torch.int32, device="cuda")
        o_na = torch.full((rows, depth + 1), -7, dtype=torch.int32, device="cuda")
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        m.spec_verify_noalloc(*args, n_na, o_na, q=dev(q), hist=dev(hist), status=status)
        torch.cuda.synchronize()
        assert torch.equal(n_ref, n_na), call
        assert torch.equal(o_ref, o_na), call
        assert int(status.item()) == 0
        # and against the oracle, row by row, unless it reports a near-tie
        n_h, o_h = n_na.cpu().numpy(), o_na.cpu().numpy()
        checked = 0
        for r in range(rows):
            p = oracle.make_params(**params[r])
            greedy = oracle.is_greedy(p)
            n, toks, mg = oracle.verify_row(lg[r], drafts[r], None if greedy else q[r], p, hist[r], u[r])
            if g.verify_near_tie(mg, n, depth, greedy):
                continue
            assert n_h[r] == n and np.array_equal(o_h[r], toks), (call, r, n_h[r], n, o_h[r], toks)
            checked += 1
        assert checked >= rows - 1


def test_noalloc_rejects_sizes_above_its_array():
    sp = m.sampling_array([dict(temperature=0.0)] * 65)
    fake = 0x10000
    rc = m.lib().spec_verify_noalloc(None, 65, 16, 64, fake, fake, None, sp, None, 0, fake, fake, fake, None, None,
                                     None)
    assert rc == 9
