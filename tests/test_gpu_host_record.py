"""The round's host record (n_acc then out_tok per row, [rows][depth+2]) that
spec_verify leaves in the caller's host buffer: page-locked memory that the
device can address is written by the verify kernel itself, other host memory
gets a copy after the kernel.  Both must equal the device outputs, for greedy
rows (one-launch argmax verify) and sampled rows (descriptor + draw path)."""
import numpy as np
import pytest
import torch

import mtp_speculative_decoding_step_gb300 as m
import oracle
import synth
from tests import gpu_common as g

pytestmark = pytest.mark.gpu
V = 2048


@pytest.mark.parametrize("pinned", [True, False])
@pytest.mark.parametrize("temperature", [0.0, 0.9])
def test_host_record_matches_device_outputs(pinned, temperature):
    rows, d = 6, 3
    lg = synth.normal(9, f"hr{temperature}", (rows, d + 1, V), std=3.0)
    am = lg.argmax(2)
    coin = synth.uniform(9, "hrc", (rows, d)) < 0.6
    drafts = np.where(coin, am[:, :d], (am[:, :d] + 1) % V).astype(np.int32)
    params = [dict(temperature=temperature)] * rows
    q = None
    if temperature > 0:
        p = oracle.make_params(temperature)
        q = np.stack([[oracle.transform(lg[r, i], p, np.zeros(0, np.int32))[0] for i in range(d)]
                      for r in range(rows)])
    u = synth.uniform(9, "hru", (rows, d + 1))
    ws = torch.zeros(m.spec_verify_workspace_bytes(rows, d, V), dtype=torch.uint8, device="cuda")
    n_acc = torch.zeros(rows, dtype=torch.int32, device="cuda")
    out = torch.zeros((rows, d + 1), dtype=torch.int32, device="cuda")
    h_out = torch.full((rows, d + 2), -7, dtype=torch.int32)
    if pinned:
        h_out = h_out.pin_memory()
    for _ in range(2):  # twice: the second call overwrites the first record
        m.spec_verify(g.to_dev(lg), g.to_dev(drafts), params, g.to_dev(u), n_acc, out, ws,
                      q=None if q is None else g.to_dev(q), h_out=h_out)
        torch.cuda.synchronize()
        rec = h_out.numpy()
        np.testing.assert_array_equal(rec[:, 0], n_acc.cpu().numpy())
        np.testing.assert_array_equal(rec[:, 1:], out.cpu().numpy())
        h_out.fill_(-7)
    if temperature == 0.0:
        # greedy: accepted prefix = drafts equal to the argmax of the row before
        for r in range(rows):
            n = 0
            while n < d and drafts[r, n] == am[r, n]:
                n += 1
            assert int(n_acc[r]) == n
