"""GPU parity of the verify-side transform on wide supports.

Top-p without top-k over the full 152,064-token vocabulary, with logits flat
enough that the kept set runs to tens of thousands of tokens, and with heavily
tied logits (a few distinct values), which push the cut into a crowded
stretch of equal keys.  The transform descriptors that spec_verify leaves in
its workspace (one 32-byte record per row and position: max transformed logit
m, normaliser S, top-k bound (key, id), top-p bound (key, id), argmax, kept
count or -1) are decoded on the host, the kept set they define is rebuilt from the
logits, and both are compared with the oracle's transform: the kept set
exactly (unless the oracle's cumulative mass lies within 1e-6 of the top-p
threshold at the cut, a counted near-tie) and S to 1e-5."""
import numpy as np
import pytest
import torch

import mtp_speculative_decoding_step_gb300 as m
import oracle
import synth
from tests import gpu_common as g

pytestmark = pytest.mark.gpu
V = synth.QWEN27B.vocab
DESC = np.dtype([("m", "<f4"), ("S", "<f4"), ("k_key", "<u4"), ("k_cut", "<i4"), ("p_key", "<u4"),
                 ("p_cut", "<i4"), ("argmax", "<i4"), ("kept", "<i4")])


def _desc_key(z: np.ndarray) -> np.ndarray:
    """Order key of a float32 array: ascending key = descending z."""
    u = z.astype(np.float32).view(np.uint32)
    asc = np.where(u & 0x80000000, ~u, u | 0x80000000).astype(np.uint32)
    return (~asc).astype(np.uint32)


def _transformed(lg, params, window):
    """Penalised, temperature-scaled logits in fp32 (the order the keys follow)."""
    z = lg.astype(np.float32).copy()
    r = np.float32(params.get("rep_penalty", 1.0))
    if r != 1.0 and window.size:
        ids = np.unique(window)
        z[ids] = np.where(z[ids] > 0, z[ids] / r, z[ids] * r)
    # + 0.0 turns -0.0 into +0.0: equal values share one key, as in the kernels
    return ((z / np.float32(params["temperature"])).astype(np.float32) + np.float32(0.0)).astype(np.float32)


def _kept_from_desc(lg, d, params, window):
    key = _desc_key(_transformed(lg, params, window))
    ids = np.arange(V)
    keep = (key < d["k_key"]) | ((key == d["k_key"]) & (ids <= d["k_cut"]))
    keep &= (key < d["p_key"]) | ((key == d["p_key"]) & (ids <= d["p_cut"]))
    return keep


CASES = [
    # (logit std, temperature, top_p, rep_penalty, quantum): quantum > 0 rounds logits to a grid
    (1.43, 0.7, 0.9, 1.0, 0.0),
    (1.0, 1.0, 0.95, 1.0, 0.0),
    (2.0, 0.7, 0.5, 1.1, 0.0),
    (3.0, 0.8, 0.99, 1.0, 0.0),
    (4.0, 0.7, 0.9, 1.0, 0.0),     # peaked: a handful of tokens kept
    (1.0, 1.0, 0.9, 1.0, 0.25),    # ~30 distinct values: crowded ties at the cut
    (0.5, 1.0, 0.6, 1.0, 1.0),     # ~5 distinct values
    (0.0, 1.0, 0.7, 1.0, 0.0),     # all logits equal
]


def test_wide_top_p_descriptors():
    R, depth = len(CASES), 1
    lg = np.zeros((R, depth + 1, V), np.float32)
    rows = []
    for r, (std, t, tp, rp, qn) in enumerate(CASES):
        x = synth.normal(60, f"flat{r}", (depth + 1, V), std=max(std, 1e-3))
        if std == 0.0:
            x = np.full_like(x, 0.25)
        if qn > 0:
            x = (np.round(x / qn) * qn).astype(np.float32)
        lg[r] = x
        rows.append(dict(temperature=t, top_p=tp, rep_penalty=rp))
    hist = synth.randint(60, "hist", (R, 64), V)
    drafts = synth.randint(60, "dr", (R, depth), V)
    q = np.full((R, depth, V), 1.0 / V, np.float32)
    u = synth.uniform(60, "u", (R, depth + 1))
    ws = torch.zeros(m.spec_verify_workspace_bytes(R, depth, V), dtype=torch.uint8, device="cuda")
    n_acc = torch.zeros(R, dtype=torch.int32, device="cuda")
    out = torch.zeros((R, depth + 1), dtype=torch.int32, device="cuda")
    m.spec_verify(g.to_dev(lg), g.to_dev(drafts), rows, g.to_dev(u), n_acc, out, ws, q=g.to_dev(q),
                  hist=g.to_dev(hist))
    torch.cuda.synchronize()
    # the descriptors lead the workspace
    desc = ws.cpu().numpy()[: R * (depth + 1) * DESC.itemsize].view(DESC).reshape(R, depth + 1)
    near = 0
    for r in range(R):
        p = oracle.make_params(**rows[r])
        for i in range(depth + 1):
            # position i's window: the history shifted by the i drafts before it
            window = np.concatenate([hist[r], drafts[r, :i]])[i:].astype(np.int32)
            probs, info = oracle.transform(lg[r, i], p, window)
            want = probs > 0
            got = _kept_from_desc(lg[r, i], desc[r, i], rows[r], window)
            if not np.array_equal(got, want):
                assert info.topp_margin < 1e-6, (r, i, int(got.sum()), int(want.sum()))
                assert abs(int(got.sum()) - int(want.sum())) <= 1, (r, i)
                near += 1
                continue
            z = _transformed(lg[r, i], rows[r], window)
            ez = np.exp(z[want].astype(np.float64) - np.float64(desc[r, i]["m"]))
            assert abs(float(desc[r, i]["S"]) - ez.sum()) <= 1e-5 * ez.sum(), (r, i)
            # the support size is recorded where the path counts it (-1: not needed)
            assert desc[r, i]["kept"] in (-1, want.sum()), (r, i)
    assert near <= 1
