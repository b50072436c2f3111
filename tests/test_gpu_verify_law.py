"""GPU verify against the exact law of rejection sampling on a V=8 vocabulary
(Leviathan/Chen; "greedy is a special case of sampled decoding", Ollama
MLX-runner commit log): the first committed token follows the target's
transformed distribution p_0 whatever q is, and given that x_1 = a was
accepted the next one follows p_1(. | a).  The CUDA kernel is evaluated at the
midpoint of every cell of the uniforms' partition (rows of one batched call)
and must reproduce the oracle's decisions cell by cell."""
import numpy as np
import pytest
import torch

import oracle
import synth
from tests import gpu_common as g
from tests import verify_law as vl

pytestmark = pytest.mark.gpu
V = 8


@pytest.mark.parametrize("params", [dict(temperature=1.0),
                                    dict(temperature=0.9, top_k=6, top_p=0.85, min_p=0.05, rep_penalty=1.2)])
def test_gpu_verify_law_v8(params):
    base = synth.normal(21, "enum:rows", (V, 3, V), std=1.5)
    base[:, 0, :] = base[0, 0]
    p = oracle.make_params(**params)
    hist = np.array([3, 5, -1, 3], np.int32)

    def window(drafts):
        i = len(drafts)
        return np.concatenate([hist[min(i, 4):], np.array(drafts, np.int32)]).astype(np.int32)

    def p_of(row, i, drafts):
        return oracle.transform(row, p, window(drafts))[0].astype(np.float64)

    q1 = oracle.transform(synth.normal(21, "enum:q1", (V,), std=1.0), p, window(()))[0]
    q2s = [oracle.transform(synth.normal(21, f"enum:q2:{a}", (V,), std=1.0), p, window((a,)))[0]
           for a in range(V)]
    cases = list(vl.enumerate_cases(lambda a: base[a], p_of, q1, lambda a: q2s[a], V))
    rig = g.Rig(synth.TINY, seed=1, rows=1, capacity=256, prefill=[0], max_depth=2)
    results = []
    near = 0
    for b0 in range(0, len(cases), 64):
        batch = cases[b0:b0 + 64]
        R = len(batch)
        lg = np.stack([c[0] for c in batch]).astype(np.float32)
        dr = np.array([c[1] for c in batch], np.int32)
        qq = np.stack([np.stack(c[2]) for c in batch]).astype(np.float32)
        uu = np.array([c[3] for c in batch], np.float32)
        hh = np.tile(hist, (R, 1))
        got = rig.verify(lg, dr, qq, [params] * R, uu, hist=hh)
        for r in range(R):
            n, out, mg = oracle.verify_row(lg[r], dr[r], qq[r], p, hist, uu[r])
            if np.min(mg) < 1e-6:
                near += 1
            else:
                assert got["n_acc"][r] == n and np.array_equal(got["out_tok"][r], out), (b0 + r, got, n, out)
            results.append((int(got["n_acc"][r]), got["out_tok"][r]))
    law1, law2, acc1 = vl.accumulate(cases, results, V)
    np.testing.assert_allclose(law1, p_of(base[0, 0], 0, ()), rtol=0, atol=5e-6)
    for a in range(V):
        if acc1[a] > 1e-9:
            np.testing.assert_allclose(law2[a] / acc1[a], p_of(base[a, 1], 1, (a,)), rtol=0, atol=5e-6)
    assert near <= 2
    rig.close()
