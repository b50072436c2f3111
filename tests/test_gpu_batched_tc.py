"""Head calls with several items (rows of a batch plus their pending pairs)
run their GEMVs on the tensor cores: the weights stream through TMA into
tcgen05 MMAs and every activation row travels as a bf16 pair (x_hi = bf16(x),
x_lo = bf16(x - x_hi)).  On a reduced bf16 head of the same family (H=512,
8/2 heads x 128, SwiGLU 1536, vocab 4096; 65536 for a head of more row
tiles than resident CTAs, 4032 for a partial last tile), batches of 8 and 20 rows with
ragged pending pairs (one pass of up to 64 items, and two passes) are compared
with the oracle: logits, the drafter's hidden state and the new KV slots
within 1e-2 of the largest magnitude (bf16 weights and cache), drafted tokens
exactly unless the oracle reports a near-tie."""
import numpy as np
import pytest

import mtp_speculative_decoding_step_gb300 as m
import oracle
import synth
from tests import gpu_common as g

pytestmark = pytest.mark.gpu
S = synth.small_shape("bf16", vocab=4096)
TOL = 1e-2


def _run(R, pend, depth, params, seed, S=S):
    prefill = [int(x) for x in 100 + synth.randint(seed, "pre", (R,), 400)]
    rig = g.Rig(S, seed=seed, rows=R, capacity=640, prefill=prefill, max_depth=depth)
    toks = [[int(t) for t in synth.randint(seed, f"tok{r}", (pend[r],), S.vocab)] for r in range(R)]
    tok, hid = rig.pairs(toks)
    hist = synth.randint(seed, "hist", (R, 64), S.vocab)
    u = synth.uniform(seed, "u", (R, depth))
    out = rig.draft(depth, pend, tok, hid, params, hist=hist, u=u)
    hh = g.to_f32(hid)
    near = 0
    for r in range(R):
        p = oracle.make_params(**params[r])
        ref = rig.oracle_draft(r, depth, toks[r], list(hh[r, :pend[r]]), p, hist=hist[r], u=u[r])
        for k in range(depth):
            assert g.max_rel(out["logits"][r, k], ref["logits"][k]) < TOL, (r, k)
            assert g.max_rel(out["hidden"][r, k], ref["h2"][k]) < TOL, (r, k)
            if ref["q"] is not None:
                assert np.max(np.abs(out["q"][r, k] - ref["q"][k])) < 1e-3 * max(ref["q"][k].max(), 1e-6)
            if g.draft_near_tie(ref["margins"][k], ref["q"] is None, 1e-3):
                near += 1
                break
            assert out["draft"][r, k] == ref["drafts"][k], (r, k)
        # the pending pairs and the first step's slot are genuine KV in both caches
        K, V = rig.kv_host()
        sl = slice(prefill[r], prefill[r] + pend[r])
        assert g.max_rel(K[r, :, sl], g.to_f32(rig.oK[r, :, sl])) < TOL, r
        assert g.max_rel(V[r, :, sl], g.to_f32(rig.oV[r, :, sl])) < TOL, r
    assert near <= max(1, R // 8)
    rig.close()


def test_batch_of_8_rows_ragged_pending_pairs():
    R = 8
    _run(R, [1, 2, 3, 4, 1, 2, 3, 4], 3, [dict(temperature=0.0)] * R, seed=70)


def test_batch_of_8_rows_mixed_sampling():
    R = 8
    params = [dict(temperature=0.0) if r % 2 == 0 else dict(temperature=0.7, top_p=0.9) for r in range(R)]
    _run(R, [1] * R, 3, params, seed=71)


def test_batch_of_8_rows_wide_vocabulary():
    # vocab 65536: 512 row tiles of the tied head, more than one wave of
    # resident CTAs
    R = 8
    params = [dict(temperature=0.0) if r % 2 == 0 else dict(temperature=0.9, top_k=40) for r in range(R)]
    _run(R, [1, 2, 1, 3, 1, 2, 1, 1], 2, params, seed=73, S=synth.small_shape("bf16", vocab=65536))


def test_batch_of_8_rows_partial_last_tile():
    # vocab 4032: the head's last 128-row tile holds 64 rows, so the in-place
    # logits epilogue's writes and per-tile argmax meet rows past the vocabulary
    R = 8
    params = [dict(temperature=0.0) if r % 2 == 0 else dict(temperature=0.9, top_k=40) for r in range(R)]
    _run(R, [1, 2, 1, 3, 1, 2, 1, 1], 2, params, seed=79, S=synth.small_shape("bf16", vocab=4032))


def test_batch_of_20_rows_two_passes():
    # 20 head items + 60 pending pairs = 80 items in the first call: two passes
    R = 20
    _run(R, [4] * R, 2, [dict(temperature=0.0)] * R, seed=72)
