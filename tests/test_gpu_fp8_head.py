"""The fp8 draft head (mtp_set_draft_head with MTP_HEAD_FP8): an e4m3 copy
of the tied output head, one fp32 scale per row, read by the drafter's logits
only. On a reduced bf16 head of the same family (H=512, vocab 4096 or 4032),
a batch of 1 and a batch of 8 are compared with the oracle quantising the
same head the same way; vocab 4096 runs the fp8 head on the tensor cores,
4032 (not a multiple of 128 rows) on the CUDA cores. Logits must agree within
1e-2 of the largest magnitude, as for every bf16 head, and drafts exactly
unless the oracle reports a near-tie. The fp8
logits must also differ from the bf16 head's, which shows that the copy is in
use, and switching back must restore the bf16 head. The same comparison runs
at the 27B shape the benchmark times (H 5120, vocab 152064, KV 4096)."""
import numpy as np
import pytest

import mtp_speculative_decoding_step_gb300 as m
import oracle
import synth
from tests import gpu_common as g

pytestmark = pytest.mark.gpu
S = synth.small_shape("bf16", vocab=4096)
TOL = 1e-2


# vocab 4096 takes the tensor-core fp8 GEMV (row groups of 128); 4032 (a
# multiple of 64 only) takes the CUDA-core one
@pytest.mark.parametrize("vocab", [4096, 4032])
@pytest.mark.parametrize("R", [1, 8])
def test_fp8_head_matches_the_oracle(R, vocab):
    depth = 2
    prefill = [40 + 7 * r for r in range(R)]
    S = synth.small_shape("bf16", vocab=vocab)
    rig = g.Rig(S, seed=61, rows=R, capacity=256, prefill=prefill, max_depth=depth)
    q, sc = oracle.quantize_rows_e4m3(rig.model.embed)
    orc_bf16 = rig.orc
    rig.orc = oracle.Head(S, rig.model.tensors, rig.model.embed, lm_fp8=(q, sc))
    m.mtp_set_draft_head(rig.h, m.MTP_HEAD_FP8)
    toks = [[int(t)] for t in synth.randint(61, "t", (R,), S.vocab)]
    tok, hid = rig.pairs(toks)
    oK, oV, olen = rig.oK.copy(), rig.oV.copy(), list(rig.olen)
    out = rig.draft(depth, [1] * R, tok, hid, [dict(temperature=0.0)] * R)
    hh = g.to_f32(hid)
    for r in range(R):
        ref = rig.oracle_draft(r, depth, toks[r], list(hh[r, :1]), oracle.make_params(0.0))
        for k in range(depth):
            assert g.max_rel(out["logits"][r, k], ref["logits"][k]) < TOL, (r, k)
            if ref["margins"][k] <= 1e-3:
                break
            assert out["draft"][r, k] == ref["drafts"][k], (r, k)
    # the bf16 head gives different logits for the same first step
    _, l_bf16 = orc_bf16.step(toks[0][0], hh[0, 0], oK[0], oV[0], olen[0])
    assert g.max_rel(out["logits"][0, 0], l_bf16) > 1e-3
    rig.close()


def test_switching_back_restores_the_bf16_head():
    depth = 1
    rig = g.Rig(S, seed=62, rows=1, capacity=128, prefill=[30], max_depth=depth)
    tok, hid = rig.pairs([[17]])
    m.mtp_set_draft_head(rig.h, m.MTP_HEAD_FP8)
    m.mtp_set_draft_head(rig.h, m.MTP_HEAD_BF16)
    out = rig.draft(depth, [1], tok, hid, [dict(temperature=0.0)])
    ref = rig.oracle_draft(0, depth, [17], list(g.to_f32(hid)[0, :1]), oracle.make_params(0.0))
    assert g.max_rel(out["logits"][0, 0], ref["logits"][0]) < TOL
    rig.close()


def test_fp8_head_at_the_27b_shape(model27):
    # the shape the benchmark times: H 5120, vocab 152064, KV 4096, depth 2;
    # the seeded case has clear argmaxes under the quantised head (top-2 gaps
    # about 0.30 on both steps), so both drafts must match exactly
    S27 = synth.QWEN27B
    rig = g.Rig(S27, seed=2, rows=1, capacity=4096 + 256, prefill=[4096], max_depth=2, model=model27)
    q, sc = oracle.quantize_rows_e4m3(rig.model.embed)
    rig.orc = oracle.Head(S27, rig.model.tensors, rig.model.embed, lm_fp8=(q, sc))
    m.mtp_set_draft_head(rig.h, m.MTP_HEAD_FP8)
    toks = [1234, 77, 150000]
    tok, hid = rig.pairs([toks])
    out = rig.draft(2, [3], tok, hid, [dict(temperature=0.0)])
    ref = rig.oracle_draft(0, 2, toks, g.to_f32(hid)[0], oracle.make_params(0.0))
    assert g.max_rel(out["logits"][0, 0], ref["logits"][0]) < TOL
    assert ref["margins"][0] > 1e-2 and out["draft"][0, 0] == ref["drafts"][0]
    assert g.max_rel(out["logits"][0, 1], ref["logits"][1]) < TOL
    assert ref["margins"][1] > 1e-2 and out["draft"][0, 1] == ref["drafts"][1]
    rig.close()
