"""Flush of completed pairs on the tcgen05 path (bf16 heads, >= 16 pairs) on a
reduced head of the same family (H=512, 8/2 heads x 128, SwiGLU 1536), against
the oracle slot by slot; and the GEMV path (< 16 pairs) on the same head.
A slot's K/V depend only on its own pair ("Ollama qwen3_5 MTP loader and
SelfDraft path": slot S pairs the token at S+1 with the target hidden at S)."""
import numpy as np
import pytest

import mtp_speculative_decoding_step_gb300 as m
import synth
from tests import gpu_common as g

pytestmark = pytest.mark.gpu
S = synth.small_shape("bf16", vocab=4096)
TOL = 1e-2


@pytest.mark.parametrize("npairs,offset", [(64, 0), (200, 77), (256, 1000), (5, 3)])
def test_flush_small_head(npairs, offset):
    rig = g.Rig(S, seed=8, rows=1, capacity=(offset + 320 + 63) // 64 * 64, prefill=[offset], max_depth=2)
    toks = synth.randint(8, f"f{npairs}:tok", (npairs,), S.vocab)
    tok, hid = rig.pairs([list(toks)], seed_tag=f"f{npairs}")
    m.mtp_flush(rig.h, [npairs], tok, hid)
    assert list(m.mtp_get_lengths(rig.h)) == [offset + npairs]
    rig.oracle_flush(0, toks, list(g.to_f32(hid)[0]))
    K, V = rig.kv_host()
    sl = slice(offset, offset + npairs)
    assert g.max_rel(K[0, :, sl], g.to_f32(rig.oK[0, :, sl])) < TOL
    assert g.max_rel(V[0, :, sl], g.to_f32(rig.oV[0, :, sl])) < TOL
    assert np.all(K[0, :, offset + npairs:offset + 320] == 0)
    rig.close()


def test_flush_two_rows_ragged():
    rig = g.Rig(S, seed=9, rows=2, capacity=512, prefill=[10, 300], max_depth=2)
    t0 = synth.randint(9, "a", (40,), S.vocab)
    t1 = synth.randint(9, "b", (7,), S.vocab)
    tok, hid = rig.pairs([list(t0), list(t1)])
    m.mtp_flush(rig.h, [40, 7], tok, hid)
    assert list(m.mtp_get_lengths(rig.h)) == [50, 307]
    hh = g.to_f32(hid)
    rig.oracle_flush(0, t0, list(hh[0, :40]))
    rig.oracle_flush(1, t1, list(hh[1, :7]))
    K, V = rig.kv_host()
    assert g.max_rel(K[0, :, 10:50], g.to_f32(rig.oK[0, :, 10:50])) < TOL
    assert g.max_rel(V[1, :, 300:307], g.to_f32(rig.oV[1, :, 300:307])) < TOL
    rig.close()
