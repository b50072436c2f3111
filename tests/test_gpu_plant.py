"""The benchmark's device-side target planting (synth/plant.cu) against
synth.plant_logits, the host rule it restates: row i gets logit[x_{i+1}] =
max + 1 when coin i is set, else second - 1 if x_{i+1} was the argmax."""
import numpy as np
import pytest

import synth

pytestmark = pytest.mark.gpu


def test_plant_device_matches_host_rule():
    import torch
    V, D = 4096, 5
    base = synth.normal(11, "plant:base", (D + 1, V), std=4.0)
    order = np.argsort(-base[:D].astype(np.float64), axis=-1, kind="stable")
    top1 = np.take_along_axis(base[:D], order[:, :1], axis=-1)[:, 0].astype(np.float32)
    top2 = np.take_along_axis(base[:D], order[:, 1:2], axis=-1)[:, 0].astype(np.float32)
    arg1 = order[:, 0].astype(np.int64)
    # drafts: argmax hits, misses and a repeated token
    drafts = np.array([arg1[0], 7, arg1[2], 7, arg1[4]], np.int32)
    coins = np.array([False, True, True, False, False])
    want = synth.plant_logits(base, drafts, coins)
    dev = torch.device("cuda", 0)
    lg = torch.from_numpy(base).to(dev).contiguous()
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)
    d, c, t1, t2, a1 = t(drafts[None]), t(coins.astype(np.uint8)), t(top1), t(top2), t(arg1)
    synth.plant_device(torch.cuda.current_stream().cuda_stream, lg.data_ptr(), V, d.data_ptr(), D,
                       c.data_ptr(), t1.data_ptr(), t2.data_ptr(), a1.data_ptr())
    got = lg.cpu().numpy()
    assert np.array_equal(got, want)
