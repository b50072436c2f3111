"""The benchmark's algorithmic byte counts, which the lm_head roofline and
the draft step's HBM fraction divide by, written out from the 27B-shaped
head's matrices (bf16 weights and K/V, fp32 logits)."""
import bench
import synth


def test_batch1_step_bytes_of_the_27b_head():
    layer, lm, kv = bench.step_bytes_of(synth.QWEN27B, 4096)
    fc = 5120 * 10240
    qkv = (24 * 256 + 2 * 4 * 256) * 5120
    o = 5120 * 24 * 256
    mlp = 3 * 17408 * 5120
    assert layer == 2 * (fc + qkv + o + mlp) == 786_432_000
    assert lm == 152064 * 5120 * 2 + 152064 * 4 + 5120 * 4 == 1_557_764_096
    assert kv == 2 * (2 * 4 * 256) * 4096 == 16_777_216
    assert layer + lm + kv == 2_360_973_312


def test_step_bytes_follow_the_shape():
    s = synth.small_shape("bf16", vocab=4096)
    layer, lm, kv = bench.step_bytes_of(s, 100)
    H, q, k, inter = 512, 8 * 128, 2 * 128, 1536
    assert layer == 2 * (H * 2 * H + (q + 2 * k) * H + H * q + 3 * inter * H)
    assert lm == 4096 * H * 2 + 4096 * 4 + H * 4
    assert kv == 2 * 2 * k * 100
