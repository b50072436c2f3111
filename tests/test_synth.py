"""The seeded input generator: Philox4x32-10 against the known-answer vectors
published with the Random123 library (Salmon et al., SC'11), and the derived
draws' basic laws."""
import numpy as np

import synth


def test_philox_known_answer_vectors():
    kat = [
        ((0, 0, 0, 0), (0, 0), (0x6627E8D5, 0xE169C58D, 0xBC57AC4C, 0x9B00DBD8)),
        ((0xFFFFFFFF,) * 4, (0xFFFFFFFF,) * 2, (0x408F276D, 0x41C83B0E, 0xA20BC7C6, 0x6D5451FD)),
        ((0x243F6A88, 0x85A308D3, 0x13198A2E, 0x03707344), (0xA4093822, 0x299F31D0),
         (0xD16CFE09, 0x94FDCCEB, 0x5001E420, 0x24126EA1)),
    ]
    for ctr, key, want in kat:
        assert list(synth.philox4x32_10(ctr, key)) == list(want)


def test_draws_are_seeded_and_distributed():
    a = synth.normal(3, "x", (200000,))
    assert np.array_equal(a, synth.normal(3, "x", (200000,)))
    assert not np.array_equal(a, synth.normal(4, "x", (200000,)))
    assert abs(a.mean()) < 0.01 and abs(a.std() - 1) < 0.01
    u = synth.uniform(3, "u", (200000,))
    assert u.min() >= 0 and u.max() < 1 and abs(u.mean() - 0.5) < 0.005
    r = synth.randint(3, "r", (200000,), 10)
    assert r.min() == 0 and r.max() == 9
    b = synth.normal(3, "x", (1000,), dtype="bf16")
    np.testing.assert_allclose(synth.bf16_to_f32(b), a[:1000], rtol=2 ** -8)


def test_planted_targets():
    base = synth.normal(1, "pl", (3, 50), std=4.0)
    out = synth.plant_logits(base, [7, 9], [True, False])
    assert out[0].argmax() == 7
    assert out[1].argmax() != 9
    np.testing.assert_array_equal(out[2], base[2])
