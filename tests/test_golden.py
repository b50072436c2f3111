"""Pins against values the pages print (fixtures under tests/golden/, each
citing its page and section): the drafter's tensor inventory, the norm
suffixes that take the +1.0 offset, and the round budget. The oracle, the
seeded model generator and the C loader (host validation only, no GPU) must
all agree with them."""
import ctypes
import pathlib

import numpy as np
import pytest

import mtp_speculative_decoding_step_gb300 as m
import oracle
import synth

GOLDEN = pathlib.Path(__file__).parent / "golden"


def _read(name):
    out = {}
    for line in (GOLDEN / name).read_text().splitlines():
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        key, val = line.split(None, 1)
        out.setdefault(key, []).append(val)
    return out


@pytest.fixture(scope="module")
def L():
    from mtp_speculative_decoding_step_gb300 import _build
    _build.build()
    return m.lib()


TENSORS = _read("drafter_tensors.txt")
CONFIG = {k: int(v[0]) for k, v in _read("drafter_config.txt").items()}


def test_fixture_counts_match_the_acceptance_criteria():
    assert len(TENSORS["tensor"]) == len(set(TENSORS["tensor"])) == 15
    assert len(TENSORS["shift"]) == len(set(TENSORS["shift"])) == 7


def test_oracle_and_generator_inventory_is_the_printed_list():
    printed = set(TENSORS["tensor"])
    assert {"mtp." + n for n in synth.INVENTORY} == printed
    assert {"mtp." + n for n in oracle.INVENTORY} == printed


def test_oracle_shift_suffixes_are_the_printed_ones():
    assert set(oracle.SHIFT_SUFFIXES) == set(TENSORS["shift"])


def test_raw_layout_shifts_exactly_the_printed_norms():
    # every raw norm weight is 0 here, so a shifted one reads 1.0 exactly
    s = synth.Shape("g", 256, 4, 2, 64, 768, 2048, dtype="f32")
    shapes = synth.tensor_shapes(s)
    t = {"mtp." + n: np.zeros(shapes[n], np.float32) for n in synth.INVENTORY}
    norms, raw = oracle.load_norms(t)
    assert raw
    want = {n for n in TENSORS["tensor"] if any(n.endswith(x) for x in TENSORS["shift"])}
    assert len(want) == 7
    assert {"mtp." + k for k in norms} == want
    for v in norms.values():
        assert np.all(v == 1.0)


def test_block_size_and_drafts_per_round():
    layers = CONFIG["mtp_num_hidden_layers"]
    assert oracle.default_block_size(layers) == CONFIG["block_size"]
    assert CONFIG["block_size"] - 1 == CONFIG["drafts_per_round"]


def test_c_abi_block_size(L):
    cfg = m.make_config(synth.small_shape(), 1, 256, 2)
    cfg.mtp_layers = CONFIG["mtp_num_hidden_layers"]
    assert L.mtp_default_block_size(ctypes.byref(cfg)) == CONFIG["block_size"]


def test_benchmarked_shape_is_the_printed_27b_config():
    assert synth.QWEN27B.hidden == CONFIG["hidden_size"]
    assert synth.QWEN27B.head_dim == CONFIG["head_dim"]


@pytest.mark.parametrize("drop", range(15))
def test_c_loader_requires_every_printed_tensor(L, drop):
    # host validation only: the pointers are never dereferenced
    FAKE = 0x10000
    s = synth.small_shape()
    shapes = synth.tensor_shapes(s)
    names = [n for i, n in enumerate(TENSORS["tensor"]) if i != drop]
    arr = (m.Tensor * len(names))()
    keep = []
    for i, full in enumerate(names):
        shp = shapes[full[len("mtp."):]]
        b = full.encode()
        keep.append(b)
        arr[i] = m.Tensor(b, FAKE, m.MTP_DTYPE_BF16, len(shp), (ctypes.c_int64 * 2)(*(list(shp) + [0, 0])[:2]))
    cfg = m.make_config(s, 1, 256, 2)
    out = ctypes.c_void_p()
    rc = L.mtp_load(ctypes.byref(cfg), arr, len(names), FAKE, None, m.KV(FAKE, FAKE, FAKE), None, None,
                    ctypes.byref(out))
    assert rc == 2 and out.value is None  # MTP_ERR_MISSING_TENSOR
