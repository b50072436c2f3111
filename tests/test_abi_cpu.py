"""Host-side checks of the C ABI that need no GPU: the library loads, exports
every symbol include/mtp.h declares, and mtp_load / spec_verify reject bad
arguments before touching the device (fail-closed named errors, "support the
qwen3_5_mtp drafter" issue: unsupported architectures and incomplete heads
fail closed; the loader never infers MTP from mtp_num_hidden_layers)."""
import ctypes
import os
import re

import pytest

import mtp_speculative_decoding_step_gb300 as m
import synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    from mtp_speculative_decoding_step_gb300 import _build
    _build.build()
    return m.lib()


def test_header_declares_exactly_the_exported_symbols(L):
    hdr = open(os.path.join(ROOT, "include", "mtp.h")).read()
    declared = set(re.findall(r"^[a-z_0-9 \*]*?\b((?:mtp|spec|kv)_[a-z_0-9]+)\(", hdr, re.M))
    assert declared == set(m.EXPORTS)
    for name in m.EXPORTS:
        assert hasattr(L, name), name


def test_block_size_and_status_strings(L):
    cfg = m.make_config(synth.TINY, 1, 256, 2)
    assert m.mtp_default_block_size(cfg) == 3
    assert m.mtp_status_str(1) == "unsupported draft architecture"
    for code in m.STATUS:
        assert m.mtp_status_str(code)


FAKE = 0x10000  # never dereferenced: every case below fails host validation


def _table(shape, raw=True, drop=None, dup=None, extra=None, bad_shape=None, dtype=None):
    shapes = synth.tensor_shapes(shape)
    names = list(synth.INVENTORY)
    if drop:
        names.remove(drop)
    if dup:
        names.append(dup)
    if extra:
        names.append(extra)
    arr = (m.Tensor * len(names))()
    keep = []
    for i, n in enumerate(names):
        shp = shapes.get(n, (3,))
        if bad_shape == n:
            shp = (shp[0] + 64,) + tuple(shp[1:])
        full = ("mtp." + n) if raw else n
        if raw == "mixed" and i == 0:
            full = n
        b = full.encode()
        keep.append(b)
        dt = m.MTP_DTYPE_BF16 if shape.dtype == "bf16" else m.MTP_DTYPE_F32
        arr[i] = m.Tensor(b, FAKE, dtype if dtype is not None else dt, len(shp),
                          (ctypes.c_int64 * 2)(*(list(shp) + [0, 0])[:2]))
    return arr, len(names), keep


def _load(L, cfg, table, embed=FAKE):
    arr, n, _ = table
    out = ctypes.c_void_p()
    kv = m.KV(FAKE, FAKE, FAKE)
    return L.mtp_load(ctypes.byref(cfg), arr, n, embed, None, kv, None, None, ctypes.byref(out))


@pytest.mark.parametrize("case,code", [
    (dict(arch="qwen3_5_moe"), 1),
    (dict(drop="layers.0.mlp.down_proj.weight"), 2),
    (dict(dup="fc.weight"), 3),
    (dict(extra="layers.0.linear_attn.in_proj.weight"), 4),
    (dict(bad_shape="layers.0.self_attn.k_proj.weight"), 5),
    (dict(dtype=m.MTP_DTYPE_F32), 5),
    (dict(layers=2), 6),
    (dict(vocab=2050), 6),
    (dict(head_dim=96), 6),
    (dict(embed=None), 7),
    (dict(raw="mixed"), 13),
])
def test_mtp_load_fails_closed(L, case, code):
    s = synth.Shape("t", 512, 8, 2, 128, 1536, case.get("vocab", 4096), dtype="bf16")
    if "head_dim" in case:
        s = synth.Shape("t", 512, 8, 2, case["head_dim"], 1536, 4096, dtype="bf16")
    cfg = m.make_config(s, 1, 256, 2, architecture=case.get("arch", "qwen3_5_mtp"))
    if "layers" in case:
        cfg.mtp_layers = case["layers"]
    table = _table(s, raw=case.get("raw", True), drop=case.get("drop"), dup=case.get("dup"),
                   extra=case.get("extra"), bad_shape=case.get("bad_shape"), dtype=case.get("dtype"))
    assert _load(L, cfg, table, embed=case.get("embed", FAKE)) == code


def test_config_layer_count_does_not_stand_in_for_tensors(L):
    # a config advertising one MTP layer with no mtp.* tensors is a missing head
    s = synth.small_shape()
    cfg = m.make_config(s, 1, 256, 2)
    arr = (m.Tensor * 0)()
    out = ctypes.c_void_p()
    rc = L.mtp_load(ctypes.byref(cfg), arr, 0, FAKE, None, m.KV(FAKE, FAKE, FAKE), None, None, ctypes.byref(out))
    assert rc == 2 and out.value is None


def test_spec_verify_rejects_bad_arguments_without_launching(L):
    sp = m.sampling_array([dict(temperature=0.0)])
    args = [None, 1, 2, 64, FAKE, FAKE, None, sp, None, 0, FAKE, FAKE, FAKE, None, None, None, FAKE]
    bad = list(args)
    bad[1] = 0
    assert L.spec_verify(*bad) == 9
    bad = list(args)
    bad[16] = None                      # no workspace
    assert L.spec_verify(*bad) == 9
    sp2 = m.sampling_array([dict(temperature=0.7, top_p=0.9)])
    bad = list(args)
    bad[7] = sp2                        # sampled row without q
    assert L.spec_verify(*bad) == 9
    sp3 = m.sampling_array([dict(temperature=0.7, top_p=1.5)])
    bad = list(args)
    bad[7] = sp3
    bad[6] = FAKE
    assert L.spec_verify(*bad) == 9
    assert m.spec_verify_workspace_bytes(8, 3, 152064) >= 8 * 4 * 32


def test_workspace_holds_the_largest_path_layout():
    # the largest of three layouts, each region 256-byte aligned:
    #  - streaming / top-k lists: descriptors (32 bytes each), accept flags and
    #    two kept-list arrays of 256 entries per (row, position);
    #  - greedy stream: one 64-bit key per (range, segment), ranges <= 2048;
    #  - flat transform: descriptors, 64 part slots (8 + 4 bytes) per task, a
    #    2048-bin fixed-point histogram and a 2048-bin one of the crossing bin's
    #    sub-bins, the min-p mass and two counters per
    #    task, a 1024-entry crossing-bin list (key, id), 64 parts x 16 warp
    #    slices of sums (2 x 8 bytes) and two counters per row
    al = lambda b: (b + 255) // 256 * 256
    for rows, depth in ((64, 3), (8, 3), (1, 2)):
        tasks = rows * (depth + 1)
        lists = al(32 * tasks) + al(4 * tasks) + 2 * al(4 * tasks * 256)
        keys = al(8 * (tasks + 2048))
        flat = (al(32 * tasks) + al(8 * tasks * 64) + al(4 * tasks * 64) + 2 * al(8 * tasks * 2048) + al(8 * tasks)
                + al(4 * tasks) + 2 * al(4 * tasks * 1024) + al(16 * rows * 64 * 16) + al(4 * rows) + al(4 * tasks)
                + al(4 * rows))
        assert m.spec_verify_workspace_bytes(rows, depth, 152064) == max(lists, keys, flat), (rows, depth)
    assert m.spec_verify_workspace_bytes(0, 3, 64) == 0


def test_binding_marshals_host_int_arrays_and_dtypes():
    import numpy as np
    import torch
    assert list(m._i32_array([3, 5])) == [3, 5]
    assert list(m._i32_array(np.array([[7], [9]], dtype=np.int64))) == [7, 9]
    assert m._dtype_code(torch.zeros(1, dtype=torch.bfloat16)) == m.MTP_DTYPE_BF16
    assert m._dtype_code(torch.zeros(1, dtype=torch.float32)) == m.MTP_DTYPE_F32


def test_draft_rejects_a_null_handle_before_any_launch(L):
    import torch

    class NullHandle:
        ptr = None

    tok = torch.zeros((1, 3), dtype=torch.int32)
    hid = torch.zeros((1, 3, 256), dtype=torch.bfloat16)
    draft = torch.zeros((1, 2), dtype=torch.int32)
    with pytest.raises(m.MTPError):
        m.mtp_draft(NullHandle(), 2, [1], tok, hid, [dict(temperature=0.0)], draft, stream=0)


def test_verify_stall_hook_rejects_bad_arguments(L):
    assert L.mtp_test_verify_stall(-1, 100) == 9
    assert L.mtp_test_verify_stall(1, 0) == 9
