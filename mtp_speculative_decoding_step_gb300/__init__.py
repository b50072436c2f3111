"""GB300 multi-token-prediction (MTP) speculative decoding step.

Thin Python binding of ``libmtp.so`` (C ABI declared in ``include/mtp.h``):
argument marshalling only.  Every step of the drafter head, the flush, the
sampling transforms, the verify and the rollback runs in the library's CUDA
kernels; there is no Python or CPU fallback.  Tensors are passed as torch
device tensors (PyTorch supplies device memory and streams only).
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmtp.so")

MTP_DTYPE_F32 = 0
MTP_DTYPE_BF16 = 1

STATUS = {
    0: "MTP_OK", 1: "MTP_ERR_UNSUPPORTED_ARCH", 2: "MTP_ERR_MISSING_TENSOR", 3: "MTP_ERR_DUP_TENSOR",
    4: "MTP_ERR_UNKNOWN_TENSOR", 5: "MTP_ERR_SHAPE", 6: "MTP_ERR_CONFIG_BOUNDS", 7: "MTP_ERR_NOT_BOUND",
    8: "MTP_ERR_KV_CAPACITY", 9: "MTP_ERR_BAD_ARG", 10: "MTP_ERR_NONFINITE", 11: "MTP_ERR_TIMEOUT",
    12: "MTP_ERR_CUDA", 13: "MTP_ERR_LAYOUT",
}

# Every symbol include/mtp.h declares.
EXPORTS = (
    "mtp_default_block_size", "mtp_status_str", "mtp_load", "mtp_free", "mtp_get_lengths",
    "mtp_set_lengths", "mtp_device_status", "mtp_flush", "mtp_draft", "spec_verify_workspace_bytes",
    "spec_verify", "kv_rollback", "mtp_profile_enable", "mtp_profile_kinds", "mtp_profile_kind_name",
    "mtp_profile_read", "mtp_kernel_launches", "spec_verify_noalloc",
    "mtp_depth_ctl_create", "mtp_depth_ctl_free", "mtp_depth_ctl_next", "mtp_depth_ctl_observe",
    "mtp_depth_ctl_state", "mtp_set_draft_head", "mtp_test_verify_stall",
)


class MTPError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {STATUS.get(code, code)}")


class Config(ctypes.Structure):
    _fields_ = [("architecture", ctypes.c_char_p), ("hidden", ctypes.c_int32), ("n_q", ctypes.c_int32),
                ("n_kv", ctypes.c_int32), ("head_dim", ctypes.c_int32), ("inter", ctypes.c_int32),
                ("vocab", ctypes.c_int32), ("mtp_layers", ctypes.c_int32), ("max_rows", ctypes.c_int32),
                ("kv_capacity", ctypes.c_int32), ("max_depth", ctypes.c_int32), ("eps", ctypes.c_float),
                ("rope_theta", ctypes.c_float), ("dtype", ctypes.c_int32)]


class Tensor(ctypes.Structure):
    _fields_ = [("name", ctypes.c_char_p), ("data", ctypes.c_void_p), ("dtype", ctypes.c_int32),
                ("ndim", ctypes.c_int32), ("shape", ctypes.c_int64 * 2)]


class Sampling(ctypes.Structure):
    _fields_ = [("temperature", ctypes.c_float), ("rep_penalty", ctypes.c_float), ("top_p", ctypes.c_float),
                ("min_p", ctypes.c_float), ("top_k", ctypes.c_int32), ("flags", ctypes.c_int32)]


class KV(ctypes.Structure):
    _fields_ = [("k", ctypes.c_void_p), ("v", ctypes.c_void_p), ("len", ctypes.c_void_p)]


_lib = None


def lib():
    """The loaded C library; raises if it has not been built (no fallback)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"libmtp.so is not built at {LIB_PATH}; run __graft_entry__.build()")
        L = ctypes.CDLL(LIB_PATH)
        vp, i32, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t
        L.mtp_default_block_size.argtypes = [ctypes.POINTER(Config)]
        L.mtp_default_block_size.restype = i32
        L.mtp_status_str.argtypes = [ctypes.c_int]
        L.mtp_status_str.restype = ctypes.c_char_p
        L.mtp_load.argtypes = [ctypes.POINTER(Config), ctypes.POINTER(Tensor), i32, vp, vp, KV, vp, vp,
                               ctypes.POINTER(vp)]
        L.mtp_free.argtypes = [vp]
        L.mtp_get_lengths.argtypes = [vp, vp]
        L.mtp_set_lengths.argtypes = [vp, vp, vp]
        L.mtp_device_status.argtypes = [vp]
        L.mtp_device_status.restype = vp
        L.mtp_flush.argtypes = [vp, vp, i32, vp, i32, vp, vp, i32]
        L.mtp_draft.argtypes = [vp, vp, i32, i32, vp, i32, vp, vp, i32, ctypes.POINTER(Sampling), vp, i32,
                                vp, vp, vp, vp, vp]
        L.spec_verify_workspace_bytes.argtypes = [i32, i32, i32]
        L.spec_verify_workspace_bytes.restype = sz
        L.spec_verify.argtypes = [vp, i32, i32, i32, vp, vp, vp, ctypes.POINTER(Sampling), vp, i32, vp, vp,
                                  vp, vp, vp, vp, vp]
        L.spec_verify_noalloc.argtypes = [vp, i32, i32, i32, vp, vp, vp, ctypes.POINTER(Sampling), vp, i32,
                                          vp, vp, vp, vp, vp, vp]
        L.mtp_test_verify_stall.argtypes = [i32, i32]
        L.kv_rollback.argtypes = [vp, vp, i32, vp, vp, i32, i32]
        L.mtp_profile_enable.argtypes = [vp, i32]
        L.mtp_profile_kinds.restype = i32
        L.mtp_profile_kind_name.argtypes = [i32]
        L.mtp_profile_kind_name.restype = ctypes.c_char_p
        L.mtp_profile_read.argtypes = [vp, vp, vp]
        L.mtp_kernel_launches.restype = ctypes.c_int64
        for name in ("mtp_load", "mtp_free", "mtp_get_lengths", "mtp_set_lengths", "mtp_flush", "mtp_draft",
                     "spec_verify", "spec_verify_noalloc", "kv_rollback", "mtp_profile_enable",
                     "mtp_profile_read", "mtp_test_verify_stall"):
            getattr(L, name).restype = ctypes.c_int
        _lib = L
    return _lib


def _check(rc: int, where: str):
    if rc != 0:
        raise MTPError(rc, where)


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


_BF16 = None


def _dtype_code(t) -> int:
    global _BF16
    if _BF16 is None:
        import torch
        _BF16 = torch.bfloat16
    return MTP_DTYPE_BF16 if t.dtype is _BF16 else MTP_DTYPE_F32


def _i32_array(values):
    """Host int32 array for a C pointer argument (a list/tuple or a numpy array)."""
    if isinstance(values, np.ndarray):
        values = values.astype(np.int32, copy=False).ravel().tolist()
    return (ctypes.c_int32 * len(values))(*values)


MTP_SAMPLE_ARGMAX_DRAFT = 1


def sampling_array(params) -> ctypes.Array:
    """params: list of dicts (temperature, rep_penalty, top_k, top_p, min_p,
    argmax_draft) or tuples (temperature, rep_penalty, top_k, top_p, min_p)."""
    arr = (Sampling * len(params))()
    for i, p in enumerate(params):
        flags = 0
        if isinstance(p, dict):
            flags = MTP_SAMPLE_ARGMAX_DRAFT if p.get("argmax_draft", False) else 0
            p = (p.get("temperature", 0.0), p.get("rep_penalty", 1.0), p.get("top_k", 0),
                 p.get("top_p", 1.0), p.get("min_p", 0.0))
        t, r, k, tp, mp = p
        arr[i] = Sampling(float(t), float(r), float(tp), float(mp), int(k), flags)
    return arr


def make_config(shape, max_rows: int, kv_capacity: int, max_depth: int,
                architecture: str = "qwen3_5_mtp") -> Config:
    return Config(architecture.encode(), shape.hidden, shape.n_q, shape.n_kv, shape.head_dim, shape.inter,
                  shape.vocab, 1, max_rows, kv_capacity, max_depth, shape.eps, shape.rope_theta,
                  MTP_DTYPE_BF16 if shape.dtype == "bf16" else MTP_DTYPE_F32)


def mtp_default_block_size(cfg: Config) -> int:
    return lib().mtp_default_block_size(ctypes.byref(cfg))


def mtp_status_str(code: int) -> str:
    return lib().mtp_status_str(code).decode()


class Handle:
    """An mtp_t plus the ctypes objects that must outlive it."""

    def __init__(self, ptr, cfg, keep):
        self.ptr = ptr
        self.cfg = cfg
        self._keep = keep

    def close(self):
        if self.ptr:
            lib().mtp_free(self.ptr)
            self.ptr = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def mtp_load(cfg: Config, tensors: dict, embed, lm_head, kv_k, kv_v, kv_len, lengths=None,
             stream=None) -> Handle:
    """tensors: name -> torch device tensor (names as in the checkpoint)."""
    names = list(tensors)
    arr = (Tensor * len(names))()
    keep = [cfg]
    for i, n in enumerate(names):
        t = tensors[n]
        b = n.encode()
        keep.append(b)
        shp = (ctypes.c_int64 * 2)(*(list(t.shape) + [0, 0])[:2])
        arr[i] = Tensor(b, _ptr(t), _dtype_code(t), t.dim(), shp)
    keep.append(arr)
    kv = KV(_ptr(kv_k), _ptr(kv_v), _ptr(kv_len))
    hl = None
    if lengths is not None:
        hl = np.ascontiguousarray(lengths, dtype=np.int32)
        keep.append(hl)
    out = ctypes.c_void_p()
    rc = lib().mtp_load(ctypes.byref(cfg), arr, len(names), _ptr(embed), _ptr(lm_head), kv,
                        hl.ctypes.data if hl is not None else None, _stream(stream), ctypes.byref(out))
    _check(rc, "mtp_load")
    return Handle(out.value, cfg, keep)


def mtp_get_lengths(h: Handle) -> np.ndarray:
    out = np.zeros(h.cfg.max_rows, np.int32)
    _check(lib().mtp_get_lengths(h.ptr, out.ctypes.data), "mtp_get_lengths")
    return out


def mtp_set_lengths(h: Handle, lengths, stream=None):
    _check(lib().mtp_set_lengths(h.ptr, _stream(stream), _i32_array(lengths)), "mtp_set_lengths")


def mtp_device_status(h: Handle) -> int:
    return lib().mtp_device_status(h.ptr)


def mtp_flush(h: Handle, pairs, tok, hid, stream=None):
    """pairs: host int list [rows]; tok [rows, pmax] int32; hid [rows, pmax, H]."""
    hp = np.ascontiguousarray(pairs, dtype=np.int32)
    rc = lib().mtp_flush(h.ptr, _stream(stream), len(hp), hp.ctypes.data, tok.shape[1], _ptr(tok), _ptr(hid),
                         _dtype_code(hid))
    _check(rc, "mtp_flush")


def mtp_draft(h: Handle, depth: int, pairs, tok, hid, params, draft, hist=None, u=None, q=None, logits=None,
              hidden=None, stream=None):
    # (on the host path between two rounds: argument marshalling kept lean)
    hp = _i32_array(pairs)
    sp = params if isinstance(params, ctypes.Array) else sampling_array(params)
    hist_w = 0 if hist is None else hist.shape[1]
    rc = lib().mtp_draft(h.ptr, stream if type(stream) is int else _stream(stream), len(hp), depth, hp,
                         tok.shape[1], _ptr(tok), _ptr(hid), _dtype_code(hid), sp, _ptr(hist), hist_w, _ptr(u),
                         _ptr(draft), _ptr(q), _ptr(logits), _ptr(hidden))
    _check(rc, "mtp_draft")


def spec_verify_workspace_bytes(rows: int, depth: int, vocab: int) -> int:
    return lib().spec_verify_workspace_bytes(rows, depth, vocab)


def spec_verify(logits, draft, params, u, n_acc, out_tok, workspace, q=None, hist=None, stats=None,
                h_out=None, status=None, stream=None):
    """logits [rows, depth+1, V] f32; draft [rows, depth] i32; u [rows, depth+1] f32;
    status: optional device int32 word (OR of 1 << MTP_ERR_* seen on the device)."""
    rows, dp1, V = logits.shape
    sp = params if isinstance(params, ctypes.Array) else sampling_array(params)
    hist_w = 0 if hist is None else hist.shape[1]
    rc = lib().spec_verify(_stream(stream), rows, dp1 - 1, V, _ptr(logits), _ptr(draft), _ptr(q), sp,
                           _ptr(hist), hist_w, _ptr(u), _ptr(n_acc), _ptr(out_tok), _ptr(stats), _ptr(h_out),
                           _ptr(status), _ptr(workspace))
    _check(rc, "spec_verify")


def spec_verify_noalloc(logits, draft, params, u, n_acc, out_tok, q=None, hist=None, stats=None, h_out=None,
                        status=None, stream=None):
    """spec_verify with the library's fixed scratch instead of a workspace
    (for callers that cannot allocate device memory)."""
    rows, dp1, V = logits.shape
    sp = params if isinstance(params, ctypes.Array) else sampling_array(params)
    hist_w = 0 if hist is None else hist.shape[1]
    rc = lib().spec_verify_noalloc(_stream(stream), rows, dp1 - 1, V, _ptr(logits), _ptr(draft), _ptr(q), sp,
                                   _ptr(hist), hist_w, _ptr(u), _ptr(n_acc), _ptr(out_tok), _ptr(stats),
                                   _ptr(h_out), _ptr(status))
    _check(rc, "spec_verify_noalloc")


def mtp_test_verify_stall(stage: int, wait_polls: int) -> None:
    """Test hook: the next streaming-path spec_verify leaves ring stage
    `stage` unfilled and gives each wait `wait_polls` polls (its waits run out
    and it reports MTP_ERR_TIMEOUT)."""
    _check(lib().mtp_test_verify_stall(int(stage), int(wait_polls)), "mtp_test_verify_stall")


def kv_rollback(h: Handle, rows: int, depth: int, n_acc=None, target_len=None, zero_tail: bool = False,
                stream=None):
    rc = lib().kv_rollback(h.ptr, _stream(stream), rows, _ptr(n_acc), _ptr(target_len), depth,
                           1 if zero_tail else 0)
    _check(rc, "kv_rollback")


PROFILE_KINDS = ("fc", "qkv", "qkv_post", "attention", "o_proj", "gate_up", "down", "lm_head", "sample",
                 "flush_fc", "flush_kv", "rollback")


def mtp_profile_enable(h: Handle, kinds=True):
    """kinds: True (all), False (off), or an iterable of kind names."""
    if kinds is True:
        mask = -1
    elif not kinds:
        mask = 0
    else:
        mask = 0
        for k in kinds:
            mask |= 1 << PROFILE_KINDS.index(k)
    _check(lib().mtp_profile_enable(h.ptr, mask), "mtp_profile_enable")


def mtp_profile_read(h: Handle) -> dict:
    n = lib().mtp_profile_kinds()
    ms = np.zeros(n, np.float32)
    cnt = np.zeros(n, np.int32)
    _check(lib().mtp_profile_read(h.ptr, ms.ctypes.data, cnt.ctypes.data), "mtp_profile_read")
    return {lib().mtp_profile_kind_name(i).decode(): (float(ms[i]), int(cnt[i])) for i in range(n)}


def mtp_kernel_launches() -> int:
    return int(lib().mtp_kernel_launches())


MTP_HEAD_BF16, MTP_HEAD_FP8 = 0, 1


def mtp_set_draft_head(h: Handle, fmt: int, stream=None) -> None:
    """MTP_HEAD_FP8: the drafter reads an e4m3 copy of the tied head (per-row
    scales); MTP_HEAD_BF16: the borrowed head itself."""
    L = lib()
    L.mtp_set_draft_head.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int32]
    _check(L.mtp_set_draft_head(h.ptr, _stream(stream), int(fmt)), "mtp_set_draft_head")


class DepthController:
    """Draft-depth controller (host-side, in libmtp): next() is the depth to
    draft this round, observe(depth, n_acc, seconds) feeds back the round run."""

    def __init__(self, max_depth: int):
        L = lib()
        L.mtp_depth_ctl_create.argtypes = [ctypes.c_int32, ctypes.POINTER(ctypes.c_void_p)]
        L.mtp_depth_ctl_next.argtypes = [ctypes.c_void_p]
        L.mtp_depth_ctl_next.restype = ctypes.c_int32
        L.mtp_depth_ctl_observe.argtypes = [ctypes.c_void_p, ctypes.c_int32, ctypes.c_int32, ctypes.c_double]
        L.mtp_depth_ctl_state.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]
        L.mtp_depth_ctl_free.argtypes = [ctypes.c_void_p]
        self.max_depth = max_depth
        self.ptr = ctypes.c_void_p()
        _check(L.mtp_depth_ctl_create(max_depth, ctypes.byref(self.ptr)), "mtp_depth_ctl_create")

    def next(self) -> int:
        return int(lib().mtp_depth_ctl_next(self.ptr))

    def observe(self, depth: int, n_acc: int, seconds: float) -> None:
        _check(lib().mtp_depth_ctl_observe(self.ptr, depth, n_acc, float(seconds)), "mtp_depth_ctl_observe")

    def state(self):
        a = np.zeros(max(self.max_depth, 1), np.float64)
        c = np.zeros(self.max_depth + 1, np.float64)
        iv = ctypes.c_int32(0)
        _check(lib().mtp_depth_ctl_state(self.ptr, a.ctypes.data, c.ctypes.data, ctypes.byref(iv)),
               "mtp_depth_ctl_state")
        return a[: self.max_depth], c, int(iv.value)

    def close(self):
        if self.ptr:
            lib().mtp_depth_ctl_free(self.ptr)
            self.ptr = ctypes.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
