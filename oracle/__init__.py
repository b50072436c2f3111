"""CPU ORACLE — test infrastructure only.

Plain restatement of one multi-token-prediction (MTP) self-speculative decoding
round: the drafter head forward, the batched flush of completed pairs, the
sampling transforms, the rejection-sampling verify and the rollback
bookkeeping.  Only ``tests/``, ``__graft_entry__.smoke()`` and the benchmark's
CPU-baseline leg may import it; the CUDA product path never does, and the two
share no code (the numerics live in ``mtp_oracle.c``).

Sources (page title, section):
  * "support the qwen3_5_mtp drafter" issue, "Where the MTP weights actually
    live": the fifteen ``mtp.*`` tensors;  "Upstream contract to port": the
    module shape, the forward, ``bind`` (borrowed tied lm_head), separate KV
    caches aligned by offsets, ``block_size = depth + 2``, and the sanitize rule
    (+1.0 on exactly seven norm suffixes, only for the raw-HF ``mtp.`` layout).
  * "Ollama qwen3_5 MTP loader and SelfDraft path", Facts: slot S pairs the
    token at S+1 with the target hidden at S; pending pairs flush in batches of
    up to 256; one head call per draft token.
  * Ollama MLX-runner commit log: greedy is the temperature-0 case of
    rejection sampling; the sampler transforms.

Parity pins for every function here live in ``tests/test_oracle_pins.py``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SO = os.path.join(_HERE, "liboracle.so")
_lib = None

# The seven RMSNorm weight suffixes that receive +1.0 in the raw-HF layout
# ("Upstream contract to port", sanitize paragraph).
SHIFT_SUFFIXES = (
    ".input_layernorm.weight",
    ".post_attention_layernorm.weight",
    ".q_norm.weight",
    ".k_norm.weight",
    "norm.weight",
    "pre_fc_norm_embedding.weight",
    "pre_fc_norm_hidden.weight",
)

INVENTORY = (
    "fc.weight", "norm.weight", "pre_fc_norm_embedding.weight", "pre_fc_norm_hidden.weight",
    "layers.0.input_layernorm.weight", "layers.0.post_attention_layernorm.weight",
    "layers.0.mlp.gate_proj.weight", "layers.0.mlp.up_proj.weight", "layers.0.mlp.down_proj.weight",
    "layers.0.self_attn.q_proj.weight", "layers.0.self_attn.k_proj.weight",
    "layers.0.self_attn.v_proj.weight", "layers.0.self_attn.o_proj.weight",
    "layers.0.self_attn.q_norm.weight", "layers.0.self_attn.k_norm.weight",
)


def build(force: bool = False) -> str:
    src = os.path.join(_HERE, "mtp_oracle.c")
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(src):
        tmp = _SO + f".{os.getpid()}.tmp"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
                               src, "-o", tmp, "-lm"])
        os.replace(tmp, _SO)
    return _SO


class _Model(ctypes.Structure):
    _fields_ = [("H", ctypes.c_int), ("nq", ctypes.c_int), ("nkv", ctypes.c_int),
                ("dh", ctypes.c_int), ("I", ctypes.c_int), ("V", ctypes.c_int),
                ("eps", ctypes.c_double), ("theta", ctypes.c_double), ("wdt", ctypes.c_int)] + \
               [(n, ctypes.c_void_p) for n in ("E", "lm", "fc", "wq", "wk", "wv", "wo", "wg", "wu", "wd")] + \
               [(n, ctypes.c_void_p) for n in ("n_emb", "n_hid", "n_in", "n_post", "n_qn", "n_kn", "n_fin")] + \
               [("lmq", ctypes.c_void_p), ("lmq_scale", ctypes.c_void_p)]


class Params(ctypes.Structure):
    """Per-row sampling parameters (temperature 0 = greedy)."""
    _fields_ = [("temperature", ctypes.c_float), ("rep_penalty", ctypes.c_float),
                ("top_p", ctypes.c_float), ("min_p", ctypes.c_float),
                ("top_k", ctypes.c_int), ("reserved", ctypes.c_int)]


class TInfo(ctypes.Structure):
    _fields_ = [("argmax", ctypes.c_int), ("kept", ctypes.c_int), ("top2_gap", ctypes.c_double),
                ("topp_margin", ctypes.c_double), ("minp_margin", ctypes.c_double)]


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        vp, ci = ctypes.c_void_p, ctypes.c_int
        lib.orc_step.argtypes = [vp, ci, vp, ci, vp, vp, ci, ci, ci, vp, vp]
        lib.orc_step.restype = ci
        lib.orc_transform.argtypes = [vp, ci, vp, vp, ci, vp, vp]
        lib.orc_draw.argtypes = [vp, ci, ctypes.c_float, vp]
        lib.orc_draw.restype = ci
        lib.orc_verify_row.argtypes = [ci, ci, vp, vp, vp, vp, vp, ci, vp, vp, vp, vp]
        lib.orc_e4m3_decode.argtypes = [ctypes.c_uint8]
        lib.orc_e4m3_decode.restype = ctypes.c_float
        lib.orc_e4m3_encode.argtypes = [ctypes.c_float]
        lib.orc_e4m3_encode.restype = ctypes.c_uint8
        lib.orc_quantize_rows_e4m3.argtypes = [vp, ci, ci, vp, vp]
        lib.orc_bf16_round.argtypes = [vp, ctypes.c_long, vp]
        lib.orc_set_threads.argtypes = [ci]
        lib.orc_threads.restype = ci
        _lib = lib
    return _lib


def set_threads(n: int) -> None:
    """Threads of the oracle's parallel loops (results do not depend on it)."""
    _load().orc_set_threads(int(n))


def threads() -> int:
    return int(_load().orc_threads())


def bf16_round_bits(x: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (uint16) of fp32 values under the oracle's rounding:
    nearest even, NaN kept a NaN."""
    x = np.ascontiguousarray(x, np.float32).ravel()
    out = np.zeros(x.shape, np.uint16)
    _load().orc_bf16_round(x.ctypes.data, x.size, out.ctypes.data)
    return out


def e4m3_encode(x: float) -> int:
    """fp8 e4m3 code of x: round to nearest even, finite values beyond 448
    saturate to 448."""
    return int(_load().orc_e4m3_encode(float(x)))


def e4m3_decode(c: int) -> float:
    return float(_load().orc_e4m3_decode(int(c)))


def quantize_rows_e4m3(w: np.ndarray):
    """Per-row fp8 e4m3 quantisation of a [rows, cols] matrix (bf16 bit
    patterns or fp32): scale = max|w| / 448 per row, code = e4m3(w / scale),
    in fp32. Returns (codes uint8 [rows, cols], scales fp32 [rows])."""
    a = np.ascontiguousarray(w)
    if a.dtype == np.uint16:
        a = (a.astype(np.uint32) << 16).view(np.float32)
    a = np.ascontiguousarray(a, dtype=np.float32)
    rows, cols = a.shape
    q = np.zeros((rows, cols), np.uint8)
    sc = np.zeros(rows, np.float32)
    _load().orc_quantize_rows_e4m3(_c(a), rows, cols, _c(q), _c(sc))
    return q, sc


def make_params(temperature=0.0, rep_penalty=1.0, top_k=0, top_p=1.0, min_p=0.0) -> Params:
    return Params(temperature, rep_penalty, top_p, min_p, top_k, 0)


def is_greedy(p: Params) -> bool:
    return p.temperature <= 0.0 or p.top_k == 1


def default_block_size(mtp_layers: int) -> int:
    """Round budget including the bonus token: depth + 2 ("Upstream contract to
    port", block_size paragraph); drafts per round = block_size - 1."""
    return int(mtp_layers) + 2


def _c(a):
    return a.ctypes.data


def _norm_vector(arr) -> np.ndarray:
    a = np.asarray(arr)
    if a.dtype == np.uint16:
        a = (a.astype(np.uint32) << 16).view(np.float32)
    return a.astype(np.float64)


def load_norms(tensors: dict) -> tuple[dict, bool]:
    """Apply the layout rule: a table whose names carry the ``mtp.`` prefix is
    raw-HF; there the seven norm suffixes get +1.0, once, and nothing else does.
    Returns (name-without-prefix -> float64 norm vector, raw_hf)."""
    names = list(tensors)
    raw = [n.startswith("mtp.") for n in names]
    if any(raw) and not all(raw):
        raise ValueError("mixed raw-HF and split layouts")
    raw_hf = all(raw) and len(names) > 0
    out = {}
    for n in names:
        base = n[4:] if raw_hf else n
        if base not in INVENTORY:
            raise ValueError(f"unknown tensor {n}")
        if np.asarray(tensors[n]).ndim == 1:
            v = _norm_vector(tensors[n])
            if raw_hf and any(n.endswith(s) for s in SHIFT_SUFFIXES):
                v = v + 1.0
            out[base] = v
    missing = [n for n in INVENTORY if n not in {(m[4:] if raw_hf else m) for m in names}]
    if missing:
        raise ValueError(f"missing tensors {missing}")
    return out, raw_hf


class Head:
    """The MTP head with its borrowed tied lm_head, on host arrays."""

    def __init__(self, shape, tensors: dict, embed: np.ndarray, lm_head: np.ndarray | None = None,
                 lm_fp8: tuple | None = None):
        """lm_fp8: (codes [V, H] uint8, scales [V] fp32) of a quantised draft
        head; the logits then use it (the embedding gather keeps `embed`)."""
        self.s = shape
        self.norms, self.raw_hf = load_norms(tensors)
        w = {(n[4:] if self.raw_hf else n): np.ascontiguousarray(a) for n, a in tensors.items()}
        self.w = w
        self.embed = np.ascontiguousarray(embed)
        self.lm = self.embed if lm_head is None else np.ascontiguousarray(lm_head)
        self.wdt = 1 if shape.dtype == "bf16" else 0
        m = _Model()
        m.H, m.nq, m.nkv, m.dh, m.I, m.V = (shape.hidden, shape.n_q, shape.n_kv, shape.head_dim,
                                            shape.inter, shape.vocab)
        m.eps, m.theta, m.wdt = shape.eps, shape.rope_theta, self.wdt
        m.E, m.lm = _c(self.embed), _c(self.lm)
        L = "layers.0."
        m.fc = _c(w["fc.weight"])
        m.wq, m.wk, m.wv, m.wo = (_c(w[L + f"self_attn.{p}_proj.weight"]) for p in "qkvo")
        m.wg, m.wu, m.wd = (_c(w[L + f"mlp.{p}_proj.weight"]) for p in ("gate", "up", "down"))
        nm = self.norms
        self._keep = [nm[k] for k in nm]
        m.n_emb = _c(nm["pre_fc_norm_embedding.weight"])
        m.n_hid = _c(nm["pre_fc_norm_hidden.weight"])
        m.n_in = _c(nm[L + "input_layernorm.weight"])
        m.n_post = _c(nm[L + "post_attention_layernorm.weight"])
        m.n_qn = _c(nm[L + "self_attn.q_norm.weight"])
        m.n_kn = _c(nm[L + "self_attn.k_norm.weight"])
        m.n_fin = _c(nm["norm.weight"])
        if lm_fp8 is not None:
            self._q = np.ascontiguousarray(lm_fp8[0], dtype=np.uint8)
            self._qs = np.ascontiguousarray(lm_fp8[1], dtype=np.float32)
            m.lmq, m.lmq_scale = _c(self._q), _c(self._qs)
        self.m = m

    # ------------------------------------------------------------------
    def step(self, tok: int, hid: np.ndarray, K: np.ndarray, V: np.ndarray, slot: int,
             logits: bool = True, kv_only: bool = False):
        """One head call at `slot` for the pair (tok, hid).  K, V: this row's
        cache [n_kv][cap][head_dim] (modified in place).  Returns (h2, logits)."""
        hid = np.ascontiguousarray(hid)
        hdt = 1 if hid.dtype == np.uint16 else 0
        if hdt == 0:
            hid = hid.astype(np.float32)
        assert K.flags.c_contiguous and V.flags.c_contiguous
        cap = K.shape[1]
        h2 = np.zeros(self.s.hidden, np.float32)
        lg = np.zeros(self.s.vocab, np.float32) if (logits and not kv_only) else None
        rc = _load().orc_step(ctypes.byref(self.m), int(tok), _c(hid), hdt, _c(K), _c(V), cap,
                              int(slot), 1 if kv_only else 0, _c(h2),
                              _c(lg) if lg is not None else None)
        if rc != 0:
            raise ValueError("bad slot or token")
        return (None if kv_only else h2), lg

    def flush(self, toks, hids, K, V, slot0: int):
        """Write completed pairs (toks[j], hids[j]) into slots slot0 + j.  For a
        one-layer head a slot's K/V depend only on its own pair (fc -> input
        norm -> k/v projection -> k_norm -> RoPE), so the flush runs exactly
        those steps; batching cannot change the result."""
        for j in range(len(toks)):
            self.step(int(toks[j]), hids[j], K, V, slot0 + j, kv_only=True)

    def draft(self, K, V, slot0: int, toks, hids, depth: int, params: Params,
              hist: np.ndarray, u_draft: np.ndarray):
        """One drafting call for one row.

        The first head call consumes the P pairs (toks, hids) at slots
        slot0..slot0+P-1: the first P-1 are pending completed pairs (flushed),
        the last is the newest pair and yields the step-1 logits.  Step k >= 2
        consumes (x_{k-1}, h2 of step k-1) at the next slot.  The draft token of
        step k comes from the transform chain under the window
        ``last W of hist ++ x_1..x_{k-1}``: argmax for greedy rows, else the
        inverse-CDF draw with u_draft[k-1] from q_k.
        Returns dict(drafts, q [depth][V] (None for greedy), logits, h2, margins)."""
        P = len(toks)
        W = len(hist)
        self.flush(toks[:P - 1], hids[:P - 1], K, V, slot0)
        slot = slot0 + P - 1
        tok, hid = int(toks[P - 1]), hids[P - 1]
        drafts, qs, lgs, h2s, margins = [], [], [], [], []
        greedy = is_greedy(params)
        for k in range(1, depth + 1):
            h2, lg = self.step(tok, hid, K, V, slot)
            lgs.append(lg)
            h2s.append(h2)
            win = np.concatenate([hist[min(k - 1, W):], np.array(drafts[max(0, k - 1 - W):], np.int32)]
                                 ).astype(np.int32)
            q, info = transform(lg, params, win)
            if greedy:
                x = info.argmax
                margins.append(info.top2_gap)
            else:
                x, mg = draw(q, float(u_draft[k - 1]))
                margins.append(mg)
                qs.append(q)
            drafts.append(int(x))
            tok, hid, slot = x, h2, slot + 1
        return dict(drafts=np.array(drafts, np.int32), q=(np.stack(qs) if qs else None),
                    logits=np.stack(lgs), h2=np.stack(h2s), margins=np.array(margins))


def transform(logits: np.ndarray, params: Params, window: np.ndarray):
    """Sampler transform chain on one row; returns (probs fp32 [V], TInfo)."""
    lg = np.ascontiguousarray(logits, dtype=np.float32)
    win = np.ascontiguousarray(window, dtype=np.int32)
    V = lg.shape[0]
    probs = np.zeros(V, np.float32)
    info = TInfo()
    _load().orc_transform(_c(lg), V, ctypes.byref(params), _c(win) if win.size else None,
                          int(win.size), _c(probs), ctypes.byref(info))
    return probs, info


def draw(weights: np.ndarray, u: float):
    """Inverse-CDF draw in ascending id order; returns (id, margin)."""
    w = np.ascontiguousarray(weights, dtype=np.float32)
    mg = ctypes.c_double(0.0)
    i = _load().orc_draw(_c(w), w.shape[0], ctypes.c_float(u), ctypes.byref(mg))
    return int(i), mg.value


def verify_row(logits: np.ndarray, drafts: np.ndarray, q, params: Params, hist: np.ndarray,
               u: np.ndarray):
    """Rejection-sampling verify of one row.  logits [d+1][V], drafts [d],
    q [d][V] or None (greedy), hist [W], u [d+1].
    Returns (n_acc, out_tok [d+1], margins [d+1])."""
    lg = np.ascontiguousarray(logits, dtype=np.float32)
    d = lg.shape[0] - 1
    V = lg.shape[1]
    dr = np.ascontiguousarray(drafts, dtype=np.int32)
    qq = None if q is None else np.ascontiguousarray(q, dtype=np.float32)
    if qq is None and not is_greedy(params):
        raise ValueError("sampled rows need q")
    hs = np.ascontiguousarray(hist, dtype=np.int32)
    uu = np.ascontiguousarray(u, dtype=np.float32)
    out = np.zeros(d + 1, np.int32)
    n = ctypes.c_int(0)
    mg = np.zeros(d + 1, np.float64)
    _load().orc_verify_row(V, d, _c(lg), _c(dr), _c(qq) if qq is not None else None,
                           ctypes.byref(params), _c(hs) if hs.size else None, int(hs.size),
                           _c(uu), _c(out), ctypes.byref(n), _c(mg))
    return n.value, out, mg


def rollback_lengths(draft_len_before: int, n_acc: int, target_len: int, depth: int):
    """Cache bookkeeping after a verify with n_acc accepted of `depth` drafts.
    Draft KV: only the slot of the first head call (the genuine pair) survives,
    so its length becomes draft_len_before + P (P = pairs of that call).  Here
    returned for P = 1.  Target KV: trimmed by block - (n_acc + 1) with
    block = depth + 1 positions verified, i.e. every verified position past the
    accepted drafts and the one committed correction or bonus token ("support
    the qwen3_5_mtp drafter" issue, comment on qualifying the qwen3_5 path)."""
    block = depth + 1
    return draft_len_before + 1, target_len - (block - (n_acc + 1))
