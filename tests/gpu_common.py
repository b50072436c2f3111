"""Shared set-up for the GPU parity tests: one synthetic head loaded both into
the CUDA library (through the C ABI) and into the CPU oracle, with separate
copies of the draft KV cache on each side."""
from __future__ import annotations

import numpy as np
import torch

import mtp_speculative_decoding_step_gb300 as m
import oracle
import synth


def to_dev(a: np.ndarray, dtype: str | None = None):
    """numpy -> cuda tensor; uint16 arrays are bf16 bit patterns."""
    if a.dtype == np.uint16:
        return torch.from_numpy(np.ascontiguousarray(a)).view(torch.bfloat16).cuda()
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def to_f32(t) -> np.ndarray:
    if isinstance(t, np.ndarray):
        return synth.bf16_to_f32(t) if t.dtype == np.uint16 else t.astype(np.float32)
    return t.detach().float().cpu().numpy()


def max_rel(got, ref) -> float:
    """max |got - ref| / max(|ref|_inf, 1e-6) over the whole tensor."""
    g = to_f32(got).astype(np.float64)
    r = to_f32(ref).astype(np.float64)
    return float(np.max(np.abs(g - r)) / max(np.max(np.abs(r)), 1e-6))


class Rig:
    def __init__(self, shape, seed, rows, capacity, prefill, max_depth, raw_hf=True, model=None):
        self.s = shape
        self.seed = seed
        self.rows = rows
        self.model = model or synth.make_model(shape, seed, raw_hf=raw_hf)
        K, V = synth.kv_prefill(shape, seed, rows, capacity, prefill)
        self.oK, self.oV = K, V                      # oracle's copies (modified in place)
        self.olen = list(prefill)
        self.kk, self.vv = to_dev(K.copy()), to_dev(V.copy())
        self.len = torch.tensor(list(prefill), dtype=torch.int32, device="cuda")
        self.dev = {n: to_dev(a) for n, a in self.model.tensors.items()}
        self.embed = to_dev(self.model.embed)
        self.cfg = m.make_config(shape, rows, capacity, max_depth)
        self.h = m.mtp_load(self.cfg, self.dev, self.embed, None, self.kk, self.vv, self.len, lengths=prefill)
        self.orc = oracle.Head(shape, self.model.tensors, self.model.embed)
        self.ws = None

    def close(self):
        self.h.close()
        self.dev = self.embed = self.kk = self.vv = None
        torch.cuda.empty_cache()

    # ---------------------------------------------------------------- inputs
    def pairs(self, toks, seed_tag="pairs"):
        """toks: list of per-row token lists (ragged). Returns device (tok, hid)
        padded to pmax; hiddens N(0,1) in the model dtype."""
        pmax = max(len(t) for t in toks)
        tok = np.zeros((self.rows, pmax), np.int32)
        for r, t in enumerate(toks):
            tok[r, :len(t)] = t
        hid = synth.normal(self.seed, seed_tag + ":hid", (self.rows, pmax, self.s.hidden), dtype=self.s.dtype)
        return to_dev(tok), to_dev(hid)

    # ---------------------------------------------------------------- GPU
    def draft(self, depth, pairs, tok, hid, params, hist=None, u=None, want_q=None):
        R, V, H = self.rows, self.s.vocab, self.s.hidden
        draft = torch.full((R, depth), -1, dtype=torch.int32, device="cuda")
        logits = torch.zeros((R, depth, V), dtype=torch.float32, device="cuda")
        hidden = torch.zeros((R, depth, H), dtype=torch.float32, device="cuda")
        sampled = any(not oracle.is_greedy(oracle.make_params(**p)) for p in params)
        q = torch.zeros((R, depth, V), dtype=torch.float32, device="cuda") if (sampled or want_q) else None
        hist_d = to_dev(hist) if hist is not None else None
        u_d = to_dev(u) if u is not None else None
        m.mtp_draft(self.h, depth, pairs[:R], tok, hid, params, draft, hist=hist_d, u=u_d, q=q, logits=logits,
                    hidden=hidden)
        torch.cuda.synchronize()
        return dict(draft=draft.cpu().numpy(), logits=logits.cpu().numpy(), hidden=hidden.cpu().numpy(),
                    q=None if q is None else q.cpu().numpy())

    def verify(self, logits, drafts, q, params, u, hist=None, stats=None):
        R, dp1, V = logits.shape
        ws_bytes = m.spec_verify_workspace_bytes(R, dp1 - 1, V)
        ws = torch.zeros(ws_bytes, dtype=torch.uint8, device="cuda")
        n_acc = torch.zeros(R, dtype=torch.int32, device="cuda")
        out = torch.zeros((R, dp1), dtype=torch.int32, device="cuda")
        m.spec_verify(to_dev(logits), to_dev(np.ascontiguousarray(drafts, np.int32)), params,
                      to_dev(np.ascontiguousarray(u, np.float32)), n_acc, out, ws,
                      q=None if q is None else to_dev(q), hist=None if hist is None else to_dev(hist),
                      stats=stats)
        torch.cuda.synchronize()
        return dict(n_acc=n_acc.cpu().numpy(), out_tok=out.cpu().numpy())

    def kv_host(self):
        return self.kk.float().cpu().numpy(), self.vv.float().cpu().numpy()

    # ---------------------------------------------------------------- oracle
    def oracle_draft(self, r, depth, toks, hids, params, hist=None, u=None):
        hist = np.zeros(0, np.int32) if hist is None else np.asarray(hist, np.int32)
        u = np.zeros(depth, np.float32) if u is None else u
        out = self.orc.draft(self.oK[r], self.oV[r], self.olen[r], list(toks), list(hids), depth, params,
                             hist, u)
        self.olen[r] += len(toks) + depth - 1
        return out

    def oracle_flush(self, r, toks, hids):
        self.orc.flush(toks, hids, self.oK[r], self.oV[r], self.olen[r])
        self.olen[r] += len(toks)


# Near-tie bands.  Accept tests: |p/q - u| < 1e-3 (the workload's stated band).
# Inverse-CDF draws: the threshold within 1e-5 of a cumulative boundary (the two
# sides' cumulative sums differ by ~1e-7 of the total).  Greedy argmax over
# recomputed logits: top-2 gap below GAP.
ACCEPT_BAND = 1e-3
DRAW_BAND = 1e-5


def verify_near_tie(mg, n, d, greedy, gap=0.0):
    """Oracle margins of one verified row -> True if any decision was a near-tie."""
    acc = mg[: min(n + 1, d)]
    if greedy:
        return bool(np.min(np.append(acc, mg[d])) <= gap)
    return bool((acc.size and np.min(acc) < ACCEPT_BAND) or mg[d] < DRAW_BAND)


def draft_near_tie(margin, greedy, gap):
    return margin <= gap if greedy else margin < DRAW_BAND


class _DevPtr:
    """A raw device pointer presented through the CUDA array interface, so
    that torch can view library-owned device memory without copying it."""

    def __init__(self, ptr: int, n: int):
        self.__cuda_array_interface__ = {"shape": (n,), "typestr": "<i4", "data": (int(ptr), False),
                                         "version": 3}


def device_i32(ptr: int, n: int = 1):
    """torch int32 view of n words at a device address owned by the library."""
    return torch.as_tensor(_DevPtr(ptr, n), device="cuda")


NONFINITE = 1 << 10   # 1 << MTP_ERR_NONFINITE
TIMEOUT = 1 << 11     # 1 << MTP_ERR_TIMEOUT
