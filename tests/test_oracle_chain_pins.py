"""Pins of the oracle's multi-step parts: how a drafting call chains its head
calls, the per-position repetition-penalty window of the draft steps and of
the verify, the verify's fallback when the residual has no mass, and the
chain-equals-block property of the verify.

Every expected value here is rebuilt by hand from the definitions: the head
calls are chained with explicit slots and hiddens, the windows are spelled out
position by position, the penalised softmax is recomputed in numpy and draws
come from numpy's cumulative sums.  Each pin is paired with a planted mistake
(a mutant chaining or window) that must change the result, so the pin can
fail."""
import numpy as np
import pytest

import oracle
import synth

P = oracle.make_params
EMPTY = np.zeros(0, np.int32)


# ---------------------------------------------------------------- helpers

def _rms(x, w, eps):
    x = np.asarray(x, np.float64)
    return x / np.sqrt(np.mean(x * x) + eps) * w


def _penalise(z, window, r):
    """Repetition penalty over the distinct valid tokens of `window`, in fp32
    (z / r where z > 0, else z * r)."""
    z = np.array(z, np.float32)
    seen = set()
    for t in window:
        t = int(t)
        if t < 0 or t >= z.size or t in seen:
            continue
        seen.add(t)
        z[t] = z[t] / np.float32(r) if z[t] > 0 else z[t] * np.float32(r)
    return z


def _softmax_p(z, window, T, r):
    """Penalised, tempered softmax with no truncation, in float64."""
    zz = _penalise(z, window, r) / np.float32(T)
    e = np.exp(zz.astype(np.float64) - zz.max())
    return e / e.sum()


def _draw(w, u):
    """Smallest id whose cumulative weight (ascending ids) exceeds u * sum;
    also the relative distance of the threshold to the nearest boundary."""
    w = np.asarray(w, np.float64)
    c = np.cumsum(w)
    thr = float(u) * c[-1]
    i = int(np.searchsorted(c, thr, side="right"))
    while w[i] == 0.0:
        i += 1
    edges = np.concatenate([[0.0], c])
    return i, float(np.min(np.abs(edges - thr)) / c[-1])


def _window(hist, drafts, i, W):
    """The penalty window of target row i (or of draft step i + 1): the last W
    tokens of the history followed by the first i drafts."""
    seq = list(hist) + list(drafts[:i])
    return np.array(seq[-W:] if W > 0 else [], np.int32)


# ------------------------------------------------- drafting call chaining

def _hand_chain(head, K, V, slot0, toks, hids, depth, chain_hidden, next_slot):
    """Chain head calls by hand: pending pairs at slot0.., the newest pair at
    slot0 + P - 1, then step k >= 2 at the slot chosen by next_slot with the
    hidden chosen by chain_hidden.  Greedy drafts (argmax, lowest id)."""
    P_ = len(toks)
    for j in range(P_ - 1):
        head.step(int(toks[j]), hids[j], K, V, slot0 + j, kv_only=True)
    slot, tok, hid = slot0 + P_ - 1, int(toks[-1]), hids[-1]
    drafts, lgs, h2s = [], [], []
    for _ in range(depth):
        h2, lg = head.step(tok, hid, K, V, slot)
        x = int(np.argmax(lg))
        drafts.append(x)
        lgs.append(lg)
        h2s.append(h2)
        tok, hid, slot = x, chain_hidden(h2), next_slot(slot)
    return np.array(drafts, np.int32), np.stack(lgs), np.stack(h2s)


@pytest.mark.parametrize("depth,npairs", [(2, 1), (3, 3)])
def test_draft_chains_prenorm_hidden_at_the_next_slots(depth, npairs):
    # Facts ("Ollama qwen3_5 MTP loader and SelfDraft path"): slot S pairs the
    # token at S+1 with the hidden at S; pending pairs go before the newest
    # pair, which yields the first draft; each later head call takes the
    # previous draft token with the head's own hidden, one slot further on.
    s = synth.TINY
    mdl = synth.make_model(s, 41)
    head = oracle.Head(s, mdl.tensors, mdl.embed)
    slot0 = 20
    toks = synth.randint(41, "chain:tok", (npairs,), s.vocab)
    hids = synth.normal(41, "chain:hid", (npairs, s.hidden))
    K1, V1 = synth.kv_prefill(s, 41, 1, 64, [slot0])
    K2, V2 = K1.copy(), V1.copy()
    out = head.draft(K1[0], V1[0], slot0, toks, hids, depth, P(0.0), EMPTY, np.zeros(depth, np.float32))
    d, lg, h2 = _hand_chain(head, K2[0], V2[0], slot0, toks, hids, depth, lambda h: h, lambda t: t + 1)
    np.testing.assert_array_equal(out["drafts"], d)
    np.testing.assert_array_equal(out["logits"], lg)
    np.testing.assert_array_equal(out["h2"], h2)
    np.testing.assert_array_equal(K1, K2)
    np.testing.assert_array_equal(V1, V2)
    # every written slot holds a value; nothing past the last head call
    last = slot0 + npairs + depth - 2
    assert np.all(np.abs(K1[0][:, slot0:last + 1]).sum(axis=-1) > 0)
    np.testing.assert_array_equal(K1[0][:, last + 1:], synth.kv_prefill(s, 41, 1, 64, [slot0])[0][0][:, last + 1:])

    # planted mistakes: chaining the final-normed hidden, or reusing the slot
    fin = head.norms["norm.weight"]
    for chain_hidden, next_slot in ((lambda h: _rms(h, fin, s.eps).astype(np.float32), lambda t: t + 1),
                                    (lambda h: h, lambda t: t)):
        K3, V3 = synth.kv_prefill(s, 41, 1, 64, [slot0])
        _, lg_m, _ = _hand_chain(head, K3[0], V3[0], slot0, toks, hids, depth, chain_hidden, next_slot)
        np.testing.assert_array_equal(lg_m[0], out["logits"][0])
        assert np.max(np.abs(lg_m[1] - out["logits"][1])) > 1e-4


def test_draft_pending_pairs_precede_the_newest_pair():
    # The newest pair sits at slot0 + P - 1 after the P - 1 pending pairs: a
    # planted mistake that writes the newest pair first moves every slot.
    s = synth.TINY
    mdl = synth.make_model(s, 43)
    head = oracle.Head(s, mdl.tensors, mdl.embed)
    toks = synth.randint(43, "pp:tok", (3,), s.vocab)
    hids = synth.normal(43, "pp:hid", (3, s.hidden))
    K1, V1 = synth.kv_prefill(s, 43, 1, 64, [8])
    K2, V2 = K1.copy(), V1.copy()
    head.draft(K1[0], V1[0], 8, toks, hids, 1, P(0.0), EMPTY, np.zeros(1, np.float32))
    for j in range(3):  # slot 8 + j holds pair j
        head.step(int(toks[j]), hids[j], K2[0], V2[0], 8 + j, kv_only=True)
    np.testing.assert_array_equal(K1, K2)
    K3, V3 = synth.kv_prefill(s, 43, 1, 64, [8])
    for j, src in enumerate((2, 0, 1)):  # mutant: newest first
        head.step(int(toks[src]), hids[src], K3[0], V3[0], 8 + j, kv_only=True)
    assert not np.array_equal(K1, K3)


def test_sampled_draft_window_grows_with_the_drafts():
    # Draft step k draws from the transform of its logits under the window
    # "last W of the history ++ x_1..x_{k-1}" (the drafts are part of the
    # sequence the step conditions on), by inverse CDF with u[k-1].
    s = synth.TINY
    mdl = synth.make_model(s, 47)
    head = oracle.Head(s, mdl.tensors, mdl.embed)
    depth, W, T, r = 3, 2, 1.0, 4.0
    prm = P(T, rep_penalty=r)
    toks = synth.randint(47, "sw:tok", (1,), s.vocab)
    hids = synth.normal(47, "sw:hid", (1, s.hidden))
    hist = synth.randint(47, "sw:hist", (5,), s.vocab).astype(np.int32)
    u = np.array([0.31, 0.62, 0.47], np.float32)
    K1, V1 = synth.kv_prefill(s, 47, 1, 64, [10])
    out = head.draft(K1[0], V1[0], 10, toks, hids, depth, prm, hist[-W:], u)
    drafts = out["drafts"]
    for k in range(depth):
        win = _window(hist[-W:], drafts, k, W)
        q = _softmax_p(out["logits"][k], win, T, r)
        np.testing.assert_allclose(out["q"][k], q, rtol=2e-5, atol=1e-9)
        x, mg = _draw(out["q"][k], u[k])
        assert mg > 1e-6 and x == drafts[k]
    # planted mistake: a window that ignores the drafts changes q at step 2
    # (x_1's own logit is penalised there only under the right reading)
    q_wrong = _softmax_p(out["logits"][1], hist[-W:], T, r)
    assert np.max(np.abs(q_wrong - out["q"][1])) > 1e-4


# ------------------------------------------- the verify's per-position window

def _expected_verify(lg, drafts, q, T, r, hist, W, u, greedy, window=_window):
    """The verify rule restated position by position with numpy (no top-k,
    top-p or min-p).  Returns (n, out_tok, min margin over the decisions)."""
    d = len(drafts)
    out = [-1] * (d + 1)
    margin = np.inf
    rows = [window(hist, drafts, i, W) for i in range(d + 1)]
    n = 0
    for i in range(1, d + 1):
        x = int(drafts[i - 1])
        if greedy:
            z = _penalise(lg[i - 1], rows[i - 1], r)
            acc = x == int(np.argmax(z))
        else:
            p = _softmax_p(lg[i - 1], rows[i - 1], T, r)
            ratio = p[x] / q[i - 1][x] if q[i - 1][x] > 0 else 0.0
            margin = min(margin, abs(ratio - u[i - 1]))
            acc = q[i - 1][x] > 0 and u[i - 1] < ratio
        if not acc:
            break
        n = i
    out[:n] = [int(x) for x in drafts[:n]]
    if greedy:
        out[n] = int(np.argmax(_penalise(lg[n], rows[n], r)))
    else:
        p = _softmax_p(lg[n], rows[n], T, r)
        w = np.maximum(p - q[n], 0) if n < d else p
        if w.sum() <= 0:
            w = p
        out[n], mg = _draw(w, u[d])
        margin = min(margin, mg)
    return n, np.array(out, np.int32), margin


def _wrong_no_drafts(hist, drafts, i, W):
    return np.array(list(hist)[-W:], np.int32)


def _wrong_untrimmed(hist, drafts, i, W):
    return np.array(list(hist) + list(drafts[:i]), np.int32)


def _wrong_off_by_one(hist, drafts, i, W):
    return _window(hist, drafts, max(i - 1, 0), W)


@pytest.mark.parametrize("W", [2, 7])
@pytest.mark.parametrize("greedy", [True, False])
def test_verify_penalty_window_per_position(W, greedy):
    # Row i of the verify is the target's distribution after x_1..x_i, so its
    # repetition window is the last W tokens of (history ++ x_1..x_i); W = 2
    # is shorter than the depth (the drafts push the history out), W = 7 longer.
    V, d, r = 12, 3, 3.0
    T = 0.0 if greedy else 1.0
    prm = P(T, rep_penalty=r)
    rng = np.random.default_rng(1000 + W + (0 if greedy else 50))
    mutants = {_wrong_no_drafts: 0, _wrong_untrimmed: 0, _wrong_off_by_one: 0}
    checked = 0
    for case in range(120):
        lg = (rng.normal(1.0, 1.0, (d + 1, V))).astype(np.float32)
        # W slots, oldest first; a window longer than the history starts empty (-1)
        hist = np.concatenate([np.full(max(W - 5, 0), -1), rng.integers(0, V, 5)]).astype(np.int32)[-W:]
        # drafts among each row's top tokens so that their penalties matter
        drafts = np.array([int(rng.choice(np.argsort(-lg[i])[:3])) for i in range(d)], np.int32)
        q = None
        if not greedy:
            q = np.stack([_softmax_p(rng.normal(0, 1.5, V).astype(np.float32), EMPTY, 1.0, 1.0)
                          for _ in range(d)]).astype(np.float32)
        u = rng.random(d + 1).astype(np.float32)
        n, out, mg = _expected_verify(lg, drafts, q, T, r, hist, W, u, greedy)
        if not greedy and mg < 1e-5:
            continue  # a decision within rounding of its threshold
        n_o, out_o, _ = oracle.verify_row(lg, drafts, q, prm, hist, u)
        assert n_o == n and np.array_equal(out_o, out), (case, n_o, n, out_o, out)
        checked += 1
        for wrong in mutants:
            nm, om, _ = _expected_verify(lg, drafts, q, T, r, hist, W, u, greedy, window=wrong)
            mutants[wrong] += int(nm != n or not np.array_equal(om, out))
    assert checked >= 100
    # every planted window mistake changes the outcome of some case (for
    # W = 7 the untrimmed window is the right one: 5 history + 3 drafts > 7
    # only at the last row)
    assert mutants[_wrong_no_drafts] > 0 and mutants[_wrong_off_by_one] > 0
    if W == 2:
        assert mutants[_wrong_untrimmed] > 0


def test_verify_residual_without_mass_draws_from_p():
    # A draft with q(x) = 0 is rejected; when q equals p the residual
    # max(p - q, 0) has no mass and the correction is drawn from p itself.
    V = 16
    lg = synth.normal(53, "res0", (2, V), std=2.0)
    prm = P(1.0, top_k=4)
    p0, _ = oracle.transform(lg[0], prm, EMPTY)
    x = int(np.argsort(-lg[0])[10])           # outside the top 4: q(x) = p(x) = 0
    assert p0[x] == 0.0
    for uu in (0.05, 0.4, 0.77, 0.98):
        n, out, _ = oracle.verify_row(lg, np.array([x], np.int32), p0[None], prm, EMPTY,
                                      np.array([0.5, uu], np.float32))
        want, mg = _draw(p0, uu)
        assert mg > 1e-6
        assert n == 0 and out[0] == want and out[1] == -1


# ------------------------------------------------------ chain equals block

def chain_of_depth_one(lg, drafts, q, prm, hist, W, u):
    """d verify calls of depth 1, chained: call j verifies x_j against rows
    j-1 and j with the window advanced by the drafts accepted so far and the
    uniforms (u[j-1], u[d]); the chain stops at the first rejection."""
    d = len(drafts)
    out = []
    for j in range(1, d + 1):
        h = _window(hist, drafts, j - 1, W)
        h = np.concatenate([np.full(W - h.size, -1, np.int32), h]) if W else EMPTY
        n, o, _ = oracle.verify_row(lg[j - 1:j + 1], drafts[j - 1:j],
                                    None if q is None else q[j - 1:j], prm, h,
                                    np.array([u[j - 1], u[d]], np.float32))
        if n == 0:
            out.append(int(o[0]))
            return j - 1, out
        out.append(int(drafts[j - 1]))
        if j == d:
            out.append(int(o[1]))
    return d, out


@pytest.mark.parametrize("greedy", [True, False])
def test_chain_of_single_token_verifies_equals_block_verify(greedy):
    # "support the qwen3_5_mtp drafter" issue, Reproduction instructions,
    # Test 3: verifying a block of T tokens must give what the single-token
    # chain gives.  Here: d depth-1 verifies chained through the accepted
    # tokens and the penalty window equal one depth-d verify.
    V, d, W = 20, 4, 3
    rng = np.random.default_rng(7 if greedy else 8)
    prm = P(0.0, rep_penalty=1.5) if greedy else P(0.9, rep_penalty=1.3, top_k=12, top_p=0.9, min_p=0.02)
    counts = np.zeros(d + 1, int)
    for case in range(150):
        lg = rng.normal(0.5, 1.5, (d + 1, V)).astype(np.float32)
        hist = rng.integers(0, V, W).astype(np.int32)
        u = rng.random(d + 1).astype(np.float32)
        if greedy:
            drafts = np.array([int(rng.choice(np.argsort(-lg[i])[:2])) for i in range(d)], np.int32)
            q = None
        else:
            q_rows, drafts = [], []
            for i in range(d):
                qi, _ = oracle.transform(lg[i] + rng.normal(0, 0.7, V).astype(np.float32), prm,
                                         _window(hist, drafts, i, W))
                drafts.append(_draw(qi, rng.random())[0])
                q_rows.append(qi)
            q, drafts = np.stack(q_rows), np.array(drafts, np.int32)
        n, out, _ = oracle.verify_row(lg, drafts, q, prm, hist, u)
        nc, oc = chain_of_depth_one(lg, drafts, q, prm, hist, W, u)
        assert nc == n and oc == list(out[:n + 1]), (case, n, out, nc, oc)
        counts[n] += 1
    assert np.count_nonzero(counts) >= 3  # several accept lengths were exercised
