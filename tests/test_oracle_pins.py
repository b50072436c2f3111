"""Pins of the CPU oracle against facts that do not come from the oracle itself:
hand-worked values of the definitions, library routines (scipy softmax,
numpy argmax/sort), special cases that reduce to textbook results, and exact
enumeration of the verify's output law.  Each test names the page passage the
fact comes from."""
import math

import numpy as np
import pytest
from scipy.special import expit, softmax

import oracle
import synth


# ---------------------------------------------------------------- helpers

def _tiny_shape(H=8, nq=2, nkv=1, dh=4, I=8, V=5, eps=1e-12, theta=100.0):
    return synth.Shape("pin", H, nq, nkv, dh, I, V, eps=eps, rope_theta=theta, dtype="f32")


def _structured(s, raw_hf=True, norms=None):
    """fp32 head with every matrix zero and every raw norm zero (shifted: 1)."""
    shapes = synth.tensor_shapes(s)
    t = {}
    for n in synth.INVENTORY:
        shp = shapes[n]
        a = np.zeros(shp, np.float32)
        if len(shp) == 1 and not raw_hf:
            a += 1.0
        t[n] = a
    if norms:
        for n, v in norms.items():
            t[n] = np.asarray(v, np.float32)
    if raw_hf:
        t = {"mtp." + n: a for n, a in t.items()}
    return t


def _w(t, name):
    return t["mtp." + name] if ("mtp." + name) in t else t[name]


def _rms(x, w, eps):
    x = np.asarray(x, np.float64)
    return x / np.sqrt(np.mean(x * x) + eps) * w


def _cache(s, cap):
    K = np.zeros((s.n_kv, cap, s.head_dim), np.float32)
    return K, K.copy()


# ------------------------------------------------ loader: +1.0 shift rule

def test_shift_applies_to_exactly_seven_norm_suffixes():
    # "Upstream contract to port", sanitize: +1.0 only for the raw-HF layout,
    # over exactly the seven norm suffixes.
    s = _tiny_shape()
    t = _structured(s, raw_hf=True)
    norms, raw = oracle.load_norms(t)
    assert raw
    shifted = [n for n, v in norms.items() if np.all(v == 1.0)]
    assert len(shifted) == 7
    mats = [n for n in synth.INVENTORY if n not in norms]
    assert len(mats) == 8 and all(not n.endswith("norm.weight") for n in mats)


def test_shift_once_equals_preshifted_and_twice_differs():
    # Facts: shifting the head's norms twice breaks acceptance; the raw and the
    # split layouts must give the same head.
    s = synth.TINY
    raw = synth.make_model(s, 3, raw_hf=True)
    split = synth.make_model(s, 3, raw_hf=False)
    a = oracle.Head(s, raw.tensors, raw.embed)
    b = oracle.Head(s, split.tensors, split.embed)
    for k in a.norms:
        np.testing.assert_allclose(a.norms[k], b.norms[k], rtol=0, atol=1e-6)
    twice = {("mtp." + n[len("mtp."):]): (v + 1.0 if v.ndim == 1 else v) for n, v in raw.tensors.items()}
    c = oracle.Head(s, twice, raw.embed)
    assert any(np.max(np.abs(c.norms[k] - a.norms[k])) > 0.5 for k in a.norms)


def test_loader_rejects_missing_unknown_and_mixed():
    s = _tiny_shape()
    t = _structured(s)
    bad = dict(t)
    del bad["mtp.fc.weight"]
    with pytest.raises(ValueError):
        oracle.load_norms(bad)
    bad = dict(t)
    bad["mtp.layers.0.linear_attn.weight"] = np.zeros(3, np.float32)
    with pytest.raises(ValueError):
        oracle.load_norms(bad)
    bad = dict(t)
    bad["norm.weight"] = bad.pop("mtp.norm.weight")
    with pytest.raises(ValueError):
        oracle.load_norms(bad)


def test_block_size_is_depth_plus_two():
    # "Upstream contract to port": mtp_num_hidden_layers 1 -> block_size 3,
    # i.e. two drafted tokens per round.
    assert oracle.default_block_size(1) == 3
    assert oracle.default_block_size(1) - 1 == 2


def test_rollback_trim_arithmetic():
    # qualify-on-the-qwen3_5-path comment: attention layers trim by
    # block_size - (max(accepted) + 1); the block here is the depth + 1
    # positions the target verified.
    assert oracle.rollback_lengths(100, 0, 500, 2) == (101, 498)
    assert oracle.rollback_lengths(100, 2, 500, 2) == (101, 500)
    assert oracle.rollback_lengths(7, 1, 9, 3) == (8, 7)


# --------------------------------------------------------- head forward

def test_fc_concat_order_norms_and_tied_head():
    # "Upstream contract to port", forward: h = fc(concat(norm_e(embed), norm_h(hidden))).
    # With fc = [0 | I] the head sees only the hidden half; with [I | 0] only
    # the embedding half. All later blocks are zero, so h2 = h0 and the
    # logits are E . norm_final(h2) (the borrowed tied head).
    s = _tiny_shape(eps=0.3)
    rng = np.random.default_rng(0)
    nw = {n: rng.normal(0, 0.2, synth.tensor_shapes(s)[n]).astype(np.float32)
          for n in ("pre_fc_norm_embedding.weight", "pre_fc_norm_hidden.weight", "norm.weight")}
    E = rng.normal(0, 1, (s.vocab, s.hidden)).astype(np.float32)
    hid = (0.2 * rng.normal(0, 1, s.hidden)).astype(np.float32)
    for half in (0, 1):
        t = _structured(s, norms=nw)
        fc = np.zeros((s.hidden, 2 * s.hidden), np.float32)
        fc[:, half * s.hidden:(half + 1) * s.hidden] = np.eye(s.hidden)
        t["mtp.fc.weight"] = fc
        h = oracle.Head(s, t, E)
        K, V = _cache(s, 4)
        h2, lg = h.step(3, hid, K, V, 0)
        src = E[3] if half == 0 else hid
        wn = nw["pre_fc_norm_embedding.weight" if half == 0 else "pre_fc_norm_hidden.weight"] + 1.0
        h0 = _rms(src, wn, 0.3)
        np.testing.assert_allclose(h2, h0, rtol=1e-6, atol=1e-6)
        f = _rms(h0.astype(np.float32), nw["norm.weight"] + 1.0, 0.3)
        np.testing.assert_allclose(lg, E.astype(np.float64) @ f, rtol=1e-5, atol=1e-5)


def _hidden_only_head(s):
    """fc = [0 | I], every other block zero, unit norm weights: h2 = h0 =
    RMSNorm_h(hidden), so the step exposes the oracle's RMSNorm alone."""
    t = _structured(s)
    fc = np.zeros((s.hidden, 2 * s.hidden), np.float32)
    fc[:, s.hidden:] = np.eye(s.hidden)
    t["mtp.fc.weight"] = fc
    return oracle.Head(s, t, np.zeros((s.vocab, s.hidden), np.float32))


def test_rmsnorm_closed_forms():
    # "Upstream contract to port", module shape: nn.RMSNorm(hidden_size, eps).
    # With every |x_i| = 1 the mean square is 1, so with eps = 1 the norm is
    # x / sqrt(2) exactly; eps outside the root would give x / 2 and a sum in
    # place of the mean x / sqrt(H + 1).
    s = _tiny_shape(eps=1.0)
    h = _hidden_only_head(s)
    sign = np.where(np.arange(s.hidden) % 3 == 0, -1.0, 1.0).astype(np.float32)
    K, V = _cache(s, 2)
    h2, _ = h.step(0, sign, K, V, 0)
    np.testing.assert_allclose(h2, sign / math.sqrt(2.0), rtol=1e-7, atol=0)
    # with a negligible eps the output has unit root mean square whatever the
    # input's scale, and scaling the input leaves it unchanged
    s = _tiny_shape(H=16, dh=8, I=16, eps=1e-12)
    h = _hidden_only_head(s)
    x = np.random.default_rng(5).normal(0, 3.0, s.hidden).astype(np.float32)
    K, V = _cache(s, 2)
    a, _ = h.step(0, x, K, V, 0)
    b, _ = h.step(0, (40.0 * x).astype(np.float32), K, V, 0)
    assert abs(math.sqrt(float(np.mean(np.asarray(a, np.float64) ** 2))) - 1.0) < 1e-6
    np.testing.assert_allclose(a, b, rtol=1e-6, atol=1e-6)


def _qk_probe(s, slot, which):
    """Head whose k (pre-norm) is sqrt(H) * e_which: hid one-hot -> h0 = sqrt(H) e_0."""
    t = _structured(s)
    fc = np.zeros((s.hidden, 2 * s.hidden), np.float32)
    fc[:, s.hidden:] = np.eye(s.hidden)
    t["mtp.fc.weight"] = fc
    wk = np.zeros((s.n_kv * s.head_dim, s.hidden), np.float32)
    wk[which, 0] = 1.0
    t["mtp.layers.0.self_attn.k_proj.weight"] = wk
    return t


@pytest.mark.parametrize("which,slot", [(0, 3), (1, 3), (0, 0), (1, 7)])
def test_rope_rotate_half_worked_values(which, slot):
    # RoPE at the drafter's own absolute offset (rotate-half pairs (i, i+d/2),
    # angle pos * theta^(-2i/d)).  k before the norm is sqrt(8)*e_which; after
    # k_norm over head_dim 4 it is 2*e_which; slot `slot` then holds the
    # rotation of that vector, worked out here by hand.
    s = _tiny_shape(theta=100.0)
    t = _qk_probe(s, slot, which)
    h = oracle.Head(s, t, np.zeros((s.vocab, s.hidden), np.float32))
    K, V = _cache(s, 8)
    hid = np.zeros(s.hidden, np.float32)
    hid[0] = 1.0
    h.step(0, hid, K, V, slot, kv_only=True)
    ang = slot * (1.0 if which == 0 else 100.0 ** -0.5)
    exp = np.zeros(4)
    exp[which] = 2 * math.cos(ang)
    exp[which + 2] = 2 * math.sin(ang)
    np.testing.assert_allclose(K[0, slot], exp, rtol=0, atol=1e-6)


def test_single_key_attention_returns_v_and_gqa_groups():
    # With one key, softmax weight is 1, so each q head returns its kv head's
    # v.  Grouped-query attention maps q head j to kv head j // (nq/nkv):
    # heads 0,1 -> kv 0; heads 2,3 -> kv 1.  W_o = I, MLP zero: h2 = h0 + o.
    s = _tiny_shape(H=8, nq=4, nkv=2, dh=2)
    rng = np.random.default_rng(1)
    t = _structured(s)
    fc = np.zeros((s.hidden, 2 * s.hidden), np.float32)
    fc[:, s.hidden:] = np.eye(s.hidden)
    t["mtp.fc.weight"] = fc
    wv = rng.normal(0, 1, (s.n_kv * s.head_dim, s.hidden)).astype(np.float32)
    t["mtp.layers.0.self_attn.v_proj.weight"] = wv
    t["mtp.layers.0.self_attn.o_proj.weight"] = np.eye(s.hidden, dtype=np.float32)
    t["mtp.layers.0.self_attn.q_proj.weight"] = rng.normal(0, 1, (8, 8)).astype(np.float32)
    t["mtp.layers.0.self_attn.k_proj.weight"] = rng.normal(0, 1, (4, 8)).astype(np.float32)
    h = oracle.Head(s, t, np.zeros((s.vocab, s.hidden), np.float32))
    K, V = _cache(s, 2)
    hid = rng.normal(0, 1, s.hidden).astype(np.float32)
    h2, _ = h.step(0, hid, K, V, 0)
    h0 = _rms(hid, 1.0, s.eps)
    v = wv.astype(np.float64) @ _rms(h0, 1.0, s.eps)
    o = np.concatenate([v[0:2], v[0:2], v[2:4], v[2:4]])
    np.testing.assert_allclose(h2, h0 + o, rtol=1e-5, atol=1e-5)


def test_two_key_softmax_scale_and_causality():
    # Attention over slots 0..S with scale 1/sqrt(head_dim); slots above S
    # are not read.  q = k = 2 e_0 rotated to position 1; slot 0 holds
    # K0 = e_0, V0 = (1, 2, 3, 4).  Scores: q.k1/2 = 2, q.K0/2 = cos(1).
    s = _tiny_shape(H=8, nq=2, nkv=1, dh=4, theta=100.0)
    t = _structured(s)
    fc = np.zeros((s.hidden, 2 * s.hidden), np.float32)
    fc[:, s.hidden:] = np.eye(s.hidden)
    t["mtp.fc.weight"] = fc
    wq = np.zeros((8, 8), np.float32)
    wq[0, 0] = 1.0
    wq[4, 0] = 1.0
    t["mtp.layers.0.self_attn.q_proj.weight"] = wq
    wk = np.zeros((4, 8), np.float32)
    wk[0, 0] = 1.0
    t["mtp.layers.0.self_attn.k_proj.weight"] = wk
    wv = np.zeros((4, 8), np.float32)
    wv[3, 0] = 1.0                         # v1 = (0, 0, 0, sqrt 8)
    t["mtp.layers.0.self_attn.v_proj.weight"] = wv
    t["mtp.layers.0.self_attn.o_proj.weight"] = np.eye(8, dtype=np.float32)
    h = oracle.Head(s, t, np.zeros((s.vocab, s.hidden), np.float32))
    K, V = _cache(s, 6)
    K[0, 0] = [1, 0, 0, 0]
    V[0, 0] = [1, 2, 3, 4]
    K[0, 2:] = 50.0                        # future slots: must not matter
    V[0, 2:] = -7.0
    hid = np.zeros(8, np.float32)
    hid[0] = 1.0
    h2, _ = h.step(0, hid, K, V, 1)
    w0, w1 = math.exp(math.cos(1.0)), math.exp(2.0)
    o = (w0 * np.array([1, 2, 3, 4]) + w1 * np.array([0, 0, 0, math.sqrt(8)])) / (w0 + w1)
    h0 = np.zeros(8)
    h0[0] = math.sqrt(8)
    np.testing.assert_allclose(h2, h0 + np.concatenate([o, o]), rtol=1e-5, atol=1e-5)


def test_swiglu_mlp_closed_form():
    # "Where the MTP weights live": mlp.{gate,up,down}_proj.  SwiGLU:
    # h2 = h1 + W_d(silu(W_g c) * (W_u c)), c = norm_post(h1), silu(g) = g*sigmoid(g).
    s = _tiny_shape(H=8, I=8)
    rng = np.random.default_rng(2)
    t = _structured(s)
    fc = np.zeros((8, 16), np.float32)
    fc[:, 8:] = np.eye(8)
    t["mtp.fc.weight"] = fc
    t["mtp.layers.0.mlp.gate_proj.weight"] = 1.5 * np.eye(8, dtype=np.float32)
    t["mtp.layers.0.mlp.up_proj.weight"] = -0.5 * np.eye(8, dtype=np.float32)
    t["mtp.layers.0.mlp.down_proj.weight"] = np.eye(8, dtype=np.float32)
    h = oracle.Head(s, t, np.zeros((s.vocab, 8), np.float32))
    K, V = _cache(s, 2)
    hid = rng.normal(0, 1, 8).astype(np.float32)
    h2, _ = h.step(0, hid, K, V, 0)
    h1 = _rms(hid, 1.0, s.eps)
    c = _rms(h1, 1.0, s.eps)
    g = 1.5 * c
    # silu from scipy's logistic function (the oracle has its own exp)
    np.testing.assert_allclose(h2, h1 + (g * expit(g)) * (-0.5 * c), rtol=1e-5, atol=1e-6)
    # and the gate's sign matters: silu is not odd (silu(-g) = silu(g) - g)
    t["mtp.layers.0.mlp.gate_proj.weight"] = -1.5 * np.eye(8, dtype=np.float32)
    h = oracle.Head(s, t, np.zeros((s.vocab, 8), np.float32))
    h2n, _ = h.step(0, hid, K, V, 0)
    np.testing.assert_allclose(h2n - h1, ((g * expit(g)) - g) * (-0.5 * c), rtol=1e-5, atol=1e-6)


def test_flush_is_batch_order_independent_and_matches_full_steps():
    # Facts: slot S pairs the token at S+1 with the target hidden at S; pending
    # pairs are written in batches.  For a one-layer head the K/V of a slot
    # depend only on that slot's pair: the KV-only flush equals full steps.
    s = synth.TINY
    m = synth.make_model(s, 5)
    h = oracle.Head(s, m.tensors, m.embed)
    toks = synth.randint(5, "ft", (6,), s.vocab)
    hids = synth.normal(5, "fh", (6, s.hidden))
    K1, V1 = synth.kv_prefill(s, 5, 1, 32, [10])
    K2, V2 = K1.copy(), V1.copy()
    h.flush(toks, hids, K1[0], V1[0], 10)
    for j in range(6):
        h.step(int(toks[j]), hids[j], K2[0], V2[0], 10 + j)
    np.testing.assert_array_equal(K1, K2)
    np.testing.assert_array_equal(V1, V2)


# ------------------------------------------------------------ transforms

P = oracle.make_params


def test_identity_params_are_plain_softmax():
    lg = synth.normal(9, "lg", (64,), std=3.0)
    pr, info = oracle.transform(lg, P(1.0), np.zeros(0, np.int32))
    np.testing.assert_allclose(pr, softmax(lg.astype(np.float64)), rtol=1e-6, atol=1e-9)
    assert info.kept == 64


def test_temperature_zero_and_top_k_one_are_argmax_point_masses():
    # Commit log: at temperature 0 the sampler yields a point mass.
    lg = synth.normal(9, "lg2", (50,), std=3.0)
    for prm in (P(0.0), P(0.7, top_k=1)):
        pr, info = oracle.transform(lg, prm, np.zeros(0, np.int32))
        assert info.argmax == int(np.argmax(lg)) and pr[info.argmax] == 1.0 and pr.sum() == 1.0
    tied = np.array([0.5, 2.0, 2.0, 1.0], np.float32)
    _, info = oracle.transform(tied, P(0.0), np.zeros(0, np.int32))
    assert info.argmax == 1


def test_temperature_scales_logits():
    lg = synth.normal(9, "lg3", (40,), std=2.0)
    pr, _ = oracle.transform(lg, P(0.5), np.zeros(0, np.int32))
    np.testing.assert_allclose(pr, softmax(lg.astype(np.float64) / 0.5), rtol=1e-5, atol=1e-9)


def test_top_p_worked_example():
    lg = np.array([1, 2, 3, 4], np.float32)
    pr, info = oracle.transform(lg, P(1.0, top_p=0.7), np.zeros(0, np.int32))
    e3, e4 = math.exp(3), math.exp(4)
    np.testing.assert_allclose(pr, [0, 0, e3 / (e3 + e4), e4 / (e3 + e4)], rtol=1e-6)
    pr, _ = oracle.transform(lg, P(1.0, top_p=0.5), np.zeros(0, np.int32))
    np.testing.assert_array_equal(pr, [0, 0, 0, 1])


def test_min_p_worked_example():
    lg = np.log(np.array([1.0, 0.5, 0.25, 0.1])).astype(np.float32)
    pr, _ = oracle.transform(lg, P(1.0, min_p=0.3), np.zeros(0, np.int32))
    np.testing.assert_allclose(pr, [2 / 3, 1 / 3, 0, 0], rtol=1e-6)


def test_top_k_ties_keep_lowest_ids():
    lg = np.array([1, 1, 1, 0], np.float32)
    pr, _ = oracle.transform(lg, P(1.0, top_k=2), np.zeros(0, np.int32))
    np.testing.assert_allclose(pr, [0.5, 0.5, 0, 0])


def test_repetition_penalty_distinct_tokens_once():
    lg = np.array([2.0, -2.0, 1.0], np.float32)
    pr, _ = oracle.transform(lg, P(1.0, rep_penalty=2.0), np.array([0, 1, 0, -1], np.int32))
    np.testing.assert_allclose(pr, softmax(np.array([1.0, -4.0, 1.0])), rtol=1e-6)


@pytest.mark.parametrize("seed", range(6))
def test_truncation_matches_sort_based_definition(seed):
    # Brute force against Python's own sort of (z desc, id asc).
    rng = np.random.default_rng(seed)
    V = 48
    lg = np.round(rng.normal(0, 2, V), 1).astype(np.float32)   # rounding creates ties
    T, k = 0.8, int(rng.integers(2, 30))
    tp, mp = float(np.float32(rng.uniform(0.3, 0.95))), float(np.float32(rng.uniform(0, 0.2)))
    pr, _ = oracle.transform(lg, P(T, top_k=k, top_p=tp, min_p=mp), np.zeros(0, np.int32))
    z = [float(np.float32(x) / np.float32(T)) for x in lg]
    order = sorted(range(V), key=lambda i: (-z[i], i))[:k]
    e = [math.exp(z[i] - z[order[0]]) for i in order]
    S = sum(e)
    keep_p = next(j + 1 for j in range(k) if sum(e[:j + 1]) >= tp * S)
    keep_m = max(1, sum(1 for x in e if x >= mp))
    kf = min(k, keep_p, keep_m)
    exp = np.zeros(V)
    for j in range(kf):
        exp[order[j]] = e[j] / sum(e[:kf])
    np.testing.assert_allclose(pr, exp, rtol=1e-6, atol=1e-9)


def test_inverse_cdf_draw_worked_values():
    w = np.array([0.1, 0.2, 0.3, 0.4], np.float32)
    for u, want in ((0.05, 0), (0.15, 1), (0.35, 2), (0.65, 3), (0.999, 3)):
        assert oracle.draw(w, u)[0] == want
        assert oracle.draw(10 * w, u)[0] == want
    z = np.array([0, 1, 0, 1], np.float32)
    assert oracle.draw(z, 0.49)[0] == 1
    assert oracle.draw(z, 0.5)[0] == 3
    assert oracle.draw(z, 0.0)[0] == 1


# ----------------------------------------------------------------- verify

def test_greedy_verify_is_argmax_prefix_plus_correction():
    # Commit log: at temperature 0 acceptance reduces to argmax-match.
    V, d = 16, 3
    lg = synth.normal(11, "gv", (d + 1, V), std=2.0)
    am = lg.argmax(1)
    for n_match in range(d + 1):
        drafts = np.array([am[i] if i < n_match else (am[i] + 1) % V for i in range(d)], np.int32)
        n, out, _ = oracle.verify_row(lg, drafts, None, P(0.0), np.zeros(0, np.int32),
                                      np.full(d + 1, 0.5, np.float32))
        assert n == n_match
        assert list(out[:n]) == list(am[:n]) and out[n] == am[n]
        assert all(out[n + 1:] == -1)


def _enumerate_verify_law(p_rows, q1, q2_of, V):
    """Exact law of the verify's committed tokens for depth 2 with identity
    params.  p_rows(a) -> target logits rows [3][V] given x_1 = a;  q1 [V];
    q2_of(a) -> q_2 given x_1 = a.  The verify is piecewise constant in the
    uniforms; it is evaluated at the midpoint of every cell of the partition
    given by the accept thresholds and the draw's cumulative sums."""
    law1 = np.zeros(V)
    law2 = np.zeros((V, V))
    acc1 = np.zeros(V)
    prm = P(1.0)

    def cells(bps):
        pts = sorted(set([0.0, 1.0] + [b for b in bps if 0.0 < b < 1.0]))
        return [((a + b) / 2, b - a) for a, b in zip(pts, pts[1:]) if b > a]

    for x1 in range(V):
        rows = p_rows(x1)
        p0 = softmax(rows[0].astype(np.float64))
        p1 = softmax(rows[1].astype(np.float64))
        p2 = softmax(rows[2].astype(np.float64))
        q2 = q2_of(x1)
        r1 = min(1.0, p0[x1] / q1[x1])
        for u1, m1 in cells([r1]):
            if u1 >= r1:       # reject at 1: residual of p0 - q1
                res = np.maximum(p0 - q1, 0)
                bps = list(np.cumsum(res) / res.sum())
                for up, mp in cells(bps):
                    n, out, _ = oracle.verify_row(rows, np.array([x1, 0], np.int32),
                                                  np.stack([q1, q2]).astype(np.float32), prm,
                                                  np.zeros(0, np.int32),
                                                  np.array([u1, 0.5, up], np.float32))
                    assert n == 0
                    law1[out[0]] += q1[x1] * m1 * mp
                continue
            for x2 in range(V):
                r2 = min(1.0, p1[x2] / q2[x2])
                for u2, m2 in cells([r2]):
                    w = p2 if u2 < r2 else np.maximum(p1 - q2, 0)
                    bps = list(np.cumsum(w) / w.sum())
                    for up, mp in cells(bps):
                        n, out, _ = oracle.verify_row(rows, np.array([x1, x2], np.int32),
                                                      np.stack([q1, q2]).astype(np.float32), prm,
                                                      np.zeros(0, np.int32),
                                                      np.array([u1, u2, up], np.float32))
                        assert n >= 1 and out[0] == x1
                        mass = q1[x1] * m1 * q2[x2] * m2 * mp
                        law1[x1] += mass
                        acc1[x1] += mass
                        law2[x1, out[1]] += mass
    return law1, law2, acc1


def test_verify_law_equals_target_by_exact_enumeration():
    # Leviathan/Chen rejection sampling ("leviathan/chen sampling", DFlash
    # commit; "greedy is a special case of sampled decoding"): the committed
    # token follows the target distribution p whatever q is; given that x_1 = a
    # was accepted, the next committed token follows p(. | a).  V = 8.
    V = 8
    base = synth.normal(21, "enum:rows", (V, 3, V), std=1.5)
    q1 = softmax(synth.normal(21, "enum:q1", (V,), std=1.0).astype(np.float64))
    q2s = softmax(synth.normal(21, "enum:q2", (V, V), std=1.0).astype(np.float64), axis=1)
    q1 = q1.astype(np.float32).astype(np.float64)
    # a real target's first row does not depend on x_1: share it across x_1
    shared = base.copy()
    shared[:, 0, :] = base[0, 0]
    law1, law2, acc1 = _enumerate_verify_law(lambda a: shared[a], q1.astype(np.float32),
                                             lambda a: q2s[a].astype(np.float32), V)
    assert abs(law1.sum() - 1.0) < 1e-6
    np.testing.assert_allclose(law1, softmax(base[0, 0].astype(np.float64)), rtol=0, atol=2e-6)
    for a in range(V):
        if acc1[a] > 1e-9:
            cond = law2[a] / acc1[a]
            np.testing.assert_allclose(cond, softmax(shared[a, 1].astype(np.float64)), rtol=0, atol=2e-6)


def test_verify_bonus_comes_from_last_row_when_all_accepted():
    # q = p exactly: every draft is accepted (ratio 1 > u), and the extra token
    # is the draw from the last row.
    V, d = 10, 2
    lg = synth.normal(31, "bonus", (d + 1, V), std=1.0)
    p = np.stack([softmax(lg[i].astype(np.float64)) for i in range(d + 1)]).astype(np.float32)
    drafts = np.array([3, 7], np.int32)
    u = np.array([0.999, 0.999, 0.37], np.float32)
    n, out, _ = oracle.verify_row(lg, drafts, p[:d], P(1.0), np.zeros(0, np.int32), u)
    assert n == 2
    assert out[2] == int(np.searchsorted(np.cumsum(p[2].astype(np.float64)), 0.37 * p[2].astype(np.float64).sum(), side="right"))


# ------------------------------------------------------------ fp8 draft head
def test_bf16_rounding_matches_torch():
    # bf16 weights and KV cache (the drafter is published in bf16, "Where the
    # MTP weights actually live"): the oracle's fp32 -> bf16 rounding against
    # PyTorch's conversion: random values, exact ties (both directions of
    # round-half-even), overflow to infinity, subnormals, signed zeros and
    # infinities; NaN inputs (with any payload) must stay NaN
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(11)
    base = [rng.normal(0, 1, 4000), rng.normal(0, 1e-3, 1000), rng.normal(0, 1e30, 1000)]
    ties = np.array([1 + 2.0 ** -8, 1 + 3 * 2.0 ** -8, -(1 + 2.0 ** -8), 2 + 2.0 ** -7, 1 + 2.0 ** -8 + 2.0 ** -20])
    special = np.array([0.0, -0.0, np.inf, -np.inf, 3.4028235e38, -3.4028235e38, 1e-40, -1e-40, 1.17549435e-38,
                        3.3895314e38, 3.3961775e38])
    x = np.concatenate(base + [ties, special]).astype(np.float32)
    got = oracle.bf16_round_bits(x)
    want = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(got, want)
    nans = np.array([0x7FC00000, 0x7FFFFFFF, 0xFFFFFFFF, 0x7F800001, 0xFFC00000], np.uint32).view(np.float32)
    b = oracle.bf16_round_bits(nans)
    assert np.all((b & 0x7F80) == 0x7F80) and np.all((b & 0x007F) != 0)


def test_e4m3_codes_match_torch_float8():
    """The oracle's e4m3 encoder against torch's float8_e4m3fn conversion
    (round to nearest even) on normals, subnormals, ties and the top of the
    range, below the point where torch turns to NaN; and every code decodes
    to torch's value."""
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(5)
    xs = np.concatenate([
        rng.standard_normal(4000) * 30, rng.standard_normal(2000) * 0.01, rng.uniform(-463.9, 463.9, 2000),
        # exact ties between neighbouring codes: the midpoints of 1.0/1.125, 1.125/1.25, of two subnormals
        np.array([1.0625, 1.1875, 3 * 2.0 ** -10, 2.0 ** -10, 448.0, -448.0, 0.0, -0.0, 2.0 ** -6, 2.0 ** -9]),
    ]).astype(np.float32)
    want = torch.from_numpy(xs).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([oracle.e4m3_encode(float(x)) for x in xs], np.uint8)
    np.testing.assert_array_equal(got, want)
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).float().numpy()
    dec = np.array([oracle.e4m3_decode(int(c)) for c in codes], np.float32)
    np.testing.assert_array_equal(dec, ref)


def test_e4m3_saturates_and_row_quantisation_bounds():
    assert oracle.e4m3_encode(500.0) == 0x7E and oracle.e4m3_encode(-1e9) == 0xFE  # +-448
    rng = np.random.default_rng(6)
    w = (rng.standard_normal((16, 300)) * rng.uniform(0.01, 3.0, (16, 1))).astype(np.float32)
    q, sc = oracle.quantize_rows_e4m3(w)
    for r in range(16):
        amax = float(np.max(np.abs(w[r])))
        assert sc[r] == np.float32(amax) / np.float32(448.0)
        # the largest magnitude takes the largest code
        assert np.max(q[r] & 0x7F) == 0x7E
        dq = np.array([oracle.e4m3_decode(int(c)) for c in q[r]], np.float64) * sc[r]
        err = np.abs(dq - w[r])
        # half a step of a 3-bit mantissa (1/16 relative) for normals, half the
        # smallest subnormal step (2^-10 * scale) below 2^-6 * scale
        bound = np.maximum(np.abs(w[r]) / 16.0, 2.0 ** -10 * sc[r]) * (1 + 1e-6)
        assert np.all(err <= bound)


def test_fp8_head_equals_the_bf16_head_on_exactly_representable_rows():
    """A head whose rows are e4m3 values scaled by max 448 quantises without
    loss, so the fp8 logits reduce to the bf16 head's."""
    s = synth.TINY
    model = synth.make_model(s, 44)
    rng = np.random.default_rng(7)
    codes = rng.integers(0, 0x7E, (s.vocab, s.hidden)).astype(np.uint8) | (rng.integers(0, 2, (s.vocab, s.hidden)) << 7).astype(np.uint8)
    codes[:, 0] = 0x7E  # each row's largest magnitude is 448: scale 1
    lm = np.array([[oracle.e4m3_decode(int(c)) for c in row] for row in codes], np.float32)
    q, sc = oracle.quantize_rows_e4m3(lm)
    np.testing.assert_array_equal(q, codes)
    np.testing.assert_array_equal(sc, np.ones(s.vocab, np.float32))
    h_ref = oracle.Head(s, model.tensors, model.embed, lm_head=lm)
    h_q = oracle.Head(s, model.tensors, model.embed, lm_head=lm, lm_fp8=(q, sc))
    K, V = synth.kv_prefill(s, 44, 1, 64, [10])
    hid = synth.normal(44, "h", (s.hidden,))
    _, l1 = h_ref.step(5, hid, K[0].copy(), V[0].copy(), 10)
    _, l2 = h_q.step(5, hid, K[0].copy(), V[0].copy(), 10)
    np.testing.assert_allclose(l2, l1, rtol=1e-6, atol=1e-6 * np.max(np.abs(l1)))
