"""The draft-depth controller ("Ollama qwen3_5 MTP loader and SelfDraft path",
Facts: depth control; Ollama MLX-runner commit "choose the speculative draft
length to maximize throughput"), host code in libmtp, on the CPU.

Rounds are simulated with known per-position acceptance a_i and a known cost
per depth, c(N). The depth the controller settles on must be the brute-force
argmax of committed(N) / c(N), with committed(N) = 1 + sum_{i<=N} prod_{j<=i}
a_j. When plain decode is best (a steep-forward target), the probe interval
must back off from 4 to 512 rounds. Probes go one past the choice, every 4
rounds while the choice keeps changing."""
import numpy as np
import pytest

import mtp_speculative_decoding_step_gb300 as m


def _best(a, cost):
    committed, run, vals = 1.0, 1.0, []
    for n in range(len(cost)):
        if n > 0:
            run *= a[n - 1]
            committed += run
        vals.append(committed / cost[n])
    return int(np.argmax(vals))


def _simulate(a, cost, rounds, seed):
    rng = np.random.default_rng(seed)
    ctl = m.DepthController(len(a))
    depths = []
    for _ in range(rounds):
        n = ctl.next()
        k = 0
        while k < n and rng.random() < a[k]:
            k += 1
        ctl.observe(n, k, cost[n] * (1.0 + 0.01 * rng.standard_normal()))
        depths.append(n)
    return ctl, depths


@pytest.mark.parametrize("a,cost", [
    ([0.8, 0.7, 0.6, 0.5, 0.4, 0.3], [1.0, 1.1, 1.2, 1.3, 1.4, 1.5, 1.6]),  # cheap drafts: go deep
    ([0.6, 0.5, 0.4, 0.3, 0.2, 0.1], [1.0, 1.2, 1.4, 1.6, 1.8, 2.0, 2.2]),
    ([0.9, 0.9, 0.9, 0.9], [1.0, 1.05, 1.1, 1.15, 1.2]),                    # best = deepest
])
def test_settles_on_the_throughput_optimum(a, cost):
    want = _best(a, cost)
    ctl, depths = _simulate(a, cost, 3000, seed=1)
    late = depths[-500:]
    # the choice is the mode of the late rounds (probes add one past it now and then)
    assert max(set(late), key=late.count) == want
    est, cst, _ = ctl.state()
    for i in range(want):
        assert abs(est[i] - a[i]) < 0.05, (i, est[i], a[i])
    ctl.close()


def test_steep_forward_target_backs_off_to_plain_decode():
    a = [0.5, 0.4, 0.3]
    cost = [1.0, 2.0, 3.0, 4.0]  # every draft costs a whole extra forward: speculation loses
    assert _best(a, cost) == 0
    ctl, depths = _simulate(a, cost, 3000, seed=2)
    assert depths[-1] in (0, 1)
    assert depths[-2000:].count(0) > 1990  # probes only, and rare
    _, _, interval = ctl.state()
    assert interval == 512
    ctl.close()


def test_probe_cadence_and_bounds():
    ctl = m.DepthController(4)
    # the floor first: plain decode until its cost is known
    assert ctl.next() == 0 and ctl.next() == 0
    ctl.observe(0, 0, 1.0)
    got = [ctl.next() for _ in range(8)]
    # no acceptance data yet: the frontier is 0, the choice is one past it
    # (depth 1, every cost alike), and every 4th round probes one deeper
    assert got.count(2) >= 1 and set(got) <= {1, 2}
    with pytest.raises(m.MTPError):
        ctl.observe(5, 0, 1.0)   # depth above max_depth
    with pytest.raises(m.MTPError):
        ctl.observe(2, 3, 1.0)   # more accepted than drafted
    with pytest.raises(m.MTPError):
        ctl.observe(2, 1, 0.0)   # no time
    ctl.close()
