"""Exact law of a depth-2 verify by enumeration (shared by the oracle pins and
the GPU tests).  The verify is piecewise constant in its uniforms; every cell
of the partition given by the accept thresholds and the draw's cumulative sums
is evaluated once, at its midpoint, and weighted by its measure."""
import numpy as np


def cells(bps):
    pts = sorted(set([0.0, 1.0] + [float(b) for b in bps if 0.0 < b < 1.0]))
    return [((a + b) / 2, b - a) for a, b in zip(pts, pts[1:]) if b > a]


def enumerate_cases(p_rows, p_of, q1, q2_of, V):
    """p_rows(a): target logits [3][V] given x_1 = a;  p_of(row_logits, i,
    drafts_so_far): transformed target distribution (float64) of row i;
    q1 [V];  q2_of(a).  Yields (logits, drafts, q, u, mass, x1, accepted_branch)."""
    for x1 in range(V):
        rows = p_rows(x1)
        p0 = p_of(rows[0], 0, ())
        p1 = p_of(rows[1], 1, (x1,))
        q2 = q2_of(x1)
        if q1[x1] <= 0:
            continue
        r1 = min(1.0, p0[x1] / q1[x1])
        for u1, m1 in cells([r1]):
            if u1 >= r1:
                res = np.maximum(p0 - q1, 0)
                w = res if res.sum() > 0 else p0
                for up, mp in cells(np.cumsum(w) / w.sum()):
                    yield rows, (x1, 0), (q1, q2), (u1, 0.5, up), q1[x1] * m1 * mp, x1, False
                continue
            for x2 in range(V):
                if q2[x2] <= 0:
                    continue
                p2 = p_of(rows[2], 2, (x1, x2))
                r2 = min(1.0, p1[x2] / q2[x2])
                for u2, m2 in cells([r2]):
                    w = p2 if u2 < r2 else np.maximum(p1 - q2, 0)
                    if w.sum() <= 0:
                        w = p1
                    for up, mp in cells(np.cumsum(w) / w.sum()):
                        yield rows, (x1, x2), (q1, q2), (u1, u2, up), q1[x1] * m1 * q2[x2] * m2 * mp, x1, True


def accumulate(cases, results, V):
    """results[i] = (n_acc, out_tok) for cases[i]."""
    law1 = np.zeros(V)
    law2 = np.zeros((V, V))
    acc1 = np.zeros(V)
    for (rows, dr, qq, uu, mass, x1, branch), (n, out) in zip(cases, results):
        law1[out[0]] += mass
        if n >= 1:
            acc1[x1] += mass
            law2[x1, out[1]] += mass
    return law1, law2, acc1
