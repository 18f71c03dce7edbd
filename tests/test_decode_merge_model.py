"""The decode merge kernel's lane logic, on the host (no GPU).

decode_merge_kernel (fa_decode_sm103.cu) gives one warp to each (b, h).  Lane s
holds split s's (m_s, l_s), 32 splits to a batch; the partial vectors are
loaded eight splits at a time, each lane holding its d/32 output columns, and
the weights w_s = 2^(m_s - M) reach the other lanes by shuffles.  This restates
that lane by lane (batches past the first 32 splits included, which the GPU
tests' split counts do not reach) and checks it against the plain merge
  M = max_s m_s,  O = sum_s 2^(m_s - M) acc_s / sum_s 2^(m_s - M) l_s
in fp64, so that only the indexing is under test.
"""
import numpy as np
import pytest

G = 8  # partial vectors in flight per lane


def warp_merge(ml, acc, n_act):
    """The kernel's steps for one warp; ml [splits][2], acc [splits][D]."""
    D = acc.shape[1]
    epl = D // 32
    lanes = range(32)

    def acc_vec(s, lane):
        return acc[s, lane * epl:(lane + 1) * epl] if s < n_act else np.zeros(epl)

    def ml_pair(s):
        return ml[s] if s < n_act else np.array([-np.inf, 0.0])

    # first G partials and the first batch of (m, l), requested together
    a = [[acc_vec(u, lane) for u in range(G)] for lane in lanes]
    mv = [ml_pair(lane) for lane in lanes]
    Ml = [mv[lane][0] for lane in lanes]
    for lane in lanes:
        for s in range(32 + lane, n_act, 32):
            Ml[lane] = max(Ml[lane], ml[s][0])
    M = max(Ml)  # the xor-shuffle maximum
    o = [np.zeros(epl) for _ in lanes]
    lsum = [0.0 for _ in lanes]
    w = [0.0 for _ in lanes]
    for g0 in range(0, n_act, G):
        if g0 % 32 == 0:
            for lane in lanes:
                if g0 > 0:
                    mv[lane] = ml_pair(g0 + lane)
                w[lane] = 2.0 ** (mv[lane][0] - M) if g0 + lane < n_act else 0.0
                lsum[lane] += w[lane] * mv[lane][1]
        if g0 > 0:
            a = [[acc_vec(g0 + u, lane) for u in range(G)] for lane in lanes]
        for lane in lanes:
            for u in range(G):
                wu = w[(g0 % 32) + u]  # __shfl_sync(w, (g0 & 31) + u)
                o[lane] = o[lane] + wu * a[lane][u]
    L = sum(lsum)  # the xor-shuffle sum
    return np.concatenate([o[lane] / L for lane in lanes])


def plain_merge(ml, acc, n_act):
    m, l = ml[:n_act, 0], ml[:n_act, 1]
    M = m.max()
    w = 2.0 ** (m - M)
    return (w[:, None] * acc[:n_act]).sum(0) / (w * l).sum()


@pytest.mark.parametrize("D", [64, 128])
def test_merge_lane_logic_matches_the_plain_merge(D):
    rng = np.random.default_rng(7 + D)
    for n_act in list(range(1, 70)) + [95, 96, 97, 128, 130]:
        splits = n_act + int(rng.integers(0, 5))  # slots past n_act hold stale data
        ml = np.stack([rng.normal(0, 3, splits), rng.uniform(0.5, 40, splits)], 1)
        acc = rng.normal(0, 5, (splits, D))
        got = warp_merge(ml, acc, n_act)
        want = plain_merge(ml, acc, n_act)
        assert np.allclose(got, want, rtol=1e-12, atol=1e-12), n_act
