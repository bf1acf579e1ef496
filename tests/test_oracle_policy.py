"""Pins of the per-frame chunking policy (Ryu & Yoo, Sec. 4.4, Eq. 6) on hand-worked cases.

T(h, k) = max((N_total + lambda h k) / K, l) + beta l,  l = max(N_1 / k, N_{h+1}),
k in {2, 4, 8, 16}; chunking only if T <= (1 - eps) T(0)."""

import oracle


def test_balanced_tiles_never_chunk():
    # 100 tiles of 100: T(0) = max(10000/10, 100) + 5 = 1005; chunking cannot lower l below 100
    h, k, cost = oracle.policy([100] * 100, K=10)
    assert (h, k) == (0, 1) and cost == 1005.0


def test_single_outlier_is_split_sixteen_ways():
    # N = [10000, 10 x 99], K = 100, lambda = 256, beta = 0.05:
    # T(0) = 10000 + 500 = 10500; T(1, 16) = max((10990 + 4096)/100, 625) + 31.25 = 656.25;
    # T(2, 16) ties with T(1, 16) and the smaller h is kept
    h, k, cost = oracle.policy([10000] + [10] * 99, K=100)
    assert (h, k) == (1, 16)
    assert abs(cost - 656.25) < 1e-9


def test_average_term_dominates_when_few_workers():
    # K = 2: every chunk raises (N_total + lambda h k)/K above T(0) = 1750
    h, k, cost = oracle.policy([1000, 900, 800, 700], K=2)
    assert (h, k, cost) == (0, 1, 1750.0)


def test_ten_percent_threshold():
    # lambda = beta = 0: [300, 250 x 3], K = 4 -> T(0) = 300, T(1, 2) = 262.5 <= 270: enabled
    assert oracle.policy([300, 250, 250, 250], K=4, lam=0.0, beta=0.0)[:2] == (1, 2)
    # [300, 280 x 3] -> T(1, 2) = 285 > 270: disabled
    h, k, cost = oracle.policy([300, 280, 280, 280], K=4, lam=0.0, beta=0.0)
    assert (h, k, cost) == (0, 1, 300.0)


def test_h_max_limits_the_search():
    counts = [5000, 4000, 3000] + [10] * 50
    h_all, k_all, _ = oracle.policy(counts, K=64)
    assert h_all >= 2
    h1, _, _ = oracle.policy(counts, K=64, h_max=1)
    assert h1 <= 1


def _golden_cases():
    import os

    path = os.path.join(os.path.dirname(__file__), "golden", "policy_eq6_cases.txt")
    for line in open(path):
        line = line.split("#", 1)[0].strip()
        if not line:
            continue
        f = [x.strip() for x in line.split(";")]
        counts = []
        for part in f[0].split(","):
            v, _, r = part.partition("x")
            counts += [int(v)] * int(r or 1)
        yield (counts, int(f[1]), float(f[2]), float(f[3]), float(f[4]), int(f[5]), int(f[6]),
               float(f[7]))


def test_golden_hand_worked_cases():
    cases = list(_golden_cases())
    assert len(cases) == 7
    for counts, K, lam, beta, eps, h, k, cost in cases:
        got = oracle.policy(counts, K=K, lam=lam, beta=beta, eps=eps)
        assert got[:2] == (h, k), (counts[:3], K, got)
        assert abs(got[2] - cost) <= 1e-9 * cost, (counts[:3], K, got)
