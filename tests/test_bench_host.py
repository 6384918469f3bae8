"""Host logic of the benchmark that needs no GPU: the acceptance diagnostics read from a call's
outputs, the per-call percentiles and the configuration object both arms print."""
import numpy as np

import bench


def test_acceptance_diagnostics_on_a_constant_rate():
    """With a constant reach-conditioned rate alpha, A is a geometric law truncated at K:
    Pr(A >= j) = alpha^j, every alpha_j^reach = alpha, and E[G] = 1 + sum_j alpha^j (the round
    progress of M7.1 0x05B).  Drawn exactly: the empirical rates match within sampling error."""
    rng = np.random.default_rng(0)
    K, alpha, n = 5, 0.7, 200_000
    acc = rng.random((n, K)) < alpha
    A = np.where(acc.all(1), K, np.argmin(acc, 1))
    d = bench.acceptance_diagnostics(A, np.zeros(n, np.int32), K)
    assert d["requests"] == n and d["K"] == K
    assert abs(sum(d["pr_A"]) - 1.0) < 1e-5
    for j in range(1, K + 1):
        assert abs(d["pr_A_ge"][j - 1] - alpha ** j) < 5e-3
        assert abs(d["alpha_reach"][j - 1] - alpha) < 1e-2
    assert abs(d["E_G"] - (1 + sum(alpha ** j for j in range(1, K + 1)))) < 2e-2


def test_acceptance_diagnostics_identities():
    """Exact identities on any sample: Pr(A = a) = s_a - s_{a+1}, Pr(A = K) = s_K, the tails are
    the products of the reach rates, and E[G] = 1 + E[A].  Requests that did not finish (status
    not OK) are left out."""
    A = np.array([0, 1, 1, 2, 3, 3, 3, 0, 2, 1, -1, -1])
    st = np.array([0] * 10 + [4, 1])
    K = 3
    d = bench.acceptance_diagnostics(A, st, K)
    ok = A[st == 0]
    assert d["requests"] == 10
    s = [1.0] + d["pr_A_ge"]
    for a in range(K):
        assert abs(d["pr_A"][a] - (s[a] - s[a + 1])) < 1e-6
    assert abs(d["pr_A"][K] - s[K]) < 1e-6
    for j in range(1, K + 1):
        assert abs(np.prod(d["alpha_reach"][:j]) - s[j]) < 1e-6
    assert abs(d["E_G"] - (1 + ok.mean())) < 1e-6
    assert abs(d["mean_A"] - ok.mean()) < 1e-6


def test_acceptance_diagnostics_unreached_positions():
    """A position no request reaches has no reach rate (None), not a rate of zero."""
    d = bench.acceptance_diagnostics(np.zeros(8, np.int64), np.zeros(8, np.int64), 3)
    assert d["alpha_reach"] == [0.0, None, None]
    assert d["pr_A_ge"] == [0.0, 0.0, 0.0] and d["E_G"] == 1.0
    assert bench.acceptance_diagnostics([], [], 3) == {"requests": 0, "K": 3}


def test_percentiles():
    ms = list(np.arange(1, 101, dtype=float))
    p = bench.percentiles(ms)
    assert p["calls"] == 100 and p["median"] == 50.5
    assert abs(p["p10"] - 10.9) < 1e-9 and abs(p["p90"] - 90.1) < 1e-9


def test_both_arms_print_the_same_config():
    """The reference arm and ours build `config` with one function from the inputs alone."""
    batches = bench.workload_batches(("c2",), 0)
    a = bench.run_config(("c2",), batches, 1)
    b = bench.run_config(("c2",), bench.workload_batches(("c2",), 0), 1)
    assert a == b
    assert a["logit_rows_per_step"] == 8 * 9
    assert a["input_bytes_per_step"] == 8 * 9 * 32000 * 2
    assert a["l2"].startswith("L2 flushed")
