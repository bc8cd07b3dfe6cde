"""Shared statistics for the Monte-Carlo checks (oracle and GPU alike).

Outcomes of one round are keyed (n, y_0, ..., y_n) as in oracle.enumerate_law.
"""
import numpy as np
import scipy.stats


def outcome_keys(out_tokens: np.ndarray, out_num_accepted: np.ndarray):
    keys = []
    for row, n in zip(out_tokens, out_num_accepted):
        keys.append((int(n),) + tuple(int(v) for v in row[: n + 1]))
    return keys


def chi_square_vs_law(keys, law: dict, min_expected: float = 5.0):
    """Goodness of fit of observed outcomes against an exact law; bins with a small
    expectation are pooled.  Returns (statistic, p-value, number of bins)."""
    N = len(keys)
    counts = {}
    for k in keys:
        counts[k] = counts.get(k, 0) + 1
    unknown = sum(c for k, c in counts.items() if k not in law)
    if unknown:
        return float("inf"), 0.0, 0
    obs, exp = [], []
    pool_o, pool_e = 0.0, 0.0
    for k, pr in law.items():
        e = pr * N
        o = counts.get(k, 0)
        if e < min_expected:
            pool_o += o
            pool_e += e
        else:
            obs.append(o)
            exp.append(e)
    if pool_e > 0:
        obs.append(pool_o)
        exp.append(pool_e)
    obs = np.asarray(obs, float)
    exp = np.asarray(exp, float)
    exp *= obs.sum() / exp.sum()
    stat, pval = scipy.stats.chisquare(obs, exp)
    return float(stat), float(pval), len(obs)


def mean_tokens_z(out_num_accepted: np.ndarray, expected: float) -> float:
    """z-score of mean(n + 1) against an expected value."""
    x = out_num_accepted.astype(np.float64) + 1.0
    se = x.std(ddof=1) / np.sqrt(x.size)
    return float((x.mean() - expected) / se)


def tree_outcome_keys(out_tokens: np.ndarray, out_num_accepted: np.ndarray, out_path: np.ndarray):
    """Tree rounds keyed (n, node_1..node_n, y_0..y_n) as in enumerate_law.tree_outcome_law."""
    keys = []
    for row, n, path in zip(out_tokens, out_num_accepted, out_path):
        n = int(n)
        keys.append((n,) + tuple(int(v) for v in path[:n]) + tuple(int(v) for v in row[: n + 1]))
    return keys
