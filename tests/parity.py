"""GPU-vs-oracle comparison of one verification round.

Contract: accepted counts and emitted ids match exactly, except where the
first disagreement sits at a near-boundary position of the float64 oracle --
an accept test with |r - p/q| < NEAR, or a final sample whose uniform lies
within NEAR of a CDF boundary.  Greedy sequences must match exactly (raw
logits are compared, no rounding involved).  Such mismatches are counted.
"""
from dataclasses import dataclass, field

import numpy as np

NEAR = 1e-5
SOFTMAX_RTOL = 1e-5


@dataclass
class ParityReport:
    positions: int = 0
    near_positions: int = 0
    mismatches_near: int = 0
    mismatches_far: int = 0
    far_detail: list = field(default_factory=list)

    def merge(self, o: "ParityReport"):
        self.positions += o.positions
        self.near_positions += o.near_positions
        self.mismatches_near += o.mismatches_near
        self.mismatches_far += o.mismatches_far
        self.far_detail += o.far_detail
        return self

    def __str__(self):
        return (f"positions={self.positions} near={self.near_positions} "
                f"mismatch_near={self.mismatches_near} mismatch_far={self.mismatches_far}")


def compare(batch, gpu_tokens, gpu_num, ref, gpu_status=None) -> ParityReport:
    rep = ParityReport()
    B = batch.B
    for b in range(B):
        g = int(batch.num_draft[b]) if 0 <= batch.num_draft[b] <= batch.gmax else 0
        sampled = batch.temperature[b] > 0
        st_ref = int(ref.seq_status[b])
        if gpu_status is not None and int(gpu_status[b]) != st_ref:
            rep.mismatches_far += 1
            rep.far_detail.append((b, "status", int(gpu_status[b]), st_ref))
            continue
        n_ref = int(ref.out_num_accepted[b])
        n_gpu = int(gpu_num[b])
        if st_ref:
            ok = n_gpu == 0 and np.all(gpu_tokens[b] == -1)
            rep.positions += 1
            if not ok:
                rep.mismatches_far += 1
                rep.far_detail.append((b, "invalid-seq", gpu_tokens[b].tolist(), n_gpu))
            continue
        evaluated = min(n_ref + 1, g)
        rep.positions += evaluated + 1
        if sampled:
            am = ref.acc_margin[b, :evaluated]
            rep.near_positions += int(np.sum(am < NEAR)) + int(ref.samp_margin[b] < NEAR)
        same = n_gpu == n_ref and np.array_equal(gpu_tokens[b], ref.out_tokens[b])
        if same:
            continue
        if not sampled:
            rep.mismatches_far += 1
            rep.far_detail.append((b, "greedy", gpu_tokens[b].tolist(), ref.out_tokens[b].tolist()))
            continue
        if n_gpu != n_ref:
            j = min(n_gpu, n_ref)
            near = j < g and ref.acc_margin[b, j] < NEAR
            what = f"accept@{j}"
        else:
            near = ref.samp_margin[b] < NEAR
            what = "sample"
        if near:
            rep.mismatches_near += 1
        else:
            rep.mismatches_far += 1
            rep.far_detail.append((b, what, gpu_tokens[b].tolist(), ref.out_tokens[b].tolist(),
                                   float(ref.samp_margin[b])))
    return rep


def read_masks(batch, num_accepted, ok=None):
    """Entries of the diagnostics the early-exit kernel must report: for each
    valid sampled sequence with cut n, the evaluated positions i <= min(n, g-1)
    (p_hat, q_hat, logz_d) and the target rows i <= n (logz_t).  ok: optional
    [B] mask of the sequences to include."""
    B, gmax = batch.B, batch.gmax
    g = np.clip(batch.num_draft.astype(np.int64), 0, gmax)
    n = np.asarray(num_accepted, np.int64)
    live = batch.temperature > 0
    if ok is not None:
        live = live & ok
    i = np.arange(gmax)[None, :]
    pos = live[:, None] & (i < g[:, None]) & (i <= n[:, None])
    i1 = np.arange(gmax + 1)[None, :]
    rows_t = live[:, None] & (i1 <= np.minimum(n, g)[:, None])
    return {"p_hat": pos, "q_hat": pos, "logz_d": pos, "logz_t": rows_t}


def softmax_close(gpu_vals, ref_vals, rtol=SOFTMAX_RTOL, atol=1e-30, need=None):
    """|gpu - ref| <= rtol * |ref| + atol where the oracle has a finite value; the
    finite-value pattern must agree.  Probabilities use rel 1e-5 (atol only
    absorbs float32 underflow); log-normalisers use atol 1e-5, since an absolute
    error d in log Z is a relative error d in every probability.
    need: the early exit reports only the rows it read -- a boolean mask of the
    entries that must be present (finite wherever the oracle is); the others may
    be missing (NaN) but, where present, must match too."""
    g = np.asarray(gpu_vals, np.float64)
    r = np.asarray(ref_vals, np.float64)
    if need is not None:
        need = np.asarray(need, bool)
        missing = need & np.isfinite(r) & ~np.isfinite(g)
        assert not missing.any(), f"{int(missing.sum())} entries the kernel read are missing"
        has = np.isfinite(g)
        assert np.all(np.isfinite(r[has])), "GPU value where the oracle has none"
    else:
        has = np.isfinite(r)
        assert np.array_equal(has, np.isfinite(g)), "finite-value pattern differs"
    if not has.any():
        return 0.0
    err = np.abs(g[has] - r[has])
    bound = rtol * np.abs(r[has]) + atol
    worst = float((err / bound).max())
    assert worst <= 1.0, (f"error {err[np.argmax(err / bound)]:.3e} at ref {r[has][np.argmax(err / bound)]:.6e} "
                          f"exceeds rtol {rtol} / atol {atol}")
    return worst


def compare_tree(tb, gpu_tokens, gpu_num, gpu_path, ref) -> ParityReport:
    """GPU-vs-oracle comparison of one tree round.  Exact match of the accepted
    path, emitted ids and count, except where the walks part at a node whose
    decision was near a boundary in the float64 oracle: a tested child there
    with |u - p/(1 - p(R))| < NEAR, or (both walks stopped there) a final draw
    within NEAR of a CDF boundary.  Greedy sequences must match exactly."""
    rep = ParityReport()
    for b in range(tb.B):
        sampled = tb.temperature[b] > 0
        n_ref, n_gpu = int(ref.out_num_accepted[b]), int(gpu_num[b])
        if int(ref.seq_status[b]):
            rep.positions += 1
            ok = n_gpu == 0 and np.all(gpu_tokens[b] == -1) and np.all(gpu_path[b] == -1)
            if not ok:
                rep.mismatches_far += 1
                rep.far_detail.append((b, "invalid-seq", gpu_tokens[b].tolist(), n_gpu))
            continue
        tested = ~np.isnan(ref.acc_margin[b])
        rep.positions += int(tested.sum()) + 1
        if sampled:
            rep.near_positions += int(np.sum(ref.acc_margin[b][tested] < NEAR)) + int(ref.samp_margin[b] < NEAR)
        same = (n_gpu == n_ref and np.array_equal(gpu_tokens[b], ref.out_tokens[b])
                and np.array_equal(gpu_path[b], ref.out_path[b]))
        if same:
            continue
        if not sampled:
            rep.mismatches_far += 1
            rep.far_detail.append((b, "greedy", gpu_path[b][:n_gpu + 1].tolist(), ref.out_path[b][:n_ref + 1].tolist()))
            continue
        # the node where the walks part: end of the common accepted prefix
        j = 0
        while j < min(n_gpu, n_ref) and gpu_path[b, j] == ref.out_path[b, j]:
            j += 1
        node = int(ref.out_path[b, j - 1]) if j else 0
        kids = [c for c in range(1, int(tb.num_nodes[b])) if tb.parent[b, c] == node]
        margins = [ref.acc_margin[b, c] for c in kids if not np.isnan(ref.acc_margin[b, c])]
        near = any(m < NEAR for m in margins)
        if j == n_gpu == n_ref:
            near = near or ref.samp_margin[b] < NEAR
        if near:
            rep.mismatches_near += 1
        else:
            rep.mismatches_far += 1
            rep.far_detail.append((b, f"part@node{node}", gpu_path[b][:n_gpu].tolist(),
                                   ref.out_path[b][:n_ref].tolist(), gpu_tokens[b][:n_gpu + 1].tolist(),
                                   ref.out_tokens[b][:n_ref + 1].tolist()))
    return rep
