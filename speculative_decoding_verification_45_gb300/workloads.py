"""Seeded synthetic inputs for the speculative-decoding verification step.

This module only builds inputs: target logits, draft logits, drafted tokens,
per-position uniforms and per-sequence temperatures.  It holds none of the
verification arithmetic (no softmax, no accept test, no residual sampling), so
both the CUDA path and the float64 oracle can be fed from it without sharing
any of the method's code.

Drafted tokens stand in for the proposer's output ("Fast Inference from
Transformers via Speculative Decoding" notes, method details, step 1: each
draft token is drawn from the draft distribution q at its position).  They are
drawn with the Gumbel-max trick, x = argmax_j (d_j / T + G_j) with G_j i.i.d.
standard Gumbel, which samples exactly from softmax(d / T) without forming it.
For greedy sequences (T = 0) the draft proposes argmax_j d_j.

All logits are drawn in float64 and rounded to the stored dtype (float32, or
bfloat16 through float32 with round-to-nearest-even); both sides of every
parity check read the rounded values.

Padding that the verifier must never read is poisoned: target rows i > g_b and
draft rows i >= g_b hold +inf, and draft token slots i >= g_b hold -1.
"""
from __future__ import annotations

import dataclasses

import numpy as np

F32 = "f32"
BF16 = "bf16"

BF16_POS_INF = np.uint16(0x7F80)


def f64_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float64 values to bfloat16 (via float32, both steps round-to-nearest-even).

    Returns the raw 16-bit patterns as uint16.  NaN maps to the quiet NaN 0x7FC0.
    """
    f = np.asarray(x, dtype=np.float64).astype(np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    rounded = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)
    nan = np.isnan(f)
    if nan.any():
        rounded[nan] = np.uint16(0x7FC0)
    return rounded


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """Widen raw bfloat16 patterns to float64 (exact)."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


def logits_as_f64(arr: np.ndarray, dtype: str) -> np.ndarray:
    """The stored logits widened exactly to float64."""
    if dtype == BF16:
        return bf16_bits_to_f64(arr)
    return np.asarray(arr, dtype=np.float32).astype(np.float64)


@dataclasses.dataclass
class Batch:
    """One verification call's inputs, host-resident.

    target      [B, gmax+1, V]  float32, or uint16 bfloat16 bit patterns
    draft       [B, gmax,   V]  same dtype as target
    tokens      [B, gmax]       int32 drafted token ids (-1 in padding)
    num_draft   [B]             int32, 0 <= num_draft[b] <= gmax
    uniforms    [B, gmax+1]     float32 in [0, 1); column i < num_draft[b] is the
                                accept-test draw of position i, column gmax the
                                draw for the final (residual or bonus) sample
    temperature [B]             float32; 0 = greedy
    """

    target: np.ndarray
    draft: np.ndarray
    tokens: np.ndarray
    num_draft: np.ndarray
    uniforms: np.ndarray
    temperature: np.ndarray
    dtype: str
    name: str = ""

    @property
    def B(self) -> int:
        return int(self.tokens.shape[0])

    @property
    def gmax(self) -> int:
        return int(self.tokens.shape[1])

    @property
    def V(self) -> int:
        return int(self.target.shape[2])

    @property
    def elem_size(self) -> int:
        return 2 if self.dtype == BF16 else 4

    def algorithmic_bytes(self) -> int:
        """Logit bytes one full verification sweep must read.

        Every target row i <= g_b, plus draft rows i < g_b of sampled (T > 0)
        sequences; greedy sequences never need q.  The 4-byte per-position
        tokens, uniforms, temperatures and outputs are included too.
        """
        g = self.num_draft.astype(np.int64)
        sampled = (self.temperature > 0).astype(np.int64)
        rows = int(((g + 1) + sampled * g).sum())
        small = 4 * (self.B * (self.gmax + self.gmax + 1 + 2) + self.B * (self.gmax + 1) + self.B)
        return rows * self.V * self.elem_size + small

    def nominal_bytes(self) -> int:
        """Bytes of every stored logit row (target and draft), read or not."""
        return (self.target.size + self.draft.size) * self.elem_size


def _round(x64: np.ndarray, dtype: str) -> np.ndarray:
    if dtype == BF16:
        return f64_to_bf16_bits(x64)
    return x64.astype(np.float32)


def _draft_token(rng: np.random.Generator, d_rounded: np.ndarray, dtype: str, temp: float) -> int:
    """Proposer stand-in: one token from softmax(d / T) by Gumbel-max, argmax d when T = 0."""
    d64 = logits_as_f64(d_rounded, dtype)
    if temp == 0.0:
        return int(np.argmax(d64))
    g = rng.gumbel(size=d64.shape[0])
    return int(np.argmax(d64 / float(temp) + g))


def _empty(B: int, gmax: int, V: int, dtype: str):
    if dtype == BF16:
        target = np.full((B, gmax + 1, V), BF16_POS_INF, dtype=np.uint16)
        draft = np.full((B, gmax, V), BF16_POS_INF, dtype=np.uint16)
    else:
        target = np.full((B, gmax + 1, V), np.inf, dtype=np.float32)
        draft = np.full((B, gmax, V), np.inf, dtype=np.float32)
    tokens = np.full((B, gmax), -1, dtype=np.int32)
    return target, draft, tokens


def _zipf_shift(rng: np.random.Generator, V: int) -> np.ndarray:
    """-1.1 * ln(rank), rank = 1 + position of the id in a random permutation."""
    perm = rng.permutation(V)
    rank = np.empty(V, dtype=np.float64)
    rank[perm] = np.arange(1, V + 1, dtype=np.float64)
    return -1.1 * np.log(rank)


# ----------------------------------------------------------------------------
# The five benchmark workloads
# ----------------------------------------------------------------------------

CONFIG_NAMES = {
    1: "B=1, gamma=4, V=1024, f32 logits, T=1.0",
    2: "B=1, gamma=5, V=32000, bf16 logits, 20 peaked ids, T=1.0 (greedy variant T=0)",
    3: "B=32, gamma=4, V=128256, bf16 logits, Zipf-shifted, draft noise sigma in {0.3,0.7,1.5}, T=0.7",
    4: "B=64, ragged gamma in [1,7], V=151936, bf16 logits, Zipf-shifted, T in {0,0.6,1.0}",
    5: "B=256, gamma=4, V=128256, bf16 logits, Zipf-shifted, draft sigma ~ U[0.2,2.0], half greedy / half T=1.0",
}


def default_seed(cfg: int) -> int:
    return 1234 + cfg


def make_config(cfg: int, seed: int | None = None, greedy: bool = False, B: int | None = None) -> Batch:
    """Build one of the five workloads (optionally with fewer sequences B)."""
    if seed is None:
        seed = default_seed(cfg)
    rng = np.random.Generator(np.random.PCG64(seed))
    if cfg == 1:
        return _cfg1(rng, B or 1)
    if cfg == 2:
        return _cfg2(rng, B or 1, greedy)
    if cfg == 3:
        return _zipf_cfg(rng, B or 32, gamma=4, V=128256, ragged=False, name="cfg3")
    if cfg == 4:
        return _zipf_cfg(rng, B or 64, gamma=7, V=151936, ragged=True, name="cfg4")
    if cfg == 5:
        return _zipf_cfg(rng, B or 256, gamma=4, V=128256, ragged=False, name="cfg5")
    raise ValueError(f"unknown config {cfg}")


def _cfg1(rng: np.random.Generator, B: int) -> Batch:
    gamma, V = 4, 1024
    target, draft, tokens = _empty(B, gamma, V, F32)
    temp = np.full(B, 1.0, dtype=np.float32)
    for b in range(B):
        t = rng.normal(0.0, 2.0, size=(gamma + 1, V))
        d = t[:gamma] + rng.normal(0.0, 0.5, size=(gamma, V))
        target[b] = _round(t, F32)
        draft[b] = _round(d, F32)
        for i in range(gamma):
            tokens[b, i] = _draft_token(rng, draft[b, i], F32, float(temp[b]))
    num_draft = np.full(B, gamma, dtype=np.int32)
    uniforms = rng.random((B, gamma + 1), dtype=np.float32)
    return Batch(target, draft, tokens, num_draft, uniforms, temp, F32, "cfg1")


def _cfg2(rng: np.random.Generator, B: int, greedy: bool) -> Batch:
    gamma, V = 5, 32000
    target, draft, tokens = _empty(B, gamma, V, BF16)
    temp = np.full(B, 0.0 if greedy else 1.0, dtype=np.float32)
    for b in range(B):
        t = rng.normal(0.0, 3.0, size=(gamma + 1, V))
        for i in range(gamma + 1):
            peaks = rng.choice(V, size=20, replace=False)
            t[i, peaks] += 8.0
        d = t[:gamma] + rng.normal(0.0, 1.0, size=(gamma, V))
        target[b] = _round(t, BF16)
        draft[b] = _round(d, BF16)
        for i in range(gamma):
            tokens[b, i] = _draft_token(rng, draft[b, i], BF16, float(temp[b]))
    num_draft = np.full(B, gamma, dtype=np.int32)
    uniforms = rng.random((B, gamma + 1), dtype=np.float32)
    return Batch(target, draft, tokens, num_draft, uniforms, temp, BF16, "cfg2-greedy" if greedy else "cfg2")


def _zipf_cfg(rng: np.random.Generator, B: int, gamma: int, V: int, ragged: bool, name: str) -> Batch:
    target, draft, tokens = _empty(B, gamma, V, BF16)
    if name == "cfg3":
        temp = np.full(B, 0.7, dtype=np.float32)
        sigma = np.array([(0.3, 0.7, 1.5)[b % 3] for b in range(B)])
    elif name == "cfg4":
        temp = np.array([(0.0, 0.6, 1.0)[b % 3] for b in range(B)], dtype=np.float32)
        sigma = np.array([(0.3, 0.7, 1.5)[b % 3] for b in range(B)])
    else:
        temp = np.array([0.0 if b % 2 == 0 else 1.0 for b in range(B)], dtype=np.float32)
        sigma = rng.uniform(0.2, 2.0, size=B)
    if ragged:
        num_draft = rng.integers(1, gamma + 1, size=B).astype(np.int32)
    else:
        num_draft = np.full(B, gamma, dtype=np.int32)
    for b in range(B):
        g = int(num_draft[b])
        shift = _zipf_shift(rng, V)
        t = rng.normal(0.0, 3.0, size=(g + 1, V)) + shift
        d = t[:g] + rng.normal(0.0, float(sigma[b]), size=(g, V))
        target[b, : g + 1] = _round(t, BF16)
        draft[b, :g] = _round(d, BF16)
        for i in range(g):
            tokens[b, i] = _draft_token(rng, draft[b, i], BF16, float(temp[b]))
    uniforms = rng.random((B, gamma + 1), dtype=np.float32)
    return Batch(target, draft, tokens, num_draft, uniforms, temp, BF16, name)


def zipf_sequences(B: int, rows: int, V: int, seed: int, sigma=(0.2, 2.0), dtype: str = BF16):
    """Rows of the large workloads' generator for the draw-rate tests: per
    sequence b one Zipf shift (a random permutation of ranks), target rows
    t_i ~ N(0, 3^2) + shift for i < rows, draft rows d_i = t_i + N(0, s_b^2)
    for i < rows - 1 with s_b ~ U[sigma], all rounded to dtype.
    Returns (target [B, rows, V], draft [B, rows - 1, V]) as bfloat16 bits
    (uint16) or float32."""
    rng = np.random.Generator(np.random.PCG64(seed))
    store = np.uint16 if dtype == BF16 else np.float32
    target = np.empty((B, rows, V), dtype=store)
    draft = np.empty((B, max(rows - 1, 0), V), dtype=store)
    for b in range(B):
        shift = _zipf_shift(rng, V)
        t = rng.normal(0.0, 3.0, size=(rows, V)) + shift
        s_b = rng.uniform(sigma[0], sigma[1])
        target[b] = _round(t, dtype)
        if rows > 1:
            draft[b] = _round(t[: rows - 1] + rng.normal(0.0, s_b, size=(rows - 1, V)), dtype)
    return target, draft


# ----------------------------------------------------------------------------
# Tiny-vocabulary batches for the distribution checks
# ----------------------------------------------------------------------------

def tiny_batch(p_rows, q_rows, N: int, seed: int, temperature: float = 1.0) -> Batch:
    """N independent copies of one round with fixed per-position distributions.

    p_rows: gamma+1 probability vectors over a tiny vocabulary (target at each
    position, the last one is the bonus position); q_rows: gamma vectors (draft).
    Logits are the float32 natural logs of the given probabilities times the
    temperature, so that softmax(logits / T) reproduces them up to float32
    rounding.  Zero probabilities become -inf logits.  Drafted tokens are drawn
    from q_rows by inverse transform on seeded uniforms.
    """
    p = np.asarray(p_rows, dtype=np.float64)
    q = np.asarray(q_rows, dtype=np.float64)
    gamma = q.shape[0]
    V = p.shape[1]
    assert p.shape == (gamma + 1, V) and q.shape == (gamma, V)
    rng = np.random.Generator(np.random.PCG64(seed))
    with np.errstate(divide="ignore"):
        tl = (np.log(p) * temperature).astype(np.float32)
        dl = (np.log(q) * temperature).astype(np.float32) if gamma else np.zeros((0, V), np.float32)
    target = np.broadcast_to(tl, (N, gamma + 1, V)).copy()
    draft = np.broadcast_to(dl, (N, gamma, V)).copy()
    tokens = np.empty((N, gamma), dtype=np.int32)
    for i in range(gamma):
        cdf = np.cumsum(q[i])
        cdf[-1] = 1.0
        x = rng.random(N)
        tokens[:, i] = np.searchsorted(cdf, x, side="right").astype(np.int32)
    tokens = np.minimum(tokens, V - 1)
    num_draft = np.full(N, gamma, dtype=np.int32)
    uniforms = rng.random((N, gamma + 1), dtype=np.float32)
    temp = np.full(N, temperature, dtype=np.float32)
    return Batch(target, draft, tokens, num_draft, uniforms, temp, F32, "tiny")


def worked_example_rows():
    """Draft gives the token 0.4, target 0.1 (the rest split so both sum to one)."""
    p = [[0.1, 0.6, 0.3], [1.0 / 3, 1.0 / 3, 1.0 / 3]]
    q = [[0.4, 0.3, 0.3]]
    return p, q


def alpha_rows(alpha: float, gamma: int):
    """Two-token rows with sum_x min(p, q) = alpha exactly, repeated gamma times.

    p = (1/2, 1/2), q = (1/2 + (1 - alpha), 1/2 - (1 - alpha)); needs alpha >= 1/2.
    """
    if not (0.5 <= alpha <= 1.0):
        raise ValueError("alpha must lie in [0.5, 1]")
    eps = 1.0 - alpha
    p = [[0.5, 0.5]] * (gamma + 1)
    q = [[0.5 + eps, 0.5 - eps]] * gamma
    return p, q


def edge_batch(kind: str, V: int = 1023, gamma: int = 3, B: int = 8, seed: int = 7,
               dtype: str = BF16) -> Batch:
    """Hand-made edge cases (see the parity tests for what each exercises).

    kinds: 'zero_draft' (num_draft = 0 everywhere), 'reject_first' (draft logits
    put all mass on a token the target gives ~0), 'accept_all' (draft equals
    target), 'greedy_ties' (T = 0, repeated maxima), 'neg_inf' (some -inf
    logits), 'mixed' (random ragged g, mixed T, generic V).
    """
    rng = np.random.Generator(np.random.PCG64(seed))
    target, draft, tokens = _empty(B, gamma, V, dtype)
    num_draft = np.full(B, gamma, dtype=np.int32)
    temp = np.full(B, 1.0, dtype=np.float32)
    for b in range(B):
        t = rng.normal(0.0, 2.0, size=(gamma + 1, V))
        d = t[:gamma] + rng.normal(0.0, 0.7, size=(gamma, V))
        g = gamma
        if kind == "zero_draft":
            g = 0
            temp[b] = (0.0, 0.8)[b % 2]
        elif kind == "reject_first":
            d[:] = -30.0
            d[:, 5] = 30.0
            t[:, 5] = -30.0
        elif kind == "accept_all":
            d = t[:gamma].copy()
        elif kind == "greedy_ties":
            temp[b] = 0.0
            t = np.round(t * 2.0) / 2.0
            for i in range(gamma + 1):
                top = t[i].max()
                ids = rng.choice(V, size=3, replace=False)
                t[i, ids] = top
        elif kind == "neg_inf":
            temp[b] = (0.0, 1.0)[b % 2]
            mask = rng.random((gamma + 1, V)) < 0.3
            t[mask] = -np.inf
            dm = rng.random((gamma, V)) < 0.3
            d[dm] = -np.inf
        elif kind == "mixed":
            g = int(rng.integers(0, gamma + 1))
            temp[b] = (0.0, 0.5, 1.3)[b % 3]
        else:
            raise ValueError(kind)
        num_draft[b] = g
        target[b, : g + 1] = _round(t[: g + 1], dtype)
        draft[b, :g] = _round(d[:g], dtype)
        for i in range(g):
            if kind == "greedy_ties":
                # propose the lowest-index maximum half of the time, another tied id otherwise
                row = logits_as_f64(target[b, i], dtype)
                tied = np.flatnonzero(row == row.max())
                tokens[b, i] = int(tied[0]) if rng.random() < 0.5 else int(tied[-1])
            else:
                tokens[b, i] = _draft_token(rng, draft[b, i], dtype, float(temp[b]))
    uniforms = rng.random((B, gamma + 1), dtype=np.float32)
    return Batch(target, draft, tokens, num_draft, uniforms, temp, dtype, f"edge-{kind}")


def random_batch(seed: int) -> Batch:
    """A seeded batch of random shape and content, for broad parity sweeps.

    B in [1, 48]; gamma_max in [0, 9] with num_draft ragged in [0, gamma_max];
    V tiny, mid-sized or up to 70000 (odd sizes included); bf16 (60 %) or
    float32; a temperature per sequence from {0, 0.05, 0.3, 0.7, 1, 1.7, 4};
    target rows N(0, s^2) with s in [0.5, 6] (plus the Zipf shift of the large
    workloads half the time), draft rows the target plus N(0, sigma^2); drafted
    ids drawn from the draft rows as the proposer stand-in does; uniforms
    U[0, 1).  About one sequence in twenty carries a data problem (a drafted id
    outside [0, V), a negative or NaN temperature, or num_draft above
    gamma_max), which must give -1 tokens and a status bit.
    """
    rng = np.random.Generator(np.random.PCG64(seed))
    B = int(rng.integers(1, 49))
    gmax = int(rng.integers(0, 10))
    pick = int(rng.integers(0, 5))
    V = [int(rng.integers(2, 64)), int(rng.integers(64, 5000)), int(rng.integers(5000, 70000)), 32000, 4097][pick]
    dtype = BF16 if rng.random() < 0.6 else F32
    target, draft, tokens = _empty(B, gmax, V, dtype)
    num_draft = rng.integers(0, gmax + 1, size=B).astype(np.int32)
    temp = rng.choice(np.array([0.0, 0.05, 0.3, 0.7, 1.0, 1.7, 4.0], np.float32), size=B).astype(np.float32)
    scale = float(rng.uniform(0.5, 6.0))
    zipf = rng.random() < 0.5
    for b in range(B):
        g = int(num_draft[b])
        t = rng.normal(0.0, scale, size=(g + 1, V))
        if zipf:
            t = t + _zipf_shift(rng, V)
        d = t[:g] + rng.normal(0.0, float(rng.uniform(0.1, 2.5)), size=(g, V))
        target[b, : g + 1] = _round(t, dtype)
        draft[b, :g] = _round(d, dtype)
        for i in range(g):
            tokens[b, i] = _draft_token(rng, draft[b, i], dtype, float(temp[b]))
    for b in range(B):
        if rng.random() >= 0.05:
            continue
        kind = int(rng.integers(0, 3))
        if kind == 0 and num_draft[b] > 0:
            tokens[b, int(rng.integers(0, num_draft[b]))] = int(rng.choice([-1, V, V + 7]))
        elif kind == 1:
            temp[b] = np.float32(rng.choice([-1.0, np.nan]))
        else:
            num_draft[b] = gmax + 1
    uniforms = rng.random((B, gmax + 1), dtype=np.float32)
    return Batch(target, draft, tokens, num_draft, uniforms, temp, dtype, f"random{seed}")


def describe(batch: Batch) -> str:
    return (f"{batch.name}: B={batch.B} gmax={batch.gmax} V={batch.V} dtype={batch.dtype} "
            f"logit bytes={batch.algorithmic_bytes()} (nominal {batch.nominal_bytes()})")


# ----------------------------------------------------------------------------
# Token contexts for the prompt-lookup proposer
# ----------------------------------------------------------------------------

def ngram_contexts(B: int, L: int, vocab: int, seed: int, copy_prob: float = 0.5, ragged: bool = True):
    """Token histories where earlier spans reappear, as in summarising or editing
    text whose output repeats the input ("Speculative Decoding", ch.5).

    Each context is built from segments of 4..32 tokens: with probability
    copy_prob a copy of an earlier span of the same context, otherwise fresh
    uniform ids in [0, vocab).  Returns (contexts int32 [B, L] padded with -1,
    lengths int32 [B]); lengths are uniform in [L/2, L] when ragged.
    """
    rng = np.random.Generator(np.random.PCG64(seed))
    ctx = np.full((B, L), -1, np.int32)
    lens = (rng.integers(L // 2, L + 1, size=B) if ragged else np.full(B, L)).astype(np.int32)
    for b in range(B):
        n = int(lens[b])
        row = []
        while len(row) < n:
            seg = int(rng.integers(4, 33))
            if row and rng.random() < copy_prob:
                start = int(rng.integers(0, len(row)))
                piece = row[start:start + seg]
            else:
                piece = list(rng.integers(0, vocab, size=seg))
            row.extend(int(t) for t in piece)
        ctx[b, :n] = row[:n]
    return ctx, lens


# ----------------------------------------------------------------------------
# Candidate trees (tree verification)
# ----------------------------------------------------------------------------

@dataclasses.dataclass
class TreeBatch:
    """One tree-verification call's inputs, host-resident.

    target      [B, N, V]  float32, or uint16 bfloat16 bit patterns; row k is the
                           target's next-token logits after the path to node k
                           (rows of nodes >= num_nodes[b] poisoned with +inf)
    parent      [B, N]     int32, parent[b, k] < k for 1 <= k < num_nodes[b]; -1 else
    tokens      [B, N]     int32 candidate id of node k (-1 for the root and padding)
    num_nodes   [B]        int32 in [1, N]
    uniforms    [B, N]     float32 in [0, 1); column k tests node k, column 0 is
                           the final sample's draw
    temperature [B]        float32; 0 = greedy
    """

    target: np.ndarray
    parent: np.ndarray
    tokens: np.ndarray
    num_nodes: np.ndarray
    uniforms: np.ndarray
    temperature: np.ndarray
    dtype: str
    name: str = "tree"

    @property
    def B(self) -> int:
        return int(self.parent.shape[0])

    @property
    def N(self) -> int:
        return int(self.parent.shape[1])

    @property
    def V(self) -> int:
        return int(self.target.shape[2])

    @property
    def elem_size(self) -> int:
        return 2 if self.dtype == BF16 else 4

    def path_bytes(self, num_accepted) -> int:
        """Logit bytes a walk must read given the accepted path lengths: the
        n_b + 1 rows of the path (root included), plus the 4-byte inputs and
        outputs."""
        rows = int((np.asarray(num_accepted, np.int64) + 1).sum())
        small = 4 * self.B * (5 * self.N + 3)
        return rows * self.V * self.elem_size + small


def tree_parents(shape: str, n: int, rng: np.random.Generator) -> np.ndarray:
    """Parent array of an n-node tree (node 0 the root, parent[0] = -1).

    'chain': one candidate per position; 'star': n-1 candidates for the first
    position; 'random': parent[k] uniform over [0, k); 'medusa': breadth-first
    levels with 4, 3, 2, 2, 1, 1, ... children per node (the top few tokens of
    each head combined, "Speculative Decoding" ch.5), cut at n nodes.
    """
    par = np.full(n, -1, np.int32)
    if shape == "chain":
        par[1:] = np.arange(n - 1)
    elif shape == "star":
        par[1:] = 0
    elif shape == "random":
        for k in range(1, n):
            par[k] = rng.integers(0, k)
    elif shape == "medusa":
        fan = [4, 3, 2, 2]
        level, k, depth = [0], 1, 0
        while k < n and level:
            nxt = []
            f = fan[depth] if depth < len(fan) else 1
            for node in level:
                for _ in range(f):
                    if k >= n:
                        break
                    par[k] = node
                    nxt.append(k)
                    k += 1
            level, depth = nxt, depth + 1
    else:
        raise ValueError(f"unknown tree shape {shape}")
    return par


def tree_batch(B: int, N: int, V: int, dtype: str = BF16, seed: int = 0, shape: str = "medusa",
               temps=(0.0, 0.6, 1.0), sigma: float = 0.7, ragged: bool = True, zipf: bool = True) -> TreeBatch:
    """Seeded candidate trees.  Per sequence: num_nodes = N (or uniform in
    [1, N] when ragged), target rows t_k ~ N(0, 3^2) (+ the Zipf shift of the
    large workloads when zipf), and the children of node k, in index order,
    carry the best ids of a noisy proposer view d_k = t_k + N(0, sigma^2) (the
    top candidates of a head, deterministic).  T_b = temps[b mod len(temps)]."""
    rng = np.random.Generator(np.random.PCG64(seed))
    if dtype == BF16:
        target = np.full((B, N, V), BF16_POS_INF, dtype=np.uint16)
    else:
        target = np.full((B, N, V), np.inf, dtype=np.float32)
    parent = np.full((B, N), -1, np.int32)
    tokens = np.full((B, N), -1, np.int32)
    num_nodes = (rng.integers(1, N + 1, size=B) if ragged else np.full(B, N)).astype(np.int32)
    temp = np.array([temps[b % len(temps)] for b in range(B)], dtype=np.float32)
    for b in range(B):
        n = int(num_nodes[b])
        par = tree_parents(shape, n, rng)
        parent[b, :n] = par
        t = rng.normal(0.0, 3.0, size=(n, V))
        if zipf:
            t += _zipf_shift(rng, V)
        rows = _round(t, dtype)
        target[b, :n] = rows
        t_rounded = logits_as_f64(rows, dtype)
        for k in range(n):
            kids = np.nonzero(par == k)[0]
            if kids.size == 0:
                continue
            d = t_rounded[k] + rng.normal(0.0, sigma, size=V)
            best = np.argsort(-d, kind="stable")[: kids.size]
            tokens[b, kids] = best.astype(np.int32)
    uniforms = rng.random((B, N), dtype=np.float32)
    return TreeBatch(target, parent, tokens, num_nodes, uniforms, temp, dtype, f"tree-{shape}")


def tree_tiny(p_rows, parent, tokens, count: int, seed: int, temperature: float = 1.0) -> TreeBatch:
    """count copies of one small tree with fixed node distributions p_rows
    (probability vectors over a tiny vocabulary; logits = ln p * T in float32,
    zero probabilities -inf) and fresh seeded uniforms per copy."""
    p = np.asarray(p_rows, dtype=np.float64)
    N, V = p.shape
    rng = np.random.Generator(np.random.PCG64(seed))
    with np.errstate(divide="ignore"):
        tl = (np.log(p) * temperature).astype(np.float32)
    target = np.broadcast_to(tl, (count, N, V)).copy()
    par = np.broadcast_to(np.asarray(parent, np.int32), (count, N)).copy()
    tok = np.broadcast_to(np.asarray(tokens, np.int32), (count, N)).copy()
    uniforms = rng.random((count, N), dtype=np.float32)
    return TreeBatch(target, par, tok, np.full(count, N, np.int32), uniforms,
                     np.full(count, temperature, np.float32), F32, "tree-tiny")
