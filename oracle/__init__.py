"""Float64 CPU oracle for the speculative-decoding verification step.

TEST INFRASTRUCTURE: only tests/, __graft_entry__.smoke() and bench.py's CPU
baseline leg (and its reference arm) may import this package.  It shares no code
with the CUDA path and never imports it.

Contents
  - spec_verify_oracle.c  the sequential float64 restatement of the step
                          (softmax at T, in-order accept test cut at the first
                          rejection, residual or bonus sample, greedy rule);
                          loaded here through ctypes as ``verify``; and the
                          walk of a candidate tree (``tree_verify``).
  - analytic.py           expected tokens per round and speedup formulas.
  - enumerate_law.py      exact outcome law of one round on tiny vocabularies
                          by brute-force enumeration of every random choice
                          (chains and candidate trees).
  - ngram.py              the prompt-lookup (n-gram) proposer, plain loops.
  - gamma_policy.py       the draft-length controller's rule, plain loops.

Parity status: every function here is pinned by -m "not gpu" tests against
values the pages print, the distribution-preservation theorem, and brute force.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "spec_verify_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None

F32 = 0
BF16 = 1

STATUS_BAD_TOKEN = 1
STATUS_BAD_TEMPERATURE = 2
STATUS_BAD_NUM_DRAFT = 4
STATUS_BAD_LOGITS = 8
STATUS_BAD_TREE = 32


def build(force: bool = False) -> str:
    """Compile the C oracle with gcc (plain -O2, IEEE semantics kept)."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-Wall", "-shared", "-fPIC", "-o", tmp, _SRC,
                               "-lm", "-lpthread"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            vp = ctypes.c_void_p
            lib.oracle_verify.argtypes = [vp, vp, ctypes.c_int, vp, vp, vp, vp, ctypes.c_int, ctypes.c_int,
                                          ctypes.c_int, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, ctypes.c_int]
            lib.oracle_verify.restype = ctypes.c_int
            lib.oracle_tree_verify.argtypes = [vp, ctypes.c_int, vp, vp, vp, vp, vp, ctypes.c_int, ctypes.c_int,
                                               ctypes.c_int, vp, vp, vp, vp, vp, vp, ctypes.c_int]
            lib.oracle_tree_verify.restype = ctypes.c_int
            lib.oracle_pick_many.argtypes = [vp, vp, ctypes.c_int, ctypes.c_int, ctypes.c_float, ctypes.c_int,
                                             ctypes.c_int, vp, ctypes.c_int, vp, vp, vp]
            lib.oracle_pick_many.restype = ctypes.c_int
            _lib = lib
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


class OracleResult:
    """Outputs of one oracle call (numpy arrays on the host)."""

    def __init__(self, B, gmax):
        self.out_tokens = np.empty((B, gmax + 1), np.int32)
        self.out_num_accepted = np.empty(B, np.int32)
        self.p_hat = np.empty((B, gmax), np.float64)
        self.q_hat = np.empty((B, gmax), np.float64)
        self.logz_t = np.empty((B, gmax + 1), np.float64)
        self.logz_d = np.empty((B, gmax), np.float64)
        self.resid_mass = np.empty(B, np.float64)
        self.acc_margin = np.empty((B, gmax), np.float64)
        self.samp_margin = np.empty(B, np.float64)
        self.seq_status = np.empty(B, np.int32)


def verify(target, draft, dtype, tokens, num_draft, uniforms, temperature, diagnostics=True,
           nthreads=None) -> OracleResult:
    """Run the oracle on host arrays.

    target [B, gmax+1, V] / draft [B, gmax, V]: float32 arrays (dtype 'f32') or
    uint16 bfloat16 bit patterns (dtype 'bf16'); draft None = point-mass
    proposals (q_i is 1 at x_i); tokens int32 [B, gmax];
    num_draft int32 [B]; uniforms float32 [B, gmax+1]; temperature float32 [B].
    """
    lib = _load()
    code = {"f32": F32, "bf16": BF16}[dtype]
    elem = np.float32 if code == F32 else np.uint16
    target = np.ascontiguousarray(target, dtype=elem)
    point = draft is None  # deterministic proposals: q_i is the point mass at x_i
    if not point:
        draft = np.ascontiguousarray(draft, dtype=elem)
    tokens = np.ascontiguousarray(tokens, dtype=np.int32)
    num_draft = np.ascontiguousarray(num_draft, dtype=np.int32)
    uniforms = np.ascontiguousarray(uniforms, dtype=np.float32)
    temperature = np.ascontiguousarray(temperature, dtype=np.float32)
    B, gmax = tokens.shape
    V = target.shape[2]
    assert target.shape == (B, gmax + 1, V) and (point or draft.shape == (B, gmax, V))
    assert uniforms.shape == (B, gmax + 1) and num_draft.shape == (B,) and temperature.shape == (B,)
    res = OracleResult(B, gmax)
    if nthreads is None:
        nthreads = os.cpu_count() or 1
    d = diagnostics
    rc = lib.oracle_verify(_ptr(target), None if point else _ptr(draft), code, _ptr(tokens), _ptr(num_draft), _ptr(uniforms),
                           _ptr(temperature), B, gmax, V, _ptr(res.out_tokens), _ptr(res.out_num_accepted),
                           _ptr(res.p_hat) if d else None, _ptr(res.q_hat) if d else None,
                           _ptr(res.logz_t) if d else None, _ptr(res.logz_d) if d else None,
                           _ptr(res.resid_mass), _ptr(res.acc_margin), _ptr(res.samp_margin),
                           _ptr(res.seq_status), int(nthreads))
    if rc != 0:
        raise ValueError("oracle_verify rejected its arguments")
    return res


def verify_batch(batch, diagnostics=True, nthreads=None, point=False) -> OracleResult:
    """Oracle on a workloads.Batch-like object (attributes as in verify()).
    point=True: deterministic proposals (q_i is the point mass at x_i; no draft rows)."""
    return verify(batch.target, None if point else batch.draft, batch.dtype, batch.tokens, batch.num_draft,
                  batch.uniforms, batch.temperature, diagnostics=diagnostics, nthreads=nthreads)


class TreeResult:
    """Outputs of one tree-oracle call (numpy arrays on the host)."""

    def __init__(self, B, N):
        self.out_tokens = np.empty((B, N), np.int32)
        self.out_num_accepted = np.empty(B, np.int32)
        self.out_path = np.empty((B, N), np.int32)
        self.acc_margin = np.empty((B, N), np.float64)
        self.samp_margin = np.empty(B, np.float64)
        self.seq_status = np.empty(B, np.int32)


def tree_verify(target, dtype, parent, tokens, num_nodes, uniforms, temperature, nthreads=None) -> TreeResult:
    """Tree oracle on host arrays: target [B, N, V] (float32, or uint16 bfloat16
    bits for 'bf16'); parent, tokens int32 [B, N]; num_nodes int32 [B];
    uniforms float32 [B, N] (column c tests node c, column 0 the final
    sample); temperature float32 [B]."""
    lib = _load()
    code = {"f32": F32, "bf16": BF16}[dtype]
    elem = np.float32 if code == F32 else np.uint16
    target = np.ascontiguousarray(target, dtype=elem)
    parent = np.ascontiguousarray(parent, dtype=np.int32)
    tokens = np.ascontiguousarray(tokens, dtype=np.int32)
    num_nodes = np.ascontiguousarray(num_nodes, dtype=np.int32)
    uniforms = np.ascontiguousarray(uniforms, dtype=np.float32)
    temperature = np.ascontiguousarray(temperature, dtype=np.float32)
    B, N, V = target.shape
    assert parent.shape == (B, N) and tokens.shape == (B, N) and uniforms.shape == (B, N)
    assert num_nodes.shape == (B,) and temperature.shape == (B,)
    res = TreeResult(B, N)
    if nthreads is None:
        nthreads = os.cpu_count() or 1
    rc = lib.oracle_tree_verify(_ptr(target), code, _ptr(parent), _ptr(tokens), _ptr(num_nodes), _ptr(uniforms),
                                _ptr(temperature), B, N, V, _ptr(res.out_tokens), _ptr(res.out_num_accepted),
                                _ptr(res.out_path), _ptr(res.acc_margin), _ptr(res.samp_margin),
                                _ptr(res.seq_status), int(nthreads))
    if rc != 0:
        raise ValueError("oracle_tree_verify rejected its arguments")
    return res


def tree_verify_batch(tb, nthreads=None) -> TreeResult:
    """Tree oracle on a workloads.TreeBatch-like object."""
    return tree_verify(tb.target, tb.dtype, tb.parent, tb.tokens, tb.num_nodes, tb.uniforms, tb.temperature,
                       nthreads=nthreads)


PICK_P = 0          # p of the row (a bonus row, or the sampler's draw)
PICK_RESIDUAL = 1   # max(0, p - q), q from a draft row
PICK_POINT = 2      # p without the point-mass draft xn


def pick_many(target_row, dtype, temperature, uniforms, mode=PICK_P, draft_row=None, xn=-1):
    """The final draw of oracle_verify for many uniforms on one decided row.

    target_row / draft_row: V logits (float32, or uint16 bfloat16 bits);
    uniforms: float32 [n].  Returns (picks int32 [n], margins float64 [n], S):
    the smallest j with u*S < C_j for each u, the distance of u to the nearer
    CDF boundary of that pick, and the total weight S."""
    lib = _load()
    code = {"f32": F32, "bf16": BF16}[dtype]
    elem = np.float32 if code == F32 else np.uint16
    t = np.ascontiguousarray(target_row, dtype=elem).reshape(-1)
    d = None if draft_row is None else np.ascontiguousarray(draft_row, dtype=elem).reshape(-1)
    u = np.ascontiguousarray(uniforms, dtype=np.float32).reshape(-1)
    picks = np.empty(u.size, np.int32)
    margins = np.empty(u.size, np.float64)
    mass = np.zeros(1, np.float64)
    rc = lib.oracle_pick_many(_ptr(t), _ptr(d), code, t.size, float(temperature), int(mode), int(xn), _ptr(u),
                              u.size, _ptr(picks), _ptr(margins), _ptr(mass))
    if rc != 0:
        raise ValueError("oracle_pick_many rejected its arguments")
    return picks, margins, float(mass[0])
