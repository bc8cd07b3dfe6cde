"""Agreement of the final draw with the float64 oracle over more than 10^5
draws each from full rows and from residual rows of the V = 128256 workload
rows (Zipf-shifted N(0, 3^2) bf16 logits, draft noise sigma ~ U[0.2, 2.0]).

The contract ("Speculative Decoding", ch.3: the method is lossless up to the
hardware's numerics) allows a GPU pick to differ from the oracle only where the
uniform lies within 1e-5 of a CDF boundary, and requires such disagreements to
stay below 0.01 % of the draws.  A V = 128256 row has ~10^5 boundaries, most
of them 1e-7 to 1e-9 apart, so this is a test of the weights' precision: each
pick is compared with oracle.pick_many on the same row and uniform.

Draws come from:
  * spec_sample (target-only / draft-side sampling): 512 rows x 200 uniforms
    (and 512 float32 rows of V = 32000 x 200);
  * spec_verify bonus rows: every draft accepted (accept uniform 0), 256
    sequences x 400 final uniforms, both kernels;
  * spec_verify residual rows: a rejection forced at position 0 (x = argmax of
    q - p, accept uniform just below 1), 256 x 400, both kernels;
  * point-mass residuals (draft_logits = NULL, x = argmax p): 256 x 100.
"""
import functools

import numpy as np
import pytest

from speculative_decoding_verification_45_gb300 import workloads
from tests.test_gpu_parity import sv  # noqa: F401

gpu = pytest.mark.gpu

V = 128256
NEAR = 1e-5
RATE = 1e-4
BELOW_ONE = np.float32(np.nextafter(np.float32(1.0), np.float32(0.0)))


@functools.lru_cache(maxsize=None)
def _rows(B, rows, seed):
    return workloads.zipf_sequences(B, rows, V, seed)


def _uniforms(n, k, seed):
    return np.random.default_rng(seed).random((k, n), dtype=np.float32)


class Tally:
    def __init__(self):
        self.picks = self.mism = self.near = self.far = 0
        self.detail = []

    def add(self, gpu_picks, ref_picks, margins):
        bad = gpu_picks != ref_picks
        self.picks += gpu_picks.size
        self.mism += int(bad.sum())
        self.near += int((margins < NEAR).sum())
        far = bad & (margins >= NEAR)
        self.far += int(far.sum())
        if far.any():
            i = int(np.argmax(far))
            self.detail.append((int(gpu_picks.flat[i]), int(ref_picks.flat[i]), float(margins.flat[i])))

    def check(self, what):
        print(f"{what}: picks={self.picks} mismatches={self.mism} (rate {self.mism / self.picks:.2e}) "
              f"near={self.near} far={self.far}")
        assert self.picks >= 100_000
        assert self.far == 0, self.detail[:5]
        assert self.mism < RATE * self.picks, f"{self.mism} of {self.picks}"


def _oracle(oracle_mod, t_rows, us, temp, mode=0, d_rows=None, xs=None):
    """[k, n] picks and margins: row b drawn with us[:, b]."""
    k, n = us.shape
    picks = np.empty((k, n), np.int32)
    margins = np.empty((k, n), np.float64)
    for b in range(n):
        p, m, _ = oracle_mod.pick_many(t_rows[b], "bf16", temp, us[:, b], mode=mode,
                                       draft_row=None if d_rows is None else d_rows[b],
                                       xn=-1 if xs is None else int(xs[b]))
        picks[:, b] = p
        margins[:, b] = m
    return picks, margins


def _bf16(a, dev):
    import torch

    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(dev)


@gpu
def test_sampler_full_rows_float32(sv, oracle_mod):
    """float32 rows (4 ids per 16-byte chunk) of the same recipe at V = 32000:
    the other chunk layout of the exact draw, 512 rows x 200 uniforms."""
    import torch

    V32 = 32000
    t, _ = workloads.zipf_sequences(512, 1, V32, 9005, dtype="f32")
    rows = t[:, 0]
    us = _uniforms(rows.shape[0], 200, 33)
    logits = torch.from_numpy(np.ascontiguousarray(rows)).to("cuda")
    temps = torch.ones(rows.shape[0], dtype=torch.float32, device="cuda")
    out = torch.empty((200, rows.shape[0]), dtype=torch.int32, device="cuda")
    u_dev = torch.from_numpy(us).to("cuda")
    for i in range(200):
        sv.sample(logits, u_dev[i], temps, out_tokens=out[i])
    torch.cuda.synchronize()
    picks = np.empty((200, rows.shape[0]), np.int32)
    margins = np.empty((200, rows.shape[0]), np.float64)
    for b in range(rows.shape[0]):
        p, m, _ = oracle_mod.pick_many(rows[b], "f32", 1.0, us[:, b])
        picks[:, b] = p
        margins[:, b] = m
    tally = Tally()
    tally.add(out.cpu().numpy(), picks, margins)
    tally.check("sampler float32 T=1")


@gpu
@pytest.mark.parametrize("temp", [1.0, 0.7])
def test_sampler_full_rows(sv, oracle_mod, temp):
    import torch

    t, _ = _rows(512, 1, 9001)
    rows = t[:, 0]
    k = 200 if temp == 1.0 else 100
    us = _uniforms(rows.shape[0], k, 31 if temp == 1.0 else 32)
    dev = "cuda"
    logits = _bf16(rows, dev)
    temps = torch.full((rows.shape[0],), temp, dtype=torch.float32, device=dev)
    out = torch.empty((k, rows.shape[0]), dtype=torch.int32, device=dev)
    u_dev = torch.from_numpy(us).to(dev)
    for i in range(k):
        sv.sample(logits, u_dev[i], temps, out_tokens=out[i])
    torch.cuda.synchronize()
    ref, margins = _oracle(oracle_mod, rows, us, temp)
    tally = Tally()
    tally.add(out.cpu().numpy(), ref, margins)
    if temp == 1.0:
        tally.check(f"sampler T={temp}")
    else:  # fewer draws: the rate bound over these alone
        assert tally.far == 0 and tally.mism < RATE * max(tally.picks, 100_000), (tally.mism, tally.picks)


def _verify_draws(sv, t, d, tokens, u0, us, kernel, point=False):
    import torch

    B = t.shape[0]
    dev = "cuda"
    tl = _bf16(t, dev)
    dl = None if point else _bf16(d, dev)
    tok = torch.from_numpy(np.ascontiguousarray(tokens, np.int32).reshape(B, 1)).to(dev)
    nd = torch.ones(B, dtype=torch.int32, device=dev)
    temps = torch.ones(B, dtype=torch.float32, device=dev)
    k = us.shape[0]
    uni = np.empty((k, B, 2), np.float32)
    uni[:, :, 0] = u0
    uni[:, :, 1] = us
    u_dev = torch.from_numpy(uni).to(dev)
    out_t = torch.empty((k, B, 2), dtype=torch.int32, device=dev)
    out_n = torch.empty((k, B), dtype=torch.int32, device=dev)
    for i in range(k):
        sv.verify(tl, dl, tok, nd, u_dev[i], temps, out_tokens=out_t[i], out_num_accepted=out_n[i], kernel=kernel)
    torch.cuda.synchronize()
    return out_t.cpu().numpy(), out_n.cpu().numpy()


@gpu
@pytest.mark.parametrize("kernel", [2, 3])
def test_verify_bonus_rows(sv, oracle_mod, kernel):
    t, d = _rows(256, 2, 9002)
    B = t.shape[0]
    us = _uniforms(B, 400, 41)
    tokens = np.zeros(B, np.int32)  # accepted whatever it is: u = 0 and p(x) > 0
    out_t, out_n = _verify_draws(sv, t, d, tokens, 0.0, us, kernel)
    assert (out_n == 1).all()
    ref, margins = _oracle(oracle_mod, t[:, 1], us, 1.0)
    tally = Tally()
    tally.add(out_t[:, :, 1], ref, margins)
    tally.check(f"bonus rows, kernel {kernel}")


@gpu
@pytest.mark.parametrize("kernel", [2, 3])
def test_verify_residual_rows(sv, oracle_mod, kernel):
    t, d = _rows(256, 2, 9003)
    B = t.shape[0]
    tf = workloads.bf16_bits_to_f64(t[:, 0])
    df = workloads.bf16_bits_to_f64(d[:, 0])
    p = np.exp(tf - tf.max(axis=1, keepdims=True))
    p /= p.sum(axis=1, keepdims=True)
    q = np.exp(df - df.max(axis=1, keepdims=True))
    q /= q.sum(axis=1, keepdims=True)
    tokens = np.argmax(q - p, axis=1).astype(np.int32)  # q(x) > p(x): rejected when u is just below 1
    us = _uniforms(B, 400, 51)
    out_t, out_n = _verify_draws(sv, t, d, tokens, BELOW_ONE, us, kernel)
    assert (out_n == 0).all()
    ref, margins = _oracle(oracle_mod, t[:, 0], us, 1.0, mode=oracle_mod.PICK_RESIDUAL, d_rows=d[:, 0])
    tally = Tally()
    tally.add(out_t[:, :, 0], ref, margins)
    tally.check(f"residual rows, kernel {kernel}")


@gpu
def test_verify_point_mass_residual_rows(sv, oracle_mod):
    t, d = _rows(256, 2, 9004)
    B = t.shape[0]
    tokens = np.argmax(workloads.bf16_bits_to_f64(t[:, 0]), axis=1).astype(np.int32)
    us = _uniforms(B, 100, 61)
    out_t, out_n = _verify_draws(sv, t, d, tokens, BELOW_ONE, us, 0, point=True)
    assert (out_n == 0).all()
    ref, margins = _oracle(oracle_mod, t[:, 0], us, 1.0, mode=oracle_mod.PICK_POINT, xs=tokens)
    tally = Tally()
    tally.add(out_t[:, :, 0], ref, margins)
    assert tally.far == 0 and tally.mism < RATE * 100_000, (tally.mism, tally.picks)
