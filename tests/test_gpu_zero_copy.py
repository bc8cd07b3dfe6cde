"""Inputs in page-locked host memory ("zero copy"): the kernels read the logits,
ids, uniforms and temperatures over the host link with no staging copy.  The
results must be the bits of the device-resident call (itself checked against
the float64 oracle in the other parity tests) and agree with the oracle; the
host checks of the binding and of spec_device_pointer reject what the GPU
cannot read."""
import ctypes

import numpy as np
import pytest

from speculative_decoding_verification_45_gb300 import workloads
from tests import parity
from tests.test_gpu_parity import sv  # noqa: F401

gpu = pytest.mark.gpu


def _pinned(dev):
    return {k: v.cpu().pin_memory() for k, v in dev.items()}


def _verify(sv, inputs, kernel, point=False):
    import torch

    args = dict(inputs)
    if point:
        args["draft_logits"] = None
    t, n = sv.verify(**args, kernel=kernel)
    torch.cuda.synchronize()
    return t.cpu().numpy(), n.cpu().numpy()


@gpu
@pytest.mark.parametrize("kernel", [0, 2, 3])
@pytest.mark.parametrize("cfg,B", [(1, None), (3, 24), (4, 16)])
def test_host_inputs_match_device_and_oracle(sv, oracle_mod, cfg, B, kernel):
    batch = workloads.make_config(cfg, B=B)
    dev = sv.to_device(batch)
    ref_t, ref_n = _verify(sv, dev, kernel)
    got_t, got_n = _verify(sv, _pinned(dev), kernel)
    np.testing.assert_array_equal(got_t, ref_t)
    np.testing.assert_array_equal(got_n, ref_n)
    rep = parity.compare(batch, got_t, got_n, oracle_mod.verify_batch(batch))
    assert rep.mismatches_far == 0, rep.far_detail[:3]


@gpu
@pytest.mark.parametrize("kernel", [0, 3])
def test_host_inputs_point_mass(sv, kernel):
    batch = workloads.make_config(3, B=16)
    dev = sv.to_device(batch)
    ref = _verify(sv, dev, kernel, point=True)
    got = _verify(sv, _pinned(dev), kernel, point=True)
    np.testing.assert_array_equal(got[0], ref[0])
    np.testing.assert_array_equal(got[1], ref[1])


@gpu
def test_host_inputs_mixed_with_device_inputs(sv):
    """Only the logits on the host, the small arrays on the device."""
    batch = workloads.make_config(4, B=8)
    dev = sv.to_device(batch)
    ref = _verify(sv, dev, 0)
    mixed = dict(dev)
    mixed["target_logits"] = dev["target_logits"].cpu().pin_memory()
    mixed["draft_logits"] = dev["draft_logits"].cpu().pin_memory()
    got = _verify(sv, mixed, 3)
    np.testing.assert_array_equal(got[0], ref[0])
    np.testing.assert_array_equal(got[1], ref[1])


@gpu
def test_host_inputs_full_size_early_exit(sv):
    """The 256-sequence, 128256-id workload the benchmark reads over the link."""
    batch = workloads.make_config(5)
    dev = sv.to_device(batch)
    ref = _verify(sv, dev, 2)
    host = _pinned(dev)
    for kernel in (3, 2):
        got = _verify(sv, host, kernel)
        np.testing.assert_array_equal(got[0], ref[0])
        np.testing.assert_array_equal(got[1], ref[1])


@gpu
@pytest.mark.parametrize("cluster", [0, 2, 8, 16])
def test_host_inputs_early_exit_cluster_sizes(sv, oracle_mod, cluster):
    """Early exit on host rows keeps the decided slices in shared memory where
    they fit (clusters of 8 and 16, and the automatic size) and reads the rows
    again where they do not (2 CTAs per sequence): the same bits either way."""
    import torch

    batch = workloads.make_config(3, B=12)
    dev = sv.to_device(batch)
    early = dict(kernel=sv.KERNEL_EARLY, cluster_size=cluster)
    ref_t, ref_n = sv.verify(**dev, **early)
    host = _pinned(dev)
    t, n = sv.verify(**host, **early)
    pt, pn = sv.verify(**{**host, "draft_logits": None}, **early)
    qt, qn = sv.verify(**{**dev, "draft_logits": None}, **early)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(t.cpu().numpy(), ref_t.cpu().numpy())
    np.testing.assert_array_equal(n.cpu().numpy(), ref_n.cpu().numpy())
    np.testing.assert_array_equal(pt.cpu().numpy(), qt.cpu().numpy())
    np.testing.assert_array_equal(pn.cpu().numpy(), qn.cpu().numpy())
    rep = parity.compare(batch, t.cpu().numpy(), n.cpu().numpy(), oracle_mod.verify_batch(batch))
    assert rep.mismatches_far == 0, rep.far_detail[:3]


@gpu
@pytest.mark.parametrize("point", [False, True])
def test_host_inputs_early_exit_float32_staged(sv, oracle_mod, point):
    """float32 rows of 128256 ids: two slices fit in shared memory from
    clusters of 8 up, so the host rows are staged; same bits as device rows at
    the same launch shape, and the oracle's answer outside its tolerance."""
    import torch

    src = workloads.make_config(4, B=12)  # ragged drafts, mixed temperatures
    f32 = lambda a: workloads.logits_as_f64(a, src.dtype).astype(np.float32)  # noqa: E731
    batch = workloads.Batch(f32(src.target), f32(src.draft), src.tokens.copy(), src.num_draft.copy(),
                            src.uniforms.copy(), src.temperature.copy(), "f32", "config 4 rows in float32")
    dev = sv.to_device(batch)
    if point:
        dev["draft_logits"] = None
    host = {k: (v.cpu().pin_memory() if v is not None else None) for k, v in dev.items()}
    early = dict(kernel=sv.KERNEL_EARLY, cluster_size=8)
    ref = sv.verify(**dev, **early)
    got = sv.verify(**host, **early)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(got[0].cpu().numpy(), ref[0].cpu().numpy())
    np.testing.assert_array_equal(got[1].cpu().numpy(), ref[1].cpu().numpy())
    if not point:
        rep = parity.compare(batch, got[0].cpu().numpy(), got[1].cpu().numpy(), oracle_mod.verify_batch(batch))
        assert rep.mismatches_far == 0, rep.far_detail[:3]


@gpu
def test_host_inputs_early_exit_rows_too_wide_to_stage(sv, oracle_mod):
    """float32 rows of 600000 ids (2.4 MB): two slices do not fit in shared
    memory at any cluster size, so pass 2 reads the rows again."""
    import torch

    rng = np.random.default_rng(17)
    B, g, V = 2, 3, 600_000
    target = (rng.standard_normal((B, g + 1, V)) * 2).astype(np.float32)
    draft = (target[:, :g] + rng.standard_normal((B, g, V)) * 0.5).astype(np.float32)
    tokens = np.stack([np.argmax(draft[b], axis=1) for b in range(B)]).astype(np.int32)
    batch = workloads.Batch(target, draft, tokens, np.full(B, g, np.int32),
                            rng.random((B, g + 1)).astype(np.float32), np.array([1.0, 0.8], np.float32), "f32",
                            "wide f32 rows")
    dev = sv.to_device(batch)
    ref = _verify(sv, dev, 2)
    got = _verify(sv, _pinned(dev), 3)
    np.testing.assert_array_equal(got[0], ref[0])
    np.testing.assert_array_equal(got[1], ref[1])
    rep = parity.compare(batch, got[0], got[1], oracle_mod.verify_batch(batch))
    assert rep.mismatches_far == 0, rep.far_detail[:3]
    torch.cuda.synchronize()


@gpu
@pytest.mark.parametrize("kernel", [0, 3])
def test_host_inputs_debug_diagnostics_identical(sv, kernel):
    """Diagnostics too: the staged early exit computes them from the same rows."""
    import torch

    batch = workloads.make_config(4, B=12)
    dev = sv.to_device(batch)
    a = sv.verify_debug(**dev, kernel=kernel)
    b = sv.verify_debug(**_pinned(dev), kernel=kernel)
    torch.cuda.synchronize()
    for k in a:
        np.testing.assert_array_equal(a[k].cpu().numpy(), b[k].cpu().numpy(), err_msg=k)


@gpu
@pytest.mark.parametrize("kind", ["mixed", "reject_first", "accept_all", "neg_inf"])
def test_host_inputs_unaligned_rows(sv, oracle_mod, kind):
    """V = 1023 bf16: rows are not 16-byte multiples, so the element-load path
    runs (no staging); host rows give the device-resident bits."""
    batch = workloads.edge_batch(kind, V=1023)
    dev = sv.to_device(batch)
    for kernel in (0, 3):
        ref = _verify(sv, dev, kernel)
        got = _verify(sv, _pinned(dev), kernel)
        np.testing.assert_array_equal(got[0], ref[0])
        np.testing.assert_array_equal(got[1], ref[1])
    rep = parity.compare(batch, got[0], got[1], oracle_mod.verify_batch(batch))
    assert rep.mismatches_far == 0, rep.far_detail[:3]


@gpu
def test_host_inputs_sample_tree_ngram(sv):
    import torch

    batch = workloads.make_config(3, B=32)
    dev = sv.to_device(batch)
    logits = dev["target_logits"][:, 0].contiguous()
    u = dev["uniforms"][:, 0].contiguous()
    a = sv.sample(logits, u, dev["temperature"])
    # named page-locked inputs, alive until the synchronisation below (the rule
    # the header states; the binding also holds them until the stream passes)
    logits_h, u_h, temp_h = logits.cpu().pin_memory(), u.cpu().pin_memory(), dev["temperature"].cpu().pin_memory()
    b = sv.sample(logits_h, u_h, temp_h)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(a.cpu().numpy(), b.cpu().numpy())

    tb = workloads.tree_batch(8, 24, 4099, "bf16", seed=3, shape="random")
    tdev = sv.tree_to_device(tb)
    ra = sv.tree_verify(**tdev)
    rb = sv.tree_verify(**_pinned(tdev))
    torch.cuda.synchronize()
    for x, y in zip(ra, rb):
        np.testing.assert_array_equal(x.cpu().numpy(), y.cpu().numpy())

    ctx, lens = workloads.ngram_contexts(16, 1024, 500, seed=5)
    ca = sv.ngram_propose(torch.from_numpy(ctx).cuda(), torch.from_numpy(lens).cuda(), 1, 4, 6)
    ctx_h, lens_h = torch.from_numpy(ctx).pin_memory(), torch.from_numpy(lens).pin_memory()
    cb = sv.ngram_propose(ctx_h, lens_h, 1, 4, 6)
    torch.cuda.synchronize()
    for x, y in zip(ca, cb):
        np.testing.assert_array_equal(x.cpu().numpy(), y.cpu().numpy())


@gpu
def test_pageable_host_tensor_rejected(sv):
    batch = workloads.make_config(1)
    dev = sv.to_device(batch)
    args = dict(dev)
    args["target_logits"] = dev["target_logits"].cpu()  # not page-locked
    with pytest.raises(ValueError, match="page-locked"):
        sv.verify(**args)


@gpu
def test_spec_device_pointer(sv):
    import torch

    lib = sv._native.load()
    out = ctypes.c_void_p()
    d = torch.empty(1024, dtype=torch.uint8, device="cuda")
    assert lib.spec_device_pointer(ctypes.c_void_p(d.data_ptr()), ctypes.byref(out)) == sv.SPEC_OK
    assert out.value == d.data_ptr()
    h = torch.empty(4096, dtype=torch.uint8).pin_memory()
    assert lib.spec_device_pointer(ctypes.c_void_p(h.data_ptr() + 256), ctypes.byref(out)) == sv.SPEC_OK
    assert out.value is not None  # with unified addressing the alias equals the host address
    pageable = np.zeros(4096, np.uint8)
    out = ctypes.c_void_p(7)
    rc = lib.spec_device_pointer(ctypes.c_void_p(pageable.ctypes.data), ctypes.byref(out))
    assert rc == sv.SPEC_ERR_INVALID_ARG and out.value == 7
    assert lib.spec_device_pointer(None, ctypes.byref(out)) == sv.SPEC_ERR_INVALID_ARG


@gpu
@pytest.mark.parametrize("seed", range(100, 116))
def test_host_inputs_random_batches(sv, oracle_mod, seed):
    """Random shapes, dtypes, temperatures and planted data problems
    (workloads.random_batch) with every input on the host: the device-resident
    bits at the same launch shape, and the oracle's answer."""
    import torch

    batch = workloads.random_batch(seed)
    kernel = (0, 3)[seed % 2]
    cluster = (0, 2, 4, 8)[(seed // 2) % 4]
    dev = sv.to_device(batch)
    st_d = torch.zeros(1, dtype=torch.int32, device="cuda")
    st_h = torch.zeros(1, dtype=torch.int32, device="cuda")
    ref = sv.verify(**dev, kernel=kernel, cluster_size=cluster, status=st_d)
    got = sv.verify(**_pinned(dev), kernel=kernel, cluster_size=cluster, status=st_h)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(got[0].cpu().numpy(), ref[0].cpu().numpy())
    np.testing.assert_array_equal(got[1].cpu().numpy(), ref[1].cpu().numpy())
    assert int(st_h.item()) == int(st_d.item())
    rep = parity.compare(batch, got[0].cpu().numpy(), got[1].cpu().numpy(), oracle_mod.verify_batch(batch))
    assert rep.mismatches_far == 0, rep.far_detail[:3]


@gpu
def test_page_locked_inputs_held_until_the_stream_passes(sv):
    """The binding keeps page-locked inputs referenced until an event recorded
    after the launch has completed, so torch's pinned-memory cache cannot hand
    a block to someone else while the kernel still reads it over the link."""
    import weakref

    import torch

    batch = workloads.make_config(5, B=32)
    dev = sv.to_device(batch)
    ref_t, ref_n = sv.verify(**dev, kernel=sv.KERNEL_EARLY)
    torch.cuda.synchronize()
    host = {k: v.cpu().pin_memory() for k, v in dev.items()}
    refs = [weakref.ref(t) for t in host.values()]
    toks, num = sv.verify(**host, kernel=sv.KERNEL_EARLY)
    del host
    assert all(r() is not None for r in refs)  # only the binding holds them now
    torch.cuda.synchronize()
    np.testing.assert_array_equal(toks.cpu().numpy(), ref_t.cpu().numpy())
    np.testing.assert_array_equal(num.cpu().numpy(), ref_n.cpu().numpy())
    sv.verify(**dev, kernel=sv.KERNEL_EARLY)  # a later call drops the references whose event has completed
    torch.cuda.synchronize()
    assert all(r() is None for r in refs)
