"""Every entry point captured into a CUDA graph and replayed (how a serving loop
launches a fixed-shape step): the replay gives the bits of the eager call.
Each call runs eagerly first, so the one-time per-device set-up (kernel
attributes, cluster occupancy queries) happens outside the capture; what the
host code does on every call (argument checks, the launch shape, the
residency check of the early-exit kernel) runs inside it."""
import numpy as np
import pytest

from speculative_decoding_verification_45_gb300 import workloads
from tests.test_gpu_parity import sv  # noqa: F401

gpu = pytest.mark.gpu


def _eager_then_replay(fn, outs):
    """Run fn eagerly, snapshot outs, clear them, capture fn, replay twice."""
    import torch

    fn()
    torch.cuda.synchronize()
    ref = [o.clone() for o in outs]
    for o in outs:
        o.fill_(-7)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=side):
        fn()
    for o in outs:
        o.fill_(-7)
    graph.replay()
    graph.replay()
    torch.cuda.synchronize()
    for r, o in zip(ref, outs):
        np.testing.assert_array_equal(o.cpu().numpy(), r.cpu().numpy())


@gpu
@pytest.mark.parametrize("kernel", [0, 2, 3])
@pytest.mark.parametrize("cfg,B", [(3, 16), (4, 24)])
def test_verify_replays_from_a_graph(sv, cfg, B, kernel):
    import torch

    batch = workloads.make_config(cfg, B=B)
    dev = sv.to_device(batch)
    ot = torch.empty((batch.B, batch.gmax + 1), dtype=torch.int32, device="cuda")
    on = torch.empty((batch.B,), dtype=torch.int32, device="cuda")
    cnt = torch.zeros(3, dtype=torch.int64, device="cuda")
    _eager_then_replay(lambda: sv.verify(**dev, out_tokens=ot, out_num_accepted=on, kernel=kernel), [ot, on])
    # counters accumulate once per launch: the eager call and two replays
    one = torch.zeros(3, dtype=torch.int64, device="cuda")
    sv.verify(**dev, kernel=kernel, counters=one)
    _eager_then_replay(lambda: sv.verify(**dev, out_tokens=ot, out_num_accepted=on, kernel=kernel, counters=cnt),
                       [ot, on])
    torch.cuda.synchronize()
    assert int(one[2]) > 0
    assert cnt.tolist() == [3 * int(x) for x in one.tolist()]


@gpu
def test_zero_copy_early_exit_replays_from_a_graph(sv):
    import torch

    batch = workloads.make_config(3, B=16)
    host = {k: v.cpu().pin_memory() for k, v in sv.to_device(batch).items()}
    ot = torch.empty((batch.B, batch.gmax + 1), dtype=torch.int32, device="cuda")
    on = torch.empty((batch.B,), dtype=torch.int32, device="cuda")
    _eager_then_replay(lambda: sv.verify(**host, out_tokens=ot, out_num_accepted=on, kernel=sv.KERNEL_EARLY),
                       [ot, on])


@gpu
def test_sample_tree_ngram_replay_from_a_graph(sv):
    import torch

    batch = workloads.make_config(5, B=64)
    dev = sv.to_device(batch)
    rows = dev["target_logits"][:, 0].contiguous()
    u = dev["uniforms"][:, -1].contiguous()
    out = torch.empty((batch.B,), dtype=torch.int32, device="cuda")
    _eager_then_replay(lambda: sv.sample(rows, u, dev["temperature"], out_tokens=out), [out])

    tb = workloads.tree_batch(8, 24, 4099, "bf16", seed=5, shape="random")
    tdev = sv.tree_to_device(tb)
    tt = torch.empty((tb.B, 24), dtype=torch.int32, device="cuda")
    tn = torch.empty((tb.B,), dtype=torch.int32, device="cuda")
    tp = torch.empty((tb.B, 24), dtype=torch.int32, device="cuda")
    _eager_then_replay(lambda: sv.tree_verify(**tdev, out_tokens=tt, out_num_accepted=tn, out_path=tp),
                       [tt, tn, tp])

    ctx, lens = workloads.ngram_contexts(16, 1024, 500, seed=9)
    ctx_d, lens_d = torch.from_numpy(ctx).cuda(), torch.from_numpy(lens).cuda()
    dt = torch.empty((16, 6), dtype=torch.int32, device="cuda")
    dn = torch.empty((16,), dtype=torch.int32, device="cuda")
    _eager_then_replay(lambda: sv.ngram_propose(ctx_d, lens_d, 1, 4, 6, out_tokens=dt, out_num=dn), [dt, dn])
