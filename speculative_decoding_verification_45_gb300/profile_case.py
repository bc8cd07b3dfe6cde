"""Run one path of the library a few times on a fixed seeded workload, for
profilers (ncu) and quick timing:

    python -m speculative_decoding_verification_45_gb300.profile_case \
        {verify,full,early,tree,sample,ngram} [--reps N] [--host] [--config C]

verify         : spec_verify with the automatic kernel choice on workload
                 --config (default 5: B=256, gamma=4, V=128256 bf16)
full / early   : the same with the full sweep / the row-ordered early exit;
                 with --host the inputs stay in page-locked host memory and
                 the kernels read them over the host link (zero copy)
tree           : spec_tree_verify, 32 sequences of 64-node Medusa-style trees
                 over V=128256 (half greedy, half T=1)
sample         : spec_sample, 256 rows of V=128256 (target-only round)
ngram          : spec_ngram_propose, 256 contexts of up to 8192 tokens

Prints the mean time per call (CUDA events over --reps back-to-back calls).
"""
from __future__ import annotations

import argparse


def main(argv=None):
    import torch

    import speculative_decoding_verification_45_gb300 as sv
    from speculative_decoding_verification_45_gb300 import workloads

    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("case", choices=["verify", "full", "early", "tree", "sample", "ngram"])
    ap.add_argument("--reps", type=int, default=10)
    ap.add_argument("--host", action="store_true", help="verify/full/early: inputs in page-locked host memory")
    ap.add_argument("--config", type=int, default=5, choices=[1, 2, 3, 4, 5],
                    help="verify/full/early: the workload (sample, tree, ngram use config 5's sizes)")
    args = ap.parse_args(argv)
    sv.build()
    torch.cuda.set_device(0)
    batch = workloads.make_config(args.config if args.case in ("verify", "full", "early") else 5)
    if args.case in ("verify", "full", "early", "sample"):
        dev = sv.to_device(batch)
        if args.host and args.case != "sample":
            dev = {k: v.cpu().pin_memory() for k, v in dev.items()}
    if args.case == "verify":
        def call():
            sv.verify(**dev)
    elif args.case == "full":
        def call():
            sv.verify(**dev, kernel=sv.KERNEL_REGISTER)
    elif args.case == "early":
        def call():
            sv.verify(**dev, kernel=sv.KERNEL_EARLY)
    elif args.case == "sample":
        rows = dev["target_logits"][:, 0].contiguous()
        u0 = dev["uniforms"][:, -1].contiguous()

        def call():
            sv.sample(rows, u0, dev["temperature"])
    elif args.case == "tree":
        tb = workloads.tree_batch(32, 64, batch.V, dtype=batch.dtype, seed=workloads.default_seed(5) + 11,
                                  shape="medusa", temps=(0.0, 1.0), ragged=False)
        tdev = sv.tree_to_device(tb)

        def call():
            sv.tree_verify(**tdev)
    else:
        ctx_np, lens_np = workloads.ngram_contexts(batch.B, 8192, batch.V, seed=workloads.default_seed(5) + 7)
        ctx, lens = torch.from_numpy(ctx_np).cuda(), torch.from_numpy(lens_np).cuda()

        def call():
            sv.ngram_propose(ctx, lens, 1, 4, batch.gmax)
    for _ in range(3):
        call()
    torch.cuda.synchronize()
    a, z = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(args.reps):
        call()
    z.record()
    torch.cuda.synchronize()
    print(f"{args.case}: {a.elapsed_time(z) / args.reps * 1e3:.2f} us per call ({args.reps} calls)")


if __name__ == "__main__":
    main()
