"""One replica rank for tests/test_multi_rank.py, launched by torch.distributed.run with the gloo
backend on CPU: runs the cross-rank steps bench.py takes between replicas and prints one JSON line."""
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import torch.distributed as dist  # noqa: E402

import bench  # noqa: E402
import synth  # noqa: E402

rank, world = int(os.environ["RANK"]), int(os.environ["WORLD_SIZE"])
dist.init_process_group("gloo")
step_ms = 10.0 + 5.0 * rank  # the last rank is the slow replica
slowest = bench.max_over_ranks(step_ms, "cpu", world)
x = synth.gen_x(4, 128, bench.rank_seed(0, rank))  # this rank's own tokens
heads = [None] * world
dist.all_gather_object(heads, x[0, :8].tobytes().hex())
print(json.dumps({"rank": rank, "slowest_ms": slowest,
                  "tokens_per_s": bench.job_tokens_per_s(world, 4, 2, slowest / 1e3),
                  "distinct_tokens": len(set(heads)) == world}), flush=True)
dist.barrier()
dist.destroy_process_group()
