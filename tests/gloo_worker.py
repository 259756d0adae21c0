"""One rank of the two-process CPU check of bench.py's multi-rank logic
(run by tests/test_multirank_gloo.py with RANK, WORLD_SIZE, MASTER_ADDR and
MASTER_PORT set; gloo backend, no GPU).  Prints one JSON line of results;
rank 0 also prints the reference arm's line before it."""
import argparse
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import torch.distributed as dist  # noqa: E402

import bench  # noqa: E402
from transformer_encoder_layer_gb300.inputs import SHAPES  # noqa: E402


def main():
    ws, rank, local = bench.dist_env()
    dist.init_process_group("gloo")
    # each rank "measured" a different time; the job takes the slowest one
    ms = bench.max_over_ranks(1.0 + 2.0 * rank, dist, "cpu")
    value = bench.whole_job_tokens_per_s(ws, 1000, ms)
    # the reference arm runs on rank 0 only; the other ranks return at once
    args = argparse.Namespace(ref_seqs=1, steps=1, warmup=0)
    bench.run_reference(args, SHAPES["tiny_d32_L32"])
    dist.barrier()
    print(json.dumps({"rank": rank, "world_size": ws, "local_rank": local,
                      "max_ms": ms, "value": value}), flush=True)
    dist.destroy_process_group()


if __name__ == "__main__":
    main()
