"""Run by tests/test_ranks_gloo.py through the N-rank launcher of bench.py
(ranks.spawn_world): joins a gloo process group from the launcher's environment
and writes its rank, world size, local rank and the result of one all-reduce."""
import json
import os
import sys


def main(outdir):
    import torch
    import torch.distributed as dist
    dist.init_process_group("gloo")
    try:
        t = torch.tensor([float(dist.get_rank() + 1)])
        dist.all_reduce(t)
        rec = {"rank": dist.get_rank(), "world": dist.get_world_size(),
               "local": int(os.environ["LOCAL_RANK"]), "sum": float(t.item())}
        with open(os.path.join(outdir, f"rank{rec['rank']}.json"), "w") as f:
            json.dump(rec, f)
    finally:
        dist.destroy_process_group()


if __name__ == "__main__":
    main(sys.argv[1])
