"""Multi-process host logic of the sharded path, on CPU with the gloo backend (world size 2):
max-over-ranks timing, barrier, per-rank seeds and the head partition. No GPU involved."""
import os
import socket

import pytest

from exact_io_aware_fa_gb300 import dist as fadist


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out_dir):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank,
                            world_size=world)
    try:
        r, w, lr = fadist.env_rank_world()
        assert (r, w, lr) == (rank, world, rank)
        fadist.barrier()
        # Each rank "measured" a different time; everyone must see the slowest.
        t_max = fadist.max_over_ranks(1.5 + rank)
        seed = fadist.rank_seed(1002, rank)
        lo, hi = fadist.partition_heads(64, rank, world)
        value = fadist.weak_scaling_value(1e12, 10, world, t_max)
        fadist.barrier()
        with open(os.path.join(out_dir, f"rank{rank}.txt"), "w") as f:
            f.write(f"{t_max} {seed} {lo} {hi} {value}\n")
    finally:
        dist.destroy_process_group()


def test_two_rank_gloo(tmp_path):
    import torch.multiprocessing as mp
    world = 2
    port = _free_port()
    mp.start_processes(_worker, args=(world, port, str(tmp_path)), nprocs=world, join=True,
                       start_method="spawn")
    rows = [open(tmp_path / f"rank{r}.txt").read().split() for r in range(world)]
    t = [float(x[0]) for x in rows]
    assert t == [2.5, 2.5]
    seeds = [int(x[1]) for x in rows]
    assert seeds == [1002, 2002]
    spans = [(int(x[2]), int(x[3])) for x in rows]
    assert spans == [(0, 32), (32, 64)]
    # value = 2 ranks * 10 steps * 1 TFLOP / 2.5 s = 8 TFLOP/s
    assert all(abs(float(x[4]) - 8.0) < 1e-12 for x in rows)


@pytest.mark.parametrize("bh,world", [(64, 1), (64, 3), (7, 4), (3, 8), (0, 2)])
def test_partition_covers_every_head_once(bh, world):
    owned = []
    sizes = []
    for r in range(world):
        lo, hi = fadist.partition_heads(bh, r, world)
        assert 0 <= lo <= hi <= bh
        owned.extend(range(lo, hi))
        sizes.append(hi - lo)
    assert owned == list(range(bh))
    assert max(sizes) - min(sizes) <= 1


def test_single_process_identity():
    assert fadist.max_over_ranks(3.25) == 3.25
    assert fadist.rank_seed(7, 0) == 7
    with pytest.raises(ValueError):
        fadist.partition_heads(4, 2, 2)
    with pytest.raises(ValueError):
        fadist.weak_scaling_value(1.0, 1, 1, 0.0)
