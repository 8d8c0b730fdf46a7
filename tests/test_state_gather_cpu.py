"""gather_states over two gloo ranks on CPU: one state per rank, stacked in
rank order, part-major, as Context.merge_states takes them."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _worker(rank, world, port, q):
    import torch
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import paged_gqa_decode_05_gb300 as pda
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    S, Hq, D = 3, 4, 8
    m = torch.full((S, Hq), float(rank))
    l = torch.full((S, Hq), 10.0 + rank)
    o = torch.arange(S * Hq * D, dtype=torch.float32).reshape(S, Hq, D) + 100 * rank
    gm, gl, go = pda.gather_states(m, l, o)
    q.put((rank, tuple(gm.shape), tuple(go.shape), gm[:, 0, 0].tolist(), gl[:, 1, 2].tolist(),
           go[:, 2, 3, 7].tolist()))
    dist.destroy_process_group()


def test_gather_states_two_gloo_ranks():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 29700 + os.getpid() % 1000
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = dict((r[0], r[1:]) for r in (q.get(timeout=5) for _ in range(2)))
    base = 2 * 4 * 8 + 3 * 8 + 7  # o[2, 3, 7] before the rank offset
    for rank in (0, 1):
        shape_m, shape_o, m0, l12, o237 = got[rank]
        assert shape_m == (2, 3, 4) and shape_o == (2, 3, 4, 8)
        assert m0 == [0.0, 1.0] and l12 == [10.0, 11.0]
        assert o237 == [float(base), float(base + 100)]
