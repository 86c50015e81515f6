"""The multi-rank host logic on CPU: world_size 2 over gloo.  Ranks own
disjoint sequences, each rank's results equal a single-process run on the same
sequences, and the timing reduction is a max over ranks."""
import os
import socket

import numpy as np
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import torch.distributed as dist
    from compressed_sparse_attention_decode_gb300 import dist as cdist
    import oracle
    from synth.workloads import WORKLOADS, scaled
    dist.init_process_group("gloo", rank=rank, world_size=world)
    r, w, _ = cdist.env()
    seqs = cdist.shard(2, r, w)
    wl = scaled(WORKLOADS[0], B=2 * w, T=1024, layers=("full", "reuse"))
    idx = {b: oracle.run_sequence(wl, b, want_out=False)["idx"][1].tolist() for b in seqs}
    t = cdist.reduce_max(1.5 + r)            # a stand-in elapsed time per rank
    cdist.barrier()
    out.put((r, seqs, idx, t))
    dist.destroy_process_group()


def test_two_ranks_shard_the_batch_with_no_exchange():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    ps = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in ps:
        p.start()
    res = sorted(q.get(timeout=120) for _ in ps)
    for p in ps:
        p.join(timeout=60)
        assert p.exitcode == 0
    (r0, s0, i0, t0), (r1, s1, i1, t1) = res
    assert s0 == [0, 1] and s1 == [2, 3]                 # disjoint, covering
    assert t0 == t1 == 2.5                                # max over ranks
    import oracle
    from synth.workloads import WORKLOADS, scaled
    wl = scaled(WORKLOADS[0], B=4, T=1024, layers=("full", "reuse"))
    for b, got in list(i0.items()) + list(i1.items()):
        want = oracle.run_sequence(wl, b, want_out=False)["idx"][1].tolist()
        assert got == want
