"""The N > 1 path on the CPU: two gloo ranks.

Every token's output depends only on its own ids, hidden and mask, so the
layer shards by tokens with replicated weights and no collective in the
data path.  Here two ranks each run the oracle on their shard of one batch
and all-gather the results: the concatenation must equal the single-process
result bit for bit.  The benchmark's max-over-ranks reduction and the
reference arm's rank-0-only output are checked on the same process group."""
import os
import socket
import subprocess
import sys

import numpy as np
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _inputs():
    import workloads as W
    wl = W.TINY.with_T(37)
    table = W.bits(W.make_table(wl))
    wts = W.make_weights(wl)
    st = W.make_step_inputs(wl)
    return wl, dict(table=table, wkv=W.bits(wts["wkv"]), q=W.bits(wts["q_weight"]),
                    k=W.bits(wts["k_weight"]), hidden=W.bits(st["hidden"]),
                    ids=st["hash_ids"].numpy(), mask=W.bits(st["token_mask"]))


def _oracle(wl, d, lo, hi):
    import oracle
    import workloads as W
    return oracle.forward(d["table"], W.row_offsets(wl.rows), np.asarray(wl.rows, np.int64),
                          np.ascontiguousarray(d["ids"][lo:hi]), wl.head_dim, d["wkv"],
                          d["hidden"][lo:hi], d["q"], d["k"], d["mask"][lo:hi], eps=wl.eps,
                          clamp=wl.clamp)


def _rank(rank, world, port, q):
    sys.path.insert(0, ROOT)
    import workloads as W
    from bench import reduce_max
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank,
                            world_size=world)
    try:
        wl, d = _inputs()
        lo, hi = W.shard_tokens(wl.T, rank, world)
        mine = _oracle(wl, d, lo, hi)["out_bf16"]
        parts = [None] * world
        dist.all_gather_object(parts, (lo, hi, mine))
        slowest = reduce_max(1.5 * (rank + 1), world, "cpu")
        if rank == 0:
            q.put((parts, slowest))
    finally:
        dist.destroy_process_group()


def test_token_shards_cover_the_batch():
    import workloads as W
    for T in (0, 1, 7, 64, 8191):
        for world in (1, 2, 3, 8):
            r = [W.shard_tokens(T, i, world) for i in range(world)]
            assert r[0][0] == 0 and r[-1][1] == T
            assert all(a[1] == b[0] for a, b in zip(r, r[1:]))
            assert max(h - l for l, h in r) - min(h - l for l, h in r) <= 1


def test_two_gloo_ranks_match_one_process():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    parts, slowest = q.get(timeout=120)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    wl, d = _inputs()
    full = _oracle(wl, d, 0, wl.T)["out_bf16"]
    parts = sorted(parts, key=lambda x: x[0])
    assert parts[0][0] == 0 and parts[-1][1] == wl.T
    assert np.array_equal(np.concatenate([p[2] for p in parts]), full)
    assert slowest == 3.0  # max over ranks of 1.5 * (rank + 1)


def test_reference_arm_prints_on_rank_zero_only():
    env = dict(os.environ, RANK="1", LOCAL_RANK="1", WORLD_SIZE="2",
               MASTER_ADDR="127.0.0.1", MASTER_PORT=str(_free_port()))
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "1"], env=env, capture_output=True,
                       text=True, timeout=120)
    assert r.returncode == 0 and r.stdout.strip() == ""
