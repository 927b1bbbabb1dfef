"""Data-parallel scaling on CPU ranks (gloo, world size 2): each rank holds a
shard of the tokens; the MAX all-reduce of the amaxes makes every rank derive
the same scale as one process that sees the whole batch.  A rank that never
joins makes the others' all-reduce fail with an error instead of hanging."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, shards, out_q, mode):
    import datetime

    import oracle as o
    from fp8_mixed_precision_amax_gb300.api import Meta, allreduce_amax
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world,
                            timeout=datetime.timedelta(seconds=10))
    try:
        if mode == "absent" and rank == 1:
            return                                  # never contributes its amax
        meta = Meta(8, device="cpu")
        x, dy = shards[rank]
        meta.amax[0] = float(o.amax(x))
        meta.amax[3] = float(o.amax(dy))
        try:
            allreduce_amax(meta)
        except Exception as e:                      # the error the test expects
            out_q.put((rank, "error", type(e).__name__))
            return
        st = o.State.initial(8)
        st.amax[:] = meta.amax.numpy()
        o.layer_update(st, o.Recipe(margin=0, history_len=8, hybrid=True))
        out_q.put((rank, "ok", st.scale.copy()))
    finally:
        if not (mode == "absent" and rank == 0):
            dist.destroy_process_group()


def _shards(seed=0):
    g = torch.Generator().manual_seed(seed)
    X = (torch.randn(64, 32, generator=g) * torch.linspace(0.1, 5, 64)[:, None]).to(torch.bfloat16)
    dY = (torch.randn(64, 16, generator=g) * 1e-3).to(torch.bfloat16)
    bits = lambda t: t.contiguous().view(torch.int16).numpy().view(np.uint16)
    return [(bits(X[:32]), bits(dY[:32])), (bits(X[32:]), bits(dY[32:]))], bits(X), bits(dY)


def test_amax_max_allreduce_gives_identical_scales():
    import oracle as o
    shards, X, dY = _shards()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, shards, q, "normal")) for r in (0, 1)]
    for p in procs:
        p.start()
    res = dict((r, (s, v)) for r, s, v in (q.get(timeout=60) for _ in procs))
    for p in procs:
        p.join(timeout=60)
    st = o.State.initial(8)
    st.amax[0], st.amax[3] = o.amax(X), o.amax(dY)
    o.layer_update(st, o.Recipe(margin=0, history_len=8, hybrid=True))
    for r in (0, 1):
        assert res[r][0] == "ok"
        assert np.array_equal(res[r][1].view(np.uint32), st.scale.view(np.uint32))


def test_rank_that_never_joins_fails_the_collective():
    shards, _, _ = _shards(1)
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, shards, q, "absent")) for r in (0, 1)]
    for p in procs:
        p.start()
    r, status, what = q.get(timeout=90)
    for p in procs:
        p.join(timeout=60)
        if p.is_alive():
            p.kill()
    assert r == 0 and status == "error"


def _fp8_worker(rank, world, port, grads, out_q):
    import datetime

    import oracle as o
    from fp8_mixed_precision_amax_gb300.api import fp8_exchange_sum, fp8_shard_len
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world,
                            timeout=datetime.timedelta(seconds=10))
    try:
        # the exchange of the FP8 all-reduce: MIN of the ranks' own scales,
        # then the library's reduce-scatter + all-gather of the FP8 codes,
        # with the oracle's sum on each rank's shard (CPU tensors)
        s = torch.tensor([float(o.local_scale(grads[rank], o.E5M2, 0))])
        dist.all_reduce(s, op=dist.ReduceOp.MIN)
        sg = np.float32(s.item())
        n = grads[rank].size
        shard = fp8_shard_len(n, world)
        q = np.zeros(world * shard, np.uint8)
        q[:n] = o.quantize(grads[rank].reshape(1, -1), sg, o.E5M2, transpose=False)[0][0]
        seen = []

        def reduce_shard(parts):
            seen.append(parts.shape)
            bits = o.dequant_sum(parts.numpy(), o.E5M2, sg)
            return torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16)

        full = fp8_exchange_sum(torch.from_numpy(q), shard, reduce_shard)
        out = full.view(torch.int16).numpy().view(np.uint16)[:n]
        out_q.put((rank, sg, out, seen))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world,n", [(3, 4096), (2, 4096 + 16), (3, 1000 * 16)])
def test_fp8_allreduce_exchange_shares_the_minimum_scale(world, n):
    """The exchange step of the FP8 all-reduce (wiki note, 'per-tensor scaling
    is the key'): gloo ranks agree on s'_g = min(s'_i), each sums only its
    own shard of every rank's codes (padded to a multiple of 16), and the
    all-gather of the shards equals the single-process reference sum."""
    import oracle as o
    from fp8_mixed_precision_amax_gb300.api import fp8_shard_len
    rng = np.random.default_rng(3 + world)
    grads = [torch.from_numpy((rng.standard_normal(n) * m).astype(np.float32))
             .to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
             for m in (1e-3, 3e-2, 5e-4)[:world]]
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_fp8_worker, args=(r, world, port, grads, q))
             for r in range(world)]
    for p in procs:
        p.start()
    res = [q.get(timeout=60) for _ in procs]
    for p in procs:
        p.join(timeout=60)
    ref, sg, _ = o.fp8_allreduce(grads, o.E5M2)
    shard = fp8_shard_len(n, world)
    assert shard % 16 == 0 and world * shard >= n > (world - 1) * shard - 16 * world
    for rank, s, out, seen in res:
        assert s == sg and np.array_equal(out, ref), rank
        assert seen == [(world, shard)], rank
