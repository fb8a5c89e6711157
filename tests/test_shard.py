"""The data-parallel split of the forward: every rank takes a contiguous
range of the flattened (batch, head) problems and computes it by pointer
offset, with no exchange.  The partition is host logic (checked here on
CPU, also across two gloo ranks); on the GPU each rank's outputs must equal
the matching rows of the whole call bit for bit, because a problem's result
does not depend on which other problems share its launch."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import exact_attention_39_gb300 as fa
from exact_attention_39_gb300 import workloads as W


def _check_tiling(bh, world, ranges):
    assert ranges[0][0] == 0 and ranges[-1][1] == bh
    for (a0, a1), (b0, b1) in zip(ranges, ranges[1:]):
        assert a1 == b0
    sizes = [h1 - h0 for h0, h1 in ranges]
    assert min(sizes) >= 0 and max(sizes) - min(sizes) <= 1
    assert sum(sizes) == bh


@pytest.mark.parametrize("world", [1, 2, 3, 4, 7, 8, 64])
def test_head_range_tiles_the_problems(world):
    for bh in list(range(0, 40)) + [256, 257, 1023]:
        _check_tiling(bh, world, [fa.head_range(bh, world, r) for r in range(world)])


def test_head_range_rejects_bad_arguments():
    for args in ((-1, 2, 0), (4, 0, 0), (4, 2, 2), (4, 2, -1)):
        with pytest.raises(ValueError):
            fa.head_range(*args)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        for bh in (1, 2, 3, 256, 257):
            mine = torch.tensor(fa.head_range(bh, world, rank), dtype=torch.int64)
            every = [torch.zeros(2, dtype=torch.int64) for _ in range(world)]
            dist.all_gather(every, mine)
            q.put((rank, bh, [tuple(t.tolist()) for t in every]))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_cover_every_problem_once():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    got = [q.get(timeout=120) for _ in range(2 * 5)]
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    for rank, bh, ranges in got:
        _check_tiling(bh, world, ranges)
        assert ranges[rank] == fa.head_range(bh, world, rank)


def test_shard_needs_contiguous_inputs():
    q = torch.zeros(1, 2, 64, 128).transpose(2, 3)
    with pytest.raises(ValueError):
        fa.fwd_shard(q, q, q, 2, 0)


@pytest.mark.gpu
@pytest.mark.parametrize("B,H,Nq,Nk,d,dtype,causal", [
    (2, 5, 300, 300, 64, "bf16", True),
    (3, 3, 200, 333, 128, "fp16", False),
    (1, 6, 1024, 1024, 64, "bf16", False),
])
def test_shards_equal_the_whole_call(B, H, Nq, Nk, d, dtype, causal):
    w = W.Workload("shard", B, H, Nq, d, dtype, causal, seed=17, Nk=Nk)
    q, k, v = (t.cuda() for t in W.make_inputs(w))
    o, lse = fa.fwd(q, k, v, causal=causal, scale=w.scale)
    o_flat, l_flat = o.reshape(B * H, Nq, d), lse.reshape(B * H, Nq)
    for world in (1, 2, 3, 4, B * H + 1):
        for rank in range(world):
            o_r, l_r, (h0, h1) = fa.fwd_shard(q, k, v, world, rank, causal=causal,
                                              scale=w.scale)
            assert o_r.shape == (h1 - h0, Nq, d) and l_r.shape == (h1 - h0, Nq)
            assert torch.equal(o_r, o_flat[h0:h1]) and torch.equal(l_r, l_flat[h0:h1])
    torch.cuda.synchronize()
    assert fa.last_device_error() == 0


@pytest.mark.gpu
def test_shards_into_preallocated_outputs():
    # the multi-GPU benchmark's call: each rank writes its problems into
    # buffers it allocated once (weak split: the global batch is world x B)
    w = W.Workload("shard_out", 4, 4, 2048, 64, "bf16", False, seed=23)
    q, k, v = (t.cuda() for t in W.make_inputs(w))
    o, lse = fa.fwd(q, k, v, scale=w.scale)
    o_flat, l_flat = o.reshape(16, 2048, 64), lse.reshape(16, 2048)
    world = 2
    for rank in range(world):
        h0, h1 = fa.head_range(16, world, rank)
        out = torch.empty(h1 - h0, 2048, 64, dtype=q.dtype, device="cuda")
        lse_r = torch.empty(h1 - h0, 2048, dtype=torch.float32, device="cuda")
        o_r, l_r, rng = fa.fwd_shard(q, k, v, world, rank, scale=w.scale, out=out, lse=lse_r)
        assert rng == (h0, h1) and o_r.data_ptr() == out.data_ptr()
        assert torch.equal(out, o_flat[h0:h1]) and torch.equal(lse_r, l_flat[h0:h1])
    with pytest.raises(ValueError):
        fa.fwd_shard(q, k, v, world, 0, out=torch.empty(1, 2048, 64, dtype=q.dtype, device="cuda"))
    torch.cuda.synchronize()
    assert fa.last_device_error() == 0
