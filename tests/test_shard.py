"""Head-sharded multi-GPU driver (exact_io_aware_17_gb300/shard.py): partition and reassembly, on the CPU.

The per-shard compute on a GPU is the library's fa_fwd / fa_bwd; here it is replaced by the fp64 oracle so
that the partition, the uneven shards, an empty shard and the gather run as real gloo ranks (world sizes 2
and 4) without a GPU.  The oracle works head by head, so the reassembled outputs must equal the unsharded
ones bit for bit."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import fa_inputs
import oracle
from exact_io_aware_17_gb300 import shard


def test_head_ranges_cover_every_head_once():
    for total in range(0, 20):
        for world in range(1, 9):
            r = shard.head_ranges(total, world)
            assert len(r) == world
            assert r[0][0] == 0 and r[-1][1] == total
            for (a0, a1), (b0, _) in zip(r, r[1:]):
                assert a1 == b0
            sizes = [b - a for a, b in r]
            assert min(sizes) >= 0 and max(sizes) - min(sizes) <= 1
            assert sizes == sorted(sizes, reverse=True)


def test_head_ranges_rejects_bad_arguments():
    with pytest.raises(ValueError):
        shard.head_ranges(4, 0)
    with pytest.raises(ValueError):
        shard.head_ranges(-1, 2)


def test_local_heads_are_views_of_the_right_heads():
    t = torch.arange(2 * 3 * 4 * 2, dtype=torch.float32).reshape(2, 3, 4, 2)
    flat = t.reshape(6, 4, 2)
    seen = []
    for rank in range(4):
        v = shard.local_heads(t, rank, 4)
        assert v.shape[0] == 1 and v.data_ptr() == flat[shard.head_ranges(6, 4)[rank][0]].data_ptr()
        seen.append(v[0])
    assert torch.equal(torch.cat(seen), flat)


def _oracle_fwd(q, k, v, scale):
    o, lse = oracle.forward(q.double().numpy(), k.double().numpy(), v.double().numpy(), scale)
    return torch.from_numpy(o), torch.from_numpy(lse)


def _oracle_bwd(q, k, v, o, do, lse, scale):
    g = oracle.backward(q.double().numpy(), k.double().numpy(), v.double().numpy(), do.double().numpy(), scale)
    return tuple(torch.from_numpy(x) for x in g)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, shape, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    B, H, N, d = shape
    inp = fa_inputs.make_inputs(B, H, N, d, "f32", seed=31, with_grad=True)
    q, k, v, do = (inp[n].double() for n in ("q", "k", "v", "do"))
    scale = d ** -0.5
    kw = dict(rank=rank, world=world, fwd=_oracle_fwd, lse_dtype=torch.float64)
    o_loc, lse_loc = shard.sharded_forward(q, k, v, scale, **kw)
    o, lse = shard.sharded_forward(q, k, v, scale, gather=True, **kw)
    grads = shard.sharded_backward(q, k, v, o, do, lse, scale, rank=rank, world=world, gather=True, bwd=_oracle_bwd)
    out[rank] = {"local_heads": int(o_loc.shape[1]), "o": o.numpy(), "lse": lse.numpy(),
                 "grads": [g.numpy() for g in grads]}
    dist.barrier()
    dist.destroy_process_group()


@pytest.mark.parametrize("world,shape", [(2, (2, 3, 17, 8)), (4, (1, 3, 9, 4)), (2, (1, 1, 5, 4))])
def test_sharded_outputs_reassemble_bitwise(world, shape):
    """Uneven shards (3 heads over 2 ranks), a rank with no head (3 heads over 4, 1 head over 2): every rank
    ends with the full outputs, equal bit for bit to the unsharded computation."""
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        out = m.dict()
        mp.start_processes(_worker, args=(world, _free_port(), shape, out), nprocs=world, join=True,
                           start_method="spawn")
        res = dict(out)
    B, H, N, d = shape
    sizes = [b - a for a, b in shard.head_ranges(B * H, world)]
    assert [res[r]["local_heads"] for r in range(world)] == sizes
    inp = fa_inputs.make_inputs(B, H, N, d, "f32", seed=31, with_grad=True)
    q, k, v, do = (inp[n].double().numpy() for n in ("q", "k", "v", "do"))
    ro, rl = oracle.forward(q, k, v, d ** -0.5)
    rg = oracle.backward(q, k, v, do, d ** -0.5)
    for r in range(world):
        assert np.array_equal(res[r]["o"], ro) and np.array_equal(res[r]["lse"], rl)
        for g, ref in zip(res[r]["grads"], rg):
            assert np.array_equal(g, ref)


@pytest.mark.gpu
@pytest.mark.parametrize("d", [64, 128])
def test_sharding_onto_one_gpu_reassembles_the_unsharded_call(d):
    """The library on one GPU, its heads split three ways (uneven: 10 heads as 4 + 3 + 3) and each shard run
    as its own call: the forward and dK, dV are bitwise equal to one unsharded call, dQ within the rounding of
    its reduce order."""
    from parity_util import need_gpu
    fa = need_gpu()
    B, H, N, world = 2, 5, 1000, 3
    inp = fa_inputs.make_inputs(B, H, N, d, "bf16", seed=4100 + d, with_grad=True)
    q, k, v, do = (inp[n].cuda() for n in ("q", "k", "v", "do"))
    scale = d ** -0.5
    o, lse = fa.fa_fwd(q, k, v, scale)
    dq, dk, dv = fa.fa_bwd(q, k, v, o, do, lse, scale)
    parts = [shard.sharded_forward(q, k, v, scale, rank=r, world=world) for r in range(world)]
    so = torch.cat([p[0][0] for p in parts]).reshape(B, H, N, d)
    sl = torch.cat([p[1][0] for p in parts]).reshape(B, H, N)
    grads = [shard.sharded_backward(q, k, v, o, do, lse, scale, rank=r, world=world) for r in range(world)]
    sdq, sdk, sdv = (torch.cat([g[i][0] for g in grads]).reshape(B, H, N, d) for i in range(3))
    torch.cuda.synchronize()
    fa.fa_check_status()
    assert [p[0].shape[1] for p in parts] == [4, 3, 3]
    assert torch.equal(so, o) and torch.equal(sl, lse)
    assert torch.equal(sdk, dk) and torch.equal(sdv, dv)
    assert (sdq.float() - dq.float()).abs().max().item() <= 1e-2 * dq.float().abs().max().item()
