"""Head sharding of a layer (one key head group per rank, no exchange on the data path).

  * the partition: every key head and value head lands on exactly one rank, each rank's packed
    channels are its q, k and v heads in order, and slicing then gathering is the identity;
  * world size 2 over gloo on the CPU: each rank runs the fp64 oracle on its own shard of one
    layer, the outputs are gathered over the process group, and the result equals the oracle
    on the whole layer exactly (every stage is head-local);
  * on the GPU: both shards through gdn_layer equal the unsharded gdn_layer bit for bit.
"""
import json
import os
import socket
import sys

import numpy as np
import pytest

import oracle
from gated_deltanet_linear_pre_gb300 import inputs as gin
from gated_deltanet_linear_pre_gb300 import shard

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
torch = pytest.importorskip("torch")

HK, HV, DK, DV = 4, 12, 16, 8  # small heads for the oracle; 3 value heads per key head as in the pages' layer


def _inputs():
    return gin.make_layer(61, [37, 0, 70], hist_nonzero=True, S0_std=0.02, dims=(HK, HV, DK, DV))


def _as_dict(inp):
    return {k: getattr(inp, k) for k in ("qkv", "conv_w", "hist", "a", "b", "A_log", "dt_bias", "z", "gamma", "S0",
                                          "cu_seqlens")}


def _layer_from(d, dims):
    return gin.LayerInputs(qkv=d["qkv"], conv_w=d["conv_w"], hist=d["hist"], a=d["a"], b=d["b"], A_log=d["A_log"],
                           dt_bias=d["dt_bias"], z=d["z"], gamma=d["gamma"], S0=d["S0"], cu_seqlens=d["cu_seqlens"],
                           dims=dims)


def test_partition_covers_every_head_once():
    for world in (1, 2, 4):
        shards = [shard.head_shard(16, 48, world, r) for r in range(world)]
        assert [s.j0 for s in shards] == list(range(0, 16, 16 // world))
        assert sum(s.hk for s in shards) == 16 and sum(s.hv for s in shards) == 48
        for s in shards:  # value head h reads key head h // 3: a shard's value heads read its key heads only
            assert all(s.j0 <= h // 3 < s.j1 for h in range(s.h0, s.h1))
        ch = np.concatenate([shard.channel_index(s, 16, 48) for s in shards])
        assert np.array_equal(np.sort(ch), np.arange(2 * 16 * 128 + 48 * 128))
    s = shard.head_shard(16, 48, 4, 1)  # q heads 4-7, k heads 20-23, v heads 12-23 of the packed order
    idx = shard.channel_index(s, 16, 48)
    assert idx[0] == 4 * 128 and idx[4 * 128] == (16 + 4) * 128 and idx[8 * 128] == (32 + 12) * 128
    with pytest.raises(ValueError):
        shard.head_shard(16, 48, 3, 0)


def test_slice_then_gather_is_the_identity():
    inp = _as_dict(_inputs())
    parts = []
    for r in range(2):
        sh = shard.head_shard(HK, HV, 2, r)
        x = shard.shard_layer_inputs(inp, sh, HK, HV, DK, DV)
        parts.append({"y": x["z"], "hist_out": x["hist"], "S_out": x["S0"]})
    full = shard.gather_outputs(parts, HK, HV, DK, DV)
    assert np.array_equal(full["y"], inp["z"])
    assert np.array_equal(full["hist_out"], inp["hist"])
    assert np.array_equal(full["S_out"], inp["S0"])


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_body(rank, world, port, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import oracle as orc
    from gated_deltanet_linear_pre_gb300 import shard as shd
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        inp = _as_dict(_inputs())
        sh = shd.head_shard(HK, HV, world, rank)
        mine = shd.shard_layer_inputs(inp, sh, HK, HV, DK, DV)
        ref = orc.layer(_layer_from(mine, (sh.hk, sh.hv, DK, DV)), hk=sh.hk, hv=sh.hv, dk=DK, dv=DV)
        out = {k: torch.from_numpy(np.ascontiguousarray(ref[k])) for k in ("y", "hist_out", "S_out")}
        gathered = {}
        for k, v in out.items():  # the only exchange: assembling full rows for the check
            bufs = [torch.empty_like(v) for _ in range(world)]
            dist.all_gather(bufs, v)
            gathered[k] = bufs
        parts = [{k: gathered[k][r].numpy() for k in gathered} for r in range(world)]
        full = shd.gather_outputs(parts, HK, HV, DK, DV)
        whole = orc.layer(_layer_from(inp, (HK, HV, DK, DV)), hk=HK, hv=HV, dk=DK, dv=DV)
        same = {k: bool(np.array_equal(full[k], whole[k])) for k in ("y", "hist_out", "S_out")}
        with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
            json.dump(same, f)
    finally:
        dist.destroy_process_group()


def test_two_ranks_over_gloo_reassemble_the_whole_layer(tmp_path):
    import torch.multiprocessing as mp
    mp.spawn(_rank_body, args=(2, _free_port(), str(tmp_path)), nprocs=2, join=True)
    for r in range(2):
        assert json.load(open(tmp_path / f"rank{r}.json")) == {"y": True, "hist_out": True, "S_out": True}


@pytest.mark.gpu
def test_shards_through_gdn_layer_equal_the_whole_layer():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import gpu_util as u
    import gated_deltanet_linear_pre_gb300 as gdn
    from gated_deltanet_linear_pre_gb300 import build
    build.build()
    inp = gin.make_layer(62, [300, 1, 130], hist_nonzero=True, S0_std=0.02)
    whole = u.run_layer(inp)
    parts = []
    for r in range(2):
        sh = shard.head_shard(16, 48, 2, r)
        x = shard.shard_layer_inputs(_as_dict(inp), sh, 16, 48)
        part = _layer_from(x, (sh.hk, sh.hv, 128, 128))
        parts.append(u.run_layer(part))
    full = shard.gather_outputs(parts, 16, 48)
    for k in ("y", "hist_out", "S_out"):
        assert np.array_equal(full[k], whole[k]), k
