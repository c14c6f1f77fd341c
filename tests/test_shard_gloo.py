"""The N > 1 path on CPU: sequences sharded over world-size-2 ``gloo`` ranks.

Each rank runs the oracle over its contiguous shard of a global batch (inputs
drawn by global sequence index, as the benchmark's ranks draw theirs), then
the ranks fold their figures with ``job_totals`` and gather their outputs.
Sharding must change nothing: the gathered outputs, codes and counters equal a
one-process run over the whole batch bit for bit, since no sequence reads
another's state.
"""

import json
import os
import socket
import subprocess
import sys
from datetime import timedelta

import numpy as np
import pytest

from kvq_inputs.gen import InputSpec
from oracle import kvq_oracle as O
from quantized_kv_cache_02_gb300.shard import Shard, job_totals, shard_range

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

# small grouped-rule workload: GQA g = 2, a prefill that flushes, then decode
# steps that cross a group boundary
CFG = dict(global_batch=5, n_kv_heads=2, n_q_heads=4, head_dim=16, residual_len=8, group=4, qmax=7,
           prefill=21, steps=6, seed=11)


def run_shard(seqs, cfg=CFG):
    """Oracle run of the sequences ``seqs``: per step, the attention outputs
    [len(seqs), Hq, d] (fp64), then the final codes and counters."""
    spec = InputSpec(seed=cfg["seed"], n_kv_heads=cfg["n_kv_heads"], n_q_heads=cfg["n_q_heads"],
                     head_dim=cfg["head_dim"], bf16=False)
    R, G, qmax = cfg["residual_len"], cfg["group"], cfg["qmax"]
    K0, V0 = spec.kv_block(0, seqs, 0, cfg["prefill"])
    state = O.append_and_partition(None, K0, V0, R, qmax, group=G)
    outs = []
    for s in range(cfg["steps"]):
        Kn, Vn = spec.kv_block(0, seqs, cfg["prefill"] + s, 1)
        state = O.append_and_partition(state, Kn, Vn, R, qmax, group=G)
        outs.append(O.decode_attention(state, spec.q_block(0, seqs, s)))
    codes = np.concatenate(state["key_q_segments"], axis=-2)
    return np.stack(outs), codes, (state["quantized_tokens"], state["total_tokens"])


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def rank_main(rank, world, port, out_dir):
    """One gloo rank (run as its own process by the test below)."""
    import torch.distributed as dist
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world,
                            timeout=timedelta(seconds=120))
    try:
        shard = shard_range(CFG["global_batch"], world, rank)
        outs, codes, ctr = run_shard(shard.seqs)
        # units processed and a per-rank "time" that differs by rank
        units, ms = job_totals(shard.count * CFG["steps"], 10.0 + rank, dist)
        gathered = [None] * world
        dist.all_gather_object(gathered, (shard.begin, shard.count, outs, codes, ctr))
        if rank == 0:
            np.save(os.path.join(out_dir, "outs.npy"), np.concatenate([g[2] for g in gathered], axis=1))
            np.save(os.path.join(out_dir, "codes.npy"), np.concatenate([g[3] for g in gathered], axis=0))
            with open(os.path.join(out_dir, "meta.json"), "w") as f:
                json.dump({"units": units, "ms": ms, "shards": [[g[0], g[1]] for g in gathered],
                           "counters": [list(g[4]) for g in gathered]}, f)
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_shard_range_partitions_the_batch():
    for batch in range(1, 41):
        for world in range(1, min(batch, 8) + 1):
            shards = [shard_range(batch, world, r) for r in range(world)]
            assert [s.begin for s in shards] == [sum(t.count for t in shards[:r]) for r in range(world)]
            assert sum(s.count for s in shards) == batch
            assert max(s.count for s in shards) - min(s.count for s in shards) <= 1
            assert all(s.count >= 1 for s in shards)
    assert shard_range(5, 2, 0) == Shard(0, 2, 0, 3)
    assert shard_range(5, 2, 1) == Shard(1, 2, 3, 2)
    for bad in [(4, 2, 2), (4, 0, 0), (4, 2, -1), (1, 2, 0)]:
        with pytest.raises(ValueError):
            shard_range(*bad)


def test_job_totals_one_process():
    assert job_totals(7, 3.5) == (7.0, 3.5)


def test_two_gloo_ranks_match_one_process(tmp_path):
    world, port = 2, _free_port()
    code = ("import sys; sys.path.insert(0, {root!r}); sys.path.insert(0, {tests!r}); "
            "import test_shard_gloo as t; t.rank_main({rank}, {world}, {port}, {out!r})")
    procs = [subprocess.Popen([sys.executable, "-c", code.format(root=ROOT, tests=os.path.join(ROOT, "tests"),
                                                                   rank=r, world=world, port=port, out=str(tmp_path))],
                              cwd=ROOT) for r in range(world)]
    try:
        rcs = [p.wait(timeout=300) for p in procs]
    finally:
        for p in procs:
            if p.poll() is None:
                p.kill()
    assert rcs == [0, 0]
    meta = json.loads((tmp_path / "meta.json").read_text())
    assert meta["shards"] == [[0, 3], [3, 2]]
    assert meta["units"] == CFG["global_batch"] * CFG["steps"]      # summed over ranks
    assert meta["ms"] == 11.0                                        # slowest rank
    outs, codes, ctr = run_shard(range(CFG["global_batch"]))
    assert all(tuple(c) == ctr for c in meta["counters"])
    np.testing.assert_array_equal(np.load(tmp_path / "codes.npy"), codes)
    np.testing.assert_array_equal(np.load(tmp_path / "outs.npy"), outs)


def test_reference_arm_runs_on_rank_zero_only(monkeypatch, capsys):
    import argparse

    import bench
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("RANK", "1")
    bench.run_reference(argparse.Namespace(steps=1, warmup=0))
    assert capsys.readouterr().out == ""
