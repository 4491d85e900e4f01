"""World-size-2 tests of the multi-process (replica) host logic of bench.py,
on CPU with the gloo backend.

The MoE block shards by independent batches: under torchrun every rank runs
the whole block on its own token draw through replicated weights, with no
data-path collective; the only cross-rank traffic is the barrier around the
timed region and the max over ranks of the elapsed time.  These tests run two
gloo ranks through exactly the helpers bench.py uses (rank_workload,
max_over_ranks, whole_job_tokens_per_s), with the oracle standing in for the
per-rank forward, and check that
  * each rank draws a different batch of the same shapes,
  * a rank's result depends only on its own batch (equal to a single-process
    oracle run of that rank's workload: nothing crosses between replicas),
  * every rank sees the slowest rank's time, and the whole-job value is all
    ranks' tokens over that time,
  * the reference arm runs on rank 0 only.
"""
import os
import socket
import types

import pytest
import torch
import torch.multiprocessing as mp

import bench
import oracle
import synth

WS = 2
STEPS = 3


def _tiny():
    return synth.custom("gloo_tiny", bs=6, hidden=128, num_experts=4, topk=2, inter=64, has_shared=True, seed=61)


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _digest(out):
    return [out["output"].view(torch.int16).to(torch.int64).sum().item(),
            out["share_output"].view(torch.int16).to(torch.int64).sum().item(),
            out["expert_token_nums"].tolist()]


def _worker(rank, port, q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    torch.distributed.init_process_group("gloo", rank=rank, world_size=WS)
    try:
        wl_r = bench.rank_workload(_tiny(), rank)
        inp = synth.make_inputs(wl_r)
        out = oracle.forward(inp, threads=1)
        elapsed = 0.25 * (rank + 1)          # rank 1 is the slow replica
        torch.distributed.barrier()
        slowest = bench.max_over_ranks(elapsed)
        value = bench.whole_job_tokens_per_s(wl_r.bs, WS, STEPS, slowest)
        q.put((rank, inp.expert_ids.tolist(), _digest(out), slowest, value))
    finally:
        torch.distributed.destroy_process_group()


@pytest.fixture(scope="module")
def gloo_results():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, port, q)) for r in range(WS)]
    for p in procs:
        p.start()
    res = {}
    for _ in range(WS):
        rank, ids, dig, slowest, value = q.get(timeout=300)
        res[rank] = (ids, dig, slowest, value)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    return res


def test_ranks_draw_distinct_batches_of_the_same_shape(gloo_results):
    ids0, ids1 = gloo_results[0][0], gloo_results[1][0]
    assert len(ids0) == len(ids1) == _tiny().bs
    assert ids0 != ids1


def test_replicas_are_independent(gloo_results):
    # each rank's result equals a single-process run of its own workload
    for rank in range(WS):
        inp = synth.make_inputs(bench.rank_workload(_tiny(), rank))
        assert gloo_results[rank][1] == _digest(oracle.forward(inp, threads=1))


def test_every_rank_sees_the_slowest_time_and_the_whole_job_value(gloo_results):
    for rank in range(WS):
        slowest, value = gloo_results[rank][2], gloo_results[rank][3]
        assert slowest == pytest.approx(0.5)
        assert value == pytest.approx(_tiny().bs * WS * STEPS / 0.5)


def test_max_over_ranks_is_the_identity_without_a_process_group():
    assert not torch.distributed.is_initialized()
    assert bench.max_over_ranks(1.25) == 1.25


def test_reference_arm_runs_on_rank_zero_only():
    args = types.SimpleNamespace(steps=1, warmup=0)
    assert bench.run_reference(args, _tiny(), 2, 1) is None
