"""The N > 1 path on CPU: world-size-2 gloo ranks.

The method's units (sequence, kv head) are independent, so the multi-GPU run
is N replicas with no collective on the data path; what crosses ranks is the
benchmark's timing: a barrier and the max over ranks.  Each rank here plans its
own replica with the C ABI (host code) and aggregates a rank-dependent step
time through bench.aggregate_over_ranks."""
import os
import socket

import pytest


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, queue):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        import synth
        import paged_kv_variable_gb300 as pkv
        case = synth.config2(draw_values=False)
        spec = case.spec
        prob = pkv.make_problem(batch=spec.batch, num_heads_q=spec.hq, num_heads_kv=spec.hkv, head_dim=spec.d,
                                page_size=spec.page_size, cache_capacity=spec.capacity, num_pages=case.num_pages,
                                cache_dtype="bf16", causal=True, softmax_scale=spec.softmax_scale)
        st = pkv.plan(prob, spec.q_lens, spec.cache_lens, spec.new_lens, num_sms=152).stats()
        units = bench.step_work(spec)["bytes"]
        t_ms = 1.0 + rank  # rank 1 is the slow one
        dist.barrier()
        t, value = bench.aggregate_over_ranks(t_ms, units, world)
        queue.put((rank, st["num_items"], t, value, units))
    finally:
        dist.destroy_process_group()


def test_two_replicas_aggregate_with_gloo():
    pytest.importorskip("torch")
    import multiprocessing as mp
    from paged_kv_variable_gb300 import build
    build.build()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=5) for _ in range(2))
    (r0, n0, t0, v0, u0), (r1, n1, t1, v1, u1) = res
    assert n0 == n1 > 0                       # identical replicas plan identically
    assert t0 == t1 == 2.0                    # max over ranks
    assert v0 == v1 == pytest.approx(2 * u0 / 2.0e-3)
