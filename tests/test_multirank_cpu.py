"""World-size-2 gloo run of the multi-rank host logic on CPU: token sharding,
the shared mean denominator and the max over ranks.  Each rank evaluates its own
shard with the oracle; summing the per-rank losses and dW reproduces the
single-process result over the whole batch (what a data-parallel run relies on)."""
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
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        from lm_head_cross_vocab_gb300 import dist as D
        from lm_head_cross_vocab_gb300 import inputs as I
        from oracle import kd_oracle as O
        assert D.world_from_env() == (rank, world, rank)
        w = I.WORKLOADS[2].scaled(n_tokens=101, d_student=16, d_teacher=24, vocab=200)
        cpu = I.make_inputs(w, "cpu")
        a, b = D.shard_rows(w.n_tokens, rank, world)
        labels = cpu["labels"][a:b]
        n_valid = D.global_valid_count(labels, w.ignore_index)
        kw = dict(variant=w.variant, t_student=w.t_student, t_teacher=w.t_teacher,
                  w_student_ce=w.w_student_ce, w_teacher_ce=w.w_teacher_ce, w_kl=w.w_kl,
                  ignore_index=w.ignore_index, num_batch_labels=n_valid)
        z_s = O.project(cpu["h_s"][a:b], cpu["w_s"])
        z_t = O.project(cpu["h_t"][a:b], cpu["w_t"])
        loss = O.forward(z_s, z_t, labels.numpy(), **kw)["loss"]
        g, _ = O.grad_logits(z_s, z_t, labels.numpy(), **kw)
        _, d_w = O.hidden_grads(cpu["h_s"][a:b], cpu["w_s"], g)
        t = torch.tensor([loss], dtype=torch.float64)
        dist.all_reduce(t)
        dw = torch.from_numpy(d_w)
        dist.all_reduce(dw)
        mx = D.max_over_ranks(float(rank + 1))
        q.put((rank, float(t.item()), dw.numpy() if rank == 0 else None, mx, n_valid, b - a))
    finally:
        dist.destroy_process_group()


def test_two_rank_data_parallel_reduces_to_the_global_batch():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    from lm_head_cross_vocab_gb300 import inputs as I
    from oracle import kd_oracle as O
    w = I.WORKLOADS[2].scaled(n_tokens=101, d_student=16, d_teacher=24, vocab=200)
    cpu = I.make_inputs(w, "cpu")
    kw = dict(variant=w.variant, t_student=w.t_student, t_teacher=w.t_teacher,
              w_student_ce=w.w_student_ce, w_teacher_ce=w.w_teacher_ce, w_kl=w.w_kl,
              ignore_index=w.ignore_index)
    z_s, z_t = O.project(cpu["h_s"], cpu["w_s"]), O.project(cpu["h_t"], cpu["w_t"])
    lab = cpu["labels"].numpy()
    ref = O.forward(z_s, z_t, lab, **kw)
    g, _ = O.grad_logits(z_s, z_t, lab, **kw)
    _, d_w = O.hidden_grads(cpu["h_s"], cpu["w_s"], g)
    assert [r[5] for r in res] == [51, 50]          # contiguous shards cover the batch
    assert res[0][4] == res[1][4] == int((lab != w.ignore_index).sum())
    assert res[0][1] == pytest.approx(ref["loss"], rel=1e-12)
    np.testing.assert_allclose(res[0][2], d_w, rtol=1e-10, atol=1e-14)
    assert res[0][3] == res[1][3] == 2.0             # max over ranks


@pytest.mark.parametrize("n,world", [(10, 3), (4096, 8), (1, 2)])
def test_shard_rows_partition(n, world):
    from lm_head_cross_vocab_gb300.dist import shard_rows
    spans = [shard_rows(n, r, world) for r in range(world)]
    assert spans[0][0] == 0 and spans[-1][1] == n
    assert all(spans[i][1] == spans[i + 1][0] for i in range(world - 1))
    assert max(b - a for a, b in spans) - min(b - a for a, b in spans) <= 1
