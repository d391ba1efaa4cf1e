"""bench.py under torchrun: independent replicas per rank (gloo, CPU). Every rank serves its own
sequences (weak scaling) with no exchange on the data path; the job time is the max over ranks.
The split is checked here with the oracle: the ranks own disjoint sequence ids that cover the
job, and each rank's results equal those of one process decoding the whole job."""
import os
import socket

import numpy as np
import pytest
import torch.multiprocessing as mp

B_PER_RANK = 2
LENS = np.array([300, 141], np.int32)  # one sequence with packed pages, one nearly all-protected


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _oracle_decode(w, inp):
    import oracle
    cfg = oracle.make_config(**w.config_kwargs())
    B = inp.seq_lens.shape[0]
    pool = np.zeros((inp.n_pages, oracle.page_bytes(cfg)), np.uint8)
    sink = np.zeros((B, cfg.n_sink, 576), np.uint16)
    ring = np.zeros((B, cfg.n_recent, 576), np.uint16)
    assert oracle.write(cfg, inp.c, inp.kr, inp.cu, np.zeros(B, np.int32), int(inp.seq_lens.max()), inp.page_table,
                        pool, sink, ring) == 0
    o, l, fl = oracle.decode(cfg, inp.q_lat, inp.q_rope, inp.page_table, inp.seq_lens, pool, sink, ring,
                             w.softmax_scale)
    assert fl == 0
    return o, l


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import torch.distributed as dist

    import bench
    import workloads
    dist.init_process_group("gloo", rank=rank, world_size=world)
    assert bench.dist_env() == (world, rank, rank)
    w = bench.replica_workload(workloads.WORKLOADS["tiny_c4r4_b1_h16_t1k"], rank)
    inp = workloads.make_inputs(w, seq_lens=LENS)
    o, l = _oracle_decode(w, inp)
    t = bench.max_over_ranks(10.0 + 5.0 * rank)
    q.put((rank, t, list(bench.replica_sequences(B_PER_RANK, rank, world)), o, l))
    dist.barrier()
    dist.destroy_process_group()


@pytest.mark.parametrize("world", [2])
def test_replicas_split_and_max_over_ranks(world):
    import bench
    import workloads
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    got = {}
    for _ in range(world):
        rank, t, ids, o, l = q.get(timeout=300)
        got[rank] = (t, ids, o, l)
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    # the job time is the slowest rank's, on every rank
    assert all(v[0] == 10.0 + 5.0 * (world - 1) for v in got.values())
    # ownership: disjoint and complete
    owned = [i for r in range(world) for i in got[r][1]]
    assert sorted(owned) == list(range(world * B_PER_RANK)) and len(set(owned)) == len(owned)
    # one process decoding the whole job as one batch: global sequence g is local row g % B of
    # the workload of rank g // B (rows, queries and page tables of the ranks concatenated)
    base = workloads.WORKLOADS["tiny_c4r4_b1_h16_t1k"]
    parts = [workloads.make_inputs(bench.replica_workload(base, r), seq_lens=LENS) for r in range(world)]
    job = parts[0]
    pt, off = [], 0
    for p_ in parts:
        pt.append(p_.page_table + off)
        off += p_.n_pages
    lens = np.concatenate([p_.seq_lens for p_ in parts])
    cu = np.zeros(len(lens) + 1, np.int32)
    cu[1:] = np.cumsum(lens)
    import dataclasses
    job = dataclasses.replace(job, seq_lens=lens, c=np.concatenate([p_.c for p_ in parts]),
                              kr=np.concatenate([p_.kr for p_ in parts]), cu=cu,
                              q_lat=np.concatenate([p_.q_lat for p_ in parts]),
                              q_rope=np.concatenate([p_.q_rope for p_ in parts]),
                              page_table=np.concatenate(pt), n_pages=off)
    o_all, l_all = _oracle_decode(base, job)
    for g in range(world * B_PER_RANK):
        r = g // B_PER_RANK
        k = got[r][1].index(g)
        np.testing.assert_array_equal(got[r][2][k], o_all[g])
        np.testing.assert_array_equal(got[r][3][k], l_all[g])
    # the replicas serve different sequences (distinct seeds)
    assert not np.array_equal(got[0][2], got[1][2])
