"""Small helpers shared by the tests: build a cache with the oracle from workload inputs."""
import numpy as np

import oracle
import workloads


def empty_cache(cfg, B, n_pages):
    pool = np.zeros((n_pages, oracle.page_bytes(cfg)), dtype=np.uint8)
    sink = np.zeros((B, cfg.n_sink, 576), dtype=np.uint16)
    ring = np.zeros((B, cfg.n_recent, 576), dtype=np.uint16)
    return pool, sink, ring


def oracle_prefill(cfg, inp: workloads.CacheInputs, chunk=None):
    """Write every prefill token with the oracle; chunk=k writes k tokens per sequence per call."""
    B = inp.seq_lens.shape[0]
    pool, sink, ring = empty_cache(cfg, B, inp.n_pages)
    if chunk is None:
        fl = oracle.write(cfg, inp.c, inp.kr, inp.cu, np.zeros(B, np.int32), int(inp.seq_lens.max(initial=1)),
                          inp.page_table, pool, sink, ring)
        assert fl == 0, fl
        return pool, sink, ring
    done = np.zeros(B, np.int32)
    while (done < inp.seq_lens).any():
        n = np.minimum(chunk, inp.seq_lens - done)
        rows_c, rows_k = [], []
        for b in range(B):
            r0 = inp.cu[b] + done[b]
            rows_c.append(inp.c[r0:r0 + n[b]])
            rows_k.append(inp.kr[r0:r0 + n[b]])
        cu = np.zeros(B + 1, np.int32)
        cu[1:] = np.cumsum(n)
        fl = oracle.write(cfg, np.concatenate(rows_c), np.concatenate(rows_k), cu, done, chunk,
                          inp.page_table, pool, sink, ring)
        assert fl == 0, fl
        done = done + n
    return pool, sink, ring
