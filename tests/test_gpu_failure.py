"""Device-side failure detection without a fault (GPU): a wait that can never complete gives up
after its bound, reports MLA_QCACHE_DEV_TIMEOUT, and the context stays usable."""
import numpy as np
import pytest
import torch

import bit_mla_kv_qcache_gb300 as q
import workloads
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu


def test_bounded_wait_reports_timeout_and_context_survives():
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    q.selftest_wait_timeout(err)
    torch.cuda.synchronize()
    assert int(err.item()) & q.DEV_TIMEOUT
    # the context still runs the hot path
    w = workloads.WORKLOADS["tiny_c4r4_b1_h16_t1k"]
    inp = workloads.make_inputs(w, seq_lens=np.array([300], np.int32))
    cache = gu.gpu_cache(w.config_kwargs(), inp)
    gu.write_rows(cache, inp.c, inp.kr, inp.seq_lens, 300)
    out, lse = cache.decode(gu.dev(inp.q_lat), gu.dev(inp.q_rope), w.softmax_scale)
    torch.cuda.synchronize()
    assert cache.error_bits() == 0 and torch.isfinite(out).all() and torch.isfinite(lse).all()
