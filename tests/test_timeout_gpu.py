"""Failure detection without a GPU fault: the bounded on-chip waits run out, report
SRKV_EFLAG_TIMEOUT to the host and let their kernel finish; the context stays usable."""
import time

import numpy as np
import pytest
import torch

from block_sparse_retrieval_gb300 import srkv, synth
from parity import check_out, gpu_decode, gpu_select, oracle_ref

pytestmark = pytest.mark.gpu

TIMEOUT = 8  # SRKV_EFLAG_TIMEOUT


def test_waits_with_no_arrival_give_up_and_report():
    flags = torch.zeros(1, dtype=torch.int32, device="cuda")
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    srkv.selftest_wait_timeout(flags)
    torch.cuda.synchronize()  # returns: the kernel finished instead of hanging
    elapsed = time.perf_counter() - t0
    assert int(flags.item()) == TIMEOUT
    assert 3.5 < elapsed < 30.0, elapsed  # two waits of 2 s each, in sequence
    # the context is intact: a decode on it still matches the oracle
    case = synth.make_case(seq_lens=[5000, 2600], num_q_heads=8, num_kv_heads=2, head_dim=128,
                           init_tokens=256, local_tokens=1024, topk_percent=0.25,
                           dense_boundary=0, seed=81, device="cuda")
    buf = gpu_select(case)
    assert int(buf.error_flags.item()) == 0
    ref = oracle_ref(case, kmax=buf.kmax)
    out = gpu_decode(case, buf, ref["sel"], ref["nsel"])
    assert int(buf.error_flags.item()) == 0
    check_out(case, out, ref["out"])
    assert np.isfinite(out).all()
