"""The largest inputs each path takes, at full parity with the oracle.

* The one-kernel path scores at most 1024 candidate blocks per (request, kv head) unit, judged
  from the block table's width: a 139 264-token request (1088 pages, 1024 candidates with an
  initial range of 1024 and a window of 7192 tokens) runs there, one page more takes the
  scoring, split decode and combine kernels.
* The selection holds every candidate's key and page on chip: 25 600 blocks is the longest
  block table it takes (3 276 800 tokens), a wider one is refused before any launch.
"""
import numpy as np
import pytest

from block_sparse_retrieval_gb300 import srkv, synth
from parity import check_fused_step, check_out, check_selection, gpu_decode, gpu_select, oracle_ref

pytestmark = pytest.mark.gpu

DEV = "cuda"
S = 128


def full_parity(case, threads=16):
    buf = gpu_select(case)
    assert int(buf.error_flags.item()) == 0
    ref = oracle_ref(case, kmax=buf.kmax, threads=threads)
    exact = check_selection(case, buf.sel.cpu().numpy(), buf.nsel.cpu().numpy(), ref)
    check_out(case, gpu_decode(case, buf, ref["sel"], ref["nsel"]), ref["out"])
    assert int(buf.error_flags.item()) == 0
    check_fused_step(case, buf, ref, exact)
    return exact


@pytest.mark.parametrize("seq_len,n,launches", [(1088 * S, 1024, 1), (1089 * S, 1025, 3)])
def test_candidate_limit_of_the_one_kernel_path(seq_len, n, launches):
    case = synth.llama8b_layer(seq_len=seq_len, device=DEV, seed=81)
    assert srkv.num_candidates(case.cfg, seq_len) == n
    assert srkv.retrieval_decode_launches(case.cfg, case.batch, case.max_blocks) == launches
    assert full_parity(case) >= 1


def test_longest_block_table():
    case = synth.make_case(seq_lens=[25600 * S], num_q_heads=4, num_kv_heads=1, head_dim=64,
                           init_tokens=1024, local_tokens=7192, topk_percent=0.2,
                           dense_boundary=0, plant_fraction=0.03, seed=82, device=DEV)
    assert case.max_blocks == 25600
    n = srkv.num_candidates(case.cfg, 25600 * S)
    assert n == 25536
    assert srkv.retrieval_decode_launches(case.cfg, case.batch, case.max_blocks) == 3
    full_parity(case)
    # with every candidate kept (p = 1) the selection is the whole candidate list
    dense = synth.Case(**{**case.__dict__, "cfg": dict(case.cfg, topk_percent=1.0)})
    buf = gpu_select(dense)
    assert int(buf.nsel[0, 0]) == n
    assert np.array_equal(buf.sel[0, 0, :n].cpu().numpy(), np.arange(8, 8 + n))
