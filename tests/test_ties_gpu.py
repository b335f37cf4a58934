"""Equal scores on the GPU: the lower block wins (the tie rule of the selection).  With keys
that are zero, every score is exactly 0 in any precision, so the selection is decided by the
tie rule alone and must equal the oracle's bit for bit: the first k candidates when every
key is zero; the blocks keyed along the group query (distinct positive scores) and then the
lowest of the zero blocks when a few are; or a group of equal positive scores that the k-th
key falls in.  This reaches the select's branch for a boundary bin that stays larger than 32
keys after every radix pass, which random scores do not, and a small bin of equal keys.
Covered on the one-kernel path, on the scoring kernel's short (n <= 1024) and long lists."""
import numpy as np
import pytest
import torch

from block_sparse_retrieval_gb300 import srkv, synth
from parity import check_out, gpu_select, oracle_ref

pytestmark = pytest.mark.gpu

DEV = "cuda"
S = 128


def tied(case, planted=()):
    """The case with every key zero, except the (block, factor) pairs in `planted`: those
    blocks of every request hold factor x the unit direction of the unit's summed query in
    every row, for every kv head."""
    cfg = case.cfg
    Hq, Hkv, d = cfg["num_q_heads"], cfg["num_kv_heads"], cfg["head_dim"]
    k = torch.zeros_like(case.k_cache)
    qsum = case.q.float().reshape(case.batch, Hkv, Hq // Hkv, d).sum(2)
    qdir = qsum / qsum.norm(dim=-1, keepdim=True)
    bt = case.block_table.cpu().numpy()
    for r in range(case.batch):
        for b, f in planted:
            if b < bt.shape[1] and bt[r, b] >= 0:  # a block the request holds
                k[int(bt[r, b])] = (f * qdir[r]).unsqueeze(1).expand(Hkv, S, d).to(k.dtype)
    return synth.Case(**{**case.__dict__, "k_cache": k})


def expected(case, planted):
    """Per unit: the planted candidates by score, then the lowest other candidates, k in
    all, ascending."""
    cfg = case.cfg
    L = case.seq_lens.cpu().numpy()
    b_lo = cfg["init_tokens"] // S
    out = []
    for r in range(case.batch):
        n = srkv.num_candidates(cfg, int(L[r]))
        k = srkv.topk_count(n, cfg["topk_percent"])
        cands = range(b_lo, b_lo + n)
        keep = [b for _, b in sorted((-f, b) for b, f in planted if b in cands)][:k]
        rest = [b for b in cands if b not in keep][:k - len(keep)]
        out.append(sorted(keep + rest))
    return out


CASES = {
    # one kernel (8 units, 64 candidates each); below the default dense boundary, so 0
    "one-kernel": lambda: synth.llama8b_layer(seq_len=16384, dense_boundary=0, device=DEV,
                                              seed=101),
    # scoring kernel, short lists (32 units)
    "short-lists": lambda: synth.ragged_batch(n_requests=4, lo=9000, hi=20000,
                                              dense_boundary=0, device=DEV, seed=102),
    # scoring kernel, long lists (1499 candidates per unit)
    "long-lists": lambda: synth.make_case(seq_lens=[200000], num_q_heads=8, num_kv_heads=2,
                                          head_dim=64, init_tokens=1024, local_tokens=7192,
                                          topk_percent=0.2, dense_boundary=0, seed=103,
                                          device=DEV),
}
PLANTED = {"all-zero": (), "three-keyed": ((13, 3.0), (9, 1.0), (40, 2.0)),
           # 10 distinct scores above 6 equal ones; with 64 candidates (k = 13) the k-th
           # key falls among the equal ones: a small boundary bin of equal keys, kept lowest
           # blocks first
           "tied-boundary": tuple((10 + j, 3.0 - 0.1 * j) for j in range(10)) +
           tuple((b, 1.5) for b in (30, 22, 45, 60, 25, 50))}


@pytest.mark.parametrize("pattern", list(PLANTED))
@pytest.mark.parametrize("name", list(CASES))
def test_ties_go_to_the_lower_block(name, pattern):
    case = tied(CASES[name](), PLANTED[pattern])
    cfg = case.cfg
    want = expected(case, PLANTED[pattern])
    ref = oracle_ref(case, kmax=srkv.kmax_bound(cfg, case.max_blocks), threads=16)
    Hkv = cfg["num_kv_heads"]
    for r in range(case.batch):  # the oracle follows the rule (a pin of the oracle itself)
        for h in range(Hkv):
            assert ref["sel"][r, h, :ref["nsel"][r, h]].tolist() == want[r], (r, h)
    # the scoring kernel
    buf = gpu_select(case)
    assert int(buf.error_flags.item()) == 0
    assert np.array_equal(buf.nsel.cpu().numpy(), ref["nsel"])
    sel = buf.sel.cpu().numpy()
    for r in range(case.batch):
        for h in range(Hkv):
            assert sel[r, h, :ref["nsel"][r, h]].tolist() == want[r], (r, h)
    # the whole step (one kernel or three), selection and output
    step = srkv.DecodeBuffers(cfg, case.batch, case.max_blocks, case.num_pages, device=DEV)
    step.reps.copy_(buf.reps)
    srkv.retrieval_decode(cfg, case.q, case.k_cache, case.v_cache, step.reps, case.block_table,
                          case.seq_lens, case.prompt_lens, step.sel, step.nsel, step.out,
                          step.workspace, step.error_flags)
    torch.cuda.synchronize()
    assert int(step.error_flags.item()) == 0
    assert np.array_equal(step.nsel.cpu().numpy(), ref["nsel"])
    sel = step.sel.cpu().numpy()
    for r in range(case.batch):
        for h in range(Hkv):
            assert sel[r, h, :ref["nsel"][r, h]].tolist() == want[r], (r, h)
    check_out(case, step.out.float().cpu().numpy(), ref["out"])
