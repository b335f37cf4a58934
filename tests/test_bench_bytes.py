"""The benchmark's algorithmic bytes (the roofline numerator) against the oracle's own
attention set.  bench.py counts the attended tokens of a (request, kv head) unit in closed
form (initial range, kept blocks clipped to the offload range, window, as a set); the oracle
attends exactly the positions whose softmax weight is nonzero.  Both must agree token for
token, page for page, and on the distinct (physical page, kv head, row) triples that a step
with shared prefix pages reads."""
import numpy as np
import pytest

import bench
import oracle
from block_sparse_retrieval_gb300 import synth

S = 128


def cases():
    mk = synth.make_case
    return {
        # unaligned initial range and window, a request shorter than both, an empty one
        "unaligned": mk(seq_lens=[3000, 5200, 130, 0, 1999], num_q_heads=4, num_kv_heads=2,
                        head_dim=64, init_tokens=1000, local_tokens=1500, topk_percent=0.3,
                        dense_boundary=0, seed=91),
        # pages of a 1024-token prefix shared by every request
        "shared-prefix": mk(seq_lens=[2600, 4100, 3333], num_q_heads=4, num_kv_heads=2,
                            head_dim=64, init_tokens=256, local_tokens=700, topk_percent=0.25,
                            dense_boundary=0, shared_prefix_tokens=1024, seed=92),
        # one prompt below the dense boundary: every candidate kept
        "dense-boundary": mk(seq_lens=[4000, 4000], prompt_lens=[3999, 4000],
                             num_q_heads=4, num_kv_heads=1, head_dim=64, init_tokens=512,
                             local_tokens=1024, topk_percent=0.2, dense_boundary=4000,
                             seed=93),
    }


def attended_positions(case, arr, r, h):
    w, _ = oracle.unit_weights(case.cfg, arr["q"], arr["k_cache"], arr["v_cache"],
                               arr["block_table"], arr["seq_lens"], arr["prompt_lens"], r, h)
    return np.flatnonzero((w != 0).any(axis=0))


@pytest.mark.parametrize("name", ["unaligned", "shared-prefix", "dense-boundary"])
def test_attended_tokens_and_pages_match_the_oracle(name):
    case = cases()[name]
    cfg = case.cfg
    arr = synth.to_oracle_arrays(case)
    ref = oracle.decode(cfg, *[arr[k] for k in ("q", "k_cache", "v_cache", "block_table",
                                               "seq_lens", "prompt_lens")])
    Ls = arr["seq_lens"]
    for r in range(case.batch):
        for h in range(cfg["num_kv_heads"]):
            L = int(Ls[r])
            pos = attended_positions(case, arr, r, h) if L > 0 else np.array([], int)
            sel = ref["sel"][r, h, :ref["nsel"][r, h]]
            toks, pages = bench.attended_tokens(L, sel, cfg["init_tokens"], cfg["local_tokens"])
            assert toks == pos.size, (name, r, h)
            assert pages == np.unique(pos // S).size, (name, r, h)


def test_unique_bytes_count_each_shared_row_once():
    case = cases()["shared-prefix"]
    cfg = case.cfg
    arr = synth.to_oracle_arrays(case)
    ref = oracle.decode(cfg, *[arr[k] for k in ("q", "k_cache", "v_cache", "block_table",
                                               "seq_lens", "prompt_lens")])
    rows = set()
    total = 0
    for r in range(case.batch):
        for h in range(cfg["num_kv_heads"]):
            pos = attended_positions(case, arr, r, h)
            total += pos.size
            rows |= {(int(arr["block_table"][r, t // S]), h, int(t % S)) for t in pos}
    row_bytes = cfg["head_dim"] * 2
    got = bench.unique_kv_bytes(case, ref["sel"], ref["nsel"], row_bytes=row_bytes)
    assert got == len(rows) * 2 * row_bytes
    assert len(rows) < total  # the shared prefix pages are attended by several requests
