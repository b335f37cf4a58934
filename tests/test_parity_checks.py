"""The parity checks themselves (CPU only): they pass the oracle's answer and reject the
errors a kernel can make.

The GPU parity tests judge the library through the comparators of ``tests/parity.py``.
Here those comparators get the oracle's own result, as the GPU would return it (outputs
rounded to bf16), which must pass; then that result with one planted error each, which
must not: a kept block swapped for the next candidate, a wrong kept count, a kept block
lost from the attention sums, an output element moved by the arithmetic bound.  Inside the
top-k gap band any valid top-k passes and an invalid one does not.
"""
import numpy as np
import pytest
import torch

import oracle
from block_sparse_retrieval_gb300 import synth
from parity import GAP, TIGHT_TOL, TOL, check_out, check_same, check_selection

KEYS = ("q", "k_cache", "v_cache", "block_table", "seq_lens", "prompt_lens")


def as_bf16(x: np.ndarray) -> np.ndarray:
    return torch.from_numpy(x).to(torch.bfloat16).double().numpy()


@pytest.fixture(scope="module")
def small():
    case = synth.make_case(seq_lens=[5000, 3000], num_q_heads=16, num_kv_heads=2, head_dim=64,
                           init_tokens=300, local_tokens=1000, topk_percent=0.3,
                           dense_boundary=0, seed=11)
    arr = synth.to_oracle_arrays(case)
    return case, arr, oracle.decode(case.cfg, *[arr[k] for k in KEYS], threads=4)


def _wide_gap_unit(ref):
    """A unit whose k-th and (k+1)-th scores are well apart, with its k and candidates."""
    B, Hkv = ref["nsel"].shape
    for r in range(B):
        for h in range(Hkv):
            s = ref["scores"][r, h]
            cand = np.flatnonzero(~np.isnan(s))
            k = int(ref["nsel"][r, h])
            if 0 < k < cand.size:
                srt = np.sort(s[cand])[::-1]
                if (srt[k - 1] - srt[k]) / np.abs(s[cand]).max() > 100 * GAP:
                    return r, h, k, cand
    raise AssertionError("no unit with a wide top-k gap")


def test_the_oracle_answer_passes(small):
    case, _, ref = small
    assert check_selection(case, ref["sel"], ref["nsel"], ref) > 0
    check_out(case, as_bf16(ref["out"]), ref["out"])
    check_same(case, as_bf16(ref["out"]), ref["out"])


def test_a_kept_block_swapped_for_the_next_candidate_is_caught(small):
    case, _, ref = small
    r, h, k, cand = _wide_gap_unit(ref)
    s = ref["scores"][r, h]
    order = cand[np.argsort(-s[cand], kind="stable")]
    sel = ref["sel"].copy()
    swapped = np.sort(np.concatenate([order[:k - 1], order[k:k + 1]]))
    sel[r, h, :k] = swapped
    with pytest.raises(AssertionError):
        check_selection(case, sel, ref["nsel"], ref)


def test_a_wrong_kept_count_is_caught(small):
    case, _, ref = small
    r, h, k, _ = _wide_gap_unit(ref)
    nsel = ref["nsel"].copy()
    nsel[r, h] = k - 1
    with pytest.raises(AssertionError):
        check_selection(case, ref["sel"], nsel, ref)


def test_inside_the_gap_band_any_valid_top_k_passes(small):
    case, _, ref = small
    r, h, k, cand = _wide_gap_unit(ref)
    s = ref["scores"][r, h]
    order = cand[np.argsort(-s[cand], kind="stable")]
    # Make the k-th and (k+1)-th candidates tie: either one completes a valid top-k.
    tied = {key: v.copy() for key, v in ref.items()}
    tied["scores"][r, h, order[k]] = s[order[k - 1]]
    alt = ref["sel"].copy()
    alt[r, h, :k] = np.sort(np.concatenate([order[:k - 1], order[k:k + 1]]))
    check_selection(case, ref["sel"], ref["nsel"], tied)
    check_selection(case, alt, ref["nsel"], tied)
    # A block from below the band is not a valid completion.
    bad = ref["sel"].copy()
    bad[r, h, :k] = np.sort(np.concatenate([order[:k - 1], order[-1:]]))
    with pytest.raises(AssertionError):
        check_selection(case, bad, ref["nsel"], tied)


def test_an_output_element_past_the_bound_is_caught(small):
    case, _, ref = small
    atol, rtol = TIGHT_TOL[case.cfg["dtype"]]
    assert atol <= TOL[case.cfg["dtype"]][0] and rtol <= TOL[case.cfg["dtype"]][1]
    want = ref["out"]
    i = np.unravel_index(np.argmax(np.abs(want)), want.shape)
    got = want.copy()
    got[i] += 0.5 * (atol + rtol * abs(want[i]))
    check_out(case, got, want)
    got[i] = want[i] + 1.5 * (atol + rtol * abs(want[i]))
    with pytest.raises(AssertionError):
        check_out(case, got, want)


def test_a_lost_kept_block_is_caught_on_a_long_layer():
    """On a 16384-token layer a kept block is 128 of ~9 900 attended tokens: dropping it moves
    the output by less than the method's tolerance but past the arithmetic bound, and past
    the tolerance between two GPU paths."""
    case = synth.llama8b_layer(seq_len=16384, seed=2)
    arr = synth.to_oracle_arrays(case)
    unit = [(0, 0)]
    ref = oracle.decode(case.cfg, *[arr[k] for k in KEYS], units=unit, threads=4)
    k = int(ref["nsel"][0, 0])
    assert k > 1
    sel, nsel = ref["sel"].copy(), ref["nsel"].copy()
    sel[0, 0, k - 1] = -1
    nsel[0, 0] = k - 1
    lost = oracle.decode(case.cfg, *[arr[key] for key in KEYS], units=unit, sel=sel, nsel=nsel,
                         threads=4)
    G = case.cfg["num_q_heads"] // case.cfg["num_kv_heads"]
    got, want = as_bf16(lost["out"]), ref["out"]
    atol, rtol = TOL[case.cfg["dtype"]]
    assert np.all(np.abs(got[0, :G] - want[0, :G]) <= atol + rtol * np.abs(want[0, :G]))
    with pytest.raises(AssertionError):
        check_out(case, got, want, unit)
    with pytest.raises(AssertionError):
        check_same(case, got[0, :G], want[0, :G])
    check_out(case, as_bf16(want), want, unit)
