"""Pins of the oracle to facts outside itself (CPU only).

Each test checks the oracle against something it does not compute itself: values
printed on the pages (``tests/golden``), exact rational arithmetic, brute-force
enumeration on tiny inputs, a library attention routine
(``torch.nn.functional.scaled_dot_product_attention`` in fp64), ``numpy.mean``, and
invariances the method must have (physical page order, prefix sharing).
"""
import itertools
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from block_sparse_retrieval_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ---- helpers that restate the pages' definitions in another form ------------------------

def widen(a: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (uint16) or float32 -> float64, exactly."""
    if a.dtype == np.uint16:
        return (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return a.astype(np.float64)


def logical_kv(arr, r: int, h: int, S: int):
    """Keys and values of request r, kv head h, gathered in token order."""
    bt, L = arr["block_table"], int(arr["seq_lens"][r])
    K = np.stack([widen(arr["k_cache"][bt[r, t // S], h, t % S]) for t in range(L)]) \
        if L else np.zeros((0, arr["k_cache"].shape[-1]))
    V = np.stack([widen(arr["v_cache"][bt[r, t // S], h, t % S]) for t in range(L)]) \
        if L else np.zeros((0, arr["v_cache"].shape[-1]))
    return K, V


def sdpa(qv: np.ndarray, K: np.ndarray, V: np.ndarray, tokens) -> np.ndarray:
    """Library softmax attention of one query over the listed tokens."""
    idx = sorted(tokens)
    q_t = torch.from_numpy(qv).reshape(1, 1, 1, -1)
    k_t = torch.from_numpy(K[idx]).reshape(1, 1, len(idx), -1)
    v_t = torch.from_numpy(V[idx]).reshape(1, 1, len(idx), -1)
    return torch.nn.functional.scaled_dot_product_attention(q_t, k_t, v_t).reshape(-1).numpy()


def exact_k(n: int, p: float) -> int:
    """Smallest integer >= p*n, with p read as the decimal it was written as."""
    return min(n, math.ceil(Fraction(repr(p)) * n)) if n > 0 else 0


def offload_blocks(L: int, S: int, INIT: int, LOCAL: int) -> list[int]:
    """Blocks that hold at least one offload token, by enumerating the tokens."""
    return sorted({t // S for t in range(max(INIT, 0), L - LOCAL)})


def attended_set(L: int, S: int, INIT: int, LOCAL: int, selected) -> set[int]:
    """initial_tokens, plus the offload tokens of the selected blocks, plus the window."""
    W = L - LOCAL
    tokens = set(range(0, min(INIT, L)))
    for b in selected:
        tokens |= {t for t in range(b * S, min(b * S + S, L)) if INIT <= t < W}
    tokens |= set(range(max(W, 0), L))
    return tokens


def small_case(seed, **kw):
    base = dict(seq_lens=[700], num_q_heads=4, num_kv_heads=2, head_dim=16, dtype=synth.F32,
                block_size=32, init_tokens=64, local_tokens=96, topk_percent=0.3,
                dense_boundary=0, seed=seed)
    base.update(kw)
    return synth.make_case(**base)


# ---- closed forms printed on the pages ------------------------------------------------------

def test_footprint_matches_survey_table():
    g = json.load(open(os.path.join(GOLDEN, "kv_footprint.json")))["kvs_gpt3_table"]
    for row in g["rows"]:
        b = oracle.kv_cache_bytes(row["batch"], g["layers"], g["tokens"], g["hidden"],
                                  g["bytes_per_value"])
        gib = b / 2**30
        printed = row["kv_gb"]
        half_unit = 0.05 if printed != int(printed) else 0.5
        assert abs(gib - printed) <= half_unit, (row, gib)
        assert round(gib / g["weights_gb"], 2) == pytest.approx(row["kv_over_weight"], abs=0.011)


def test_footprint_atb_example_and_its_printed_slip():
    g = json.load(open(os.path.join(GOLDEN, "kv_footprint.json")))["atb_llama2_70b"]
    b = oracle.kv_cache_bytes(1, g["layers"], g["seq_len"], g["hidden"], g["bytes_per_value"])
    assert b == g["formula_bytes"] == 2 * 80 * 2048 * 8192 * 2
    # The page's 10.7 GB is twice the product of its own factors.
    assert abs(2 * b / 1e9 - g["printed_gb"]) < 0.05


# ---- k and the candidate range --------------------------------------------------------------

@pytest.mark.parametrize("n,p,k", [(448, 0.2, 90), (445, 0.2, 89), (26, 0.2, 6), (960, 0.1, 96),
                                   (960, 0.2, 192), (960, 0.4, 384), (960, 1.0, 960),
                                   (0, 0.2, 0), (100, 0.0, 0), (5, 0.01, 1), (1, 0.2, 1),
                                   # p * n rounds to just above a whole number in binary
                                   (100, 0.07, 7), (50, 0.14, 7), (25, 0.28, 7), (100, 0.55, 55)])
def test_topk_count_worked_values(n, p, k):
    assert oracle.topk_count(n, p) == k


def test_topk_count_equals_exact_rational_ceiling():
    """Every ratio in hundredths (some of them, 0.07 or 0.55, give products p * n that round to
    just above a whole number in binary), a third and 1."""
    for p in [i / 100 for i in range(0, 101)] + [1 / 3]:
        for n in range(0, 2049):
            assert oracle.topk_count(n, p) == exact_k(n, p), (n, p)


def test_candidate_count_by_token_enumeration():
    rng = np.random.default_rng(0)
    for _ in range(300):
        S = int(rng.choice([1, 4, 16, 128]))
        L = int(rng.integers(0, 3000))
        INIT = int(rng.integers(0, 700))
        LOCAL = int(rng.integers(0, 900))
        assert oracle.num_candidates(L, S, INIT, LOCAL) == len(offload_blocks(L, S, INIT, LOCAL))
    # The workloads' defaults: 65536 tokens -> 448 candidates; 131072 -> 960; tiny -> 26.
    assert oracle.num_candidates(65536, 128, 1024, 7192) == 448
    assert oracle.num_candidates(131072, 128, 1024, 7192) == 960
    assert oracle.num_candidates(4096, 128, 256, 512) == 26


# ---- representation vectors -------------------------------------------------------------------

@pytest.mark.parametrize("dtype", [synth.BF16, synth.F32])
def test_block_reps_equal_numpy_mean(dtype):
    case = small_case(3, dtype=dtype, seq_lens=[300, 257, 64], head_dim=32)
    arr = synth.to_oracle_arrays(case)
    reps = oracle.block_reps(case.cfg, arr["k_cache"], arr["page_ids"], arr["page_valid"])
    K = widen(arr["k_cache"])
    for i, (p, v) in enumerate(zip(arr["page_ids"], arr["page_valid"])):
        np.testing.assert_allclose(reps[i], K[p, :, :v, :].mean(axis=1), rtol=0, atol=1e-13)


def test_block_rep_of_equal_keys_is_that_key():
    case = small_case(4, dtype=synth.BF16)
    arr = synth.to_oracle_arrays(case)
    k = arr["k_cache"].copy()
    k[5, 1, :, :] = k[5, 1, 0, :]
    reps = oracle.block_reps(case.cfg, k, [5], [32])
    assert np.array_equal(reps[0, 1], widen(k[5, 1, 0]))


# ---- attention against a library routine -------------------------------------------------------

def check_against_sdpa(case, token_sets):
    """token_sets(r, L) -> set of attended tokens, for every unit of the case."""
    arr = synth.to_oracle_arrays(case)
    res = oracle.decode(case.cfg, **{k: arr[k] for k in ("q", "k_cache", "v_cache",
                                                         "block_table", "seq_lens",
                                                         "prompt_lens")})
    c = case.cfg
    G = c["num_q_heads"] // c["num_kv_heads"]
    for r in range(case.batch):
        L = int(arr["seq_lens"][r])
        for h in range(c["num_kv_heads"]):
            K, V = logical_kv(arr, r, h, c["block_size"])
            toks = token_sets(r, h, L, res)
            for j in range(G):
                want = sdpa(widen(arr["q"][r, h * G + j]), K, V, toks)
                np.testing.assert_allclose(res["out"][r, h * G + j], want, rtol=1e-12,
                                           atol=1e-12)
    return res


@pytest.mark.parametrize("dtype", [synth.BF16, synth.F32])
def test_ratio_one_is_dense_attention(dtype):
    case = small_case(5, dtype=dtype, topk_percent=1.0, seq_lens=[700, 333, 1024])
    check_against_sdpa(case, lambda r, h, L, res: set(range(L)))


def test_short_prompt_is_dense_attention():
    case = small_case(6, topk_percent=0.2, dense_boundary=800, seq_lens=[700, 799],
                      prompt_lens=[700, 799])
    res = check_against_sdpa(case, lambda r, h, L, res: set(range(L)))
    # Every candidate is selected for a dense request.
    for r, L in enumerate((700, 799)):
        assert res["nsel"][r, 0] == len(offload_blocks(L, 32, 64, 96))


def test_prompt_at_boundary_is_sparse():
    case = small_case(6, topk_percent=0.2, dense_boundary=700, seq_lens=[700])
    res = oracle.decode(case.cfg, **{k: v for k, v in synth.to_oracle_arrays(case).items()
                                     if k not in ("page_ids", "page_valid")})
    n = len(offload_blocks(700, 32, 64, 96))
    assert res["nsel"][0, 0] == exact_k(n, 0.2) < n


def test_default_boundary_32k_is_strict():
    """The pages' DENSE_BOUNDARY of 32K = 32768: a prompt of 32767 tokens is attended densely,
    one of 32768 is not (the comparison is a strict "less than")."""
    case = small_case(9, topk_percent=0.2, dense_boundary=32768, seq_lens=[33000, 33000],
                      prompt_lens=[32767, 32768], head_dim=8)
    arr = synth.to_oracle_arrays(case)
    res = oracle.decode(case.cfg, *[arr[k] for k in ("q", "k_cache", "v_cache", "block_table",
                                                      "seq_lens", "prompt_lens")], threads=4)
    n = len(offload_blocks(33000, 32, 64, 96))
    assert res["nsel"][0, 0] == n
    assert res["nsel"][1, 0] == exact_k(n, 0.2) < n


def test_without_prompt_lengths_a_prompt_is_its_sequence():
    """With no prompt lengths given, DENSE_BOUNDARY is compared with the sequence length: the
    request below the boundary is attended densely, the other one is not."""
    case = small_case(8, topk_percent=0.2, dense_boundary=800, seq_lens=[700, 900],
                      prompt_lens=[700, 900])
    arr = synth.to_oracle_arrays(case)
    args = [arr[k] for k in ("q", "k_cache", "v_cache", "block_table", "seq_lens")]
    given = oracle.decode(case.cfg, *args, arr["prompt_lens"])
    absent = oracle.decode(case.cfg, *args, None)
    for key in ("sel", "nsel", "out"):
        np.testing.assert_array_equal(absent[key], given[key])
    assert absent["nsel"][0, 0] == len(offload_blocks(700, 32, 64, 96))
    n = len(offload_blocks(900, 32, 64, 96))
    assert absent["nsel"][1, 0] == exact_k(n, 0.2) < n


def test_ratio_zero_is_sinks_plus_window():
    case = small_case(7, topk_percent=0.0, seq_lens=[700, 190, 40])
    check_against_sdpa(case, lambda r, h, L, res: attended_set(L, 32, 64, 96, []))


def test_softmax_weights_sum_to_one_and_vanish_off_the_set():
    case = small_case(8, seq_lens=[900])
    arr = synth.to_oracle_arrays(case)
    args = {k: arr[k] for k in ("q", "k_cache", "v_cache", "block_table", "seq_lens",
                                "prompt_lens")}
    res = oracle.decode(case.cfg, **args)
    for h in range(2):
        w, _ = oracle.unit_weights(case.cfg, **args, r=0, h=h)
        toks = attended_set(900, 32, 64, 96, res["sel"][0, h, :res["nsel"][0, h]])
        off = [t for t in range(900) if t not in toks]
        assert np.all(np.abs(w.sum(axis=1) - 1.0) < 1e-12)
        assert np.all(w >= 0) and np.all(w[:, off] == 0)
    ones = dict(args, v_cache=np.ones_like(arr["v_cache"]))
    out = oracle.decode(case.cfg, **ones)["out"]
    np.testing.assert_allclose(out, 1.0, rtol=0, atol=1e-12)


# ---- selection by brute force ---------------------------------------------------------------------

def brute_force_unit(arr, cfg, r, h):
    """Best k-subset by total score (ties: lexicographically smallest), enumerated."""
    S, INIT, LOCAL = cfg["block_size"], cfg["init_tokens"], cfg["local_tokens"]
    G = cfg["num_q_heads"] // cfg["num_kv_heads"]
    L = int(arr["seq_lens"][r])
    K, V = logical_kv(arr, r, h, S)
    cands = offload_blocks(L, S, INIT, LOCAL)
    k = exact_k(len(cands), cfg["topk_percent"])
    qs = [widen(arr["q"][r, h * G + j]) for j in range(G)]
    score = {b: sum(float(qj @ K[b * S:min(b * S + S, L)].mean(axis=0)) for qj in qs)
             for b in cands}
    best, best_sum = None, -math.inf
    for sub in itertools.combinations(cands, k):     # ascending tuples, lexicographic order
        s = sum(score[b] for b in sub)
        if best is None or s > best_sum + 1e-9 * (1 + abs(best_sum)):
            best, best_sum = sub, s
    toks = attended_set(L, S, INIT, LOCAL, best or ())
    outs = [sdpa(qj, K, V, toks) for qj in qs]
    return list(best or ()), outs


def test_selection_and_output_match_brute_force():
    rng = np.random.default_rng(11)
    for trial in range(40):
        S = int(rng.choice([8, 16, 32]))
        INIT = int(rng.integers(0, 3 * S))
        LOCAL = int(rng.integers(0, 4 * S))
        L = int(rng.integers(1, INIT + LOCAL + 12 * S))
        case = small_case(100 + trial, seq_lens=[L], block_size=S, init_tokens=INIT,
                          local_tokens=LOCAL, topk_percent=float(rng.choice([0.2, 0.34, 0.5])),
                          dtype=int(rng.integers(0, 2)), head_dim=8)
        arr = synth.to_oracle_arrays(case)
        res = oracle.decode(case.cfg, **{k: arr[k] for k in ("q", "k_cache", "v_cache",
                                                             "block_table", "seq_lens",
                                                             "prompt_lens")})
        for h in range(2):
            sel, outs = brute_force_unit(arr, case.cfg, 0, h)
            got = res["sel"][0, h, :res["nsel"][0, h]].tolist()
            assert got == sel, (trial, h, L, S, INIT, LOCAL)
            for j in range(2):
                np.testing.assert_allclose(res["out"][0, h * 2 + j], outs[j], rtol=1e-12,
                                           atol=1e-12)


def test_exact_ties_go_to_the_lower_block():
    # Every offload block gets identical keys, so every score ties exactly.
    case = small_case(12, seq_lens=[600], topk_percent=0.25)
    arr = synth.to_oracle_arrays(case)
    k = arr["k_cache"].copy()
    bt = arr["block_table"][0]
    for b in offload_blocks(600, 32, 64, 96):
        k[bt[b]] = k[bt[offload_blocks(600, 32, 64, 96)[0]]]
    arr["k_cache"] = k
    res = oracle.decode(case.cfg, **{x: arr[x] for x in ("q", "k_cache", "v_cache",
                                                         "block_table", "seq_lens",
                                                         "prompt_lens")})
    cands = offload_blocks(600, 32, 64, 96)
    kk = exact_k(len(cands), 0.25)
    for h in range(2):
        assert res["sel"][0, h, :res["nsel"][0, h]].tolist() == cands[:kk]
        assert brute_force_unit(arr, case.cfg, 0, h)[0] == cands[:kk]


def test_block_size_one_is_token_level_topk():
    case = small_case(13, seq_lens=[260], block_size=1, init_tokens=20, local_tokens=30,
                      topk_percent=0.1)
    arr = synth.to_oracle_arrays(case)
    res = oracle.decode(case.cfg, **{x: arr[x] for x in ("q", "k_cache", "v_cache",
                                                         "block_table", "seq_lens",
                                                         "prompt_lens")})
    for h in range(2):
        K, V = logical_kv(arr, 0, h, 1)
        qs = [widen(arr["q"][0, 2 * h + j]) for j in range(2)]
        qsum = qs[0] + qs[1]
        offload = np.arange(20, 230)
        s = K[offload] @ qsum
        order = np.lexsort((offload, -s))                 # score desc, then token asc
        chosen = sorted(offload[order[:exact_k(210, 0.1)]].tolist())
        assert res["sel"][0, h, :res["nsel"][0, h]].tolist() == chosen
        toks = set(range(20)) | set(chosen) | set(range(230, 260))
        for j in range(2):
            np.testing.assert_allclose(res["out"][0, 2 * h + j], sdpa(qs[j], K, V, toks),
                                       rtol=1e-12, atol=1e-12)


# ---- invariances ------------------------------------------------------------------------------------

def decode_all(case_cfg, arr):
    return oracle.decode(case_cfg, **{x: arr[x] for x in ("q", "k_cache", "v_cache",
                                                          "block_table", "seq_lens",
                                                          "prompt_lens")})


def test_physical_page_permutation_changes_nothing():
    case = small_case(14, seq_lens=[700, 450], shuffle=False)
    arr = synth.to_oracle_arrays(case)
    base = decode_all(case.cfg, arr)
    rng = np.random.default_rng(1)
    perm = rng.permutation(arr["k_cache"].shape[0])
    moved = dict(arr)
    moved["k_cache"] = np.empty_like(arr["k_cache"])
    moved["v_cache"] = np.empty_like(arr["v_cache"])
    moved["k_cache"][perm] = arr["k_cache"]
    moved["v_cache"][perm] = arr["v_cache"]
    bt = arr["block_table"].copy()
    bt[bt >= 0] = perm[bt[bt >= 0]]
    moved["block_table"] = bt
    other = decode_all(case.cfg, moved)
    for key in ("out", "sel", "nsel"):
        assert np.array_equal(base[key], other[key])


def test_prefix_sharing_changes_nothing():
    shared = small_case(15, seq_lens=[500, 640, 590], shared_prefix_tokens=256)
    arr = synth.to_oracle_arrays(shared)
    base = decode_all(shared.cfg, arr)
    # Give every request its own copy of the shared pages.
    bt = arr["block_table"].copy()
    k, v = [arr["k_cache"]], [arr["v_cache"]]
    nxt = arr["k_cache"].shape[0]
    for r in range(1, 3):
        for b in range(256 // 32):
            k.append(arr["k_cache"][bt[r, b]][None])
            v.append(arr["v_cache"][bt[r, b]][None])
            bt[r, b] = nxt
            nxt += 1
    copied = dict(arr, k_cache=np.concatenate(k), v_cache=np.concatenate(v), block_table=bt)
    other = decode_all(shared.cfg, copied)
    for key in ("out", "sel", "nsel"):
        assert np.array_equal(base[key], other[key])


def test_planted_blocks_are_selected():
    case = synth.llama8b_layer(seq_len=12288, init_tokens=1024, local_tokens=2048,
                               plant_fraction=0.05, seed=21)
    arr = synth.to_oracle_arrays(case)
    res = decode_all(case.cfg, arr)
    # A planted block: its keys were moved along the group's query direction.
    bt = arr["block_table"][0]
    K = widen(arr["k_cache"])
    G = 4
    for h in range(8):
        qd = sum(widen(arr["q"][0, h * G + j]) for j in range(G))
        qd /= np.linalg.norm(qd)
        planted = [b for b in offload_blocks(12288, 128, 1024, 2048)
                   if K[bt[b], h].mean(axis=0) @ qd > 0.35]
        assert planted, h
        assert set(planted) <= set(res["sel"][0, h, :res["nsel"][0, h]].tolist())


def test_empty_sequence_gives_zero_output():
    case = small_case(16, seq_lens=[0, 100])
    res = decode_all(case.cfg, synth.to_oracle_arrays(case))
    assert np.all(res["out"][0] == 0) and np.all(res["nsel"][0] == 0)


def test_candidate_scores_match_enumeration():
    # LOCAL below the block size makes the partially filled last block a candidate.
    rng = np.random.default_rng(17)
    for trial in range(30):
        S = int(rng.choice([8, 16, 32]))
        L = int(rng.integers(S + 1, 20 * S))
        if L % S == 0:
            L += 1
        INIT, LOCAL = int(rng.integers(0, 2 * S)), int(rng.integers(0, L % S))
        case = small_case(300 + trial, seq_lens=[L], block_size=S, init_tokens=INIT,
                          local_tokens=LOCAL, head_dim=8, dtype=int(rng.integers(0, 2)))
        arr = synth.to_oracle_arrays(case)
        res = decode_all(case.cfg, arr)
        cands = offload_blocks(L, S, INIT, LOCAL)
        assert cands[-1] == (L - 1) // S            # the partial block is a candidate
        for h in range(2):
            K, _ = logical_kv(arr, 0, h, S)
            qsum = widen(arr["q"][0, 2 * h]) + widen(arr["q"][0, 2 * h + 1])
            for b in range(case.max_blocks):
                got = res["scores"][0, h, b]
                if b in cands:
                    want = float(qsum @ K[b * S:min(b * S + S, L)].mean(axis=0))
                    assert abs(got - want) <= 1e-12 * (1 + abs(want)), (trial, b)
                else:
                    assert math.isnan(got)


# ---- E4M3 compressed pages (OCP 8-bit floating point, "E4M3") -----------------------------

def test_e4m3_values_match_the_library_format():
    """Every code's value against PyTorch's float8_e4m3fn, the same OCP format, and the
    specification's landmarks."""
    codes = np.arange(256, dtype=np.uint8)
    got = oracle.e4m3_value(codes)
    lib = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    nan = (codes & 0x7F) == 0x7F
    assert np.isnan(got[nan]).all() and np.isnan(lib[nan]).all()
    np.testing.assert_array_equal(got[~nan], lib[~nan])
    assert got[0x7E] == 448.0 and got[0xFE] == -448.0          # largest finite
    assert got[0x08] == 2.0 ** -6 and got[0x07] == 7 / 8 * 2.0 ** -6  # normal / subnormal edge
    assert got[0x01] == 2.0 ** -9 and got[0x38] == 1.0
    assert math.copysign(1.0, got[0x80]) == -1.0 and got[0x80] == 0.0


def test_e4m3_rounding_matches_the_library_and_ties_go_even():
    rng = np.random.default_rng(3)
    x = np.concatenate([rng.uniform(-448, 448, 4000), rng.normal(0, 1, 4000),
                        rng.normal(0, 2.0 ** -7, 2000)]).astype(np.float32)
    lib = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    np.testing.assert_array_equal(oracle.e4m3_code(x.astype(np.float64)), lib)
    # exact midpoints between neighbouring codes go to the even code
    vals = oracle.e4m3_value(np.arange(0x7F, dtype=np.uint8))
    mids = (vals[:-1] + vals[1:]) / 2
    want = np.where(np.arange(0x7E) % 2 == 0, np.arange(0x7E), np.arange(1, 0x7F))
    np.testing.assert_array_equal(oracle.e4m3_code(mids), want)
    # saturation past the largest finite value, both signs
    np.testing.assert_array_equal(oracle.e4m3_code([449.0, 1e9, -500.0]), [0x7E, 0x7E, 0xFE])
    # a (positive) NaN gets the library's NaN code
    nan = torch.tensor([float("nan")]).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    np.testing.assert_array_equal(oracle.e4m3_code([float("nan")]), nan)


def test_e4m3_quantiser_scale_and_error_bound():
    """R10: the largest magnitude of a row lands on +-448, and every value comes back within
    half a unit in the last place of its binade (relative 2^-4 for normals)."""
    cfg = dict(num_q_heads=4, num_kv_heads=2, head_dim=64, block_size=128, init_tokens=0,
               local_tokens=0, topk_percent=0.2, dense_boundary=0, dtype=0)
    rng = np.random.default_rng(5)
    x = (rng.normal(0, 1, (3, 2, 128, 64)) * rng.uniform(0.01, 50, (3, 2, 128, 1)))
    x[1, 0, 7] = 0.0  # an all-zero row
    bits = (torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16).view(torch.int16)
            .numpy().view(np.uint16))
    codes, scales = oracle.quantize_e4m3(cfg, bits)
    xs = widen(bits)
    amax = np.abs(xs).max(-1)
    np.testing.assert_array_equal(scales, np.where(amax > 0, (amax.astype(np.float32)
                                                              / np.float32(448)), 1.0))
    assert (scales[1, 0, 7] == 1.0) and (codes[1, 0, 7] == 0).all()
    top = np.abs(xs).argmax(-1)
    lead = np.take_along_axis(codes, top[..., None], -1)[..., 0]
    assert np.all((lead & 0x7F)[amax > 0] == 0x7E)
    deq = oracle.e4m3_value(codes) * scales[..., None]
    y = np.abs(xs / scales[..., None])
    ulp_half = np.where(y >= 2.0 ** -6, 2.0 ** (np.floor(np.log2(np.maximum(y, 2.0 ** -6))) - 4),
                        2.0 ** -10)
    assert np.all(np.abs(deq - xs) <= (ulp_half * 1.0001 + 1e-12) * scales[..., None])


def test_e4m3_quantiser_matches_the_library_pipeline():
    """R10 against PyTorch doing the same steps in fp32: the row's largest magnitude, the scale
    max / 448, the quotient x / scale, its float8_e4m3fn code.  Besides random rows, rows
    whose fp32 quotient lands exactly on the midpoint between two codes while the exact
    quotient lies just above it (x = 4.875 in a row of largest magnitude 52: 42.0 in fp32,
    42.0000012 exactly): the fp32 quotient goes to the even code, 40, not to 44."""
    cfg = dict(num_q_heads=4, num_kv_heads=2, head_dim=64, block_size=128, init_tokens=0,
               local_tokens=0, topk_percent=0.2, dense_boundary=0, dtype=0)
    rng = np.random.default_rng(9)
    x = (rng.normal(0, 1, (2, 2, 128, 64)) * rng.uniform(0.01, 50, (2, 2, 128, 1)))
    pairs = [(52.0, 4.875), (9.25, -6.9375), (58.0, -10.875), (22.0, 4.125), (13.0, 9.75),
             (5.625, 4.21875), (40.5, 30.375), (50.0, -37.5), (39.5, -7.40625), (25.0, -4.6875)]
    for i, (amax, v) in enumerate(pairs):
        row = x[0, 0, i]
        row *= 0.5 * amax / np.abs(row).max()
        row[0], row[1] = amax, v
    t = torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16)
    bits = t.view(torch.int16).numpy().view(np.uint16)
    codes, scales = oracle.quantize_e4m3(cfg, bits)
    xf = t.float()
    lib_scale = xf.abs().amax(-1) / 448.0
    lib_scale = torch.where(lib_scale > 0, lib_scale, torch.ones_like(lib_scale))
    lib_codes = (xf / lib_scale[..., None]).to(torch.float8_e4m3fn).view(torch.uint8)
    np.testing.assert_array_equal(scales, lib_scale.numpy())
    np.testing.assert_array_equal(codes, lib_codes.numpy())
    assert codes[0, 0, 0, 1] == 0x62  # 4.875 in the row of 52: 40, the even neighbour of 42


def test_e4m3_pages_decode_as_the_equivalent_bf16_cache():
    """A compressed cache whose values code x scale are exact in bf16 (power-of-two
    scales) decodes exactly like that bf16 cache given the same selection: pins the per-row
    scale indexing and the reading of codes."""
    case = synth.make_case(seq_lens=[1500, 900], num_q_heads=8, num_kv_heads=2, head_dim=64,
                           init_tokens=256, local_tokens=384, topk_percent=0.3,
                           dense_boundary=0, seed=21)
    arr = synth.to_oracle_arrays(case)
    cfg = case.cfg
    rng = np.random.default_rng(9)
    P, Hkv, S, d = arr["k_cache"].shape
    kc = rng.integers(0, 256, (P, Hkv, S, d)).astype(np.uint8)
    vc = rng.integers(0, 256, (P, Hkv, S, d)).astype(np.uint8)
    kc[(kc & 0x7F) == 0x7F] = 0x38  # no NaN codes
    vc[(vc & 0x7F) == 0x7F] = 0x38
    ks = (2.0 ** rng.integers(-8, 3, (P, Hkv, S))).astype(np.float32)
    vs = (2.0 ** rng.integers(-8, 3, (P, Hkv, S))).astype(np.float32)

    def as_bf16(codes, scales):  # code x scale: 4 significant bits, exact in bf16
        v = (oracle.e4m3_value(codes) * scales[..., None]).astype(np.float32)
        return (v.view(np.uint32) >> 16).astype(np.uint16)

    kb, vb = as_bf16(kc, ks), as_bf16(vc, vs)
    ref = oracle.decode(cfg, arr["q"], kb, vb, arr["block_table"], arr["seq_lens"],
                        arr["prompt_lens"])
    got = oracle.decode(dict(cfg, dtype=2), arr["q"], kc, vc, arr["block_table"],
                        arr["seq_lens"], arr["prompt_lens"], sel=ref["sel"], nsel=ref["nsel"],
                        k_scale=ks, v_scale=vs)
    np.testing.assert_array_equal(got["out"], ref["out"])


def test_e4m3_pages_accuracy_against_bf16():
    """Accuracy of the compressed pages (oracle against oracle, fp64): with the selection of
    the full-precision cache (R11), the output over E4M3 pages stays within 10 % of the
    largest output magnitude of the unit, and within 2.5 % on average.  (Measured on the
    16384-token Llama-3-8B layer: 3.7 % max, 0.7 % mean.)"""
    case = synth.make_case(seq_lens=[6000, 3500], num_q_heads=8, num_kv_heads=2,
                           head_dim=128, init_tokens=512, local_tokens=1024, topk_percent=0.2,
                           dense_boundary=0, plant_fraction=0.05, seed=23)
    arr = synth.to_oracle_arrays(case)
    ref = oracle.decode(case.cfg, arr["q"], arr["k_cache"], arr["v_cache"], arr["block_table"],
                        arr["seq_lens"], arr["prompt_lens"], threads=4)
    kc, ks = oracle.quantize_e4m3(case.cfg, arr["k_cache"])
    vc, vs = oracle.quantize_e4m3(case.cfg, arr["v_cache"])
    got = oracle.decode(dict(case.cfg, dtype=2), arr["q"], kc, vc, arr["block_table"],
                        arr["seq_lens"], arr["prompt_lens"], sel=ref["sel"], nsel=ref["nsel"],
                        k_scale=ks, v_scale=vs, threads=4)
    G = case.cfg["num_q_heads"] // case.cfg["num_kv_heads"]
    for r in range(case.batch):
        for h in range(case.cfg["num_kv_heads"]):
            o = ref["out"][r, h * G:(h + 1) * G]
            e = np.abs(got["out"][r, h * G:(h + 1) * G] - o)
            top = np.abs(o).max()
            assert e.max() <= 0.10 * top, (r, h, e.max(), top)
            assert e.mean() <= 0.025 * top, (r, h, e.mean(), top)


def test_e4m3_decode_refuses_to_select_on_its_own():
    """R11: over compressed pages the selection must come from the full-precision keys, which
    the E4M3 decode does not see, so a call without a selection is refused instead of scoring
    the dequantised keys."""
    case = synth.make_case(seq_lens=[1500], num_q_heads=4, num_kv_heads=1, head_dim=128,
                           init_tokens=256, local_tokens=512, topk_percent=0.2,
                           dense_boundary=0, seed=24)
    arr = synth.to_oracle_arrays(case)
    kc, ks = oracle.quantize_e4m3(case.cfg, arr["k_cache"])
    vc, vs = oracle.quantize_e4m3(case.cfg, arr["v_cache"])
    with pytest.raises(ValueError):
        oracle.decode(dict(case.cfg, dtype=2), arr["q"], kc, vc, arr["block_table"],
                      arr["seq_lens"], arr["prompt_lens"], k_scale=ks, v_scale=vs)
    ref = oracle.decode(case.cfg, arr["q"], arr["k_cache"], arr["v_cache"], arr["block_table"],
                        arr["seq_lens"], arr["prompt_lens"])
    got = oracle.decode(dict(case.cfg, dtype=2), arr["q"], kc, vc, arr["block_table"],
                        arr["seq_lens"], arr["prompt_lens"], sel=ref["sel"], nsel=ref["nsel"],
                        k_scale=ks, v_scale=vs)
    assert np.isfinite(got["out"]).all()
