"""GPU parity of the compressed pages: srkv_quantize_kv_fp8 against the oracle's E4M3
quantiser (bit-exact codes and scales), and srkv_retrieval_decode_fp8 against the oracle's
decode of its own codes (the selection of the full-precision cache, as the library takes it
from the vectors of the bf16 keys)."""
import numpy as np
import pytest
import torch

import oracle
from block_sparse_retrieval_gb300 import srkv, synth
from parity import check_out, check_selection, gpu_select, oracle_ref

pytestmark = pytest.mark.gpu

DEV = "cuda"


def quantize(case):
    P = case.num_pages
    ids = torch.arange(P, dtype=torch.int32, device=DEV)
    k8 = torch.empty(case.k_cache.shape, dtype=torch.uint8, device=DEV)
    v8 = torch.empty_like(k8)
    ks = torch.empty(case.k_cache.shape[:3], dtype=torch.float32, device=DEV)
    vs = torch.empty_like(ks)
    flags = torch.zeros(1, dtype=torch.int32, device=DEV)
    srkv.quantize_kv_fp8(case.cfg, case.k_cache, case.v_cache, ids, k8, v8, ks, vs, flags)
    torch.cuda.synchronize()
    assert int(flags.item()) == 0
    return k8, v8, ks, vs


def test_quantizer_matches_the_oracle_bit_for_bit():
    case = synth.llama8b_layer(seq_len=4096, device=DEV, seed=71)
    k8, v8, ks, vs = quantize(case)
    arr = synth.to_oracle_arrays(case)
    for got_c, got_s, src in ((k8, ks, arr["k_cache"]), (v8, vs, arr["v_cache"])):
        codes, scales = oracle.quantize_e4m3(case.cfg, src)
        np.testing.assert_array_equal(got_c.cpu().numpy(), codes)
        np.testing.assert_array_equal(got_s.cpu().numpy(), scales)


def test_quantizer_d64_and_zero_rows_match_the_oracle():
    case = synth.make_case(seq_lens=[3000, 1500], num_q_heads=4, num_kv_heads=2, head_dim=64,
                           seed=73, device=DEV)
    k = case.k_cache.clone()
    k[0, 1, 5:9] = 0      # all-zero rows: scale 1, codes 0
    k[1, 0, 100] *= 1e4   # a large row: the scale follows its maximum
    case = synth.Case(**{**case.__dict__, "k_cache": k})
    k8, v8, ks, vs = quantize(case)
    arr = synth.to_oracle_arrays(case)
    for got_c, got_s, src in ((k8, ks, arr["k_cache"]), (v8, vs, arr["v_cache"])):
        codes, scales = oracle.quantize_e4m3(case.cfg, src)
        np.testing.assert_array_equal(got_c.cpu().numpy(), codes)
        np.testing.assert_array_equal(got_s.cpu().numpy(), scales)
    assert (ks[0, 1, 5:9] == 1).all() and (k8[0, 1, 5:9] == 0).all()


def test_quantizer_rows_on_a_code_midpoint_match_the_oracle():
    """Rows whose fp32 quotient x / scale lands exactly on the midpoint between two codes while
    the exact quotient lies just above it (4.875 in a row of largest magnitude 52: 42.0 in
    fp32): the fp32 quotient's tie goes to the even code on both sides."""
    case = synth.make_case(seq_lens=[1024], num_q_heads=4, num_kv_heads=2, head_dim=64,
                           seed=74, device=DEV)
    pairs = [(52.0, 4.875), (9.25, -6.9375), (58.0, -10.875), (22.0, 4.125), (13.0, 9.75),
             (5.625, 4.21875), (40.5, 30.375), (50.0, -37.5), (39.5, -7.40625), (25.0, -4.6875)]
    k = case.k_cache.clone()
    for i, (amax, v) in enumerate(pairs):
        row = k[0, 0, i].float()
        row = row * (0.5 * amax / row.abs().max())
        row[0], row[1] = amax, v
        k[0, 0, i] = row.to(torch.bfloat16)
    case = synth.Case(**{**case.__dict__, "k_cache": k})
    k8, _, ks, _ = quantize(case)
    codes, scales = oracle.quantize_e4m3(case.cfg, synth.to_oracle_arrays(case)["k_cache"])
    np.testing.assert_array_equal(k8.cpu().numpy(), codes)
    np.testing.assert_array_equal(ks.cpu().numpy(), scales)
    assert int(k8[0, 0, 0, 1]) == 0x62


def test_quantizer_leaves_other_pages_and_flags_bad_ids():
    case = synth.llama8b_layer(seq_len=2048, device=DEV, seed=72)
    P = case.num_pages
    k8 = torch.full(case.k_cache.shape, 0x5A, dtype=torch.uint8, device=DEV)
    v8 = torch.full_like(k8, 0x5A)
    ks = torch.full(case.k_cache.shape[:3], -1.0, dtype=torch.float32, device=DEV)
    vs = torch.full_like(ks, -1.0)
    flags = torch.zeros(1, dtype=torch.int32, device=DEV)
    ids = torch.tensor([3, P + 5, 1], dtype=torch.int32, device=DEV)
    srkv.quantize_kv_fp8(case.cfg, case.k_cache, case.v_cache, ids, k8, v8, ks, vs, flags)
    torch.cuda.synchronize()
    assert int(flags.item()) & 1  # SRKV_EFLAG_PAGE_RANGE
    untouched = [p for p in range(P) if p not in (1, 3)]
    assert (k8[untouched] == 0x5A).all() and (ks[untouched] == -1).all()
    assert (ks[[1, 3]] > 0).all()


def fp8_call(case, reps, q8):
    k8, v8, ks, vs = q8
    b = srkv.DecodeBuffers(case.cfg, case.batch, case.max_blocks, case.num_pages, device=DEV)
    b.reps.copy_(reps)
    srkv.retrieval_decode_fp8(case.cfg, case.q, k8, v8, ks, vs, b.reps, case.block_table,
                              case.seq_lens, case.prompt_lens, b.sel, b.nsel, b.out,
                              b.workspace, b.error_flags)
    torch.cuda.synchronize()
    assert int(b.error_flags.item()) == 0
    return b


CASES = {
    # one kernel (8 units)
    "llama8b-16k": lambda: synth.llama8b_layer(seq_len=16384, device=DEV, seed=73),
    # scoring + split decode + combine (32 units)
    "ragged-4": lambda: synth.ragged_batch(n_requests=4, lo=9000, hi=20000, device=DEV, seed=74),
    "short-and-empty": lambda: synth.make_case(seq_lens=[700, 1, 0, 129, 130, 1030, 9000],
                                               num_q_heads=8, num_kv_heads=2, head_dim=128,
                                               init_tokens=1024, local_tokens=1024,
                                               topk_percent=0.2, dense_boundary=0, seed=75,
                                               device=DEV),
}


@pytest.mark.parametrize("name", list(CASES))
def test_fp8_decode_parity(name):
    case = CASES[name]()
    base = gpu_select(case)  # vectors of the bf16 keys, and the bf16 selection
    q8 = quantize(case)
    got = fp8_call(case, base.reps, q8)
    # the selection is the bf16 one (same vectors)
    assert np.array_equal(got.sel.cpu().numpy(), base.sel.cpu().numpy())
    assert np.array_equal(got.nsel.cpu().numpy(), base.nsel.cpu().numpy())
    arr = synth.to_oracle_arrays(case)
    ref16 = oracle_ref(case, arr, kmax=base.kmax)
    exact = check_selection(case, got.sel.cpu().numpy(), got.nsel.cpu().numpy(), ref16)
    kc, ks = oracle.quantize_e4m3(case.cfg, arr["k_cache"])
    vc, vs = oracle.quantize_e4m3(case.cfg, arr["v_cache"])
    ref8 = oracle.decode(dict(case.cfg, dtype=2), arr["q"], kc, vc, arr["block_table"],
                         arr["seq_lens"], arr["prompt_lens"], sel=ref16["sel"],
                         nsel=ref16["nsel"], k_scale=ks, v_scale=vs, threads=8)
    if exact == case.batch * case.cfg["num_kv_heads"]:
        check_out(case, got.out.float().cpu().numpy(), ref8["out"])


def test_fp8_decode_rejects_what_it_does_not_cover():
    case = synth.make_case(seq_lens=[3000], num_q_heads=4, num_kv_heads=2, head_dim=64,
                           init_tokens=256, local_tokens=512, topk_percent=0.2,
                           dense_boundary=0, seed=76, device=DEV)
    b = srkv.DecodeBuffers(case.cfg, case.batch, case.max_blocks, case.num_pages, device=DEV)
    k8 = torch.zeros(case.k_cache.shape, dtype=torch.uint8, device=DEV)
    ks = torch.ones(case.k_cache.shape[:3], dtype=torch.float32, device=DEV)
    with pytest.raises(RuntimeError, match="unsupported"):
        srkv.retrieval_decode_fp8(case.cfg, case.q, k8, k8, ks, ks, b.reps, case.block_table,
                                  case.seq_lens, case.prompt_lens, b.sel, b.nsel, b.out,
                                  b.workspace, b.error_flags)
