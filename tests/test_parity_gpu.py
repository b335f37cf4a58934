"""GPU parity: libsrkv (through its C ABI) against the oracle on seeded synthetic caches.

Small cases are checked in full; the full-size workloads on sampled (request, kv head)
units, in the launch configuration the benchmark uses.
"""
import numpy as np
import pytest
import torch

import oracle
from block_sparse_retrieval_gb300 import srkv, synth
from parity import check_fused_step, check_out, check_selection, gpu_decode, gpu_select, oracle_ref

pytestmark = pytest.mark.gpu

DEV = "cuda"


def small_cases():
    mk = synth.make_case
    return {
        "tiny": lambda: synth.tiny(device=DEV),
        "llama8b-16k": lambda: synth.llama8b_layer(seq_len=16384, device=DEV),
        "ragged-4": lambda: synth.ragged_batch(n_requests=4, lo=9000, hi=20000, device=DEV),
        # 24 and 12 (request, kv head) units: one kernel on clusters of 5 and of 10 (the
        # largest size whose clusters are all resident)
        "ragged-3": lambda: synth.ragged_batch(n_requests=3, lo=9000, hi=20000, seed=21,
                                               device=DEV),
        "h4-3req": lambda: mk(seq_lens=[11000, 7000, 15000], num_q_heads=16, num_kv_heads=4,
                              head_dim=128, init_tokens=1024, local_tokens=2048,
                              topk_percent=0.2, dense_boundary=0, seed=22, device=DEV),
        "dense-p1.0": lambda: synth.dense_vs_sparse(1.0, batch=2, seq_len=24576, device=DEV),
        "sparse-p0.1": lambda: synth.dense_vs_sparse(0.1, batch=2, seq_len=24576, device=DEV),
        "sparse-p0.4": lambda: synth.dense_vs_sparse(0.4, batch=2, seq_len=24576, device=DEV),
        "prefix-shared-8": lambda: synth.prefix_shared(n_requests=8, prefix=4096, lo=1024,
                                                       hi=4096, local_tokens=2048, device=DEV),
        "g8-d64": lambda: mk(seq_lens=[5000, 3000], num_q_heads=16, num_kv_heads=2, head_dim=64,
                             init_tokens=300, local_tokens=1000, topk_percent=0.3,
                             dense_boundary=0, seed=11, device=DEV),
        "g1": lambda: mk(seq_lens=[6100, 4000], num_q_heads=4, num_kv_heads=4, head_dim=128,
                         init_tokens=512, local_tokens=1024, topk_percent=0.25,
                         dense_boundary=0, seed=12, device=DEV),
        "g2-p0": lambda: mk(seq_lens=[7000], num_q_heads=8, num_kv_heads=4, head_dim=128,
                            init_tokens=256, local_tokens=512, topk_percent=0.0,
                            dense_boundary=0, seed=13, device=DEV),
        "g16-simt": lambda: mk(seq_lens=[3000, 2500], num_q_heads=32, num_kv_heads=2,
                               head_dim=128, init_tokens=256, local_tokens=512,
                               topk_percent=0.2, dense_boundary=0, seed=14, device=DEV),
        "f32-d128": lambda: mk(seq_lens=[4500, 2000], num_q_heads=8, num_kv_heads=2,
                               head_dim=128, dtype=synth.F32, init_tokens=256,
                               local_tokens=512, topk_percent=0.2, dense_boundary=0, seed=15,
                               device=DEV),
        "short-and-empty": lambda: mk(seq_lens=[700, 1, 0, 129, 130, 1030, 9000],
                                      num_q_heads=8, num_kv_heads=2, head_dim=128,
                                      init_tokens=1024, local_tokens=1024, topk_percent=0.2,
                                      dense_boundary=0, seed=16, device=DEV),
        "unaligned-init-no-window": lambda: mk(seq_lens=[9000, 9100, 2600], num_q_heads=8,
                                               num_kv_heads=2, head_dim=128, init_tokens=1000,
                                               local_tokens=0, topk_percent=0.3,
                                               dense_boundary=0, seed=17, device=DEV),
        "unaligned-both": lambda: mk(seq_lens=[9000, 9100, 2600, 2400], num_q_heads=8,
                                     num_kv_heads=2, head_dim=128, init_tokens=1000,
                                     local_tokens=1500, topk_percent=0.3, dense_boundary=0,
                                     seed=18, device=DEV),
        # more (request, kv head) units than split CTAs: the per-unit combine
        "many-units": lambda: mk(seq_lens=[1500 + 97 * i for i in range(20)], num_q_heads=32,
                                 num_kv_heads=8, head_dim=128, init_tokens=256,
                                 local_tokens=512, topk_percent=0.2, dense_boundary=0, seed=20,
                                 device=DEV),
        # p * n just above a whole number in binary (0.07 x 100 = 7.000000000000001): the
        # kept count is 7 of 100 on both sides, and 55 of 100 at 0.55
        "binary-ratio-0.07": lambda: mk(seq_lens=[21016, 21016 + 6400], num_q_heads=32,
                                        num_kv_heads=8, head_dim=128, topk_percent=0.07,
                                        dense_boundary=0, seed=23, device=DEV),
        "binary-ratio-0.55": lambda: mk(seq_lens=[21016], num_q_heads=32, num_kv_heads=8,
                                        head_dim=128, topk_percent=0.55, dense_boundary=0,
                                        seed=24, device=DEV),
        "dense-boundary": lambda: mk(seq_lens=[9000, 12000, 12000], prompt_lens=[9000, 11999, 12000],
                                     num_q_heads=8, num_kv_heads=2, head_dim=128,
                                     init_tokens=1024, local_tokens=2048, topk_percent=0.2,
                                     dense_boundary=12000, seed=19, device=DEV),
    }


CASES = small_cases()


@pytest.mark.parametrize("name", list(CASES))
def test_small_case_parity(name):
    case = CASES[name]()
    buf = gpu_select(case)
    assert int(buf.error_flags.item()) == 0
    arr = synth.to_oracle_arrays(case)
    # representation vectors
    reps = oracle.block_reps(case.cfg, arr["k_cache"], arr["page_ids"], arr["page_valid"])
    got_reps = buf.reps[case.page_ids.long()].double().cpu().numpy()
    np.testing.assert_allclose(got_reps, reps, rtol=0, atol=1e-5)
    # selection
    ref = oracle_ref(case, arr, kmax=buf.kmax)
    gsel, gnsel = buf.sel.cpu().numpy(), buf.nsel.cpu().numpy()
    exact = check_selection(case, gsel, gnsel, ref)
    # attention with the oracle's selection
    out = gpu_decode(case, buf, ref["sel"], ref["nsel"])
    assert int(buf.error_flags.item()) == 0
    check_out(case, out, ref["out"])
    check_fused_step(case, buf, ref, exact)


def test_empty_request_gives_zero_output():
    case = CASES["short-and-empty"]()
    buf = gpu_select(case)
    out = gpu_decode(case, buf, buf.sel.cpu().numpy(), buf.nsel.cpu().numpy())
    assert np.all(out[2] == 0)


def test_output_is_deterministic_and_page_order_invariant():
    case = synth.llama8b_layer(seq_len=20000, device=DEV, shuffle=False, seed=31)
    buf = gpu_select(case)
    sel, nsel = buf.sel.cpu().numpy(), buf.nsel.cpu().numpy()
    a = gpu_decode(case, buf, sel, nsel).copy()
    b = gpu_decode(case, buf, sel, nsel).copy()
    assert np.array_equal(a, b)
    # the same logical cache on a permuted set of physical pages
    perm = torch.randperm(case.num_pages, generator=torch.Generator().manual_seed(5))
    k2 = torch.empty_like(case.k_cache)
    v2 = torch.empty_like(case.v_cache)
    k2[perm.to(DEV)] = case.k_cache
    v2[perm.to(DEV)] = case.v_cache
    bt = case.block_table.clone()
    ok = bt >= 0
    bt[ok] = perm.to(DEV).to(torch.int32)[bt[ok].long()]
    moved = synth.Case(cfg=case.cfg, q=case.q, k_cache=k2, v_cache=v2, block_table=bt,
                       seq_lens=case.seq_lens, prompt_lens=case.prompt_lens,
                       page_ids=perm.to(DEV).to(torch.int32)[case.page_ids.long()],
                       page_valid=case.page_valid)
    buf2 = gpu_select(moved)
    assert np.array_equal(buf2.sel.cpu().numpy(), sel)
    c = gpu_decode(moved, buf2, sel, nsel)
    assert np.array_equal(a, c)


def test_one_kernel_output_is_reproducible_when_the_release_carries_every_kept_block():
    """The one-kernel path assigns each streaming CTA's first 16 kept blocks with the release:
    with k = 90 and 11 streaming CTAs per unit every kept block is assigned that way, so the
    output is bitwise the same on every call."""
    case = synth.llama8b_layer(device=DEV, seed=33)
    assert srkv.retrieval_decode_launches(case.cfg, case.batch, case.max_blocks) == 1
    reps = gpu_select(case).reps
    outs = []
    for _ in range(3):
        b = srkv.DecodeBuffers(case.cfg, case.batch, case.max_blocks, case.num_pages,
                               device=DEV)
        b.reps.copy_(reps)
        srkv.retrieval_decode(case.cfg, case.q, case.k_cache, case.v_cache, b.reps,
                              case.block_table, case.seq_lens, case.prompt_lens, b.sel, b.nsel,
                              b.out, b.workspace, b.error_flags)
        torch.cuda.synchronize()
        assert int(b.error_flags.item()) == 0
        assert int(b.nsel.max().item()) <= 16 * 11
        outs.append(b.out.clone())
    assert torch.equal(outs[0], outs[1]) and torch.equal(outs[0], outs[2])


# ---- device-side checks: bad inputs are skipped and flagged, never faulted -----------------

def test_bad_page_ids_are_flagged():
    case = synth.llama8b_layer(seq_len=12000, device=DEV, local_tokens=2048, seed=41)
    buf = gpu_select(case)
    bt = case.block_table.clone()
    bt[0, 20] = case.num_pages + 5          # a selected-or-candidate block
    bt[0, 0] = -7                           # an init block
    bad = synth.Case(**{**case.__dict__, "block_table": bt})
    buf.error_flags.zero_()
    srkv.score_topk(case.cfg, case.q, buf.reps, bt, case.seq_lens, case.prompt_lens, buf.sel,
                    buf.nsel, buf.error_flags)
    gpu_decode(bad, buf, buf.sel.cpu().numpy(), buf.nsel.cpu().numpy())
    assert int(buf.error_flags.item()) & srkv.EFLAG_PAGE_RANGE


def test_bad_lengths_and_selection_are_flagged():
    case = synth.llama8b_layer(seq_len=12000, device=DEV, local_tokens=2048, seed=42)
    buf = gpu_select(case)
    sel = buf.sel.cpu().numpy()
    nsel = buf.nsel.cpu().numpy()
    # nsel beyond kmax, entries that are not candidates, a descending pair
    nsel2 = nsel.copy()
    nsel2[0, 0] = buf.kmax + 3
    sel2 = sel.copy()
    sel2[0, 1, 0] = 10 ** 6
    sel2[0, 2, :2] = sel2[0, 2, 1::-1]
    buf.error_flags.zero_()
    gpu_decode(case, buf, sel2, nsel2)
    assert int(buf.error_flags.item()) & srkv.EFLAG_SELECTION
    long = synth.Case(**{**case.__dict__,
                         "seq_lens": torch.tensor([10 ** 7], dtype=torch.int32, device=DEV)})
    buf.error_flags.zero_()
    gpu_decode(long, buf, sel, nsel)
    assert int(buf.error_flags.item()) & srkv.EFLAG_SEQ_LEN


# ---- full-size workloads, sampled units ---------------------------------------------------

def sampled_units(case, n, seed):
    rng = np.random.default_rng(seed)
    Hkv = case.cfg["num_kv_heads"]
    picks = rng.choice(case.batch * Hkv, size=min(n, case.batch * Hkv), replace=False)
    return [(int(u) // Hkv, int(u) % Hkv) for u in sorted(picks)]


FULL = {
    "llama8b-65536": lambda: synth.llama8b_layer(device=DEV),
    "ragged-16x[32768,131072]": lambda: synth.ragged_batch(device=DEV),
    "dense-vs-sparse-4x131072-p0.2": lambda: synth.dense_vs_sparse(0.2, device=DEV),
    "dense-vs-sparse-4x131072-p1.0": lambda: synth.dense_vs_sparse(1.0, device=DEV),
    "prefix-shared-64": lambda: synth.prefix_shared(device=DEV),
}


@pytest.mark.parametrize("name", list(FULL))
def test_full_size_sampled(name):
    case = FULL[name]()
    buf = gpu_select(case)
    assert int(buf.error_flags.item()) == 0
    units = None if name == "llama8b-65536" else sampled_units(case, 6, seed=len(name))
    arr = synth.to_oracle_arrays(case)
    ref = oracle_ref(case, arr, units=units, kmax=buf.kmax, threads=16)
    exact = check_selection(case, buf.sel.cpu().numpy(), buf.nsel.cpu().numpy(), ref, units)
    out = gpu_decode(case, buf, ref["sel"], ref["nsel"])
    check_out(case, out, ref["out"], units)
    assert int(buf.error_flags.item()) == 0
    assert exact >= 1
    assert check_fused_step(case, buf, ref, exact, units) >= 1


def test_retrieval_decode_paths():
    """One kernel for a batch whose clusters are all resident (clusters of 4 for up to 36
    units at a top-k ratio <= 0.3; clusters of 8 or more for up to 15 units at any ratio),
    three otherwise."""
    small = synth.llama8b_layer(seq_len=16384, device=DEV)
    two = synth.ragged_batch(n_requests=2, lo=9000, hi=20000, device=DEV)  # 16 units
    mid = synth.ragged_batch(n_requests=4, lo=9000, hi=20000, device=DEV)  # 32 units
    big = synth.ragged_batch(n_requests=5, lo=9000, hi=20000, device=DEV)  # 40 units
    assert srkv.retrieval_decode_launches(small.cfg, small.batch, small.max_blocks) == 1
    assert srkv.retrieval_decode_launches(two.cfg, two.batch, two.max_blocks) == 1
    assert srkv.retrieval_decode_launches(dict(two.cfg, topk_percent=0.4), two.batch,
                                          two.max_blocks) == 3
    assert srkv.retrieval_decode_launches(mid.cfg, mid.batch, mid.max_blocks) == 1
    wide = dict(mid.cfg, topk_percent=0.4)
    assert srkv.retrieval_decode_launches(wide, mid.batch, mid.max_blocks) == 3
    assert srkv.retrieval_decode_launches(big.cfg, big.batch, big.max_blocks) == 3
    f32 = CASES["f32-d128"]()
    assert srkv.retrieval_decode_launches(f32.cfg, f32.batch, f32.max_blocks) == 3
