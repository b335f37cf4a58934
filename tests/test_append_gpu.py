"""Decode-time maintenance through the C ABI: srkv_append_kv writes each request's new token
into its page and keeps that page's representation vector equal to a fresh build; a decode
step after a run of appends matches the oracle on the grown cache."""
import numpy as np
import pytest
import torch

import oracle
from block_sparse_retrieval_gb300 import srkv, synth
from parity import check_out, check_selection, oracle_ref

pytestmark = pytest.mark.gpu
DEV = "cuda"


def grown_case(dtype, head_dim, n_new, seed):
    # pages for the final lengths exist; the run starts n_new tokens earlier
    final = [9000 + n_new - 9000 % 128 + 120, 5000]  # request 0 crosses a page boundary
    case = synth.make_case(seq_lens=final, num_q_heads=8, num_kv_heads=2, head_dim=head_dim,
                           dtype=dtype, init_tokens=1024, local_tokens=2048, topk_percent=0.2,
                           dense_boundary=0, seed=seed, device=DEV)
    return case, case.seq_lens - n_new


@pytest.mark.parametrize("dtype,head_dim", [(synth.BF16, 128), (synth.F32, 64)])
def test_append_writes_rows_and_keeps_reps_current(dtype, head_dim):
    n_new = 24
    case, lens = grown_case(dtype, head_dim, n_new, seed=61)
    cfg, B, Hkv = case.cfg, case.batch, case.cfg["num_kv_heads"]
    buf = srkv.DecodeBuffers(cfg, B, case.max_blocks, case.num_pages, device=DEV)
    k_ref, v_ref = case.k_cache.clone(), case.v_cache.clone()
    g = torch.Generator(device=DEV).manual_seed(7)
    touched = set()
    bt = case.block_table.cpu().numpy()
    for _ in range(n_new):
        kn = torch.randn(B, Hkv, head_dim, generator=g, device=DEV).to(case.k_cache.dtype)
        vn = torch.randn(B, Hkv, head_dim, generator=g, device=DEV).to(case.k_cache.dtype)
        srkv.append_kv(cfg, kn, vn, case.k_cache, case.v_cache, case.block_table, lens,
                       buf.reps, buf.error_flags)
        L = lens.cpu().numpy()
        for r in range(B):
            page = int(bt[r, L[r] // 128])
            k_ref[page, :, L[r] % 128] = kn[r]
            v_ref[page, :, L[r] % 128] = vn[r]
            touched.add((page, int(L[r]) % 128 + 1, r))
        lens += 1
    torch.cuda.synchronize()
    assert int(buf.error_flags.item()) == 0
    assert torch.equal(case.k_cache, k_ref) and torch.equal(case.v_cache, v_ref)
    # every touched page's vector equals a fresh build over its rows so far (latest count)
    latest = {}
    for page, valid, r in touched:
        latest[page] = max(latest.get(page, 0), valid)
    pages = torch.tensor(sorted(latest), dtype=torch.int32, device=DEV)
    valid = torch.tensor([latest[p] for p in sorted(latest)], dtype=torch.int32, device=DEV)
    fresh = torch.zeros_like(buf.reps)
    srkv.build_block_reps(cfg, case.k_cache, pages, valid, fresh)
    torch.cuda.synchronize()
    assert torch.equal(buf.reps[pages.long()], fresh[pages.long()])


def test_decode_after_appends_matches_the_oracle():
    n_new = 40
    case, lens = grown_case(synth.BF16, 128, n_new, seed=62)
    cfg, B, Hkv = case.cfg, case.batch, case.cfg["num_kv_heads"]
    buf = srkv.DecodeBuffers(cfg, B, case.max_blocks, case.num_pages, device=DEV)
    # vectors of the prefix as prefill leaves them, then token by token
    L0 = lens.cpu().numpy()
    ids, valid = [], []
    bt = case.block_table.cpu().numpy()
    for r in range(B):
        for b in range((int(L0[r]) + 127) // 128):
            ids.append(int(bt[r, b]))
            valid.append(min(128, int(L0[r]) - b * 128))
    srkv.build_block_reps(cfg, case.k_cache, torch.tensor(ids, dtype=torch.int32, device=DEV),
                          torch.tensor(valid, dtype=torch.int32, device=DEV), buf.reps)
    g = torch.Generator(device=DEV).manual_seed(9)
    for _ in range(n_new):
        kn = torch.randn(B, Hkv, 128, generator=g, device=DEV).to(torch.bfloat16)
        vn = torch.randn(B, Hkv, 128, generator=g, device=DEV).to(torch.bfloat16)
        srkv.append_kv(cfg, kn, vn, case.k_cache, case.v_cache, case.block_table, lens,
                       buf.reps, buf.error_flags)
        lens += 1
    grown = synth.Case(**{**case.__dict__, "seq_lens": lens, "prompt_lens": lens.clone()})
    srkv.retrieval_decode(cfg, grown.q, grown.k_cache, grown.v_cache, buf.reps,
                          grown.block_table, grown.seq_lens, grown.prompt_lens, buf.sel,
                          buf.nsel, buf.out, buf.workspace, buf.error_flags)
    torch.cuda.synchronize()
    assert int(buf.error_flags.item()) == 0
    ref = oracle_ref(grown, kmax=buf.kmax)
    exact = check_selection(grown, buf.sel.cpu().numpy(), buf.nsel.cpu().numpy(), ref)
    if exact == B * Hkv:
        check_out(grown, buf.out.float().cpu().numpy(), ref["out"])


def test_append_beyond_the_table_is_flagged_and_writes_nothing():
    case = synth.make_case(seq_lens=[256], num_q_heads=8, num_kv_heads=2, head_dim=128,
                           init_tokens=0, local_tokens=128, dense_boundary=0, seed=63,
                           device=DEV)
    buf = srkv.DecodeBuffers(case.cfg, 1, case.max_blocks, case.num_pages, device=DEV)
    before = case.k_cache.clone()
    kn = torch.ones(1, 2, 128, dtype=torch.bfloat16, device=DEV)
    full = torch.tensor([case.max_blocks * 128], dtype=torch.int32, device=DEV)
    srkv.append_kv(case.cfg, kn, kn, case.k_cache, case.v_cache, case.block_table, full,
                   buf.reps, buf.error_flags)
    torch.cuda.synchronize()
    assert int(buf.error_flags.item()) & srkv.EFLAG_SEQ_LEN
    assert torch.equal(case.k_cache, before)
