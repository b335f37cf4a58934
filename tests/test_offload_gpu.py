"""GPU parity of the offload tier (openGauss page, "Overall Solution": blocks past the offload
boundary live off the accelerator, their representation vectors stay resident, and only the
topK blocks are fetched): srkv_retrieval_decode_tiered with pages in a pinned host pool
against srkv_retrieval_decode on the same pages in device memory, and against the oracle.
"""
import ctypes

import numpy as np
import pytest
import torch

from block_sparse_retrieval_gb300 import srkv, synth
from parity import check_out, check_same, check_selection, gpu_select, oracle_ref

pytestmark = pytest.mark.gpu

DEV = "cuda"
INVALID_ARG, UNSUPPORTED = 1, 2  # srkv_status values


def candidate_pages(case) -> np.ndarray:
    """Physical pages that hold only offload-range tokens of some request: blocks b with
    INIT <= b*S and (b+1)*S <= L - LOCAL (the pages the method moves off the device)."""
    cfg = case.cfg
    S = 128
    bt = case.block_table.cpu().numpy()
    out = np.zeros(case.num_pages, bool)
    for r, L in enumerate(case.seq_lens.cpu().numpy()):
        W = int(L) - cfg["local_tokens"]
        for b in range(-(-cfg["init_tokens"] // S), max(W, 0) // S):
            if bt[r, b] >= 0:
                out[bt[r, b]] = True
    return out


def split_pools(case, reps: torch.Tensor, to_host: np.ndarray):
    """The same logical cache with the pages marked `to_host` in a pinned host pool: device
    pool first (ids 0..), host pool after it; block table and vectors renumbered."""
    P = case.num_pages
    dev_ids = np.nonzero(~to_host)[0]
    host_ids = np.nonzero(to_host)[0]
    new_id = np.empty(P, np.int64)
    new_id[dev_ids] = np.arange(len(dev_ids))
    new_id[host_ids] = len(dev_ids) + np.arange(len(host_ids))
    d_idx = torch.from_numpy(dev_ids).to(DEV)
    h_idx = torch.from_numpy(host_ids).to(DEV)
    k_dev = case.k_cache[d_idx].contiguous()
    v_dev = case.v_cache[d_idx].contiguous()
    k_host = case.k_cache[h_idx].cpu().contiguous().pin_memory()
    v_host = case.v_cache[h_idx].cpu().contiguous().pin_memory()
    reps2 = torch.empty_like(reps)
    reps2[torch.from_numpy(new_id).to(DEV)] = reps
    bt = case.block_table.cpu().numpy().copy()
    ok = bt >= 0
    bt[ok] = new_id[bt[ok]]
    return k_dev, v_dev, k_host, v_host, reps2, torch.from_numpy(bt).to(DEV)


def run_both(case, to_host):
    """(all-device call, tiered call) buffers on the same logical cache."""
    base = gpu_select(case)
    dev = srkv.DecodeBuffers(case.cfg, case.batch, case.max_blocks, case.num_pages, device=DEV)
    dev.reps.copy_(base.reps)
    srkv.retrieval_decode(case.cfg, case.q, case.k_cache, case.v_cache, dev.reps,
                          case.block_table, case.seq_lens, case.prompt_lens, dev.sel, dev.nsel,
                          dev.out, dev.workspace, dev.error_flags)
    k_dev, v_dev, k_host, v_host, reps2, bt2 = split_pools(case, base.reps, to_host)
    tie = srkv.DecodeBuffers(case.cfg, case.batch, case.max_blocks, case.num_pages, device=DEV)
    tie.reps.copy_(reps2)
    srkv.retrieval_decode_tiered(case.cfg, case.q, k_dev, v_dev, k_host, v_host, tie.reps, bt2,
                                 case.seq_lens, case.prompt_lens, tie.sel, tie.nsel, tie.out,
                                 tie.workspace, tie.error_flags)
    torch.cuda.synchronize()
    assert int(dev.error_flags.item()) == 0
    assert int(tie.error_flags.item()) == 0
    return dev, tie


CASES = {
    # one kernel (8 units), d 128
    "llama8b-16k": lambda: synth.llama8b_layer(seq_len=16384, device=DEV, seed=51),
    # scoring + split decode + combine (32 units)
    "ragged-4": lambda: synth.ragged_batch(n_requests=4, lo=9000, hi=20000, device=DEV, seed=52),
    # one kernel, d 64, group 8
    "g8-d64": lambda: synth.make_case(seq_lens=[5000, 3000], num_q_heads=16, num_kv_heads=2,
                                      head_dim=64, init_tokens=300, local_tokens=1000,
                                      topk_percent=0.3, dense_boundary=0, seed=53, device=DEV),
}


@pytest.mark.parametrize("name", list(CASES))
def test_offloaded_candidates_match_device_pages(name):
    case = CASES[name]()
    to_host = candidate_pages(case)
    assert to_host.sum() > 0
    dev, tie = run_both(case, to_host)
    # the selection is a function of the vectors alone: identical
    assert np.array_equal(dev.nsel.cpu().numpy(), tie.nsel.cpu().numpy())
    assert np.array_equal(dev.sel.cpu().numpy(), tie.sel.cpu().numpy())
    got = tie.out.float().cpu().numpy()
    want = dev.out.float().cpu().numpy()
    units = case.batch * case.cfg["num_kv_heads"]
    if srkv.retrieval_decode_launches(case.cfg, case.batch, case.max_blocks) == 3:
        # the split decode partitions the pages statically: the same sums in the same order
        assert np.array_equal(got, want)
    else:
        # one kernel: CTAs take kept blocks from a shared pool, so the partials' split
        # depends on timing; equal up to rounding
        check_same(case, got, want)
    ref = oracle_ref(case, kmax=dev.kmax)
    exact = check_selection(case, tie.sel.cpu().numpy(), tie.nsel.cpu().numpy(), ref)
    if exact == units:
        check_out(case, got, ref["out"])


def test_random_pages_on_host_including_window():
    """Any page may live in the host pool, also initial and window pages (list A)."""
    case = synth.llama8b_layer(seq_len=16384, device=DEV, seed=54)
    to_host = np.random.default_rng(3).random(case.num_pages) < 0.5
    dev, tie = run_both(case, to_host)
    assert np.array_equal(dev.sel.cpu().numpy(), tie.sel.cpu().numpy())
    check_same(case, tie.out.float().cpu().numpy(), dev.out.float().cpu().numpy())


def test_all_pages_on_host_split_path():
    case = synth.ragged_batch(n_requests=5, lo=6000, hi=12000, device=DEV, seed=55)  # 40 units
    to_host = np.ones(case.num_pages, bool)
    to_host[0] = False  # the device pool is never empty
    dev, tie = run_both(case, to_host)
    assert np.array_equal(dev.sel.cpu().numpy(), tie.sel.cpu().numpy())
    if srkv.retrieval_decode_launches(case.cfg, case.batch, case.max_blocks) == 3:
        assert np.array_equal(tie.out.float().cpu().numpy(), dev.out.float().cpu().numpy())
    else:
        check_same(case, tie.out.float().cpu().numpy(), dev.out.float().cpu().numpy())


def test_host_pool_arguments_are_checked():
    case = synth.llama8b_layer(seq_len=12000, device=DEV, seed=56)
    buf = gpu_select(case)
    lib = srkv.load()
    c = srkv.config(case.cfg)
    pageable = np.zeros(case.k_cache[:1].numel(), np.uint16)  # ordinary (pageable) memory
    p = ctypes.c_void_p(pageable.ctypes.data)

    def call(cfg, kh, vh, n_host):
        return lib.srkv_retrieval_decode_tiered(
            ctypes.byref(cfg), ctypes.c_void_p(case.q.data_ptr()),
            ctypes.c_void_p(case.k_cache.data_ptr()), ctypes.c_void_p(case.v_cache.data_ptr()),
            case.num_pages, kh, vh, n_host, ctypes.c_void_p(buf.reps.data_ptr()),
            ctypes.c_void_p(case.block_table.data_ptr()), case.max_blocks,
            ctypes.c_void_p(case.seq_lens.data_ptr()), None, case.batch,
            ctypes.c_void_p(buf.sel.data_ptr()), buf.kmax, ctypes.c_void_p(buf.nsel.data_ptr()),
            ctypes.c_void_p(buf.out.data_ptr()), ctypes.c_void_p(buf.workspace.data_ptr()),
            buf.workspace.numel(), None, None)

    assert call(c, p, p, 1) == INVALID_ARG          # pageable host memory
    assert call(c, None, None, 1) == INVALID_ARG    # missing pool
    assert call(c, None, None, -1) == INVALID_ARG   # negative size
    f32 = dict(case.cfg, dtype=synth.F32)
    pinned = torch.zeros(8, dtype=torch.int32).pin_memory()
    pp = ctypes.c_void_p(pinned.data_ptr())
    assert call(srkv.config(f32), pp, pp, 1) == UNSUPPORTED  # needs the bf16 decode
    with pytest.raises(ValueError):
        srkv.retrieval_decode_tiered(case.cfg, case.q, case.k_cache, case.v_cache,
                                     case.k_cache[:1].cpu(), case.v_cache[:1].cpu(), buf.reps,
                                     case.block_table, case.seq_lens, None, buf.sel, buf.nsel,
                                     buf.out, buf.workspace)
