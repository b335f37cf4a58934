"""Helpers for the GPU parity tests: run the library on a synthetic case and compare with
the oracle under the rules of the method's statement:

  * selected block ids equal the oracle's exactly wherever the top-k boundary gap
    (s_(k) - s_(k+1)) / max_b |s_b| exceeds 1e-4; inside that band any selection that is a
    valid top-k within the band is accepted (scores are fp32 on the GPU, fp64 in the oracle);
  * attention outputs are compared with the oracle's own selection fed to the GPU decode:
    |gpu - oracle| <= 2e-2 + 1e-2 |oracle| for bf16 inputs, 1e-5 + 1e-5 |oracle| for fp32;
    bf16 outputs must also meet a tighter bound set by the GPU arithmetic (TIGHT_TOL).
"""
from __future__ import annotations

import os

import numpy as np
import torch

import oracle
from block_sparse_retrieval_gb300 import srkv, synth

GAP = 1e-4
TOL = {synth.BF16: (2e-2, 1e-2), synth.F32: (1e-5, 1e-5)}
# The method's bf16 tolerance is loose against the size of an attention output over many
# tokens: on a 16384-token layer the outputs are ~1e-2, and dropping a whole kept block moves
# them by ~3e-3, a sixth of it.  So bf16 outputs must also meet a bound set by the GPU's
# arithmetic: fp32 sums, softmax weights entering the P.V products as 16-bit values (each
# within 2^-8 relative, independent roundings that average out over the tokens) and one
# rounding of the output to bf16 (within 2^-8 relative).  Emulating those roundings on the
# parity cases gives errors of ~1e-4 to 2e-3, at most 0.4 of this bound, which a lost block
# exceeds.
TIGHT_TOL = {synth.BF16: (2e-3, 1e-2), synth.F32: (1e-5, 1e-5)}
ORACLE_KEYS = ("q", "k_cache", "v_cache", "block_table", "seq_lens", "prompt_lens")


def gpu_select(case, buf=None):
    cfg = case.cfg
    buf = buf or srkv.DecodeBuffers(cfg, case.batch, case.max_blocks, case.num_pages,
                                    device=case.q.device)
    srkv.build_block_reps(cfg, case.k_cache, case.page_ids, case.page_valid, buf.reps,
                          buf.error_flags)
    srkv.score_topk(cfg, case.q, buf.reps, case.block_table, case.seq_lens, case.prompt_lens,
                    buf.sel, buf.nsel, buf.error_flags)
    torch.cuda.synchronize()
    return buf


def gpu_decode(case, buf, sel: np.ndarray, nsel: np.ndarray) -> np.ndarray:
    dev = case.q.device
    kmax = buf.kmax
    s = np.full((case.batch, case.cfg["num_kv_heads"], kmax), -1, np.int32)
    s[:, :, :min(kmax, sel.shape[2])] = sel[:, :, :kmax]
    srkv.sparse_paged_decode(case.cfg, case.q, case.k_cache, case.v_cache, case.block_table,
                             case.seq_lens, torch.from_numpy(s).to(dev),
                             torch.from_numpy(np.ascontiguousarray(nsel)).to(dev), buf.out,
                             buf.workspace, buf.error_flags)
    torch.cuda.synchronize()
    return buf.out.float().cpu().numpy()


def oracle_ref(case, arr=None, units=None, kmax=None, threads=8):
    arr = arr or synth.to_oracle_arrays(case)
    return oracle.decode(case.cfg, *[arr[k] for k in ORACLE_KEYS], units=units, kmax=kmax,
                         threads=threads)


def check_selection(case, gpu_sel: np.ndarray, gpu_nsel: np.ndarray, ref: dict, units=None):
    """Returns the number of units compared exactly (gap above the threshold)."""
    B, Hkv = gpu_nsel.shape
    units = units or [(r, h) for r in range(B) for h in range(Hkv)]
    exact = 0
    for r, h in units:
        k = int(ref["nsel"][r, h])
        assert int(gpu_nsel[r, h]) == k, (r, h, int(gpu_nsel[r, h]), k)
        want = ref["sel"][r, h, :k]
        got = gpu_sel[r, h, :k]
        scores = ref["scores"][r, h]
        cand = np.flatnonzero(~np.isnan(scores))
        n = cand.size
        if k == 0 or k == n:
            assert np.array_equal(got, want), (r, h)
            exact += 1
            continue
        s_sorted = np.sort(scores[cand])[::-1]
        scale = max(np.abs(scores[cand]).max(), 1e-300)
        gap = (s_sorted[k - 1] - s_sorted[k]) / scale
        if gap > GAP:
            assert np.array_equal(got, want), (r, h, gap)
            exact += 1
        else:
            assert np.all(np.diff(got) > 0), (r, h)
            assert np.all(~np.isnan(scores[got])), (r, h)
            band = GAP * scale
            assert scores[got].min() >= s_sorted[k - 1] - band, (r, h)
            assert np.all(np.isin(cand[scores[cand] > s_sorted[k - 1] + band], got)), (r, h)
    return exact


# Two GPU decode paths over the same selection differ only in how the attended pages are
# split into partials (fp32 sums in another order) and in the rounding of the output: a few
# units in the last place of the output's dtype.  Much tighter than the method's tolerance
# against the oracle, so that a lost or doubled partial (an error of the size of the output
# itself, ~1e-2 here) cannot hide inside it.
SAME_TOL = {synth.BF16: (1e-3, 1e-2), synth.F32: (1e-6, 1e-5)}


def check_same(case, got: np.ndarray, want: np.ndarray):
    atol, rtol = SAME_TOL[case.cfg["dtype"]]
    err = np.abs(got - want)
    bad = err > atol + rtol * np.abs(want)
    assert not bad.any(), f"{bad.sum()} elements off between paths, max err {err.max():.3e}"
    return float(err.max())


def check_out(case, got: np.ndarray, want: np.ndarray, units=None):
    atol, rtol = TOL[case.cfg["dtype"]]
    G = case.cfg["num_q_heads"] // case.cfg["num_kv_heads"]
    if units is None:
        g, w = got, want
    else:
        heads = [(r, h * G + j) for r, h in units for j in range(G)]
        g = np.stack([got[r, qh] for r, qh in heads])
        w = np.stack([want[r, qh] for r, qh in heads])
    err = np.abs(g - w)
    bad = err > atol + rtol * np.abs(w)
    assert not bad.any(), f"{bad.sum()} elements off, max err {err.max():.3e}"
    tatol, trtol = TIGHT_TOL[case.cfg["dtype"]]
    ratio = float((err / (tatol + trtol * np.abs(w))).max()) if err.size else 0.0
    if os.environ.get("SRKV_PARITY_VERBOSE"):
        print(f"[parity] {case.name}: max err {err.max() if err.size else 0.0:.3e}, "
              f"{ratio:.3f} of the arithmetic bound")
    assert ratio <= 1.0, f"max err {err.max():.3e} is {ratio:.2f} x the arithmetic bound"
    return float(err.max())


def check_fused_step(case, buf, ref, exact_score_topk, units=None):
    """srkv_retrieval_decode (scoring, then the decode behind it) against the oracle."""
    fused = srkv.DecodeBuffers(case.cfg, case.batch, case.max_blocks, case.num_pages,
                               device=case.q.device)
    fused.reps.copy_(buf.reps)
    srkv.retrieval_decode(case.cfg, case.q, case.k_cache, case.v_cache, fused.reps,
                          case.block_table, case.seq_lens, case.prompt_lens, fused.sel,
                          fused.nsel, fused.out, fused.workspace, fused.error_flags)
    torch.cuda.synchronize()
    assert int(fused.error_flags.item()) == 0
    fsel, fnsel = fused.sel.cpu().numpy(), fused.nsel.cpu().numpy()
    exact = check_selection(case, fsel, fnsel, ref, units)
    got = fused.out.float().cpu().numpy()
    # The split decode fed the fused selection computes the same sums, but the fused call
    # spreads the initial and window pages over fewer CTAs (the scoring CTAs hold the other
    # SMs), so the partials split at other pages: equal up to rounding, not to the bit.
    again = gpu_decode(case, buf, fsel, fnsel)
    check_same(case, got, again)
    n_units = len(units) if units else case.batch * case.cfg["num_kv_heads"]
    if exact == n_units:
        check_out(case, got, ref["out"], units)
    return exact
