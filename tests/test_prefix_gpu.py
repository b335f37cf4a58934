"""GPU parity of the shared-prefix calls (cascade attention over a prefix of pages every
request of the batch maps to the same physical pages) through the C ABI.

* srkv_sparse_paged_decode_prefix, fed the oracle's selection, against the oracle on every
  unit (the method's tolerance), and against srkv_sparse_paged_decode on the same selection
  (the tight same-sums tolerance: only the split into partials differs);
* srkv_retrieval_decode_prefix against srkv_retrieval_decode: the same selection to the bit,
  outputs within the same-sums tolerance, and bitwise equal on a second call;
* query groups of 8, 4, 2 and 1 heads, a batch that is not a multiple of the requests an
  item takes, requests whose length ends inside or at the end of the prefix, a dense
  request, a declared prefix shorter than the shared one, and a block table that breaks the
  contract (flagged);
* the full 64-request workload (16384 shared tokens) on sampled units against the oracle and
  on every unit against the plain call.
"""
import numpy as np
import pytest
import torch

from block_sparse_retrieval_gb300 import srkv, synth
from parity import check_out, check_same, check_selection, gpu_decode, gpu_select, oracle_ref

pytestmark = pytest.mark.gpu

DEV = "cuda"
S = 128


def prefix_case(name):
    mk = synth.make_case
    return {
        # 8 requests, 64/8 heads (group 8), 32 shared blocks
        "g8": lambda: synth.prefix_shared(n_requests=8, prefix=4096, lo=1024, hi=4096,
                                          local_tokens=2048, device=DEV),
        # 19 requests of group 4 (one partial item of 32 requests), window inside the prefix
        "g4-19": lambda: mk(seq_lens=[3072 + 97 * i for i in range(19)], num_q_heads=16,
                            num_kv_heads=4, head_dim=128, init_tokens=512, local_tokens=1024,
                            topk_percent=0.25, dense_boundary=0, shared_prefix_tokens=3072,
                            seed=101, device=DEV),
        # group 2: a request that ends exactly at the prefix, one a token past it, a dense one
        "g2-edges": lambda: mk(seq_lens=[2048, 2049, 5000, 2048 + 700, 7000],
                               prompt_lens=[2048, 2049, 5000, 2748, 2000], num_q_heads=8,
                               num_kv_heads=4, head_dim=128, init_tokens=300, local_tokens=900,
                               topk_percent=0.3, dense_boundary=2040, shared_prefix_tokens=2048,
                               seed=102, device=DEV),
        # group 1: 150 requests, two items of 128
        "g1-150": lambda: mk(seq_lens=[1024 + 11 * i for i in range(150)], num_q_heads=2,
                             num_kv_heads=2, head_dim=128, init_tokens=256, local_tokens=512,
                             topk_percent=0.2, dense_boundary=0, shared_prefix_tokens=1024,
                             seed=103, device=DEV),
    }[name]()


def shared_blocks(case):
    """Leading logical blocks every request maps to the same page (whole pages only)."""
    bt = case.block_table.cpu().numpy()
    L = case.seq_lens.cpu().numpy()
    n = 0
    while n < bt.shape[1] and all(n < L[r] // S for r in range(case.batch)) and \
            np.all(bt[:, n] == bt[0, n]):
        n += 1
    return n


def decode_prefix(case, buf, sel, nsel, prefix_blocks):
    s = np.full((case.batch, case.cfg["num_kv_heads"], buf.kmax), -1, np.int32)
    s[:, :, :min(buf.kmax, sel.shape[2])] = sel[:, :, :buf.kmax]
    out = torch.full_like(buf.out, float("nan"))
    buf.error_flags.zero_()
    srkv.sparse_paged_decode_prefix(case.cfg, case.q, case.k_cache, case.v_cache,
                                    case.block_table, case.seq_lens, prefix_blocks,
                                    torch.from_numpy(s).to(DEV),
                                    torch.from_numpy(np.ascontiguousarray(nsel)).to(DEV), out,
                                    buf.workspace, buf.error_flags)
    torch.cuda.synchronize()
    return out.float().cpu().numpy()


def retrieval(case, reps, prefix_blocks):
    buf = srkv.DecodeBuffers(case.cfg, case.batch, case.max_blocks, case.num_pages, device=DEV,
                             prefix=True)
    buf.reps.copy_(reps)
    if prefix_blocks is None:
        srkv.retrieval_decode(case.cfg, case.q, case.k_cache, case.v_cache, buf.reps,
                              case.block_table, case.seq_lens, case.prompt_lens, buf.sel,
                              buf.nsel, buf.out, buf.workspace, buf.error_flags)
    else:
        srkv.retrieval_decode_prefix(case.cfg, case.q, case.k_cache, case.v_cache, buf.reps,
                                     case.block_table, case.seq_lens, case.prompt_lens,
                                     prefix_blocks, buf.sel, buf.nsel, buf.out, buf.workspace,
                                     buf.error_flags)
    torch.cuda.synchronize()
    assert int(buf.error_flags.item()) == 0
    return buf


@pytest.mark.parametrize("name", ["g8", "g4-19", "g2-edges", "g1-150"])
def test_prefix_decode_matches_the_oracle_and_the_plain_decode(name):
    case = prefix_case(name)
    ps = shared_blocks(case)
    assert ps >= 8
    buf = srkv.DecodeBuffers(case.cfg, case.batch, case.max_blocks, case.num_pages, device=DEV,
                             prefix=True)
    gpu_select(case, buf)
    assert int(buf.error_flags.item()) == 0
    ref = oracle_ref(case, kmax=buf.kmax)
    got = decode_prefix(case, buf, ref["sel"], ref["nsel"], ps)
    assert int(buf.error_flags.item()) == 0
    check_out(case, got, ref["out"])
    plain = gpu_decode(case, buf, ref["sel"], ref["nsel"])
    check_same(case, got, plain)
    # a declared prefix shorter than the shared one: the rest goes through the split decode
    half = decode_prefix(case, buf, ref["sel"], ref["nsel"], ps // 2)
    assert int(buf.error_flags.item()) == 0
    check_same(case, half, plain)
    # no prefix: the plain call's result
    none = decode_prefix(case, buf, ref["sel"], ref["nsel"], 0)
    assert np.array_equal(none, plain)


@pytest.mark.parametrize("name", ["g8", "g2-edges"])
def test_retrieval_prefix_selects_the_same_and_is_reproducible(name):
    case = prefix_case(name)
    ps = shared_blocks(case)
    base = gpu_select(case)
    plain = retrieval(case, base.reps, None)
    a = retrieval(case, base.reps, ps)
    b = retrieval(case, base.reps, ps)
    assert np.array_equal(a.nsel.cpu().numpy(), plain.nsel.cpu().numpy())
    assert np.array_equal(a.sel.cpu().numpy(), plain.sel.cpu().numpy())
    check_same(case, a.out.float().cpu().numpy(), plain.out.float().cpu().numpy())
    assert torch.equal(a.out, b.out)
    ref = oracle_ref(case, kmax=a.kmax)
    if check_selection(case, a.sel.cpu().numpy(), a.nsel.cpu().numpy(), ref) == \
            case.batch * case.cfg["num_kv_heads"]:
        check_out(case, a.out.float().cpu().numpy(), ref["out"])


def test_a_table_that_breaks_the_prefix_contract_is_flagged():
    case = prefix_case("g8")
    ps = shared_blocks(case)
    buf = srkv.DecodeBuffers(case.cfg, case.batch, case.max_blocks, case.num_pages, device=DEV,
                             prefix=True)
    gpu_select(case, buf)
    sel, nsel = buf.sel.cpu().numpy(), buf.nsel.cpu().numpy()
    bt = case.block_table.clone()
    bt[3, 5] = bt[3, ps + 1]  # request 3 maps a prefix block elsewhere
    bad = synth.Case(**{**case.__dict__, "block_table": bt})
    decode_prefix(bad, buf, sel, nsel, ps)
    assert int(buf.error_flags.item()) & srkv.EFLAG_PREFIX


def sampled_units(case, n, seed):
    rng = np.random.default_rng(seed)
    Hkv = case.cfg["num_kv_heads"]
    picks = rng.choice(case.batch * Hkv, size=min(n, case.batch * Hkv), replace=False)
    return [(int(u) // Hkv, int(u) % Hkv) for u in sorted(picks)]


def test_full_prefix_shared_workload():
    case = synth.prefix_shared(device=DEV)
    ps = shared_blocks(case)
    assert ps == 16384 // S
    base = gpu_select(case)
    plain = retrieval(case, base.reps, None)
    got = retrieval(case, base.reps, ps)
    assert np.array_equal(got.sel.cpu().numpy(), plain.sel.cpu().numpy())
    check_same(case, got.out.float().cpu().numpy(), plain.out.float().cpu().numpy())
    units = sampled_units(case, 6, seed=5)
    ref = oracle_ref(case, units=units, kmax=got.kmax, threads=16)
    check_selection(case, got.sel.cpu().numpy(), got.nsel.cpu().numpy(), ref, units)
    out = decode_prefix(case, got, ref["sel"], ref["nsel"], ps)
    assert int(got.error_flags.item()) == 0
    check_out(case, out, ref["out"], units)
