"""The Python binding checks tensor shapes against the configuration before anything reaches
the library (which sees only pointers, so a tensor of the wrong shape would be read or
written out of its bounds).  Runs on CPU: with every shape right, a call gets as far as the
device check; with one shape wrong, it stops at the shape check."""
import pytest
import torch

from block_sparse_retrieval_gb300 import srkv

CFG = dict(num_q_heads=8, num_kv_heads=2, head_dim=64, block_size=128, init_tokens=256,
           local_tokens=512, topk_percent=0.2, dense_boundary=0, dtype=srkv.BF16)
B, MAXB, P, KMAX = 3, 10, 24, 4
bf, i32, f32, u8 = torch.bfloat16, torch.int32, torch.float32, torch.uint8


def step_args():
    return dict(q=torch.zeros(B, 8, 64, dtype=bf), k_cache=torch.zeros(P, 2, 128, 64, dtype=bf),
                v_cache=torch.zeros(P, 2, 128, 64, dtype=bf),
                reps=torch.zeros(P, 2, 64, dtype=f32),
                block_table=torch.zeros(B, MAXB, dtype=i32), seq_lens=torch.zeros(B, dtype=i32),
                prompt_lens=torch.zeros(B, dtype=i32), sel=torch.zeros(B, 2, KMAX, dtype=i32),
                nsel=torch.zeros(B, 2, dtype=i32), out=torch.zeros(B, 8, 64, dtype=bf),
                workspace=torch.zeros(256, dtype=u8))


def call_retrieval(**over):
    a = {**step_args(), **over}
    srkv.retrieval_decode(CFG, a["q"], a["k_cache"], a["v_cache"], a["reps"], a["block_table"],
                          a["seq_lens"], a["prompt_lens"], a["sel"], a["nsel"], a["out"],
                          a["workspace"])


def call_sparse(**over):
    a = {**step_args(), **over}
    srkv.sparse_paged_decode(CFG, a["q"], a["k_cache"], a["v_cache"], a["block_table"],
                             a["seq_lens"], a["sel"], a["nsel"], a["out"], a["workspace"])


def call_score(**over):
    a = {**step_args(), **over}
    srkv.score_topk(CFG, a["q"], a["reps"], a["block_table"], a["seq_lens"], a["prompt_lens"],
                    a["sel"], a["nsel"])


def call_noalloc(**over):
    a = {**step_args(), **over}
    srkv.sparse_paged_decode_noalloc(CFG, a["q"], a["k_cache"], a["v_cache"], a["block_table"],
                                     a["seq_lens"], a["sel"], a["nsel"], a["out"])


def call_tiered(**over):
    a = {**step_args(), "k_host": torch.zeros(5, 2, 128, 64, dtype=bf),
         "v_host": torch.zeros(5, 2, 128, 64, dtype=bf),
         "reps": torch.zeros(P + 5, 2, 64, dtype=f32), **over}
    srkv.retrieval_decode_tiered(CFG, a["q"], a["k_cache"], a["v_cache"], a["k_host"],
                                 a["v_host"], a["reps"], a["block_table"], a["seq_lens"],
                                 a["prompt_lens"], a["sel"], a["nsel"], a["out"], a["workspace"])


def call_fp8(**over):
    cfg = dict(CFG, head_dim=128)
    a = {**step_args(), "q": torch.zeros(B, 8, 128, dtype=bf),
         "out": torch.zeros(B, 8, 128, dtype=bf), "reps": torch.zeros(P, 2, 128, dtype=f32),
         "k_fp8": torch.zeros(P, 2, 128, 128, dtype=u8),
         "v_fp8": torch.zeros(P, 2, 128, 128, dtype=u8),
         "k_scale": torch.zeros(P, 2, 128, dtype=f32), "v_scale": torch.zeros(P, 2, 128, dtype=f32),
         **over}
    srkv.retrieval_decode_fp8(cfg, a["q"], a["k_fp8"], a["v_fp8"], a["k_scale"], a["v_scale"],
                              a["reps"], a["block_table"], a["seq_lens"], a["prompt_lens"],
                              a["sel"], a["nsel"], a["out"], a["workspace"])


def call_reps(**over):
    a = {**step_args(), "page_ids": torch.zeros(7, dtype=i32),
         "valid": torch.zeros(7, dtype=i32), **over}
    srkv.build_block_reps(CFG, a["k_cache"], a["page_ids"], a["valid"], a["reps"])


def call_append(**over):
    a = {**step_args(), "k_new": torch.zeros(B, 2, 64, dtype=bf),
         "v_new": torch.zeros(B, 2, 64, dtype=bf), **over}
    srkv.append_kv(CFG, a["k_new"], a["v_new"], a["k_cache"], a["v_cache"], a["block_table"],
                   a["seq_lens"], a["reps"])


def call_quantize(**over):
    a = {**step_args(), "page_ids": torch.zeros(7, dtype=i32),
         "k_fp8": torch.zeros(P, 2, 128, 64, dtype=u8), "v_fp8": torch.zeros(P, 2, 128, 64, dtype=u8),
         "k_scale": torch.zeros(P, 2, 128, dtype=f32), "v_scale": torch.zeros(P, 2, 128, dtype=f32),
         **over}
    srkv.quantize_kv_fp8(CFG, a["k_cache"], a["v_cache"], a["page_ids"], a["k_fp8"], a["v_fp8"],
                         a["k_scale"], a["v_scale"])


def call_sparse_prefix(**over):
    a = {**step_args(), **over}
    srkv.sparse_paged_decode_prefix(CFG, a["q"], a["k_cache"], a["v_cache"], a["block_table"],
                                    a["seq_lens"], 2, a["sel"], a["nsel"], a["out"],
                                    a["workspace"])


def call_retrieval_prefix(**over):
    a = {**step_args(), **over}
    srkv.retrieval_decode_prefix(CFG, a["q"], a["k_cache"], a["v_cache"], a["reps"],
                                 a["block_table"], a["seq_lens"], a["prompt_lens"], 2, a["sel"],
                                 a["nsel"], a["out"], a["workspace"])


def _host_args(over):
    return {**step_args(), "out_host": torch.zeros(B, 8, 64, dtype=bf),
            "staging": torch.zeros(4096, dtype=u8), **over}


def call_host(**over):
    a = _host_args(over)
    srkv.retrieval_decode_host(CFG, a["q"], a["seq_lens"], a["prompt_lens"], a["out_host"],
                               a["staging"], a["k_cache"], a["v_cache"], a["reps"],
                               a["block_table"], a["sel"], a["nsel"], a["out"], a["workspace"])


def call_host_step(**over):
    a = _host_args(over)
    srkv.HostDecodeStep(CFG, a["q"], a["seq_lens"], a["prompt_lens"], a["out_host"],
                        a["staging"], a["k_cache"], a["v_cache"], a["reps"], a["block_table"],
                        a["sel"], a["nsel"], a["out"], a["workspace"])


CALLS = {"retrieval_decode": call_retrieval, "sparse_paged_decode": call_sparse,
         "retrieval_decode_host": call_host, "HostDecodeStep": call_host_step,
         "sparse_paged_decode_prefix": call_sparse_prefix,
         "retrieval_decode_prefix": call_retrieval_prefix,
         "score_topk": call_score, "sparse_paged_decode_noalloc": call_noalloc,
         "retrieval_decode_tiered": call_tiered, "retrieval_decode_fp8": call_fp8,
         "build_block_reps": call_reps, "append_kv": call_append,
         "quantize_kv_fp8": call_quantize}


@pytest.mark.parametrize("name", list(CALLS))
def test_right_shapes_reach_the_device_check(name):
    with pytest.raises(ValueError, match="CUDA tensor|pinned host tensor"):
        CALLS[name]()


WRONG = [
    ("retrieval_decode", dict(q=torch.zeros(B, 4, 64, dtype=bf))),            # heads
    ("retrieval_decode", dict(out=torch.zeros(B, 8, 32, dtype=bf))),          # head dim
    ("retrieval_decode", dict(sel=torch.zeros(B, 3, KMAX, dtype=i32))),       # kv heads
    ("retrieval_decode", dict(seq_lens=torch.zeros(B + 1, dtype=i32))),       # batch
    ("retrieval_decode", dict(reps=torch.zeros(P - 1, 2, 64, dtype=f32))),    # too few pages
    ("retrieval_decode", dict(v_cache=torch.zeros(P - 2, 2, 128, 64, dtype=bf))),
    ("retrieval_decode", dict(k_cache=torch.zeros(P, 2, 64, 64, dtype=bf))),  # page size
    ("sparse_paged_decode", dict(nsel=torch.zeros(B * 2, dtype=i32))),       # flattened
    ("sparse_paged_decode", dict(block_table=torch.zeros(B * MAXB, dtype=i32))),
    ("sparse_paged_decode_prefix", dict(sel=torch.zeros(B, 1, KMAX, dtype=i32))),
    ("retrieval_decode_prefix", dict(reps=torch.zeros(P - 1, 2, 64, dtype=f32))),
    ("score_topk", dict(prompt_lens=torch.zeros(B, 1, dtype=i32))),
    ("score_topk", dict(reps=torch.zeros(P, 1, 64, dtype=f32))),
    ("sparse_paged_decode_noalloc", dict(q=torch.zeros(B, 8, 64, 1, dtype=bf))),
    ("retrieval_decode_tiered", dict(reps=torch.zeros(P + 4, 2, 64, dtype=f32))),  # host pages
    ("retrieval_decode_tiered", dict(v_host=torch.zeros(4, 2, 128, 64, dtype=bf))),
    ("retrieval_decode_fp8", dict(k_scale=torch.zeros(P, 2, dtype=f32))),
    ("retrieval_decode_fp8", dict(v_fp8=torch.zeros(P, 2, 128, 64, dtype=u8))),
    ("build_block_reps", dict(valid=torch.zeros(6, dtype=i32))),
    ("build_block_reps", dict(reps=torch.zeros(P - 1, 2, 64, dtype=f32))),
    ("append_kv", dict(k_new=torch.zeros(B, 8, 64, dtype=bf))),
    ("quantize_kv_fp8", dict(v_scale=torch.zeros(P, 2, 64, dtype=f32))),
    ("quantize_kv_fp8", dict(k_fp8=torch.zeros(P - 1, 2, 128, 64, dtype=u8))),
    ("retrieval_decode_host", dict(out_host=torch.zeros(B, 8, 32, dtype=bf))),
    ("retrieval_decode_host", dict(q=torch.zeros(B - 1, 8, 64, dtype=bf))),
    ("HostDecodeStep", dict(out_host=torch.zeros(B + 1, 8, 64, dtype=bf))),
    ("HostDecodeStep", dict(seq_lens=torch.zeros(B, 1, dtype=i32))),
]


@pytest.mark.parametrize("name,over", WRONG, ids=[f"{n}-{i}" for i, (n, _) in enumerate(WRONG)])
def test_wrong_shapes_stop_before_the_library(name, over):
    with pytest.raises(ValueError, match="shape|rows"):
        CALLS[name](**over)


def test_a_missing_library_fails_loudly(monkeypatch, tmp_path):
    """No library, no answer: the binding has no other way to compute anything."""
    monkeypatch.setattr(srkv, "_lib", None)
    monkeypatch.setattr(srkv, "LIB_PATH", str(tmp_path / "libsrkv.so"))
    with pytest.raises(RuntimeError, match="missing"):
        srkv.load()
    with pytest.raises(RuntimeError, match="missing"):
        srkv.host_staging_size(CFG, B)
