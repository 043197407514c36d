"""Paged cross-attention decode (Whisper-style: a non-causal cache of encoder
states written once and read by every decode step; M* "Speech recognition:
Whisper and Qwen3-ASR", "Graph") through qa_decode_attn with as many query
heads as KV heads, against the fp64 oracle.

The cache holds 1500 encoder frames per request (30 s at the Whisper encoder
rate); each step brings a fresh query; the pages are never rewritten, so
consecutive steps read identical K/V.
"""
import numpy as np
import pytest

import oracle
import workloads as wl
from _util import assert_close, bits, f64, to_dev

pytestmark = pytest.mark.gpu
import torch  # noqa: E402

import paged_kv_gqa_attention_gb300 as qa  # noqa: E402


def _cross_cache(seed, lengths, heads=8):
    n_pages = sum(-(-L // 16) for L in lengths) + 3
    return wl.decode_workload(seed, lengths, num_pages=n_pages, max_pages=max(-(-L // 16) for L in lengths),
                              hq=heads, hkv=heads)


@pytest.mark.parametrize("heads", [8, 4, 1])
def test_steps_over_a_cache_written_once(heads):
    w = _cross_cache(300 + heads, (1500, 1500, 1500, 1500), heads)
    kp, vp = to_dev(w["k_pages"]), to_dev(w["v_pages"])
    pt, sl = to_dev(w["page_table"]), to_dev(w["seq_lens"])
    before_k, before_v = bits(kp), bits(vp)
    rng = wl.rng_for(400 + heads)
    for step in range(3):
        q = wl.normal_bf16(rng, (4, heads, wl.D_DEC))
        out = qa.qa_decode_attn(to_dev(q), kp, vp, pt, sl, debug_checks=True)
        torch.cuda.synchronize()
        ref = oracle.decode(q, w["k_pages"], w["v_pages"], w["page_table"], w["seq_lens"])
        assert_close(f64(out), ref, f"cross-attention step {step}, {heads} heads")
    # read-only: the cache is untouched
    np.testing.assert_array_equal(bits(kp), before_k)
    np.testing.assert_array_equal(bits(vp), before_v)


def test_mixed_encoder_lengths():
    # requests with shorter audio have shorter caches (1500 frames is the cap)
    w = _cross_cache(310, (1500, 750, 16, 1, 1499, 333))
    out = qa.qa_decode_attn(to_dev(w["q"]), to_dev(w["k_pages"]), to_dev(w["v_pages"]), to_dev(w["page_table"]),
                            to_dev(w["seq_lens"]), debug_checks=True)
    torch.cuda.synchronize()
    ref = oracle.decode(w["q"], w["k_pages"], w["v_pages"], w["page_table"], w["seq_lens"])
    assert_close(f64(out), ref, "mixed cross-attention lengths")
