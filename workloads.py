"""Seeded synthetic inputs for the five attention workloads.

This module is shared by the tests, the smoke check and the benchmark.  It
holds input generation only -- lengths, page assignment, random values and
their rounding to bf16 -- and none of the attention arithmetic: it never
gathers through a page table, masks, normalises or attends.

Recipe (identical for every consumer):

* ``numpy.random.Generator(PCG64(seed))`` with seed = the workload number 1..5;
* draw order: lengths -> page permutation -> q -> k -> v (prefill/decode), or
  lengths -> q -> k -> v (window);
* values are N(0, 1) float32 rounded to bf16 with round-to-nearest-even and
  kept as their uint16 bit patterns, so the oracle and the GPU see identical
  bits;
* decode-append inputs (the new token's pre-norm q/k/v and the two RMSNorm
  gains) come after those draws, or from the stream PCG64([seed, 1]) when
  they extend a named workload, so that workload's own draws stay unchanged;
* a KV pool starts as all-NaN sentinels (bf16 0x7FC0); pages are handed to the
  requests in the order of a seeded permutation of the whole pool; each
  request's page-table row is padded with -1; slots past a request's length
  keep the sentinel, so any stray read shows up as NaN.

Shapes follow the Qwen3-ASR attention dims (qwenasr.cpp ARCHITECTURE.md,
"GGUF layout" and "Windowed audio tower"): decoder 16 query / 8 KV heads of
128, encoder 14 heads of 64, pages of 16 tokens.  No public dataset is used:
the length mixes stand in for LibriSpeech-style audio durations (see the
per-workload docstrings).
"""
from __future__ import annotations

import math

import numpy as np

BF16_NAN = 0x7FC0
PAGE_SIZE = 16
HQ, HKV, D_DEC = 16, 8, 128
HE, D_ENC = 14, 64


def rng_for(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(seed))


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bit patterns, round to nearest even (finite inputs)."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    r = (u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)
    return r.astype(np.uint16)


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns -> float64 (exact)."""
    u = np.ascontiguousarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return u.view(np.float32).astype(np.float64)


def normal_bf16(rng: np.random.Generator, shape) -> np.ndarray:
    return bf16_bits(rng.standard_normal(size=shape, dtype=np.float32))


def cu_from_lengths(lengths) -> np.ndarray:
    return np.concatenate([[0], np.cumsum(np.asarray(lengths, dtype=np.int64))]).astype(np.int32)


def _assign_pages(rng, lengths, num_pages, max_pages):
    """Hand out pages to requests by walking a seeded permutation of the pool."""
    perm = rng.permutation(num_pages).astype(np.int32)
    table = np.full((len(lengths), max_pages), -1, dtype=np.int32)
    cursor = 0
    for b, L in enumerate(lengths):
        n = -(-int(L) // PAGE_SIZE)
        if n > max_pages or cursor + n > num_pages:
            raise ValueError("pool too small for the drawn lengths")
        table[b, :n] = perm[cursor:cursor + n]
        cursor += n
    return table


def _fill_pool(rng, lengths, table, num_pages, hkv, d):
    """Pool [P, 16, hkv, d] of sentinels with each request's rows drawn in
    request order and laid into its pages."""
    pool = np.full((num_pages, PAGE_SIZE, hkv, d), BF16_NAN, dtype=np.uint16)
    for b, L in enumerate(lengths):
        L = int(L)
        if L == 0:
            continue
        n = -(-L // PAGE_SIZE)
        rows = np.full((n * PAGE_SIZE, hkv, d), BF16_NAN, dtype=np.uint16)
        rows[:L] = normal_bf16(rng, (L, hkv, d))
        pool[table[b, :n]] = rows.reshape(n, PAGE_SIZE, hkv, d)
    return pool


def decode_workload(seed: int, lengths, num_pages: int, max_pages: int,
                    hq: int = HQ, hkv: int = HKV, d: int = D_DEC) -> dict:
    """Batched single-token decode over a paged pool with the given lengths."""
    rng = rng_for(seed)
    return _decode_from_rng(rng, np.asarray(lengths, np.int32), num_pages, max_pages, hq, hkv, d)


def _decode_from_rng(rng, lengths, num_pages, max_pages, hq, hkv, d):
    table = _assign_pages(rng, lengths, num_pages, max_pages)
    q = normal_bf16(rng, (len(lengths), hq, d))
    k_pages = _fill_pool(rng, lengths, table, num_pages, hkv, d)
    v_pages = _fill_pool(rng, lengths, table, num_pages, hkv, d)
    return dict(kind="decode", q=q, k_pages=k_pages, v_pages=v_pages, page_table=table,
                seq_lens=lengths.astype(np.int32), num_pages=num_pages, max_pages=max_pages)


def prefill_workload(seed: int, lengths, num_pages: int, max_pages: int,
                     hq: int = HQ, hkv: int = HKV, d: int = D_DEC, rng=None) -> dict:
    """Packed causal prefill of requests with the given lengths, plus an
    all-sentinel destination pool and a page table for the page write."""
    rng = rng_for(seed) if rng is None else rng
    lengths = np.asarray(lengths, np.int32)
    table = _assign_pages(rng, lengths, num_pages, max_pages)
    T = int(lengths.sum())
    q = normal_bf16(rng, (T, hq, d))
    k = normal_bf16(rng, (T, hkv, d))
    v = normal_bf16(rng, (T, hkv, d))
    pool_shape = (num_pages, PAGE_SIZE, hkv, d)
    return dict(kind="prefill", q=q, k=k, v=v, cu_seqlens=cu_from_lengths(lengths),
                page_table=table, k_pages=np.full(pool_shape, BF16_NAN, np.uint16),
                v_pages=np.full(pool_shape, BF16_NAN, np.uint16), num_pages=num_pages,
                max_pages=max_pages, lengths=lengths)


def window_workload(seed: int, token_counts, h: int = HE, d: int = D_ENC, rng=None) -> dict:
    """Packed encoder tokens of requests with the given token counts.  The
    window plan (cu_windows) is not made here: it is the method's."""
    rng = rng_for(seed) if rng is None else rng
    token_counts = np.asarray(token_counts, np.int32)
    T = int(token_counts.sum())
    q = normal_bf16(rng, (T, h, d))
    k = normal_bf16(rng, (T, h, d))
    v = normal_bf16(rng, (T, h, d))
    return dict(kind="window", q=q, k=k, v=v, token_counts=token_counts)


def chunk_workload(seed: int, past_lengths, new_lengths, num_pages: int, max_pages: int,
                   hq: int = HQ, hkv: int = HKV, d: int = D_DEC, rng=None) -> dict:
    """Chunked prefill: request r already holds past_lengths[r] positions in
    its pages (random K/V there, NaN sentinels in every other slot) and brings
    new_lengths[r] packed rows.  Draw order: pages -> cached K -> cached V ->
    q -> k -> v."""
    rng = rng_for(seed) if rng is None else rng
    past = np.asarray(past_lengths, np.int32)
    new = np.asarray(new_lengths, np.int32)
    table = _assign_pages(rng, past + new, num_pages, max_pages)
    k_pages = _fill_pool(rng, past, table, num_pages, hkv, d)
    v_pages = _fill_pool(rng, past, table, num_pages, hkv, d)
    T = int(new.sum())
    q = normal_bf16(rng, (T, hq, d))
    k = normal_bf16(rng, (T, hkv, d))
    v = normal_bf16(rng, (T, hkv, d))
    return dict(kind="chunk", q=q, k=k, v=v, cu_seqlens=cu_from_lengths(new), n_past=past.copy(),
                page_table=table, k_pages=k_pages, v_pages=v_pages, num_pages=num_pages, max_pages=max_pages,
                lengths=new)


# --------------------------------------------------------------------------
# The five named workloads.

def encoder_tokens_for_frames(n_frames: int) -> int:
    """Encoder tokens for n mel frames under the recipe's rule: 13 per full
    100-frame chunk, and ceil(r / 8) for a final chunk of r frames (three
    stride-2 convolutions)."""
    return 13 * (n_frames // 100) + -(-(n_frames % 100) // 8)


# Decode-append parameters of the Qwen3 Thinker (qwenasr.cpp ARCHITECTURE.md,
# "GGUF layout": rope.freq_base 1e6; the RMS epsilon key carries no value
# there, and the Qwen3 decoders of the TTS page state 1e-6).
ROPE_THETA = 1.0e6
RMS_EPS = 1.0e-6


def append_inputs(rng: np.random.Generator, batch: int, hq: int = HQ, hkv: int = HKV, d: int = D_DEC,
                  x_scale: float = 1.0) -> dict:
    """Pre-norm q/k/v projections of one new token per request (N(0, 1) times
    x_scale, rounded to bf16) and the two [d] RMSNorm gains (U[0.5, 1.5],
    bf16-representable, stored as float32).  Draw order q, k, v, q gain, k gain."""
    def proj(shape):
        return bf16_bits(rng.standard_normal(size=shape, dtype=np.float32) * np.float32(x_scale))

    def gain():
        g = bf16_bits(rng.uniform(0.5, 1.5, size=d).astype(np.float32))
        return bf16_to_f64(g).astype(np.float32)

    q, k, v = proj((batch, hq, d)), proj((batch, hkv, d)), proj((batch, hkv, d))
    return dict(q_new=q, k_new=k, v_new=v, q_gain=gain(), k_gain=gain(), rope_theta=ROPE_THETA, rms_eps=RMS_EPS)


def decode_append_workload(seed: int, lengths, num_pages: int, max_pages: int, x_scale: float = 1.0) -> dict:
    """decode_workload plus the new token of every request: seq_lens count it,
    its slot (position seq_lens - 1) already holds random K/V that the append
    overwrites."""
    rng = rng_for(seed)
    w = _decode_from_rng(rng, np.asarray(lengths, np.int32), num_pages, max_pages, HQ, HKV, D_DEC)
    w.update(append_inputs(rng, len(lengths), x_scale=x_scale))
    return w


def with_append(w: dict, seed: int) -> dict:
    """A named decode workload plus new-token inputs drawn from a second
    stream of the same seed (the workload's own draws are unchanged)."""
    w = dict(w)
    w.update(append_inputs(np.random.Generator(np.random.PCG64([seed, 1])), len(w["seq_lens"])))
    return w


def tiny(seed: int = 1) -> dict:
    """1 request, prefill of 64 tokens into a 4-page pool whose page table is
    a random permutation of the 4 pages, then one decode query over the 64
    cached positions."""
    rng = rng_for(seed)
    lengths = np.array([64], np.int32)
    pre = prefill_workload(seed, lengths, num_pages=4, max_pages=4, rng=rng)
    pre["decode_q"] = normal_bf16(rng, (1, HQ, D_DEC))
    pre["seq_lens"] = lengths.copy()
    pre["name"] = "tiny decode+prefill (1 request, 64 tokens, 4-page pool)"
    return pre


def decode_0p6b(seed: int = 2) -> dict:
    """32 requests, context ~ U{200..2000} (audio prefix at 12.5 tokens/s for
    1-30 s plus ~40 prompt tokens plus generated tokens), 4096-page pool."""
    rng = rng_for(seed)
    lengths = rng.integers(200, 2000, size=32, endpoint=True).astype(np.int32)
    w = _decode_from_rng(rng, lengths, 4096, 125, HQ, HKV, D_DEC)
    w["name"] = "batched decode 0.6B (B=32, L~U[200,2000], 4096-page pool)"
    return w


def prefill_bucket(seed: int = 3) -> dict:
    """16 requests, length ceil(13 * d) + 40 for d ~ U[1, 30] s, 512-page pool."""
    rng = rng_for(seed)
    dur = rng.uniform(1.0, 30.0, size=16)
    lengths = np.array([math.ceil(13.0 * x) + 40 for x in dur], np.int32)
    w = prefill_workload(seed, lengths, num_pages=512, max_pages=27, rng=rng)
    w["name"] = "ragged causal prefill (16 requests, ceil(13 d)+40 tokens, d~U[1,30] s)"
    return w


def window_aut(seed: int = 4) -> dict:
    """8 requests of d ~ U[10, 1200] s audio, floor(100 d) mel frames each,
    13 encoder tokens per 100 frames, 14 heads of 64."""
    rng = rng_for(seed)
    dur = rng.uniform(10.0, 1200.0, size=8)
    counts = np.array([encoder_tokens_for_frames(int(math.floor(100.0 * x))) for x in dur],
                      np.int32)
    w = window_workload(seed, counts, rng=rng)
    w["name"] = "AuT windowed attention (8 requests, d~U[10,1200] s, 14x64 heads)"
    return w


def decode_1p7b(seed: int = 5) -> dict:
    """64 requests, context ~ U{2000..16000}, 65536-page pool (2 GiB per K/V)."""
    rng = rng_for(seed)
    lengths = rng.integers(2000, 16000, size=64, endpoint=True).astype(np.int32)
    w = _decode_from_rng(rng, lengths, 65536, 1000, HQ, HKV, D_DEC)
    w["name"] = "long-context decode 1.7B (B=64, L~U[2000,16000], 65536-page pool)"
    return w


def chunk_reprefill(seed: int = 7) -> dict:
    """Chunked prefill of a bucket of 16 requests whose audio prompt is
    already cached (n_past = ceil(13 d) + 40 for d ~ U[1, 30] s, the prefill
    bucket's recipe) and that bring 16..128 new tokens each (an assistant
    prefix for re-transcription); 512-page pool."""
    rng = rng_for(seed)
    dur = rng.uniform(1.0, 30.0, size=16)
    past = np.array([math.ceil(13.0 * x) + 40 for x in dur], np.int32)
    new = rng.integers(16, 128, size=16, endpoint=True).astype(np.int32)
    w = chunk_workload(seed, past, new, num_pages=512, max_pages=40, rng=rng)
    w["name"] = "chunked prefill (16 requests, cached ceil(13 d)+40, 16..128 new tokens)"
    return w


WORKLOADS = {1: tiny, 2: decode_0p6b, 3: prefill_bucket, 4: window_aut, 5: decode_1p7b}


# --------------------------------------------------------------------------
# AuT encoder layer around the window attention (qwenasr.cpp ARCHITECTURE.md,
# "Windowed audio tower" and "GGUF layout": d_model 896, 14 heads of 64, FFN
# 3584 on the 0.6B; LayerNorm with bias, biases on every projection).  The
# checkpoint's weights are not available: they are drawn at random, with the
# scales of a freshly initialised layer.

ENC_D, ENC_FFN = 896, 3584
ENC_LN_EPS = 1.0e-5


def encoder_weights(rng: np.random.Generator, d: int = ENC_D, d_ffn: int = ENC_FFN) -> dict:
    """Synthetic bf16 weights of one encoder layer, PyTorch Linear layout
    (out, in).  Draw order: ln1 gain, ln1 bias, Wqkv, bqkv, Wo, bo, ln2 gain,
    ln2 bias, W1, b1, W2, b2.  Matrices ~ N(0, 1 / fan_in), biases and
    LayerNorm biases ~ N(0, 0.1^2), LayerNorm gains ~ U[0.5, 1.5]."""
    def mat(n_out, n_in):
        return bf16_bits(rng.standard_normal(size=(n_out, n_in), dtype=np.float32) * np.float32(n_in ** -0.5))

    def vec(n):
        return bf16_bits(rng.standard_normal(size=n, dtype=np.float32) * np.float32(0.1))

    def gain(n):
        return bf16_bits(rng.uniform(0.5, 1.5, size=n).astype(np.float32))

    w = {}
    w["ln1_g"], w["ln1_b"] = gain(d), vec(d)
    w["w_qkv"], w["b_qkv"] = mat(3 * d, d), vec(3 * d)
    w["w_o"], w["b_o"] = mat(d, d), vec(d)
    w["ln2_g"], w["ln2_b"] = gain(d), vec(d)
    w["w_fc1"], w["b_fc1"] = mat(d_ffn, d), vec(d_ffn)
    w["w_fc2"], w["b_fc2"] = mat(d, d_ffn), vec(d)
    return w


def encoder_layer_workload(seed: int, token_counts, d: int = ENC_D, h: int = HE, d_ffn: int = ENC_FFN,
                           rng=None) -> dict:
    """Packed encoder states x [T, d] ~ N(0, 1) (bf16) of requests with the
    given token counts, then the layer's weights.  The window plan is the
    method's (not made here)."""
    rng = rng_for(seed) if rng is None else rng
    token_counts = np.asarray(token_counts, np.int32)
    T = int(token_counts.sum())
    x = normal_bf16(rng, (T, d))
    w = dict(kind="encoder_layer", x=x, token_counts=token_counts, n_heads=h, d_ffn=d_ffn, eps=ENC_LN_EPS)
    w["weights"] = encoder_weights(rng, d, d_ffn)
    return w


def encoder_layer_aut(seed: int = 4) -> dict:
    """The AuT window workload's requests (8 requests, d ~ U[10, 1200] s,
    13 tokens per 100 mel frames) through one 0.6B encoder layer: x [T, 896]
    and the layer's weights drawn after the token counts."""
    rng = rng_for(seed)
    dur = rng.uniform(10.0, 1200.0, size=8)
    counts = np.array([encoder_tokens_for_frames(int(math.floor(100.0 * x))) for x in dur], np.int32)
    w = encoder_layer_workload(seed, counts, rng=rng)
    w["name"] = "AuT encoder layer (8 requests, d~U[10,1200] s, d_model 896, 14x64 heads, FFN 3584)"
    return w
