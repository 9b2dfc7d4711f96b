"""Non-absorbed 128-head attention in numpy fp64: an independent pin for the oracle.

TEST INFRASTRUCTURE ONLY (same rule as the rest of ``oracle/``).

MLA caches one latent c_t (512 kv_c dims) plus a shared 64-dim k_rope per token.
Written out without absorption, head h sees explicit keys and values

    k_{h,t} = [ W_UK[h] @ c_t ; k_rope_t ]      (128 + 64 = 192 dims)
    v_{h,t} =   W_UV[h] @ c_t                    (128 dims)

and runs ordinary scaled dot-product softmax attention with its query
[q_nope_h ; q_pe_h].  The absorbed form folds W_UK into the query
(q_lat = W_UK[h]^T q_nope_h) and W_UV into the output, so that
W_UV[h] @ (absorbed output) equals this function's output.  This is the identity
behind the absorbed decode that engines run
[dp-attention-expert-parallel-mla-kv-replication (inferenceinterviews.com),
"A strong answer"; MLA 的 TP 切分 (10100.com), section 一: kv_lora_rank = 512,
qk_rope_head_dim = 64 shared by all heads, per-head K of 128 + 64 = 192 dims].

This module shares no code with ``mla_oracle.c``: it works on logical token rows
(no paging) with numpy linear algebra.
"""
from __future__ import annotations

import numpy as np

KV_LORA_RANK = 512
ROPE_DIM = 64


def mha_nonabsorbed(q_nope, q_pe, w_uk, w_uv, rows, softmax_scale):
    """Explicit-K/V multi-head attention for one request.

    q_nope: [H, dn] fp64, q_pe: [H, 64], w_uk: [H, dn, 512], w_uv: [H, dv, 512],
    rows: [L, 576] fp64 latent rows in logical token order (L >= 1).
    Returns [H, dv] fp64.
    """
    rows = np.asarray(rows, np.float64)
    c = rows[:, :KV_LORA_RANK]                      # [L, 512]
    k_rope = rows[:, KV_LORA_RANK:]                 # [L, 64], shared by all heads
    assert k_rope.shape[1] == ROPE_DIM
    H = q_nope.shape[0]
    k_nope = np.einsum("hik,tk->hti", w_uk, c)      # [H, L, dn]
    v = np.einsum("hik,tk->hti", w_uv, c)           # [H, L, dv]
    k = np.concatenate([k_nope, np.broadcast_to(k_rope, (H,) + k_rope.shape)], axis=2)
    q = np.concatenate([q_nope, q_pe], axis=1)      # [H, dn + 64]
    scores = np.einsum("hd,htd->ht", q, k) * softmax_scale
    scores -= scores.max(axis=1, keepdims=True)
    w = np.exp(scores)
    w /= w.sum(axis=1, keepdims=True)
    return np.einsum("ht,hti->hi", w, v)


def softmax_attention(q, keys, values, softmax_scale):
    """Textbook single-query attention, one head: softmax(scale * K q) @ V."""
    s = softmax_scale * (np.asarray(keys, np.float64) @ np.asarray(q, np.float64))
    s -= s.max()
    w = np.exp(s)
    w /= w.sum()
    return w @ np.asarray(values, np.float64)
