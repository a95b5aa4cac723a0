"""Plain float64 definition of the attention forward (oracle; test-only).

Follows the standard definition on the "flash attention v3 paper" search page
(first snippet): for Q, K, V of shape (N, d), S = Q K^T, P = row-softmax(S),
O = P V.  That snippet leaves out the scale and the mask; the scale is taken
from the FA2 pseudocode on "Hacker News Digest — gpu-computing" (section
"Алгоритм Flash Attention 2": S = Q K^T * scale, scale = DIM**-0.5, here the
fp32 value the caller passes) and the mask is the lower-triangular causal
mask (key j visible to query i iff j <= i).

Readings taken where the pages are silent:
  * grouped-query attention: query head hq reads kv head hq // (Hq // Hkv),
    i.e. each kv head serves Hq/Hkv consecutive query heads;
  * causal alignment is top-left (j <= i) for any Nq, Nkv;
  * LSE_i = natural log of the sum over visible keys of exp(scale * q_i . k_j);
  * the scale is the float32 value handed to the kernel, promoted exactly to
    float64.

No blocking beyond splitting query rows into groups to bound memory: every
score row is materialised in full over all keys, then softmaxed in two passes
(max, then exp/sum).  Inputs are upcast exactly to float64 (bf16 and fp32 are
subsets of float64).
"""

import math

import numpy as np
import torch


def kv_head_index(hq, Hq, Hkv):
    """KV head read by query head ``hq`` (consecutive groups of Hq/Hkv)."""
    return hq // (Hq // Hkv)


def visible(rows, Nkv, causal):
    """Boolean [len(rows), Nkv]: True where key j is visible to query row i.

    ``rows`` are absolute query indices.  Non-causal: every key is visible.
    Causal (top-left): key j is visible to query i iff j <= i.
    """
    rows = torch.as_tensor(rows, dtype=torch.int64).reshape(-1, 1)
    cols = torch.arange(Nkv, dtype=torch.int64).reshape(1, -1)
    if not causal:
        return torch.ones(rows.shape[0], Nkv, dtype=torch.bool)
    return cols <= rows


def scale_fp64(scale):
    """The fp32 value the kernel receives, promoted exactly to float64."""
    return float(np.float32(scale))


def _check_shapes(q, k, v):
    B, Hq, Nq, D = q.shape
    Bk, Hkv, Nkv, Dk = k.shape
    if k.shape != v.shape or Bk != B or Dk != D:
        raise ValueError("k and v must be [B, Hkv, Nkv, D] matching q")
    if Hkv < 1 or Hq % Hkv != 0:
        raise ValueError("Hq must be a multiple of Hkv")
    return B, Hq, Hkv, Nq, Nkv, D


def _row_block(qrows, kh, vh, rows, scale64, causal):
    """Exact attention for a set of query rows against one kv head.

    qrows [r, D] float64, kh/vh [Nkv, D] float64, rows = absolute indices.
    Returns (O [r, D], LSE [r]) in float64.
    """
    S = (qrows @ kh.T) * scale64                      # scores, full rows
    mask = visible(rows, kh.shape[0], causal)
    S = S.masked_fill(~mask, -math.inf)
    m = S.max(dim=1, keepdim=True).values             # pass 1: row max
    E = torch.exp(S - m)                              # pass 2: exp / sum
    l = E.sum(dim=1, keepdim=True)
    P = E / l
    O = P @ vh
    lse = m.squeeze(1) + torch.log(l.squeeze(1))
    return O, lse


def attention_fp64(q, k, v, scale, causal, block_rows=1024):
    """O, LSE of the attention forward, in float64, for [B,H,N,D] inputs.

    q: [B, Hq, Nq, D]; k, v: [B, Hkv, Nkv, D] (any float dtype, upcast
    exactly).  Returns O float64 [B, Hq, Nq, D] and LSE float64 [B, Hq, Nq].
    """
    B, Hq, Hkv, Nq, Nkv, D = _check_shapes(q, k, v)
    s64 = scale_fp64(scale)
    O = torch.empty(B, Hq, Nq, D, dtype=torch.float64)
    L = torch.empty(B, Hq, Nq, dtype=torch.float64)
    for b in range(B):
        for hq in range(Hq):
            hk = kv_head_index(hq, Hq, Hkv)
            kh = k[b, hk].to(torch.float64)
            vh = v[b, hk].to(torch.float64)
            for r0 in range(0, Nq, block_rows):
                r1 = min(Nq, r0 + block_rows)
                rows = torch.arange(r0, r1)
                o, lse = _row_block(q[b, hq, r0:r1].to(torch.float64), kh, vh,
                                    rows, s64, causal)
                O[b, hq, r0:r1] = o
                L[b, hq, r0:r1] = lse
    return O, L


def attention_rows_fp64(q, k, v, scale, causal, b, hq, rows):
    """O and LSE for selected query rows of one (batch, query head).

    Used to check full-size launches on sampled outputs.  ``rows`` is a list
    or tensor of absolute query indices.  Returns (O [r, D], LSE [r]) float64.
    """
    B, Hq, Hkv, Nq, Nkv, D = _check_shapes(q, k, v)
    rows = torch.as_tensor(rows, dtype=torch.int64)
    hk = kv_head_index(hq, Hq, Hkv)
    qrows = q[b, hq].index_select(0, rows).to(torch.float64)
    return _row_block(qrows, k[b, hk].to(torch.float64),
                      v[b, hk].to(torch.float64), rows, scale_fp64(scale),
                      causal)


def probabilities_fp64(q, k, v, scale, causal):
    """The full probability matrix P [B, Hq, Nq, Nkv] in float64 (small
    shapes only), built exactly as in ``attention_fp64``."""
    B, Hq, Hkv, Nq, Nkv, D = _check_shapes(q, k, v)
    s64 = scale_fp64(scale)
    P = torch.empty(B, Hq, Nq, Nkv, dtype=torch.float64)
    rows = torch.arange(Nq)
    for b in range(B):
        for hq in range(Hq):
            hk = kv_head_index(hq, Hq, Hkv)
            S = (q[b, hq].to(torch.float64) @ k[b, hk].to(torch.float64).T) * s64
            S = S.masked_fill(~visible(rows, Nkv, causal), -math.inf)
            E = torch.exp(S - S.max(dim=1, keepdim=True).values)
            P[b, hq] = E / E.sum(dim=1, keepdim=True)
    return P
