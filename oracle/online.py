"""The tiled online-softmax recurrences, in float64 (oracle; test-only).

These restate the method itself, not the definition, so the CPU tests can
check that the recurrence the GPU kernel implements reaches the plain
definition in ``attention.py`` (the pages call the method exact).

Loop nest: the FA2 pseudocode on "Hacker News Digest — gpu-computing",
section "Алгоритм Flash Attention 2": for each (batch, query tile) set the
output tile to zero, then for each key/value tile form the scaled scores,
apply the online softmax in place and accumulate the product with the value
tile; finally store the output tile.

Two forms of the per-tile update:

``online_normalised_fp64`` — the recurrence of section "v1 — базовая версия",
item 3, exactly as printed there, which renormalises at every tile:
    m = max(m_prev, m_cur)
    d = d_prev * exp(m_prev - m) + sum exp(S - m)
    O = O_prev * (d_prev / d) * exp(m_prev - m) + (exp(S - m) / d) @ V
Reading taken: m_cur is the row max of the current (masked) score tile.

``online_deferred_fp64`` — the same running max and denominator (called l
here), with the division by l deferred to the end: the accumulator is
rescaled by exp(m_prev - m) and the tile's exp(S - m) @ V is added; O = acc/l
after the last tile, and LSE = m + ln l.  This is the form the GPU kernel
uses.
"""

import math

import torch

from .attention import kv_head_index, scale_fp64, visible


def _tiles(q, k, v, scale, causal, block_m, block_n):
    """Yield (b, hq, rows, qt, [(cols, Kt, Vt), ...]) in the pseudocode's
    loop order, with tensors in float64."""
    B, Hq, Nq, D = q.shape
    Hkv, Nkv = k.shape[1], k.shape[2]
    for b in range(B):
        for hq in range(Hq):
            hk = kv_head_index(hq, Hq, Hkv)
            for r0 in range(0, Nq, block_m):
                rows = torch.arange(r0, min(Nq, r0 + block_m))
                qt = q[b, hq, r0:r0 + len(rows)].to(torch.float64)
                kv = []
                for c0 in range(0, Nkv, block_n):
                    c1 = min(Nkv, c0 + block_n)
                    kv.append((torch.arange(c0, c1),
                               k[b, hk, c0:c1].to(torch.float64),
                               v[b, hk, c0:c1].to(torch.float64)))
                yield b, hq, rows, qt, kv


def _masked_scores(qt, Kt, rows, cols, s64, causal):
    S = (qt @ Kt.T) * s64
    if causal:
        vis = visible(rows, int(cols[-1]) + 1, True)[:, int(cols[0]):]
        S = S.masked_fill(~vis, -math.inf)
    return S


def _safe_exp_diff(a, b):
    """exp(a - b) with exp(-inf - (-inf)) read as 0 (an all-masked prefix)."""
    out = torch.exp(a - b)
    return torch.where(torch.isneginf(a) & torch.isneginf(b),
                       torch.zeros_like(out), out)


def online_normalised_fp64(q, k, v, scale, causal, block_m=128, block_n=128):
    """Tile-by-tile forward with per-tile renormalisation (the printed v1
    recurrence).  Returns O [B,Hq,Nq,D] and LSE [B,Hq,Nq] in float64."""
    B, Hq, Nq, D = q.shape
    s64 = scale_fp64(scale)
    O = torch.zeros(B, Hq, Nq, D, dtype=torch.float64)
    L = torch.zeros(B, Hq, Nq, dtype=torch.float64)
    for b, hq, rows, qt, kv in _tiles(q, k, v, scale, causal, block_m, block_n):
        r = len(rows)
        m = torch.full((r, 1), -math.inf, dtype=torch.float64)
        d = torch.zeros(r, 1, dtype=torch.float64)
        o = torch.zeros(r, D, dtype=torch.float64)
        for cols, Kt, Vt in kv:
            S = _masked_scores(qt, Kt, rows, cols, s64, causal)
            m_cur = S.max(dim=1, keepdim=True).values
            m_new = torch.maximum(m, m_cur)
            corr = _safe_exp_diff(m, m_new)
            e = _safe_exp_diff(S, m_new)
            d_new = d * corr + e.sum(dim=1, keepdim=True)
            ratio = torch.where(d_new > 0, d / d_new, torch.zeros_like(d))
            inv = torch.where(d_new > 0, 1.0 / d_new, torch.zeros_like(d))
            o = o * ratio * corr + (e * inv) @ Vt
            m, d = m_new, d_new
        O[b, hq, rows] = o
        L[b, hq, rows] = (m + torch.log(d)).squeeze(1)
    return O, L


def online_deferred_fp64(q, k, v, scale, causal, block_m=128, block_n=128):
    """Tile-by-tile forward with the division by l deferred to the end.
    Returns O [B,Hq,Nq,D] and LSE [B,Hq,Nq] in float64."""
    B, Hq, Nq, D = q.shape
    s64 = scale_fp64(scale)
    O = torch.zeros(B, Hq, Nq, D, dtype=torch.float64)
    L = torch.zeros(B, Hq, Nq, dtype=torch.float64)
    for b, hq, rows, qt, kv in _tiles(q, k, v, scale, causal, block_m, block_n):
        r = len(rows)
        m = torch.full((r, 1), -math.inf, dtype=torch.float64)
        l = torch.zeros(r, 1, dtype=torch.float64)
        acc = torch.zeros(r, D, dtype=torch.float64)
        for cols, Kt, Vt in kv:
            S = _masked_scores(qt, Kt, rows, cols, s64, causal)
            m_new = torch.maximum(m, S.max(dim=1, keepdim=True).values)
            corr = _safe_exp_diff(m, m_new)
            e = _safe_exp_diff(S, m_new)
            l = l * corr + e.sum(dim=1, keepdim=True)
            acc = acc * corr + e @ Vt
            m = m_new
        O[b, hq, rows] = acc / l
        L[b, hq, rows] = (m + torch.log(l)).squeeze(1)
    return O, L
