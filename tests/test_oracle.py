"""Pins of the CPU oracle to things other than itself (CPU only).

Each test checks the oracle against what the pages and the mathematics fix:
hand-derived closed forms (tests/golden/closed_forms.json), invariants of
the softmax, special cases with textbook answers, the online recurrence the
pages print, an independent pure-Python triple loop and a library routine.
The last group plants mistakes in the oracle and checks that the pins catch
each one.
"""

import json
import math
import os

import pytest
import torch

import oracle
from oracle import attention as oatt
from exact_io_aware_fa2_gb300.workloads import (WORKLOADS, Workload,
                                                make_custom, make_inputs)

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "closed_forms.json")
F64 = torch.float64


def _load_golden():
    with open(GOLDEN) as f:
        return json.load(f)["cases"]


def _t(x):
    return torch.tensor(x, dtype=F64)


def _rand(B, Hq, Hkv, Nq, Nkv, D, seed, std=1.0):
    g = torch.Generator().manual_seed(seed)
    q = torch.randn(B, Hq, Nq, D, generator=g, dtype=F64) * std
    k = torch.randn(B, Hkv, Nkv, D, generator=g, dtype=F64)
    v = torch.randn(B, Hkv, Nkv, D, generator=g, dtype=F64)
    return q, k, v


# --------------------------------------------------------------- closed forms

@pytest.mark.parametrize("case", _load_golden(), ids=lambda c: c["name"])
def test_golden_closed_forms(case):
    q, k, v = _t(case["q"]), _t(case["k"]), _t(case["v"])
    o_ref, lse_ref = _t(case["o"]), _t(case["lse"])
    O, L = oracle.attention_fp64(q, k, v, case["scale"], case["causal"])
    assert torch.allclose(O, o_ref, atol=1e-12, rtol=0)
    assert torch.allclose(L, lse_ref, atol=1e-12, rtol=0)
    # the probability matrix, against the weights the derivation names
    P = oracle.probabilities_fp64(q, k, v, case["scale"], case["causal"])
    assert torch.allclose(P, _t(case["p"]), atol=1e-12, rtol=0)
    # the brute force and both recurrences reach the same closed form
    Ob, Lb = oracle.attention_loops(case["q"], case["k"], case["v"],
                                    case["scale"], case["causal"])
    assert torch.allclose(_t(Ob), o_ref, atol=1e-12, rtol=0)
    assert torch.allclose(_t(Lb), lse_ref, atol=1e-12, rtol=0)
    for fn in (oracle.online_normalised_fp64, oracle.online_deferred_fp64):
        Oo, Lo = fn(q, k, v, case["scale"], case["causal"], 2, 2)
        assert torch.allclose(Oo, o_ref, atol=1e-12, rtol=0)
        assert torch.allclose(Lo, lse_ref, atol=1e-12, rtol=0)


# ----------------------------------------------------------------- invariants

@pytest.mark.parametrize("causal", [False, True])
def test_rows_of_p_sum_to_one(causal):
    q, k, v = _rand(2, 4, 2, 37, 37, 16, 1, std=2.0)
    P = oracle.probabilities_fp64(q, k, v, 0.25, causal)
    assert (P >= 0).all()
    assert torch.allclose(P.sum(-1), torch.ones(2, 4, 37, dtype=F64),
                          atol=1e-12, rtol=0)
    if causal:  # no weight above the diagonal
        assert torch.all(P.triu(diagonal=1) == 0)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("Hq,Hkv", [(4, 4), (8, 2), (6, 1)])
def test_p_times_v_is_the_output_of_mha_on_repeated_kv(Hq, Hkv, causal):
    """P from probabilities_fp64, applied to V, gives the output that the
    (golden-pinned) attention_fp64 computes for plain multi-head attention
    on K and V repeated per query head: this fixes P's scale, mask and GQA
    head map together (a wrong one changes the weights of some row)."""
    q, k, v = _rand(2, Hq, Hkv, 29, 41, 8, 15, std=2.0)
    g = Hq // Hkv
    scale = 0.37
    P = oracle.probabilities_fp64(q, k, v, scale, causal)
    kr, vr = k.repeat_interleave(g, dim=1), v.repeat_interleave(g, dim=1)
    O, L = oracle.attention_fp64(q, kr, vr, scale, causal)
    assert torch.allclose(P @ vr, O, atol=1e-12, rtol=0)
    # ln of the largest weight of a row is that row's largest score minus
    # LSE; the scores come from the MHA inputs, not from P
    S = (q @ kr.transpose(-1, -2)) * oatt.scale_fp64(scale)
    if causal:
        S = S.masked_fill(~oatt.visible(torch.arange(29), 41, True), -math.inf)
    assert torch.allclose(P.max(-1).values.log(),
                          S.max(-1).values - L, atol=1e-12, rtol=0)


@pytest.mark.parametrize("causal", [False, True])
def test_identical_keys_give_mean_of_visible_v(causal):
    q, _, v = _rand(1, 2, 2, 40, 40, 8, 2)
    krow = torch.randn(8, dtype=F64, generator=torch.Generator().manual_seed(9))
    k = krow.expand(1, 2, 40, 8).clone()
    scale = 0.3
    O, L = oracle.attention_fp64(q, k, v, scale, causal)
    for h in range(2):
        for i in range(40):
            n = i + 1 if causal else 40
            mean = v[0, h, :n].mean(0)
            assert torch.allclose(O[0, h, i], mean, atol=1e-12, rtol=0)
            s = float(oatt.scale_fp64(scale)) * float(q[0, h, i] @ krow)
            assert abs(float(L[0, h, i]) - (s + math.log(n))) < 1e-12


@pytest.mark.parametrize("causal", [False, True])
def test_constant_v_rows_return_that_row(causal):
    q, k, _ = _rand(2, 2, 1, 33, 50, 16, 3, std=3.0)
    row = torch.linspace(-2, 5, 16, dtype=F64)
    v = row.expand(2, 1, 50, 16).clone()
    O, _ = oracle.attention_fp64(q, k, v, 0.25, causal)
    assert torch.allclose(O, row.expand_as(O), atol=1e-12, rtol=0)


def test_causal_query0_returns_v0():
    q, k, v = _rand(2, 3, 3, 20, 20, 8, 4, std=2.0)
    scale = 0.35
    O, L = oracle.attention_fp64(q, k, v, scale, True)
    assert torch.equal(O[:, :, 0], v[:, :, 0])
    s = oatt.scale_fp64(scale) * (q[:, :, 0] * k[:, :, 0]).sum(-1)
    assert torch.allclose(L[:, :, 0], s, atol=1e-12, rtol=0)


def test_causal_rows_ignore_future_keys():
    q, k, v = _rand(1, 2, 2, 24, 24, 8, 5)
    O, L = oracle.attention_fp64(q, k, v, 0.4, True)
    i = 11
    k2, v2 = k.clone(), v.clone()
    k2[:, :, i + 1:] += 5.0
    v2[:, :, i + 1:] -= 3.0
    O2, L2 = oracle.attention_fp64(q, k2, v2, 0.4, True)
    assert torch.equal(O[:, :, :i + 1], O2[:, :, :i + 1])
    assert torch.equal(L[:, :, :i + 1], L2[:, :, :i + 1])
    assert not torch.allclose(O[:, :, i + 1:], O2[:, :, i + 1:])


@pytest.mark.parametrize("causal", [False, True])
def test_scale_zero_gives_mean(causal):
    q, k, v = _rand(1, 2, 2, 17, 17, 8, 6, std=5.0)
    O, L = oracle.attention_fp64(q, k, v, 0.0, causal)
    for i in range(17):
        n = i + 1 if causal else 17
        assert torch.allclose(O[0, :, i], v[0, :, :n].mean(1), atol=1e-12,
                              rtol=0)
        assert torch.allclose(L[0, :, i], torch.full((2,), math.log(n),
                                                     dtype=F64),
                              atol=1e-12, rtol=0)


@pytest.mark.parametrize("causal", [False, True])
def test_single_key_returns_v0(causal):
    q, k, v = _rand(2, 2, 2, 5, 1, 8, 7, std=4.0)
    O, _ = oracle.attention_fp64(q, k, v, 0.7, causal)
    assert torch.equal(O, v[:, :, :1].expand_as(O))


@pytest.mark.parametrize("shape,causal", [
    ((1, 2, 2, 300, 300, 16), False),
    ((1, 2, 2, 300, 300, 16), True),
    ((2, 4, 2, 129, 257, 8), False),
    ((2, 4, 2, 257, 129, 8), True),
    ((1, 1, 1, 1, 1, 4), True),
])
def test_online_recurrences_equal_two_pass(shape, causal):
    q, k, v = _rand(*shape, seed=8, std=4.0)
    O, L = oracle.attention_fp64(q, k, v, 0.3, causal)
    for fn in (oracle.online_normalised_fp64, oracle.online_deferred_fp64):
        Oo, Lo = fn(q, k, v, 0.3, causal, block_m=128, block_n=128)
        assert torch.allclose(Oo, O, atol=1e-12, rtol=0)
        assert torch.allclose(Lo, L, atol=1e-12, rtol=0)


def test_online_recurrence_large_logits():
    """Logits near +-100 (the large-logit workload's range): the running max
    keeps every exp in range and both recurrences still match."""
    q, k, v = _rand(1, 1, 1, 256, 512, 32, 9, std=3.0)
    k[:, :, ::97] *= 8
    O, L = oracle.attention_fp64(q, k, v, 1.0, True)
    assert torch.isfinite(O).all() and torch.isfinite(L).all()
    assert float(L.max()) > 50
    for fn in (oracle.online_normalised_fp64, oracle.online_deferred_fp64):
        Oo, Lo = fn(q, k, v, 1.0, True)
        assert torch.allclose(Oo, O, atol=1e-11, rtol=0)
        assert torch.allclose(Lo, L, atol=1e-11, rtol=0)


def test_joint_permutation_of_keys_and_values_noncausal():
    q, k, v = _rand(1, 2, 2, 31, 45, 8, 10)
    perm = torch.randperm(45, generator=torch.Generator().manual_seed(1))
    O, L = oracle.attention_fp64(q, k, v, 0.5, False)
    O2, L2 = oracle.attention_fp64(q, k[:, :, perm], v[:, :, perm], 0.5, False)
    assert torch.allclose(O, O2, atol=1e-12, rtol=0)
    assert torch.allclose(L, L2, atol=1e-12, rtol=0)


@pytest.mark.parametrize("causal", [False, True])
def test_gqa_equals_mha_on_repeated_kv(causal):
    q, k, v = _rand(2, 8, 2, 40, 40, 8, 11)
    O, L = oracle.attention_fp64(q, k, v, 0.5, causal)
    kr = k.repeat_interleave(4, dim=1)
    vr = v.repeat_interleave(4, dim=1)
    O2, L2 = oracle.attention_fp64(q, kr, vr, 0.5, causal)
    assert torch.equal(O, O2) and torch.equal(L, L2)


def test_rows_variant_matches_full():
    q, k, v = _rand(2, 4, 2, 70, 90, 8, 12)
    O, L = oracle.attention_fp64(q, k, v, 0.5, True, block_rows=16)
    rows = [0, 5, 63, 64, 69]
    for b in range(2):
        for h in range(4):
            o, l = oracle.attention_rows_fp64(q, k, v, 0.5, True, b, h, rows)
            assert torch.allclose(o, O[b, h, rows], atol=1e-13, rtol=0)
            assert torch.allclose(l, L[b, h, rows], atol=1e-13, rtol=0)


# ------------------------------------------------- independent implementations

def _tiny_cases():
    g = torch.Generator().manual_seed(13)
    out = []
    for idx in range(8):
        B = int(torch.randint(1, 3, (1,), generator=g))
        Hkv = int(torch.randint(1, 3, (1,), generator=g))
        Hq = Hkv * int(torch.randint(1, 3, (1,), generator=g))
        Nq = int(torch.randint(1, 34, (1,), generator=g))
        Nkv = int(torch.randint(1, 34, (1,), generator=g))
        D = int(torch.randint(1, 17, (1,), generator=g))
        out.append((B, Hq, Hkv, Nq, Nkv, D, idx % 2 == 1, 100 + idx))
    return out


@pytest.mark.parametrize("B,Hq,Hkv,Nq,Nkv,D,causal,seed", _tiny_cases())
def test_oracle_equals_pure_python_loops(B, Hq, Hkv, Nq, Nkv, D, causal, seed):
    q, k, v = _rand(B, Hq, Hkv, Nq, Nkv, D, seed, std=2.0)
    O, L = oracle.attention_fp64(q, k, v, 0.6, causal)
    Ob, Lb = oracle.attention_loops(q.tolist(), k.tolist(), v.tolist(),
                                    oatt.scale_fp64(0.6), causal)
    assert torch.allclose(O, _t(Ob), atol=1e-12, rtol=0)
    assert torch.allclose(L, _t(Lb), atol=1e-12, rtol=0)


@pytest.mark.parametrize("Nq,Nkv,causal", [(64, 64, False), (64, 64, True),
                                           (40, 72, False), (72, 40, True)])
def test_oracle_equals_torch_sdpa_fp64(Nq, Nkv, causal):
    q, k, v = _rand(2, 4, 2, Nq, Nkv, 16, 14, std=2.0)
    scale = 0.37
    O, _ = oracle.attention_fp64(q, k, v, scale, causal)
    mask = oatt.visible(torch.arange(Nq), Nkv, causal)
    ref = torch.nn.functional.scaled_dot_product_attention(
        q, k.repeat_interleave(2, 1), v.repeat_interleave(2, 1),
        attn_mask=mask, scale=oatt.scale_fp64(scale))
    assert torch.allclose(O, ref, atol=1e-10, rtol=0)


def test_oracle_on_bf16_inputs_upcasts_exactly():
    q, k, v = make_inputs(WORKLOADS["tiny_128_d64"])
    assert q.dtype == torch.bfloat16
    O, L = oracle.attention_fp64(q, k, v, WORKLOADS["tiny_128_d64"].scale,
                                 False)
    O2, L2 = oracle.attention_fp64(q.double(), k.double(), v.double(),
                                   WORKLOADS["tiny_128_d64"].scale, False)
    assert torch.equal(O, O2) and torch.equal(L, L2)


# ------------------------------------------------------------ planted mistakes

def _golden_pins_pass():
    """True iff every golden closed form still holds for attention_fp64 and
    probabilities_fp64 (looked up in the module, so a planted mistake in
    either one is what runs)."""
    for case in _load_golden():
        q, k, v = _t(case["q"]), _t(case["k"]), _t(case["v"])
        O, L = oatt.attention_fp64(q, k, v, case["scale"], case["causal"])
        P = oatt.probabilities_fp64(q, k, v, case["scale"], case["causal"])
        if not (torch.allclose(O, _t(case["o"]), atol=1e-9) and
                torch.allclose(L, _t(case["lse"]), atol=1e-9) and
                torch.allclose(P, _t(case["p"]), atol=1e-9)):
            return False
    return True


def _probabilities_variant(scale_used, head_map, axis, masked):
    """probabilities_fp64 with one planted mistake: the scale it applies,
    the kv head it reads, the axis it normalises over, or the mask."""
    def fn(q, k, v, scale, causal):
        B, Hq, Nq, _ = q.shape
        Hkv, Nkv = k.shape[1], k.shape[2]
        P = torch.empty(B, Hq, Nq, Nkv, dtype=F64)
        for b in range(B):
            for hq in range(Hq):
                hk = head_map(hq, Hq, Hkv)
                S = (q[b, hq].double() @ k[b, hk].double().T) * \
                    scale_used(scale)
                if masked:
                    S = S.masked_fill(~oatt.visible(torch.arange(Nq), Nkv,
                                                    causal), -math.inf)
                E = torch.exp(S - S.max(dim=axis, keepdim=True).values)
                P[b, hq] = E / E.sum(dim=axis, keepdim=True)
        return P
    return fn


_GQA = oatt.kv_head_index
_SCALE = oatt.scale_fp64


def _row_block_no_lse_max(qrows, kh, vh, rows, s64, causal):
    S = (qrows @ kh.T) * s64
    S = S.masked_fill(~oatt.visible(rows, kh.shape[0], causal), -math.inf)
    m = S.max(dim=1, keepdim=True).values
    E = torch.exp(S - m)
    l = E.sum(1, keepdim=True)
    return (E / l) @ vh, torch.log(l.squeeze(1))        # dropped "+ m"


def _row_block_unnormalised(qrows, kh, vh, rows, s64, causal):
    S = (qrows @ kh.T) * s64
    S = S.masked_fill(~oatt.visible(rows, kh.shape[0], causal), -math.inf)
    m = S.max(dim=1, keepdim=True).values
    E = torch.exp(S - m)
    l = E.sum(1, keepdim=True)
    return E @ vh, m.squeeze(1) + torch.log(l.squeeze(1))  # dropped "/ l"


def _row_block_transposed_v(qrows, kh, vh, rows, s64, causal):
    S = (qrows @ kh.T) * s64
    S = S.masked_fill(~oatt.visible(rows, kh.shape[0], causal), -math.inf)
    m = S.max(dim=1, keepdim=True).values
    E = torch.exp(S - m)
    l = E.sum(1, keepdim=True)
    return (E / l) @ kh, m.squeeze(1) + torch.log(l.squeeze(1))  # K for V


MUTANTS = {
    "gqa_modulo_mapping": ("kv_head_index",
                           lambda hq, Hq, Hkv: hq % Hkv),
    "causal_mask_reversed": ("visible",
                             lambda rows, Nkv, causal: (
                                 torch.ones(len(rows), Nkv, dtype=torch.bool)
                                 if not causal else
                                 torch.arange(Nkv).reshape(1, -1) >=
                                 torch.as_tensor(rows).reshape(-1, 1))),
    "causal_bottom_right": ("visible",
                            lambda rows, Nkv, causal: (
                                torch.ones(len(rows), Nkv, dtype=torch.bool)
                                if not causal else
                                torch.arange(Nkv).reshape(1, -1) <=
                                torch.as_tensor(rows).reshape(-1, 1) + 1)),
    "scale_dropped": ("scale_fp64", lambda s: 1.0),
    "lse_without_max": ("_row_block", _row_block_no_lse_max),
    "output_not_normalised": ("_row_block", _row_block_unnormalised),
    "keys_used_as_values": ("_row_block", _row_block_transposed_v),
    "p_scale_dropped": ("probabilities_fp64", _probabilities_variant(
        lambda s: 1.0, _GQA, 1, True)),
    "p_gqa_modulo_mapping": ("probabilities_fp64", _probabilities_variant(
        _SCALE, lambda hq, Hq, Hkv: hq % Hkv, 1, True)),
    "p_normalised_over_queries": ("probabilities_fp64", _probabilities_variant(
        _SCALE, _GQA, 0, True)),
    "p_mask_dropped": ("probabilities_fp64", _probabilities_variant(
        _SCALE, _GQA, 1, False)),
}


def test_pins_pass_on_unmodified_oracle():
    assert _golden_pins_pass()
    # the planted variant without a mistake passes too
    oracle_p = oatt.probabilities_fp64
    try:
        oatt.probabilities_fp64 = _probabilities_variant(_SCALE, _GQA, 1, True)
        assert _golden_pins_pass()
    finally:
        oatt.probabilities_fp64 = oracle_p


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_is_caught(name, monkeypatch):
    attr, fn = MUTANTS[name]
    monkeypatch.setattr(oatt, attr, fn)
    assert not _golden_pins_pass(), f"mutant {name} slipped through the pins"


# ---------------------------------------------------------- input generator

def test_workload_recipe_is_deterministic_and_bf16():
    w = WORKLOADS["tiny_128_d64"]
    a = make_inputs(w, seed=0)
    b = make_inputs(w, seed=0)
    c = make_inputs(w, seed=1)
    for x, y, z in zip(a, b, c):
        assert x.dtype == torch.bfloat16 and x.shape == (1, 1, 128, 64)
        assert torch.equal(x, y) and not torch.equal(x, z)
    assert w.scale == float(torch.tensor(0.125, dtype=torch.float32))


def test_workload_spike_rows():
    w = Workload("spiky", 1, 2, 2, 64, 200, 16, True, q_std=3.0,
                 k_spike_frac=0.01, k_spike_mult=8.0)
    q, k, v = make_inputs(w, seed=0)
    g = torch.Generator().manual_seed(0)
    q0 = torch.randn(1, 2, 64, 16, generator=g) * 3.0
    k0 = torch.randn(1, 2, 200, 16, generator=g)
    torch.randn(1, 2, 200, 16, generator=g)
    for h in range(2):
        rows = torch.randperm(200, generator=g)[:2]
        k0[0, h, rows] *= 8.0
        others = torch.ones(200, dtype=torch.bool)
        others[rows] = False
        assert torch.equal(k[0, h, rows].float(),
                           (k0[0, h, rows]).to(torch.bfloat16).float())
    assert torch.equal(q, q0.to(torch.bfloat16))
    assert torch.equal(k, k0.to(torch.bfloat16))


def test_headline_workload_shape():
    w = WORKLOADS["pages_b1_h8_q4096_kv8192_d128"]
    assert (w.B, w.Hq, w.Hkv, w.Nq, w.Nkv, w.D, w.causal) == \
        (1, 8, 8, 4096, 8192, 128, False)
    assert w.flops == 4 * 8 * 4096 * 8192 * 128
    assert WORKLOADS["causal_b4_h16_n2048_d64"].flops == \
        4 * 4 * 16 * 2048 * 2048 * 64 / 2


def test_make_custom_shapes():
    q, k, v = make_custom(2, 4, 2, 129, 257, 64)
    assert q.shape == (2, 4, 129, 64) and k.shape == (2, 2, 257, 64)
