"""Seeded synthetic inputs for the attention forward.

This module holds only the input recipe (shapes, value distributions, seed):
no attention arithmetic.  Both the GPU tests/benchmark and the CPU oracle
consume what it generates; neither side's arithmetic lives here.

The shapes are the workloads the pages benchmark or that this library is
specified on.  The one shape the pages print is the RTX 5090 benchmark of
"Hacker News Digest — gpu-computing", section "Flash Attention на 5090 в CUDA
C++" (bs=1, heads=8, q=4096, kv=8192, BF16; head_dim 128 from the note that
head_dim=128 fits in registers).  The other four are the tiny parity case,
a causal D=64 batch, causal grouped-query attention and a long causal
sequence with large logits.

Recipe (all configs): one CPU ``torch.Generator`` seeded with ``seed``
draws Q, then K, then V as float32 ``randn`` (Q multiplied by ``q_std`` in
float32 first), each rounded to bf16 (round-to-nearest-even).  For the
large-logit config, after V, each (batch, kv head) draws
``randperm(Nkv)[:round(0.01 * Nkv)]`` and multiplies those K rows by 8 in
float32 before the bf16 rounding (exact either way).  The scale is the
float32 value of 1/sqrt(D).
"""

import math
from dataclasses import dataclass, asdict

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    Hq: int
    Hkv: int
    Nq: int
    Nkv: int
    D: int
    causal: bool
    q_std: float = 1.0
    k_spike_frac: float = 0.0
    k_spike_mult: float = 1.0
    # Q and K quantised per tensor to e4m3 (the fa_fwd_qk8 path)
    qk8: bool = False
    # Q and K quantised to MXFP8: e4m3 with a power-of-two scale per 32
    # head-dim elements (the fa_fwd_mxfp8 path)
    mx: bool = False

    @property
    def scale(self):
        """float32 value of 1/sqrt(D), as a Python float."""
        return float(torch.tensor(1.0 / math.sqrt(self.D), dtype=torch.float32))

    @property
    def flops(self):
        """Algorithmic flops of the forward: 4*B*Hq*Nq*Nkv*D, halved if
        causal (the metric's convention)."""
        f = 4.0 * self.B * self.Hq * self.Nq * self.Nkv * self.D
        return f / 2 if self.causal else f

    def as_dict(self):
        return asdict(self)


WORKLOADS = {
    w.name: w for w in [
        Workload("tiny_128_d64", 1, 1, 1, 128, 128, 64, False),
        Workload("pages_b1_h8_q4096_kv8192_d128", 1, 8, 8, 4096, 8192, 128,
                 False),
        Workload("causal_b4_h16_n2048_d64", 4, 16, 16, 2048, 2048, 64, True),
        Workload("causal_gqa_b2_hq32_hkv8_n8192_d128", 2, 32, 8, 8192, 8192,
                 128, True),
        Workload("causal_b1_h16_n32768_d128_large_logits", 1, 16, 16, 32768,
                 32768, 128, True, q_std=3.0, k_spike_frac=0.01,
                 k_spike_mult=8.0),
        # Few query rows over a long key sequence (a decode/prefill-chunk
        # shape): 32 query blocks, so the split-KV schedule is what fills
        # the GPU.  Not one of the pages' shapes; it measures that schedule.
        Workload("splitkv_b1_hq32_hkv8_q128_kv32768_d128", 1, 32, 8, 128,
                 32768, 128, False),
        # The pages' shape with wide heads (head_dim 192 and 256), run by
        # the one-tile-per-CTA kernel.
        Workload("wide_b1_h8_q4096_kv8192_d192", 1, 8, 8, 4096, 8192, 192,
                 False),
        Workload("wide_b1_h8_q4096_kv8192_d256", 1, 8, 8, 4096, 8192, 256,
                 False),
        Workload("wide_causal_b1_h8_n8192_d256", 1, 8, 8, 8192, 8192, 256,
                 True),
        # The decode/prefill-chunk shape with wide heads: split-KV on the
        # one-tile kernel.
        Workload("splitkv_b1_hq32_hkv8_q128_kv32768_d256", 1, 32, 8, 128,
                 32768, 256, False),
        # The pages' shape at head dim 64.
        Workload("d64_b1_h8_q4096_kv8192", 1, 8, 8, 4096, 8192, 64, False),
        # The pages' shape with e4m3 Q and K (per-tensor descales).
        Workload("qk8_b1_h8_q4096_kv8192_d128", 1, 8, 8, 4096, 8192, 128,
                 False, qk8=True),
        # The pages' shape with MXFP8 Q and K (a scale per 32 elements).
        Workload("mxfp8_b1_h8_q4096_kv8192_d128", 1, 8, 8, 4096, 8192, 128,
                 False, mx=True),
        # The pages' shape with 5 heads: 80 tile pairs fill 53% of the 152
        # SMs, so the stream schedule (equal K/V-block shares per CTA) runs
        # it.  Not one of the pages' shapes; it measures that schedule.
        Workload("stream_b1_h5_q4096_kv8192_d128", 1, 5, 5, 4096, 8192, 128,
                 False),
        # 200 tile pairs (1.3 waves of one pair per SM): stream schedule.
        Workload("stream_b1_h25_q2048_kv8192_d128", 1, 25, 25, 2048, 8192,
                 128, False),
    ]
}

# The configuration the throughput metric is quoted on (the pages' shape).
HEADLINE = "pages_b1_h8_q4096_kv8192_d128"


def make_inputs(w, seed=0, device="cpu"):
    """Generate (q, k, v) bf16 tensors [B,H,N,D] for workload ``w``.

    Always drawn on the CPU generator (so every consumer sees identical
    values), then moved to ``device``.
    """
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    q = torch.randn(w.B, w.Hq, w.Nq, w.D, generator=g, dtype=torch.float32)
    if w.q_std != 1.0:
        q.mul_(w.q_std)
    k = torch.randn(w.B, w.Hkv, w.Nkv, w.D, generator=g, dtype=torch.float32)
    v = torch.randn(w.B, w.Hkv, w.Nkv, w.D, generator=g, dtype=torch.float32)
    if w.k_spike_frac > 0:
        n = int(round(w.k_spike_frac * w.Nkv))
        for b in range(w.B):
            for h in range(w.Hkv):
                rows = torch.randperm(w.Nkv, generator=g)[:n]
                k[b, h, rows] *= w.k_spike_mult
    out = tuple(t.to(torch.bfloat16) for t in (q, k, v))
    if device != "cpu":
        out = tuple(t.to(device) for t in out)
    return out


def make_custom(B, Hq, Hkv, Nq, Nkv, D, seed=0, q_std=1.0):
    """Seeded N(0,1) bf16 inputs of an arbitrary shape (edge-case tests)."""
    w = Workload("custom", B, Hq, Hkv, Nq, Nkv, D, False, q_std=q_std)
    return make_inputs(w, seed)


def make_custom_on_device(B, Hq, Hkv, Nq, Nkv, D, seed=0, device="cuda"):
    """Seeded N(0,1) bf16 inputs drawn directly on a device, for shapes too
    large to draw on the host (maximum-size tests).  Q, then K, then V from
    one generator seeded with ``seed`` on that device."""
    gen = torch.Generator(device=device).manual_seed(seed)
    out = []
    for shape in ((B, Hq, Nq, D), (B, Hkv, Nkv, D), (B, Hkv, Nkv, D)):
        out.append(torch.randn(shape, generator=gen, device=device,
                               dtype=torch.bfloat16))
    return tuple(out)


E4M3_MAX = 448.0


def quantize_e4m3(t):
    """Per-tensor e4m3 quantisation of a bf16 tensor: descale = amax / 448,
    values t / descale rounded to e4m3.  Returns (t8, descale)."""
    amax = float(t.float().abs().max())
    descale = amax / E4M3_MAX if amax > 0 else 1.0
    return (t.float() / descale).to(torch.float8_e4m3fn), descale


def make_qk8_inputs(B, Hq, Hkv, Nq, Nkv, D, seed=0, q_std=1.0):
    """Seeded inputs of the e4m3 Q/K path: the N(0,1) bf16 Q, K, V of
    make_custom with Q and K quantised per tensor.  Returns
    (q8, k8, v, q_descale, k_descale)."""
    q, k, v = make_custom(B, Hq, Hkv, Nq, Nkv, D, seed=seed, q_std=q_std)
    q8, qd = quantize_e4m3(q)
    k8, kd = quantize_e4m3(k)
    return q8, k8, v, qd, kd


MX_BLOCK = 32
E4M3_MIN_NORMAL_EXP = -6


def quantize_mxfp8(t):
    """MXFP8 quantisation of a [..., D] tensor along its last dimension: for
    every block of 32 consecutive elements, the smallest power of two 2^e
    with amax / 2^e <= 448 (e clamped to [-127, 127]; e = -127 for an
    all-zero block) is the block's scale, stored as the ue8m0 byte e + 127,
    and the elements become e4m3 values of t / 2^e (round to nearest; the
    division is exact).  Returns (t8 float8_e4m3fn, scales uint8 [..., D/32]).
    This is the input recipe of the MXFP8 path, not part of the method."""
    x = t.float()
    D = x.shape[-1]
    if D % MX_BLOCK:
        raise ValueError("last dimension must be a multiple of 32")
    xb = x.reshape(*x.shape[:-1], D // MX_BLOCK, MX_BLOCK)
    amax = xb.abs().amax(dim=-1)
    e = torch.where(amax > 0, torch.ceil(torch.log2(amax / E4M3_MAX)),
                    torch.full_like(amax, -127.0))
    # log2 rounding can land one short of the bound: fix by one step
    e = torch.where(amax / torch.exp2(e) > E4M3_MAX, e + 1, e)
    e = e.clamp(-127, 127)
    q8 = (xb / torch.exp2(e).unsqueeze(-1)).reshape(x.shape).to(
        torch.float8_e4m3fn)
    return q8, (e + 127).to(torch.uint8)


def dequantize_mxfp8(t8, scales):
    """The exact values an MXFP8 pair (e4m3 t8, ue8m0 scales) stands for,
    in float64: t8 times 2^(byte - 127) per 32-element block."""
    x = t8.to(torch.float64)
    D = x.shape[-1]
    s = torch.exp2(scales.to(torch.float64) - 127.0)
    return (x.reshape(*x.shape[:-1], D // MX_BLOCK, MX_BLOCK) *
            s.unsqueeze(-1)).reshape(x.shape)


def make_mxfp8_inputs(B, Hq, Hkv, Nq, Nkv, D, seed=0, q_std=1.0):
    """Seeded inputs of the MXFP8 path: the N(0,1) bf16 Q, K, V of
    make_custom with Q and K quantised to MXFP8.  Returns
    (q8, k8, v, q_scale, k_scale)."""
    q, k, v = make_custom(B, Hq, Hkv, Nq, Nkv, D, seed=seed, q_std=q_std)
    q8, qs = quantize_mxfp8(q)
    k8, ks = quantize_mxfp8(k)
    return q8, k8, v, qs, ks
