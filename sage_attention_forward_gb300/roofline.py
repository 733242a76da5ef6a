"""Work and traffic accounting for the attention forward and the Sage prepare.

These are the algorithmic counts the throughput metric and the roofline
fractions are computed from; they do not depend on how a kernel is written.

* Attention FLOPs: 4 * B * H * S^2 * D -- two GEMMs of 2*S*S*D each per
  (batch, head).  This is the count the aiter pull request
  "gfx1201_sage_prepare / gfx1201_sage_attention" divides by the time to
  report TFLOPS (How to reproduce, with D = 128) and the `4 * n * n * d`
  of the ai-infra handbook chapter "Kernel acceleration: attention,
  compilation and fusion" (block_profile table, row "attention (Flash)").
* Attention minimum bytes (flash form): read Q, K, V once and write O once,
  the `flash` term of the same chapter's attn_bytes example (section
  "Attention: from O(N^2) memory to blocks").
* Naive bytes: write the N x N scores, read them back, plus Q, K, V and O
  (same example's `naive` term).
* Prepare bytes: read Q, K, V (BF16), read V a second time (the per-channel
  V maximum must be known before any V element can be encoded), write the
  INT8 Q/K and e4m3 V at the padded length, their FP32 scales, and the
  optional norm weights and RoPE tables.
"""
from __future__ import annotations


def attention_flops(B: int, H: int, S: int, D: int = 128) -> int:
    return 4 * B * H * S * S * D


def score_matrix_bytes(S: int, H: int, B: int = 1, elem: int = 2) -> int:
    return B * H * S * S * elem


def flash_bytes(B: int, H: int, S: int, D: int = 128, elem: int = 2) -> int:
    """Q, K, V read once, O written once."""
    return 4 * B * S * H * D * elem


def naive_bytes(B: int, H: int, S: int, D: int = 128, elem: int = 2) -> int:
    """Scores written and read back, plus the flash traffic."""
    return 2 * score_matrix_bytes(S, H, B, elem) + flash_bytes(B, H, S, D, elem)


def sage_fwd_min_bytes(B: int, H: int, S: int, S_pad: int, D: int = 128) -> int:
    """INT8 Q/K + e4m3 V read once, BF16 O written once, plus the scales."""
    codes = 3 * B * H * S_pad * D
    scales = 2 * B * H * (S_pad // 32) * 4 + B * H * D * 4
    return codes + scales + B * S * H * D * 2


def prepare_bytes(B: int, H: int, S: int, S_pad: int, D: int = 128, rms_norm: bool = False,
                  rope_dim: int = 0) -> int:
    read = 3 * B * S * H * D * 2          # Q, K, V in BF16
    reread_v = B * S * H * D * 2          # second pass over V after its channel maxima are known
    write = 3 * B * H * S_pad * D         # INT8 Q, K and e4m3 V (1 byte each)
    scales = 2 * B * H * (S_pad // 32) * 4 + B * H * D * 4
    extra = 0
    if rms_norm:
        extra += 2 * D * 2
    if rope_dim:
        extra += 2 * S * rope_dim * 2     # cos and sin tables, read once
    return read + reread_v + write + scales + extra


def prepare_smooth_k_bytes(B: int, H: int, S: int, S_pad: int, D: int = 128, rms_norm: bool = False,
                           rope_dim: int = 0) -> int:
    """prepare_bytes plus K smoothing: one more pass over K for its block sums,
    which are written once and read once, and the per-channel means."""
    extra_k = B * S * H * D * 2
    partials = 2 * B * H * (S_pad // 32) * D * 4
    means = 2 * B * H * D * 4
    return prepare_bytes(B, H, S, S_pad, D, rms_norm, rope_dim) + extra_k + partials + means


# Dense tcgen05 MMA throughput per SM per clock on the GB300, measured by a probe
# that issues back-to-back 128 x 128 (x 16 or x 32) MMAs from one thread and times
# them with %clock64: kind::f16 (BF16 or FP16 operands, FP32 accumulator)
# 8188 FLOP/clk/SM, kind::f8f6f4 with e4m3 operands 16376 FLOP/clk/SM.  The
# clock-normalised roof of a kernel is this rate x SMs x its own average SM clock,
# which takes the power-capped clock of a long run out of the fraction.
TC_FLOP_PER_CLK_SM = {"f16": 8188.0, "e4m3": 16376.0}


def sage_flop_per_clk_sm() -> float:
    """The Sage forward's mixed rate: half of the FLOPs (Q K^T, INT8 codes widened to
    FP16) at the kind::f16 rate, half (P V) at the e4m3 rate."""
    return 2.0 / (1.0 / TC_FLOP_PER_CLK_SM["f16"] + 1.0 / TC_FLOP_PER_CLK_SM["e4m3"])


def clock_peak_tflops(flop_per_clk_sm: float, n_sms: int, sm_mhz: float) -> float:
    return flop_per_clk_sm * n_sms * sm_mhz * 1e6 / 1e12
