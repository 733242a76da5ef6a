"""Seeded synthetic inputs for the attention forward and its Sage variant.

This module only draws random tensors and lays them out; it holds none of
the method's arithmetic.  Both the CUDA path (tests, bench) and the CPU
oracle receive the tensors it makes, so the two sides always see the same
bytes.

The workloads are shaped like the diffusion-transformer self-attention
shapes quoted by the ai-infra handbook chapter "Kernel acceleration:
attention, compilation and fusion" (section "Attention: from O(N^2) memory
to blocks", its byte table: FLUX 1024^2, FLUX 2048^2, Wan 2.1 720p,
HunyuanVideo 720p), at head dimension 128 as the aiter pull request
"gfx1201_sage_prepare / gfx1201_sage_attention" fixes it (Technical
Details).  No public dataset is involved: every tensor is drawn from a
seeded generator.

Recipes (one per named workload):
  tiny        B=1 H=2  S=512     Q,K,V ~ N(0,1)
  flux1024    B=1 H=24 S=4608    Q,K,V ~ N(0,1); K[:, :, h, d] += mu[h, d],
                                 mu ~ N(0, 0.5^2) per (head, channel)
  flux2048    B=2 H=24 S=16896   Q,K,V ~ N(0,1); RMSNorm weights for Q and K
                                 ~ U(0.5, 1.5) (BF16, [128]), eps 1e-6;
                                 rotate-half RoPE tables for rope_dim 64,
                                 positions 0..S-1, base 10000
  wan720p     B=1 H=40 S=76112   Q,K,V ~ N(0,1); a token set T of
                                 floor(0.05*S) rows (seeded randperm) is
                                 scaled x8 in Q, K and V (all heads/channels)
  hunyuan720p B=1 H=24 S=119056  Q,K,V ~ N(0,1) stored [B,H,S,D] and passed
                                 as the [B,S,H,D] permuted view (head stride
                                 S*128, sequence stride 128)
  profile_small B=1 H=8 S=32768  Q,K,V ~ N(0,1): the same kernels at a size a
                                 profiler replay finishes quickly
Values are drawn in FP32 and rounded to BF16 by torch's cast.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

HEAD_DIM = 128


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    S: int
    seed: int
    k_channel_offset_std: float = 0.0   # flux1024: per-(head, channel) K mean offset
    q_channel_offset_std: float = 0.0   # Q smoothing cases: per-(head, channel) Q mean offset
    outlier_frac: float = 0.0           # wan720p: fraction of tokens scaled
    outlier_gain: float = 1.0
    head_major_storage: bool = False    # hunyuan720p: [B,H,S,D] storage
    rms_norm: bool = False              # flux2048: fused QK RMSNorm
    rope_dim: int = 0                   # flux2048: fused rotate-half RoPE
    rope_base: float = 10000.0
    rms_eps: float = 1e-6
    D: int = HEAD_DIM

    @property
    def softmax_scale(self) -> float:
        return 1.0 / math.sqrt(self.D)

    @property
    def flops(self) -> int:
        return 4 * self.B * self.H * self.S * self.S * self.D


WORKLOADS = {
    "tiny": Workload("tiny", 1, 2, 512, 1000),
    "flux1024": Workload("flux1024", 1, 24, 4608, 1001, k_channel_offset_std=0.5),
    "flux2048": Workload("flux2048", 2, 24, 16896, 1002, rms_norm=True, rope_dim=64),
    "wan720p": Workload("wan720p", 1, 40, 76112, 1003, outlier_frac=0.05, outlier_gain=8.0),
    "hunyuan720p": Workload("hunyuan720p", 1, 24, 119056, 1004, head_major_storage=True),
}

# A smaller case of the same recipe for profiler captures (each capture replays
# a kernel many times): B=1 H=8 S=32768, Q/K/V ~ N(0,1), 64 MiB per tensor.
WORKLOADS["profile_small"] = Workload("profile_small", 1, 8, 32768, 1005)

# The workload the throughput metric is quoted on.
HEADLINE = "wan720p"


def small_case(B: int, H: int, S: int, seed: int, **kw) -> Workload:
    """A ragged or edge-case shape with the plain N(0,1) recipe."""
    return Workload(f"B{B}H{H}S{S}", B, H, S, seed, **kw)


@dataclass
class Inputs:
    wl: Workload
    q: torch.Tensor            # BF16 [B, S, H, D] (possibly a strided view)
    k: torch.Tensor
    v: torch.Tensor
    q_norm_w: torch.Tensor | None = None   # BF16 [D]
    k_norm_w: torch.Tensor | None = None
    rope_cos: torch.Tensor | None = None   # BF16 [S, rope_dim]
    rope_sin: torch.Tensor | None = None
    outlier_tokens: torch.Tensor | None = None  # int64 token indices
    extra: dict = field(default_factory=dict)


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def rope_tables(S: int, rope_dim: int, base: float = 10000.0):
    """Rotate-half RoPE cos/sin tables, BF16 [S, rope_dim].

    These are inputs of the prepare stage (the caller owns them), drawn from
    the usual 1-D position recipe: angle(s, i) = s * base^(-2i/rope_dim) for
    i < rope_dim/2, evaluated in FP64, the half-table repeated so that
    channel i and channel i + rope_dim/2 share one angle, then rounded to
    BF16.
    """
    half = rope_dim // 2
    i = torch.arange(half, dtype=torch.float64)
    inv_freq = base ** (-2.0 * i / rope_dim)
    pos = torch.arange(S, dtype=torch.float64)
    ang = pos[:, None] * inv_freq[None, :]
    ang = torch.cat([ang, ang], dim=1)
    return torch.cos(ang).to(torch.bfloat16), torch.sin(ang).to(torch.bfloat16)


def make_inputs(wl: Workload, device="cpu") -> Inputs:
    """Draw the workload's tensors on `device` (CPU draws are what the oracle sees)."""
    g = _gen(wl.seed, device)
    B, H, S, D = wl.B, wl.H, wl.S, wl.D
    if wl.head_major_storage:
        shape = (B, H, S, D)
    else:
        shape = (B, S, H, D)

    def draw():
        return torch.randn(shape, generator=g, device=device, dtype=torch.float32)

    q = draw().to(torch.bfloat16)
    k = draw()
    if wl.k_channel_offset_std > 0:
        mu = torch.randn((H, D), generator=g, device=device, dtype=torch.float32) * wl.k_channel_offset_std
        if wl.head_major_storage:
            k = k + mu[None, :, None, :]
        else:
            k = k + mu[None, None, :, :]
    k = k.to(torch.bfloat16)
    v = draw().to(torch.bfloat16)

    inp = Inputs(wl, q, k, v)
    if wl.outlier_frac > 0:
        n_out = int(math.floor(wl.outlier_frac * S))
        perm = torch.randperm(S, generator=g, device=device)
        tok = perm[:n_out]
        inp.outlier_tokens = tok.cpu()
        gain = torch.tensor(wl.outlier_gain, dtype=torch.bfloat16, device=device)
        for t in (q, k, v):
            # [B, S, H, D] layout here (outliers are not combined with head-major storage)
            t[:, tok] = t[:, tok] * gain
    if wl.q_channel_offset_std > 0:
        # drawn after everything else, so that the other tensors match the recipe without it
        mu = torch.randn((H, D), generator=g, device=device, dtype=torch.float32) * wl.q_channel_offset_std
        mu = mu[None, :, None, :] if wl.head_major_storage else mu[None, None, :, :]
        q = (q.float() + mu).to(torch.bfloat16)
        inp.q = q
    if wl.head_major_storage:
        inp.q = q.permute(0, 2, 1, 3)
        inp.k = k.permute(0, 2, 1, 3)
        inp.v = v.permute(0, 2, 1, 3)
    if wl.rms_norm:
        inp.q_norm_w = (torch.rand(D, generator=g, device=device) + 0.5).to(torch.bfloat16)
        inp.k_norm_w = (torch.rand(D, generator=g, device=device) + 0.5).to(torch.bfloat16)
    if wl.rope_dim:
        c, s = rope_tables(S, wl.rope_dim, wl.rope_base)
        inp.rope_cos, inp.rope_sin = c.to(device), s.to(device)
    return inp


def wide_bf16(seed: int, shape, lo_exp: int, hi_exp: int) -> torch.Tensor:
    """BF16 values of random sign with magnitudes m * 2^e, m ~ U[1, 2) and the
    integer e ~ U[lo_exp, hi_exp): inputs at the ends of the BF16 range
    (subnormals from e = -133, near the maximum up to e = 127)."""
    g = _gen(seed, "cpu")
    e = torch.randint(lo_exp, hi_exp, shape, generator=g).to(torch.float64)
    m = 1.0 + torch.rand(shape, generator=g, dtype=torch.float64)
    sign = torch.where(torch.rand(shape, generator=g) < 0.5, -1.0, 1.0).to(torch.float64)
    return (sign * m * torch.pow(2.0, e)).to(torch.bfloat16)


def to_device(inp: Inputs, device) -> Inputs:
    """Copy every tensor to `device`, keeping the logical strides of q/k/v."""
    def mv(t):
        if t is None:
            return None
        if t.dim() == 4 and not t.is_contiguous():
            # keep the permuted-view layout: copy the storage order, then re-view
            base = t.permute(0, 2, 1, 3).contiguous().to(device)
            return base.permute(0, 2, 1, 3)
        return t.to(device)
    out = Inputs(inp.wl, mv(inp.q), mv(inp.k), mv(inp.v), mv(inp.q_norm_w), mv(inp.k_norm_w),
                 mv(inp.rope_cos), mv(inp.rope_sin), inp.outlier_tokens, dict(inp.extra))
    return out


def sample_rows(wl: Workload, n: int, seed: int = 7, outlier_tokens=None, must_include_tail: bool = True):
    """Pick (b, s, h) query rows for row-sampled comparisons.

    Always includes every row of the ragged last 128-row tile (when S is not a
    multiple of 128), a share of outlier tokens when the workload has them, and
    the rest uniformly at random.  Returns an int64 tensor [n, 3].
    """
    g = torch.Generator().manual_seed(seed)
    rows = []
    B, H, S = wl.B, wl.H, wl.S
    if must_include_tail:
        tail0 = (S // 128) * 128
        if tail0 == S:
            tail0 = S - 128 if S >= 128 else 0
        for s in range(tail0, S):
            b = int(torch.randint(B, (1,), generator=g))
            h = int(torch.randint(H, (1,), generator=g))
            rows.append((b, s, h))
    if outlier_tokens is not None and len(outlier_tokens):
        n_out = n // 4
        idx = torch.randint(len(outlier_tokens), (n_out,), generator=g)
        for i in idx.tolist():
            rows.append((int(torch.randint(B, (1,), generator=g)), int(outlier_tokens[i]),
                         int(torch.randint(H, (1,), generator=g))))
    while len(rows) < n:
        rows.append((int(torch.randint(B, (1,), generator=g)), int(torch.randint(S, (1,), generator=g)),
                     int(torch.randint(H, (1,), generator=g))))
    return torch.tensor(rows[:max(n, len(rows))], dtype=torch.int64)
