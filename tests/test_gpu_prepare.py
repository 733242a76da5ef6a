"""sage_prepare (CUDA, through the C ABI) is bit-exact against the oracle:
INT8 Q/K codes, e4m3 V codes and all FP32 scales, on every workload and on
small ragged shapes, with and without the fused RMSNorm + RoPE."""
import dataclasses
import math

import numpy as np
import pytest
import torch

import oracle
import sage_attention_forward_gb300 as sa
from workloads import make_inputs, rope_tables, small_case, to_device, wide_bf16

pytestmark = pytest.mark.gpu


def assert_prepared_equal(prep, exp, what=""):
    for name in ("q_i8", "k_i8", "v_fp8", "q_scale", "k_scale", "v_scale"):
        got = getattr(prep, name).cpu()
        ref = exp[name]
        if got.dtype == torch.float32:
            same = torch.equal(got.view(torch.int32), ref.view(torch.int32))
        else:
            same = torch.equal(got, ref)
        if not same:
            diff = (got.view(torch.uint8) != ref.view(torch.uint8)) if got.dtype != torch.float32 else (got != ref)
            idx = diff.nonzero()[:5].tolist()
            raise AssertionError(f"{what}: {name} differs at {int(diff.sum())} places, first {idx}")


def run(inp, dev, S_pad=None, **kw):
    g = to_device(inp, dev)
    norm = {}
    if g.q_norm_w is not None:
        norm = dict(q_norm_w=g.q_norm_w, k_norm_w=g.k_norm_w, rms_eps=inp.wl.rms_eps)
    rope = {}
    if g.rope_cos is not None:
        rope = dict(rope_cos=g.rope_cos, rope_sin=g.rope_sin, rope_dim=inp.wl.rope_dim)
    prep = sa.sage_prepare(g.q, g.k, g.v, softmax_scale=inp.wl.softmax_scale, S_pad=S_pad, **norm, **rope, **kw)
    torch.cuda.synchronize()
    exp = oracle.prepare(inp.q, inp.k, inp.v, inp.wl.softmax_scale, S_pad=prep.S_pad,
                         q_norm_w=inp.q_norm_w, k_norm_w=inp.k_norm_w, rms_eps=inp.wl.rms_eps,
                         rope_cos=inp.rope_cos, rope_sin=inp.rope_sin, rope_dim=inp.wl.rope_dim)
    return prep, exp


@pytest.mark.parametrize("B,H,S", [(1, 1, 1), (1, 3, 31), (2, 1, 33), (1, 2, 127), (1, 3, 129), (2, 2, 200),
                                   (1, 1, 1000)])
def test_small_ragged_bit_exact(cuda_dev, B, H, S):
    inp = make_inputs(small_case(B, H, S, 200 + S))
    prep, exp = run(inp, cuda_dev)
    assert_prepared_equal(prep, exp, f"B{B} H{H} S{S}")


@pytest.mark.parametrize("H", [32, 33])
def test_both_quantiser_layouts_bit_exact(cuda_dev, H):
    # the quantiser takes four warps per 32-row block up to 4096 blocks per task and two
    # beyond: S = 4000 pads to 4096 rows, 128 blocks a head, so 32 heads sit exactly at the
    # bound and 33 just past it; RMSNorm and RoPE on, a ragged last block
    inp = make_inputs(small_case(1, H, 4000, 4000 + H, rms_norm=True, rope_dim=64))
    prep, exp = run(inp, cuda_dev)
    assert prep.S_pad == 4096 and H * prep.S_pad // 32 in (4096, 4224)
    assert_prepared_equal(prep, exp, f"H={H}")


def test_extra_padding_is_zero(cuda_dev):
    inp = make_inputs(small_case(1, 2, 100, 3))
    prep, exp = run(inp, cuda_dev, S_pad=512)
    assert_prepared_equal(prep, exp, "S_pad 512")
    assert (prep.q_i8[:, :, 100:] == 0).all() and (prep.v_fp8[..., 100:] == 0).all()


@pytest.mark.parametrize("rope_dim", [0, 32, 64, 96, 128])
@pytest.mark.parametrize("norm", [False, True])
def test_norm_rope_bit_exact(cuda_dev, rope_dim, norm):
    if rope_dim == 0 and not norm:
        pytest.skip("covered by the plain cases")
    inp = make_inputs(small_case(2, 3, 300, 300 + rope_dim, rms_norm=norm, rope_dim=rope_dim))
    prep, exp = run(inp, cuda_dev)
    assert_prepared_equal(prep, exp, f"norm={norm} rope_dim={rope_dim}")


def test_norm_with_zero_eps_and_ragged_tail(cuda_dev):
    """rms_eps = 0 (a valid argument): the padding rows of the last 32-row block,
    zeros whose RMSNorm factor would be infinite, still code to 0 and leave the
    block's maximum alone; the S real rows are bit-exact against the oracle."""
    inp = make_inputs(dataclasses.replace(small_case(1, 2, 300, 63, rms_norm=True, rope_dim=64), rms_eps=0.0))
    prep, exp = run(inp, cuda_dev)
    assert_prepared_equal(prep, exp, "rms_eps 0, S 300")
    assert (prep.q_i8[:, :, 300:] == 0).all() and (prep.k_i8[:, :, 300:] == 0).all()


def test_fused_equals_unfused(cuda_dev):
    """Prepare with RMSNorm + RoPE fused equals prepare without them applied to the
    normalised, rotated BF16 tensors (aiter pull request, Test Result: fused == unfused)."""
    inp = make_inputs(small_case(1, 4, 500, 41, rms_norm=True, rope_dim=64))
    prep, _ = run(inp, cuda_dev)
    qn = oracle.norm_rope(inp.q, inp.q_norm_w, inp.wl.rms_eps, inp.rope_cos, inp.rope_sin, 64).to(cuda_dev)
    kn = oracle.norm_rope(inp.k, inp.k_norm_w, inp.wl.rms_eps, inp.rope_cos, inp.rope_sin, 64).to(cuda_dev)
    plain = sa.sage_prepare(qn, kn, inp.v.to(cuda_dev), softmax_scale=inp.wl.softmax_scale)
    torch.cuda.synchronize()
    for name in ("q_i8", "k_i8", "v_fp8", "q_scale", "k_scale", "v_scale"):
        assert torch.equal(getattr(prep, name), getattr(plain, name)), name


def test_extreme_magnitudes_bit_exact(cuda_dev):
    """Q/K blocks at the ends of the BF16 range: blocks whose largest |x| is so
    small that 127 / max overflows to infinity (every code is then +-127),
    subnormal blocks, blocks near the BF16 maximum and blocks spanning 2^-120 to
    2^120; V of magnitudes 2^-100 to 2^100.  Bit-exact against the oracle."""
    S, H = 256, 2
    ranges = [(-130, -123), (-120, 120), (100, 127), (-133, -126), (-20, 20), (-126, -100), (0, 1), (-60, 60)]
    def qk(seed):
        return torch.cat([wide_bf16(seed + i, (1, 32, H, 128), lo, hi) for i, (lo, hi) in enumerate(ranges)], dim=1)
    inp = make_inputs(small_case(1, H, S, 61))
    inp.q, inp.k, inp.v = qk(100), qk(200), wide_bf16(300, (1, S, H, 128), -100, 100)
    prep, exp = run(inp, cuda_dev)
    assert_prepared_equal(prep, exp, "extreme magnitudes")
    codes = prep.q_i8[0, 0, :32].cpu()
    assert (codes.abs() == 127).all()                     # the overflowing block


def test_norm_rope_extreme_tables_bit_exact(cuda_dev):
    """RMSNorm weights of magnitude 2^-100 to 2^20 (Q) and 2^-125 to 2^-95 (K),
    RoPE tables of 2^-60 to 2^10 (any BF16 tables are valid input): K's rounded
    products reach the BF16 subnormal range and below (7 % of its values end
    subnormal, 15 % zero), where eager BF16 rounds the binary32 result and the
    prepare rounds a BF16 product directly.  Bit-exact against the oracle."""
    S, H, rd = 256, 2, 64
    inp = make_inputs(small_case(1, H, S, 62, rms_norm=True, rope_dim=rd))
    inp.q_norm_w, inp.k_norm_w = wide_bf16(400, (128,), -100, 20), wide_bf16(401, (128,), -125, -95)
    inp.rope_cos, inp.rope_sin = wide_bf16(402, (S, rd), -60, 10), wide_bf16(403, (S, rd), -60, 10)
    prep, exp = run(inp, cuda_dev)
    assert_prepared_equal(prep, exp, "extreme norm weights and RoPE tables")


@pytest.mark.parametrize("name", ["tiny", "flux1024", "flux2048", "wan720p", "hunyuan720p"])
def test_workloads_bit_exact(cuda_dev, workload_inputs, name):
    cpu, g = workload_inputs(name)
    kw = {}
    if g.q_norm_w is not None:
        kw.update(q_norm_w=g.q_norm_w, k_norm_w=g.k_norm_w, rms_eps=cpu.wl.rms_eps)
    if g.rope_cos is not None:
        kw.update(rope_cos=g.rope_cos, rope_sin=g.rope_sin, rope_dim=cpu.wl.rope_dim)
    prep = sa.sage_prepare(g.q, g.k, g.v, softmax_scale=cpu.wl.softmax_scale, **kw)
    torch.cuda.synchronize()
    exp = oracle.prepare(cpu.q, cpu.k, cpu.v, cpu.wl.softmax_scale, S_pad=prep.S_pad, q_norm_w=cpu.q_norm_w,
                         k_norm_w=cpu.k_norm_w, rms_eps=cpu.wl.rms_eps, rope_cos=cpu.rope_cos,
                         rope_sin=cpu.rope_sin, rope_dim=cpu.wl.rope_dim)
    assert_prepared_equal(prep, exp, name)


def test_deterministic_non_default_stream(cuda_dev):
    inp = make_inputs(small_case(1, 3, 777, 42, rms_norm=True, rope_dim=32))
    g = to_device(inp, cuda_dev)
    kw = dict(q_norm_w=g.q_norm_w, k_norm_w=g.k_norm_w, rope_cos=g.rope_cos, rope_sin=g.rope_sin, rope_dim=32)
    a = sa.sage_prepare(g.q, g.k, g.v, **kw)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        b = sa.sage_prepare(g.q, g.k, g.v, stream=s, **kw)
    s.synchronize()
    torch.cuda.synchronize()
    for name in ("q_i8", "k_i8", "v_fp8", "q_scale", "k_scale", "v_scale"):
        assert torch.equal(getattr(a, name), getattr(b, name)), name
