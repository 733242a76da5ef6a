"""The C ABI loads, exports what include/sageattn.h declares, and rejects bad
arguments on the host before touching the GPU (CPU-only tests)."""
import ctypes
import os
import re

import pytest

import sage_attention_forward_gb300 as sa

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "sageattn.h")

I64x3 = ctypes.c_int64 * 3


def declared_functions():
    text = open(HEADER).read()
    return re.findall(r"ATTN_API\s+[\w\s\*]+?\b(\w+)\s*\(", text)


def test_every_declared_symbol_is_exported():
    names = declared_functions()
    assert {"attn_fwd_bf16", "sage_prepare", "sage_attn_fwd"} <= set(names)
    L = sa.lib()
    for n in names:
        assert hasattr(L, n), n


def test_status_names_and_padded_length():
    L = sa.lib()
    for code, name in sa.STATUS.items():
        assert L.attn_status_name(code).decode() == name
    assert sa.sage_padded_len(1) == 128 and sa.sage_padded_len(128) == 128 and sa.sage_padded_len(129) == 256
    assert sa.sage_padded_len(76112) == 76160 and sa.sage_padded_len(119056) == 119168
    assert L.sage_prepare_workspace_size(2, 3) == 2 * 3 * 128 * 4
    assert L.sage_attn_workspace_size(1, 40, 76160) == 4 * 40 * 76160 * 128


FAKE = 0x10000  # an aligned non-null address; validation never dereferences it


def call_fwd(q=FAKE, k=FAKE, v=FAKE, o=FAKE, B=1, S=256, H=2, D=128, qs=(256 * 2 * 128, 256, 128), scale=0.088):
    L = sa.lib()
    st = I64x3(*qs)
    return L.attn_fwd_bf16(q, k, v, o, B, S, H, D, st, st, st, st, scale, None)


@pytest.mark.parametrize("kw,status", [
    (dict(D=64), 3),
    (dict(B=0), 0),                    # no query rows: an empty problem, nothing happens
    (dict(H=0, q=0, k=0, v=0, o=0), 0),   # ... and its pointers are not looked at
    (dict(S=0), 1),                    # no keys: attention is undefined
    (dict(H=-1), 1),
    (dict(q=0), 1),
    (dict(o=FAKE + 8), 2),
    (dict(qs=(256 * 2 * 128, 260, 128)), 2),
    (dict(qs=(256 * 2 * 128, -256, 128)), 1),
    (dict(scale=float("inf")), 1),
    (dict(B=65536, H=16384), 1),       # B*H*S_pad/128 = 2^31 CTAs: beyond the grid
    (dict(B=300, H=300, q=0), 1),      # 90000 heads are accepted (then the NULL q is reported)
])
def test_attn_fwd_bf16_rejects_bad_arguments(kw, status):
    assert call_fwd(**kw) == status
    if status:
        assert sa.lib().attn_last_error().decode() != ""


def call_prepare(rope_dim=0, S_pad=256, qn=None, kn=None, ws_bytes=10**6, cos=None):
    L = sa.lib()
    st = I64x3(256 * 2 * 128, 256, 128)
    return L.sage_prepare(FAKE, FAKE, FAKE, 1, 256, 2, 128, st, st, st, 0.088, qn, kn, 1e-6, cos, cos, rope_dim,
                          S_pad, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, ws_bytes, None)


@pytest.mark.parametrize("kw,status", [
    (dict(rope_dim=48, cos=FAKE), 1),
    (dict(rope_dim=64, cos=None), 1),
    (dict(S_pad=200), 1),
    (dict(S_pad=128), 1),
    (dict(qn=FAKE, kn=None), 1),
    (dict(qn=FAKE + 4, kn=FAKE), 2),
    (dict(ws_bytes=16), 1),
])
def test_sage_prepare_rejects_bad_arguments(kw, status):
    assert call_prepare(**kw) == status


def call_prepare_smooth(k_mean=FAKE, ws_bytes=None, S_pad=256, rope_dim=0):
    L = sa.lib()
    st = I64x3(256 * 2 * 128, 256, 128)
    if ws_bytes is None:
        ws_bytes = L.sage_prepare_smooth_k_workspace_size(1, 2, S_pad)
    return L.sage_prepare_smooth_k(FAKE, FAKE, FAKE, 1, 256, 2, 128, st, st, st, 0.088, None, None, 1e-6, None, None,
                                   rope_dim, S_pad, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, k_mean, FAKE, ws_bytes, None)


def test_sage_prepare_smooth_k_workspace_and_rejections():
    L = sa.lib()
    # V maxima (B*H*128 words) + one float per (b, h, 32-row block, channel)
    assert L.sage_prepare_smooth_k_workspace_size(2, 3, 256) == 2 * 3 * 128 * 4 + 2 * 3 * 8 * 128 * 4
    assert L.sage_prepare_smooth_k_workspace_size(0, 3, 256) == 0
    assert call_prepare_smooth(k_mean=None) == 1
    assert call_prepare_smooth(k_mean=FAKE + 4) == 2
    assert call_prepare_smooth(ws_bytes=L.sage_prepare_workspace_size(1, 2)) == 1   # the plain size is too small
    assert call_prepare_smooth(S_pad=200) == 1
    assert call_prepare_smooth(rope_dim=64) == 1                                       # tables missing


def test_sage_attn_fwd_rejects_bad_arguments():
    L = sa.lib()
    st = I64x3(256 * 2 * 128, 256, 128)
    ok_ws = L.sage_attn_workspace_size(1, 2, 256)
    assert L.sage_attn_fwd(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, st, 1, 256, 2, 128, 192, FAKE, ok_ws, None) == 1
    assert L.sage_attn_fwd(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, st, 1, 256, 2, 128, 256, FAKE, 64, None) == 1
    assert L.sage_attn_fwd(FAKE, FAKE + 1, FAKE, FAKE, FAKE, FAKE, FAKE, st, 1, 256, 2, 128, 256, FAKE, ok_ws,
                           None) == 2
    assert L.sage_attn_fwd(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, st, 1, 256, 2, 96, 256, FAKE, ok_ws, None) == 3


def test_sage_attn_fwd_pv16_rejects_bad_arguments():
    L = sa.lib()
    st = I64x3(256 * 2 * 128, 256, 128)
    ws = L.sage_attn_workspace_size(1, 2, 256)

    def call(q8=FAKE, v=FAKE, vst=st, S_pad=256, D=128, ws_bytes=ws):
        return L.sage_attn_fwd_pv16(q8, FAKE, FAKE, FAKE, v, vst, FAKE, st, 1, 256, 2, D, S_pad, FAKE, ws_bytes, None)

    assert call(q8=None) == 1
    assert call(v=None) == 1
    assert call(v=FAKE + 2) == 2
    assert call(vst=I64x3(256 * 2 * 128, 250, 128)) == 2      # s-stride not a multiple of 8 elements
    assert call(S_pad=200) == 1
    assert call(ws_bytes=ws - 1) == 1
    assert call(D=64) == 3


def test_selftest_rejects_bad_pointers():
    L = sa.lib()
    assert L.attn_selftest_wait_timeout(None, FAKE, FAKE, FAKE, None) == 1
    assert L.attn_selftest_wait_timeout(FAKE, FAKE, FAKE, FAKE + 8, None) == 2


def test_sage_attention_one_call_rejects_bad_arguments():
    L = sa.lib()
    st = I64x3(256 * 2 * 128, 256, 128)
    ws = L.sage_attention_workspace_size(1, 2, 256, 0, 0, 0)
    # FP16 Q and K codes, their scales, Q's block means (Q smoothing), e4m3 V^T, V scales and
    # channel maxima, 256-byte pieces
    qmean = 2 * (256 // 32) * 128 * 2
    assert ws == 2 * (2 * 256 * 128 * 2) + 2 * 256 + qmean + 2 * 128 * 256 + 1024 + 1024
    # Q coded inside the forward: no Q codes, scales or means
    assert L.sage_attention_workspace_size(1, 2, 256, 0, 0, 1) == ws - (2 * 256 * 128 * 2) - 256 - qmean
    assert L.sage_attention_workspace_size(1, 2, 256, 0, 1, 0) < ws       # no V in the 16-bit mode
    assert L.sage_attention_workspace_size(1, 2, 256, 1, 0, 0) > ws       # K smoothing adds its sums

    # Q and K coded on load with the 16-bit P V: nothing is prepared, no workspace at all
    assert L.sage_attention_workspace_size(1, 2, 256, 0, 1, 2) == 0
    assert 0 < L.sage_attention_workspace_size(1, 2, 256, 0, 0, 2) < L.sage_attention_workspace_size(1, 2, 256, 0, 0, 1)

    def call(smooth=0, pv=0, o=FAKE, ws_bytes=ws, S=256, qload=0, smooth_q=0, ws_ptr=FAKE):
        return L.sage_attention(FAKE, FAKE, FAKE, 1, S, 2, 128, st, st, st, 0.088, None, None, 1e-6, None, None, 0,
                                smooth_q, smooth, pv, qload, o, st, ws_ptr, ws_bytes, None)

    assert call(pv=0, qload=2, ws_ptr=None, ws_bytes=0) == 1     # e4m3 V still needs its workspace
    if call(pv=1, qload=2, ws_ptr=None, ws_bytes=0) != 0:        # accepted; fails later only for want of a GPU
        assert b"workspace" not in L.attn_last_error()
    assert call(smooth=1, qload=2) == 3          # K's sequence mean needs a pass of its own

    assert call(smooth=2) == 1
    assert call(smooth_q=2) == 1
    assert call(smooth_q=1, qload=1) == 3       # Q coded on load has no block means
    assert call(pv=-1) == 1
    assert call(qload=3) == 1
    assert call(o=FAKE + 2) == 2
    assert call(ws_bytes=ws - 1) == 1
    assert call(S=0) == 1


def test_smoothed_prepare_and_forward_reject_bad_arguments():
    L = sa.lib()
    st = I64x3(256 * 2 * 128, 256, 128)

    def prep(smooth_q=1, smooth_k=0, q_mean=FAKE, k_mean=FAKE):
        return L.sage_prepare_smoothed(FAKE, FAKE, FAKE, 1, 256, 2, 128, st, st, st, 0.088, None, None, 1e-6, None,
                                       None, 0, 256, smooth_q, smooth_k, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, q_mean,
                                       k_mean, FAKE, 1 << 20, None)

    assert prep(smooth_q=2) == 1
    assert prep(smooth_k=-1) == 1
    assert prep(q_mean=None) == 1
    assert prep(q_mean=FAKE + 4) == 2
    assert prep(smooth_q=0, smooth_k=1, k_mean=None) == 1
    ws = L.sage_attn_workspace_size(1, 2, 256)
    assert L.sage_attn_fwd_smooth_q(FAKE, None, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, st, 1, 256, 2, 128, 256, FAKE, ws,
                                    None) == 1
    assert L.sage_attn_fwd_smooth_q(FAKE, FAKE + 8, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, st, 1, 256, 2, 128, 256, FAKE,
                                    ws, None) == 2
    assert L.sage_attn_fwd_pv16_smooth_q(FAKE, None, FAKE, FAKE, FAKE, FAKE, st, FAKE, st, 1, 256, 2, 128, 256, FAKE,
                                         ws, None) == 1


def test_e4m3_encode_rejects_bad_arguments():
    L = sa.lib()
    assert L.sage_e4m3_encode(None, None, 0, None) == 0          # nothing to encode: nothing is touched
    assert L.sage_e4m3_encode(FAKE, FAKE, -1, None) == 1
    assert L.sage_e4m3_encode(None, FAKE, 16, None) == 1
    assert L.sage_e4m3_encode(FAKE, None, 16, None) == 1


def test_product_path_does_not_import_the_oracle():
    import subprocess
    import sys
    code = ("import sys, sage_attention_forward_gb300 as s; s.lib(); "
            "assert not any(m == 'oracle' or m.startswith('oracle.') for m in sys.modules), 'oracle imported'")
    subprocess.run([sys.executable, "-c", code], check=True, cwd=ROOT)
