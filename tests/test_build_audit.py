"""GPU-free resource audit of the compiled kernels (the RDNAttention README,
section "Tests": a check that needs only the compiler and fails on any register
spill).  Every kernel of the library is cross-compiled for sm_103a with
``-Xptxas -v``. The test requires that none spills. It also requires that the
attention kernel stays within the per-thread register budget of its launch:
320 threads (10 warps) per CTA, one CTA per SM. Two of the SM's four
sub-partitions then hold three warps, and 3 x 32 x regs must fit a
sub-partition's 16384 registers, so regs <= 170, or 168 in the allocation's
8-register granules.
"""
import os
import re
import subprocess

import pytest

from sage_attention_forward_gb300 import build as lib_build

REG_BUDGET_ATTN = 168
# The two opt-in instantiations that code K tiles on load run the row coder inside the
# softmax loop, next to the loop's own state; a few words of that state go to local memory
# there (measured 16 and 94 bytes of spill stores plus loads).  Any other kernel, and any
# growth past this, fails.
KLOAD_SPILL_BUDGET = 128


def is_k_on_load(name):
    return "attn_fwd_kernel" in name and "ELb1ELb1E" in name


def ptxas_report(src, tmp_path):
    """Compile one translation unit with the library's own flags; return
    {function: {"regs": n, "spill": bytes, "entry": bool}} from ptxas's
    statistics (kernels, and device functions compiled as calls)."""
    out = tmp_path / (os.path.basename(src) + ".o")
    cmd = [lib_build.nvcc()] + lib_build._flags(["-Xptxas", "-v"]) + ["-c", src, "-o", str(out)]
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stderr[-3000:]
    kernels, current = {}, None
    for line in (r.stdout + r.stderr).splitlines():
        m = re.search(r"Compiling entry function '([^']+)'", line)
        if m:
            current = m.group(1)
            kernels[current] = {"regs": None, "spill": None, "entry": True}
            continue
        m = re.search(r"Function properties for (\S+)", line)
        if m:
            current = m.group(1)
            # a called function is reported once per kernel that calls it: keep the worst
            kernels.setdefault(current, {"regs": None, "spill": None, "entry": False})
            continue
        if current is None:
            continue
        m = re.search(r"(\d+) bytes spill stores, (\d+) bytes spill loads", line)
        if m:
            kernels[current]["spill"] = max(kernels[current]["spill"] or 0, int(m.group(1)) + int(m.group(2)))
        m = re.search(r"Used (\d+) registers", line)
        if m:
            kernels[current]["regs"] = int(m.group(1))
    return kernels


@pytest.mark.parametrize("src", lib_build.SOURCES)
def test_no_kernel_spills(src, tmp_path):
    kernels = ptxas_report(os.path.join(lib_build.CSRC, src), tmp_path)
    if src != "api.cu":                              # api.cu holds host entry points
        assert kernels, f"{src}: no kernels in the ptxas report"
    for name, st in kernels.items():
        assert st["spill"] is not None, f"{name}: incomplete report {st}"
        assert st["regs"] is not None or not st["entry"], f"{name}: incomplete report {st}"
        if st["entry"] and is_k_on_load(name):
            assert st["spill"] <= KLOAD_SPILL_BUDGET, f"{name} spills: {st}"
        else:
            assert st["spill"] == 0, f"{name} spills: {st}"
    if src == "attn_fwd.cu":
        attn = {n: st for n, st in kernels.items() if "attn_fwd_kernel" in n and st["entry"]}
        # the BF16, Sage FP8-PV and Sage 16-bit-PV modes, the two Sage modes also with Q
        # quantised on load, and with Q and K quantised on load
        assert len(attn) == 7, sorted(attn)
        for name, st in attn.items():
            assert st["regs"] <= REG_BUDGET_ATTN, f"{name} uses {st['regs']} registers"
