"""The library's own linkage, the check the RDNA2 DiT flash-kernel note reports
(Results and Reproducibility / Provenance: the note's kernel links against the base
runtime and the operating system's libraries and nothing more): the built
libsageattn.so needs the CUDA runtime and the C/C++ system libraries and nothing
else -- no cuBLAS, cuDNN or other kernel library.  The TMA descriptor
encoder is reached through the runtime's driver entry point, so libcuda is not
linked either.  Reads the dynamic section with readelf; no GPU involved."""
import re
import shutil
import subprocess

import pytest

from sage_attention_forward_gb300 import build as lib_build

ALLOWED = re.compile(r"^(libcudart\.so\.\d+|libstdc\+\+\.so\.\d+|libgcc_s\.so\.\d+|libc\.so\.\d+|libm\.so\.\d+|"
                     r"libdl\.so\.\d+|libpthread\.so\.\d+|librt\.so\.\d+|ld-linux[-\w]*\.so\.\d+)$")


def test_library_links_only_the_cuda_runtime():
    if shutil.which("readelf") is None:
        pytest.skip("readelf not available")
    lib = lib_build.build()
    out = subprocess.run(["readelf", "-d", lib], capture_output=True, text=True, check=True).stdout
    needed = re.findall(r"\(NEEDED\)\s+Shared library: \[([^\]]+)\]", out)
    assert any(n.startswith("libcudart.so") for n in needed), needed
    extra = [n for n in needed if not ALLOWED.match(n)]
    assert not extra, f"unexpected dependencies: {extra}"
