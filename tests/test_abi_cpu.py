"""C-ABI checks that need no GPU: the library builds/loads, exports every
function include/*.h declares, and rejects bad arguments on the host before
touching the device."""
import ctypes
import glob
import os
import re
import subprocess

import pytest

import nvfp4_bit_quantized_quantize_gb300 as nv
from nvfp4_bit_quantized_quantize_gb300 import build as nvbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        src = open(h).read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        names |= set(re.findall(r"^\s*[A-Za-z_][\w\s\*]*?\b(nvfp4_\w+)\s*\(", src, flags=re.M))
    return names


@pytest.fixture(scope="module")
def lib():
    nvbuild.build()
    return nv.load()


def test_header_declares_the_boundary():
    names = _declared()
    for n in ["nvfp4_quantize", "nvfp4_quantize_2d", "nvfp4_rht_quantize", "nvfp4_gemm", "nvfp4_sf_bytes",
              "nvfp4_workspace_bytes", "nvfp4_workspace_init", "nvfp4_device_status", "nvfp4_status_str"]:
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", nv.LIB_PATH], capture_output=True, text=True).stdout
    exported = set(re.findall(r"\bT (nvfp4_\w+)$", out, flags=re.M))
    declared = _declared()
    assert declared, "no declarations found"
    assert declared <= exported, declared - exported
    assert set(nv.EXPORTS) == declared
    for n in declared:
        assert hasattr(lib, n)


def test_sizes_and_status_strings(lib):
    assert nv.nvfp4_sf_bytes(256, 256) == 256 * 16
    assert nv.nvfp4_sf_bytes(1, 16) == 512
    assert nv.nvfp4_sf_bytes(129, 1040) == 256 * 68
    assert nv.nvfp4_workspace_bytes() == 256
    assert nv.nvfp4_status_str(0) == "ok"
    assert nv.nvfp4_status_str(4) == "non-finite input"


def test_host_validation_rejects_before_launch(lib):
    # null pointers and bad shapes return synchronously, no device touched
    L = lib
    fake = 1 << 20  # aligned, never dereferenced
    assert L.nvfp4_quantize(None, 16, 16, 16, 0, 0, fake, fake, fake, fake, None) == 1
    assert L.nvfp4_quantize(fake, 16, 16, 16, 7, 0, fake, fake, fake, fake, None) == 1
    assert L.nvfp4_quantize(fake, 16, 24, 24, 0, 0, fake, fake, fake, fake, None) == 2
    assert L.nvfp4_quantize(fake, 0, 16, 16, 0, 0, fake, fake, fake, fake, None) == 2
    assert L.nvfp4_quantize(fake + 8, 16, 16, 16, 0, 0, fake, fake, fake, fake, None) == 3
    assert L.nvfp4_quantize(fake, 16, 32, 36, 0, 0, fake, fake, fake, fake, None) == 3
    assert L.nvfp4_quantize_2d(fake, 24, 32, 32, fake, fake, fake, None, fake, fake, None) == 1
    assert L.nvfp4_quantize_2d(fake, 24, 32, 32, fake, fake, None, None, fake, fake, None) == 2
    assert L.nvfp4_rht_quantize(fake, 24, 32, 32, 1, 0, 0, fake, fake, fake, fake, None) == 2
    # GEMM: any M, N > 0; K a positive multiple of 32
    assert L.nvfp4_gemm(fake, fake, fake, fake, fake, fake, 0, 128, 64, fake, 128, 0, fake, None) == 2
    assert L.nvfp4_gemm(fake, fake, fake, fake, fake, fake, 128, 0, 64, fake, 128, 0, fake, None) == 2
    assert L.nvfp4_gemm(fake, fake, fake, fake, fake, fake, 128, 128, 80, fake, 128, 0, fake, None) == 2
    assert L.nvfp4_gemm(fake, fake, fake, fake, fake, fake, 128, 128, 0, fake, 128, 0, fake, None) == 2
    assert L.nvfp4_gemm(fake, fake, fake, fake, fake, fake, 100, 130, 64, fake, 128, 0, fake, None) == 2
    assert L.nvfp4_gemm(fake, fake, fake, fake, fake, fake, 100, 130, 64, fake, 134, 1, fake, None) == 3
    assert L.nvfp4_gemm(fake, fake, fake, fake, fake, fake, 128, 128, 64, fake, 128, 5, fake, None) == 1
    assert L.nvfp4_gemm(fake, fake, fake, fake, fake, fake, 128, 128, 64, fake, 132, 0, fake, None) == 3
    # dual quantizer: T % 16 and C % 16
    assert L.nvfp4_quantize_dual(fake, 32, 40, 40, 0, 0, fake, fake, fake, 1, 1, 0, fake, fake, fake, fake,
                                 None) == 2
    assert L.nvfp4_quantize_dual(fake, 24, 32, 32, 0, 0, fake, fake, fake, 1, 1, 0, fake, fake, fake, fake,
                                 None) == 2
    assert L.nvfp4_quantize_dual(fake, 32, 32, 32, 0, 0, fake, fake, fake, 1, 3, 0, fake, fake, fake, fake,
                                 None) == 1
    assert L.nvfp4_quantize_dual(fake, 32, 32, 32, 0, 0, fake, fake, fake, 1, 1, 0, None, fake, fake, fake,
                                 None) == 1
    # GEMM with output maxima: M % 16, N % 16, an amax buffer, bf16 output rows of 16-byte multiples
    assert L.nvfp4_gemm_amax(fake, fake, fake, fake, fake, fake, 24, 32, 64, fake, 32, 0, fake, fake, None) == 2
    assert L.nvfp4_gemm_amax(fake, fake, fake, fake, fake, fake, 32, 40, 64, fake, 40, 0, fake, fake, None) == 2
    assert L.nvfp4_gemm_amax(fake, fake, fake, fake, fake, fake, 32, 32, 80, fake, 32, 0, fake, fake, None) == 2
    assert L.nvfp4_gemm_amax(fake, fake, fake, fake, fake, fake, 32, 32, 64, fake, 32, 0, None, fake, None) == 1
    assert L.nvfp4_gemm_amax(fake, fake, fake, fake, fake, fake, 32, 32, 64, fake, 36, 0, fake, fake, None) == 3
    assert L.nvfp4_gemm_amax(fake, fake, fake, fake, fake, fake, 32, 32, 64, fake, 32, 0, fake + 2, fake, None) == 3
    # one-read dual quantizer: an amax buffer (4-byte aligned), then the dual quantizer's rules
    assert L.nvfp4_quantize_dual_from_amax(fake, 32, 32, 32, None, 0, 0, fake, fake, fake, 1, 1, 0, fake, fake,
                                           fake, fake, None) == 1
    assert L.nvfp4_quantize_dual_from_amax(fake, 32, 32, 32, fake + 2, 0, 0, fake, fake, fake, 1, 1, 0, fake,
                                           fake, fake, fake, None) == 3
    assert L.nvfp4_quantize_dual_from_amax(fake, 24, 32, 32, fake, 0, 0, fake, fake, fake, 1, 1, 0, fake, fake,
                                           fake, fake, None) == 2
    assert L.nvfp4_workspace_init(None, None) == 1
    # noise meter: cols % 16, 8-byte aligned sums
    assert L.nvfp4_quant_noise(fake, 16, 24, 24, fake, fake, fake, fake, None) == 2
    assert L.nvfp4_quant_noise(fake, 16, 32, 32, fake, fake, fake, fake + 4, None) == 3
    assert L.nvfp4_quant_noise(fake, 16, 32, 32, None, fake, fake, fake, None) == 1
    # MXFP4: 32-element blocks; its GEMM has the same shape rules as NVFP4's
    assert L.nvfp4_mxfp4_quantize(fake, 16, 48, 48, fake, fake, fake, None) == 2
    assert L.nvfp4_mxfp4_quantize(fake, 16, 64, 64, fake, fake, None, None) == 1
    assert L.nvfp4_mxfp4_gemm(fake, fake, fake, fake, 128, 128, 80, fake, 128, 0, fake, None) == 2
    assert L.nvfp4_mxfp4_gemm(fake, fake, fake, fake, 128, 128, 64, fake, 132, 0, fake, None) == 3
    # allocation-free quantizer: mode, shape, alignment
    assert L.nvfp4_quantize_noalloc(fake, 16, 16, 16, 5, 0, fake, fake, fake, None) == 1
    assert L.nvfp4_quantize_noalloc(fake, 16, 24, 24, 0, 0, fake, fake, fake, None) == 2
    assert L.nvfp4_quantize_noalloc(fake + 8, 16, 16, 16, 0, 0, fake, fake, fake, None) == 3
