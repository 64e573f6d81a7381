"""The quantizer kernels form rn(bamax / 6) (the block-scale step) as
rn(b * rn(1/6)) corrected once with the exact fused-multiply-add residual when
b >= 2^-124, and by division below that.  This checks, on the host in IEEE
binary32 with a hardware fused multiply-add, that the shortcut equals the
correctly rounded quotient for every binary32 b in [2^-124, FLT_MAX]."""
import os
import platform
import subprocess
import tempfile

SRC = r"""
#include <stdio.h>
#include <stdint.h>
#include <string.h>
#include <math.h>
int main(void)
{
    volatile float six = 6.0f;
    const float r6 = 0x1.555556p-3f;
    if (r6 != 1.0f / six) { printf("bad reciprocal\n"); return 2; }
    unsigned long long bad = 0;
    for (uint32_t u = 0x01800000u; u < 0x7F800000u; ++u) {
        float b, q1, ref;
        memcpy(&b, &u, 4);
        ref = b / six;
        float q0 = b * r6;
        q1 = fmaf(fmaf(-6.0f, q0, b), r6, q0);
        if (memcmp(&q1, &ref, 4) != 0)
            ++bad;
    }
    printf("%llu\n", bad);
    return bad != 0;
}
"""


def test_fma_corrected_division_by_six_is_exact():
    with tempfile.TemporaryDirectory() as d:
        c = os.path.join(d, "div6.c")
        exe = os.path.join(d, "div6")
        open(c, "w").write(SRC)
        flags = ["-O2", "-ffp-contract=off", "-fno-fast-math"]
        if platform.machine() in ("x86_64", "AMD64"):
            flags.append("-mfma")  # fmaf as one instruction (aarch64 has it in the base ISA)
        subprocess.check_call(["gcc", *flags, c, "-o", exe, "-lm"])
        out = subprocess.run([exe], capture_output=True, text=True, timeout=600)
        assert out.returncode == 0 and out.stdout.strip() == "0", out.stdout
