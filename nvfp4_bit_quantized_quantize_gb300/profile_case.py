"""Run one kernel of the library on synthetic device data, for profiling.

  python -m nvfp4_bit_quantized_quantize_gb300.profile_case gemm M N K [reps]
  python -m nvfp4_bit_quantized_quantize_gb300.profile_case quantize ROWS COLS rn|sr [reps]
  python -m nvfp4_bit_quantized_quantize_gb300.profile_case quantize_2d ROWS COLS [reps]
  python -m nvfp4_bit_quantized_quantize_gb300.profile_case rht T C rn|sr [reps]
  python -m nvfp4_bit_quantized_quantize_gb300.profile_case dual T C rn|sr [reps]
  python -m nvfp4_bit_quantized_quantize_gb300.profile_case noise ROWS COLS [reps]

Inputs are made on the device (random codes and E4M3 scales for the GEMM,
N(0,1) bf16 for the quantizers); each case runs 2 warm-up launches and then
`reps` launches (default 3), then prints the mean time per launch from CUDA
events.  Numbers printed while a profiler is attached are not benchmarks.
"""
from __future__ import annotations

import sys

import torch

import nvfp4_bit_quantized_quantize_gb300 as nv


def _time(fn, reps):
    for _ in range(2):
        fn()
    torch.cuda.synchronize()
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(reps):
        fn()
    b.record()
    torch.cuda.synchronize()
    return a.elapsed_time(b) / reps


def main(argv):
    kind = argv[0]
    torch.manual_seed(0)
    ws = nv.alloc_workspace()
    if kind == "gemm":
        M, N, K = (int(v) for v in argv[1:4])
        reps = int(argv[4]) if len(argv) > 4 else 3
        a = torch.randint(0, 256, (M, K // 2), dtype=torch.uint8, device="cuda")
        b = torch.randint(0, 256, (N, K // 2), dtype=torch.uint8, device="cuda")
        sfa = torch.randint(0x30, 0x48, (nv.nvfp4_sf_bytes(M, K),), dtype=torch.uint8, device="cuda")
        sfb = torch.randint(0x30, 0x48, (nv.nvfp4_sf_bytes(N, K),), dtype=torch.uint8, device="cuda")
        ga = torch.ones(1, device="cuda")
        gb = torch.ones(1, device="cuda")
        d = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
        ms = _time(lambda: nv.nvfp4_gemm(a, sfa, ga, b, sfb, gb, M, N, K, d, N, nv.OUT_BF16, ws), reps)
        print(f"gemm {M}x{N}x{K}: {ms:.4f} ms, {2 * M * N * K / ms / 1e9:.1f} TFLOP/s")
    else:
        R, C = int(argv[1]), int(argv[2])
        mode = nv.SR if (len(argv) > 3 and argv[3] == "sr") else nv.RN
        rest = argv[4:] if kind in ("quantize", "rht", "dual") else argv[3:]
        reps = int(rest[0]) if rest else 3
        x = torch.randn((R, C), dtype=torch.bfloat16, device="cuda")
        if kind == "quantize":
            q, sf, g = nv.alloc_quantized(R, C)
            fn = lambda: nv.nvfp4_quantize(x, R, C, C, mode, 1, q, sf, g, ws)
        elif kind == "quantize_2d":
            q, sf, g = nv.alloc_quantized(R, C)
            qT, sfT, _ = nv.alloc_quantized(C, R)
            fn = lambda: nv.nvfp4_quantize_2d(x, R, C, C, q, sf, qT, sfT, g, ws)
        elif kind == "rht":
            q, sf, g = nv.alloc_quantized(C, R)
            fn = lambda: nv.nvfp4_rht_quantize(x, R, C, C, 5, mode, 1, q, sf, g, ws)
        elif kind == "noise":
            q, sf, g = nv.alloc_quantized(R, C)
            nv.nvfp4_quantize(x, R, C, C, nv.RN, 0, q, sf, g, ws)
            sums = torch.empty(2, dtype=torch.float64, device="cuda")
            fn = lambda: nv.nvfp4_quant_noise(x, R, C, C, q, sf, g, sums)
        elif kind == "dual":
            q, sf, g = nv.alloc_quantized(R, C)
            qT, sfT, gT = nv.alloc_quantized(C, R)
            fn = lambda: nv.nvfp4_quantize_dual(x, R, C, C, mode, 1, q, sf, g, 5, mode, 2, qT, sfT, gT, ws)
        else:
            raise SystemExit(__doc__)
        ms = _time(fn, reps)
        print(f"{kind} {R}x{C}: {ms:.4f} ms")
    st = nv.nvfp4_device_status(ws)
    if st != 0:
        raise SystemExit(f"device status {nv.nvfp4_status_str(st)}")


if __name__ == "__main__":
    main(sys.argv[1:])
