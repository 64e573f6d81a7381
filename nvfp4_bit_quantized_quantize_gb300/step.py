"""One NVFP4 training step of a linear-layer pair: the pass -> operand wiring.

The MLP of a transformer block without an activation function (the workload
names none): an up projection W_up [F, D] and a down projection W_down [D, F]
over T tokens, forward and backward, as the recipe assigns the formats
("Entrenamiento de Modelos de Lenguaje con 4 Bits de Precisión", "Metodología
de Entrenamiento": 2-D block scaling for weights, random Hadamard transforms on
the Wgrad inputs, stochastic rounding of gradients; "FP4 All the Way",
"Describir": round-to-nearest in the forward pass, stochastic rounding in the
backward pass):

  Fprop up     H  = X  W_up^T      A = X   1x16 RN        B = W_up    2-D RN
  Fprop down   Y  = H  W_down^T    A = H   1x16 RN        B = W_down  2-D RN
  Dgrad down   dH = dY W_down      A = dY  1x16 SR        B = W_down^T (the 2-D transposed output, g of W_down)
  Wgrad down   dW_down = dY^T H    A = dY^T RHT + SR      B = H^T     RHT + RN (one sign diagonal)
  Dgrad up     dX = dH W_up        A = dH  1x16 SR        B = W_up^T  (the 2-D transposed output, g of W_up)
  Wgrad up     dW_up = dH^T X      A = dH^T RHT + SR      B = X^T     RHT + RN

Every activation or gradient is quantized once, into both its 1x16 row form
(Fprop/Dgrad operand) and its Hadamard-transformed, token-contiguous form
(Wgrad operand).  The step's inputs X and dY go through nvfp4_quantize_dual
(an amax pass, then the quantization).  H and dH are written by the step's own
GEMMs: those run as nvfp4_gemm_amax, whose epilogue also reduces both tensor
amaxes of its output, and nvfp4_quantize_dual_from_amax then quantizes them in
one read.  Every GEMM has bf16 output.  Twelve launches per step, all library
kernels; this module only allocates buffers and strings the calls together.

Seeds: the Hadamard sign diagonal uses ``seed + 1`` for every Wgrad operand (so
that the transforms cancel in dY^T X); stochastic rounding of dY uses
``16 seed + 3`` (row form) and ``16 seed + 4`` (transformed form), of dH
``16 seed + 5`` and ``16 seed + 6``.
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import Callable

import nvfp4_bit_quantized_quantize_gb300 as nv


@dataclass(frozen=True)
class Launch:
    kind: str          # "quantize_dual", "quantize_dual_from_amax", "quantize_2d_t" or "gemm"
    shape: tuple       # (mode, rows, cols) for quantizers, (M, N, K) for GEMMs
    label: str         # which pass / tensor
    fn: Callable[[], None]


@dataclass(frozen=True)
class GemmWiring:
    """Which quantized operands, tensor scales and output one GEMM uses
    (names of MlpStep attributes; A and B are (codes, scales, g) triples)."""
    label: str
    a: str
    b: str
    b_scale_of: str    # the triple whose g scales B (the transposed weights reuse the weight's g)
    out: str
    mnk: tuple


class MlpStep:
    """Buffers and launches of one forward+backward step.

    ``slots`` independent copies of the step's inputs (X, W_up, W_down,
    dY_down) and results (Y, dX, dW_up, dW_down) let a caller copy the next
    step's inputs in and the previous step's results out while a step runs;
    the quantized operands and the intermediates H, dH are shared."""

    IN = ("X", "W_up", "W_down", "dY_down")
    OUT = ("Y", "dX", "dW_up", "dW_down")

    def __init__(self, T: int, D: int, F: int, seed: int, device, slots: int = 1):
        import torch

        self.T, self.D, self.F, self.seed = T, D, F, seed
        self.rht_seed = seed + 1
        self.sr_seeds = {"dY": (16 * seed + 3, 16 * seed + 4), "dH": (16 * seed + 5, 16 * seed + 6)}
        self.device = device
        bf = torch.bfloat16
        e = lambda *s: torch.empty(s, dtype=bf, device=device)
        in_shapes = {"X": (T, D), "W_up": (F, D), "W_down": (D, F), "dY_down": (T, D)}
        out_shapes = {"Y": (T, D), "dX": (T, D), "dW_up": (F, D), "dW_down": (D, F)}
        self.inputs = [{k: e(*s) for k, s in in_shapes.items()} for _ in range(slots)]
        self.outputs = [{k: e(*s) for k, s in out_shapes.items()} for _ in range(slots)]
        self.H, self.dH = e(T, F), e(T, F)
        q = lambda r, c: nv.alloc_quantized(r, c, device)
        # row forms (K = the contiguous axis) and transposed / Hadamard forms
        self.xq, self.xT = q(T, D), q(D, T)
        self.wuq, self.wuqT = q(F, D), q(D, F)
        self.hq, self.hT = q(T, F), q(F, T)
        self.wdq, self.wdqT = q(D, F), q(F, D)
        self.dyq, self.dyT = q(T, D), q(D, T)
        self.dhq, self.dhT = q(T, F), q(F, T)
        # (max |.|, max |RHT(.)|) of H and dH, from the GEMMs that write them
        self.amax = {k: torch.zeros(2, dtype=torch.float32, device=device) for k in ("H", "dH")}
        self.ws = nv.alloc_workspace(device)
        self.ws_side = nv.alloc_workspace(device)  # for launches on a second stream
        self._side = None
        self._plans = {}

    # the six GEMMs: D[M, N] = ga gb sum_k A[M, K] B[N, K]
    def wiring(self):
        T, D, F = self.T, self.D, self.F
        return [
            GemmWiring("fprop_up", "xq", "wuq", "wuq", "H", (T, F, D)),
            GemmWiring("fprop_down", "hq", "wdq", "wdq", "Y", (T, D, F)),
            GemmWiring("dgrad_down", "dyq", "wdqT", "wdq", "dH", (T, F, D)),
            GemmWiring("wgrad_down", "dyT", "hT", "hT", "dW_down", (D, F, T)),
            GemmWiring("dgrad_up", "dhq", "wuqT", "wuq", "dX", (T, D, F)),
            GemmWiring("wgrad_up", "dhT", "xT", "xT", "dW_up", (F, D, T)),
        ]

    def tensor(self, name: str, slot: int = 0):
        if name in self.IN:
            return self.inputs[slot][name]
        if name in self.OUT:
            return self.outputs[slot][name]
        return getattr(self, name)

    def launches(self, slot: int = 0, stream=None, ws=None) -> list:
        T, D, F = self.T, self.D, self.F
        x, wu, wd, dy = (self.inputs[slot][k] for k in self.IN)
        ws, rs = (self.ws if ws is None else ws), self.rht_seed
        (dy_r, dy_t), (dh_r, dh_t) = self.sr_seeds["dY"], self.sr_seeds["dH"]

        def dual(src, C, rows_q, t_q, mode, seed, seed_t, label):
            sh = ("sr" if mode == nv.SR else "rn", T, C)
            if label in self.amax:  # written by a GEMM of this step, which reduced its amaxes
                am = self.amax[label]
                fn = lambda: nv.nvfp4_quantize_dual_from_amax(src, T, C, C, am, mode, seed, *rows_q, rs, mode,
                                                              seed_t, *t_q, ws, stream)
                return Launch("quantize_dual_from_amax", sh, label, fn)
            fn = lambda: nv.nvfp4_quantize_dual(src, T, C, C, mode, seed, *rows_q, rs, mode, seed_t, *t_q, ws,
                                                stream)
            return Launch("quantize_dual", sh, label, fn)

        def w2d(w, R, C, wq, wqT, label):
            fn = lambda: nv.nvfp4_quantize_2d(w, R, C, C, wq[0], wq[1], wqT[0], wqT[1], wq[2], ws, stream)
            return Launch("quantize_2d_t", ("rn", R, C), label, fn)

        gemms = {}
        for w in self.wiring():
            a, b, bs = getattr(self, w.a), getattr(self, w.b), getattr(self, w.b_scale_of)
            out = self.tensor(w.out, slot)
            M, N, K = w.mnk
            if w.out in self.amax:
                fn = (lambda a=a, b=b, bs=bs, out=out, M=M, N=N, K=K, am=self.amax[w.out]:
                      nv.nvfp4_gemm_amax(a[0], a[1], a[2], b[0], b[1], bs[2], M, N, K, out, N, rs, am, ws, stream))
            else:
                fn = (lambda a=a, b=b, bs=bs, out=out, M=M, N=N, K=K:
                      nv.nvfp4_gemm(a[0], a[1], a[2], b[0], b[1], bs[2], M, N, K, out, N, nv.OUT_BF16, ws, stream))
            gemms[w.label] = Launch("gemm", (M, N, K), w.label, fn)
        return [
            dual(x, D, self.xq, self.xT, nv.RN, 0, 0, "X"),
            w2d(wu, F, D, self.wuq, self.wuqT, "W_up"),
            gemms["fprop_up"],
            dual(self.H, F, self.hq, self.hT, nv.RN, 0, 0, "H"),
            w2d(wd, D, F, self.wdq, self.wdqT, "W_down"),
            gemms["fprop_down"],
            dual(dy, D, self.dyq, self.dyT, nv.SR, dy_r, dy_t, "dY"),
            gemms["dgrad_down"],
            gemms["wgrad_down"],
            dual(self.dH, F, self.dhq, self.dhT, nv.SR, dh_r, dh_t, "dH"),
            gemms["dgrad_up"],
            gemms["wgrad_up"],
        ]

    def run(self, slot: int = 0, stream=None) -> None:
        """The twelve launches in order on one stream."""
        for l in self.launches(slot, stream):
            l.fn()

    def run_overlapped(self, slot: int = 0, stream=None, side=None) -> None:
        """The same launches with each weight-gradient GEMM on a second stream,
        beside the data-gradient work that does not depend on it: dW_down =
        dY^T H runs beside dH = dY W_down and dH's quantization, dW_up = dH^T X
        beside dX = dH W_up.  The four GEMMs are persistent kernels with no
        grid-wide barrier, so the second one's CTAs take the SMs the first
        one's last, partial wave of tiles leaves idle.  The cooperative
        quantizers (which wait on a grid-wide barrier) never overlap anything:
        the side stream forks after them and joins before the step ends.  The
        side GEMMs use their own workspace (self.ws_side)."""
        import torch

        main = stream if stream is not None else torch.cuda.current_stream()
        side = side if side is not None else self.side_stream()
        key = (slot, main, side)
        if key not in self._plans:
            self._plans[key] = ({l.label: l for l in self.launches(slot, main)},
                                {l.label: l for l in self.launches(slot, side, ws=self.ws_side)})
        ls, wg = self._plans[key]
        for name in ("X", "W_up", "fprop_up", "H", "W_down", "fprop_down", "dY"):
            ls[name].fn()
        fork_a = torch.cuda.Event()
        fork_a.record(main)
        ls["dgrad_down"].fn()
        side.wait_event(fork_a)          # dY's and H's Hadamard forms are ready
        wg["wgrad_down"].fn()
        ls["dH"].fn()
        fork_b = torch.cuda.Event()
        fork_b.record(main)
        ls["dgrad_up"].fn()
        side.wait_event(fork_b)          # dH's Hadamard form is ready
        wg["wgrad_up"].fn()
        join = torch.cuda.Event()
        join.record(side)
        main.wait_event(join)

    def side_stream(self):
        import torch

        if self._side is None:
            self._side = torch.cuda.Stream(device=self.device)
        return self._side
