"""Parity of the composed forward+backward step (the pass -> operand wiring).

The twelve launches of ``MlpStep`` (nvfp4_bit_quantized_quantize_gb300/step.py)
run on the GPU; every stage is then checked against the oracle on that
stage's own inputs.  The expected operands below are written out here, not
read from ``MlpStep.wiring()``, so a wrong operand, transposition, tensor
scale or seed in the step fails:

  GEMM          A (M x K)                          B (N x K)                         g of B
  fprop_up      X     1x16 RN                      W_up    2-D RN                     W_up
  fprop_down    H     1x16 RN                      W_down  2-D RN                     W_down
  dgrad_down    dY    1x16 SR, seed 16s+3          W_down^T (2-D, transposed codes)   W_down
  wgrad_down    dY^T  RHT(seed s+1) + SR, 16s+4    H^T   RHT(seed s+1) + RN           H^T
  dgrad_up      dH    1x16 SR, seed 16s+5          W_up^T  (2-D, transposed codes)    W_up
  wgrad_up      dH^T  RHT(seed s+1) + SR, 16s+6    X^T   RHT(seed s+1) + RN           X^T

("Entrenamiento ...", "Metodología de Entrenamiento": 2-D scaling for
weights, random Hadamard transforms for Wgrad, stochastic rounding of
gradients; "FP4 All the Way", "Describir": nearest rounding forward.)

Quantized operands must be bit-exact (codes, scale bytes with padding, tensor
scale); GEMM outputs (bf16) within 1e-5 * ga gb sum_k |a b| + 2^-8 |ref|.
H and dH, the GPU's own bf16 GEMM outputs, are the inputs of the next stage
on both sides, so each stage is checked on exactly the data it consumed.
"""
import concurrent.futures as cf

import numpy as np
import pytest
import torch

import nvfp4_bit_quantized_quantize_gb300 as nv
import oracle as O
from nvfp4_bit_quantized_quantize_gb300 import synth
from nvfp4_bit_quantized_quantize_gb300.step import MlpStep

pytestmark = pytest.mark.gpu


def _bits(t):
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def _trip(tr):
    q, sf, g = tr
    return q.cpu().numpy(), sf.cpu().numpy(), float(g.cpu()[0])


def _run(T, D, F, seed):
    """Inputs as the 7B-MLP workload draws them (X with 0.1% outliers x100,
    weights N(0, 0.02), dY N(0, 1e-3)), at the given shape."""
    host = {
        "X": synth.normal_bf16((T, D), seed, 0, 1.0, 0.0, 0.001, 100.0),
        "W_up": synth.normal_bf16((F, D), seed, 1, 0.02),
        "W_down": synth.normal_bf16((D, F), seed, 2, 0.02),
        "dY_down": synth.normal_bf16((T, D), seed, 3, 1e-3),
    }
    st = MlpStep(T, D, F, seed, "cuda")
    for k, v in host.items():
        st.inputs[0][k].copy_(torch.from_numpy(v.view(np.int16)).view(torch.bfloat16))
    st.run()
    torch.cuda.synchronize()
    assert nv.nvfp4_device_status(st.ws) == 0
    return st, host


def _expected_operands(st, host, pool):
    """Oracle quantizations of every operand, from the host inputs and the
    GPU's H and dH.  Returns name -> (codes, scales, g) and, for the 2-D
    weights, their transposed (codes, scales)."""
    s = st.seed
    rht = s + 1
    H, dH = _bits(st.H), _bits(st.dH)
    jobs = {
        "xq": (O.quantize, host["X"], O.RN, 0),
        "xT": (O.rht_quantize, host["X"], rht, O.RN, 0),
        "W_up": (O.quantize_2d, host["W_up"]),
        "hq": (O.quantize, H, O.RN, 0),
        "hT": (O.rht_quantize, H, rht, O.RN, 0),
        "W_down": (O.quantize_2d, host["W_down"]),
        "dyq": (O.quantize, host["dY_down"], O.SR, 16 * s + 3),
        "dyT": (O.rht_quantize, host["dY_down"], rht, O.SR, 16 * s + 4),
        "dhq": (O.quantize, dH, O.SR, 16 * s + 5),
        "dhT": (O.rht_quantize, dH, rht, O.SR, 16 * s + 6),
    }
    futs = {k: pool.submit(j[0], *j[1:]) for k, j in jobs.items()}
    out = {k: f.result() for k, f in futs.items()}
    for w, (n, nT) in (("W_up", ("wuq", "wuqT")), ("W_down", ("wdq", "wdqT"))):
        q, sf, qT, sfT, g = out.pop(w)
        out[n] = (q, sf, g)
        out[nT] = (qT, sfT, g)       # the transposed codes keep the weight's tensor scale
    return out


# GEMM -> (A, B, output, (M, N, K) in terms of T, D, F)
GEMMS = {
    "fprop_up": ("xq", "wuq", "H", lambda T, D, F: (T, F, D)),
    "fprop_down": ("hq", "wdq", "Y", lambda T, D, F: (T, D, F)),
    "dgrad_down": ("dyq", "wdqT", "dH", lambda T, D, F: (T, F, D)),
    "wgrad_down": ("dyT", "hT", "dW_down", lambda T, D, F: (D, F, T)),
    "dgrad_up": ("dhq", "wuqT", "dX", lambda T, D, F: (T, D, F)),
    "wgrad_up": ("dhT", "xT", "dW_up", lambda T, D, F: (F, D, T)),
}


# the transposed weight codes carry no tensor scale of their own: the GEMM
# takes the weight's (the 2-D quantizer writes only that one)
G_OF = {"wuqT": "wuq", "wdqT": "wdq"}


def _check_operands(st, exp):
    for name, (q, sf, g) in exp.items():
        gq, gsf, _ = _trip(getattr(st, name))
        gg = float(getattr(st, G_OF.get(name, name))[2].cpu()[0])
        assert np.array_equal(gq, q), f"{name}: codes differ"
        assert np.array_equal(gsf, sf), f"{name}: scale bytes differ"
        assert gg == g, f"{name}: tensor scale {gg} != {g}"


def _gpu_out(st, name):
    return st.tensor(name).float().cpu().numpy().astype(np.float64)


@pytest.mark.parametrize("T,D,F", [(256, 128, 384), (384, 320, 1056)])
def test_step_wiring_full_compare(T, D, F):
    st, host = _run(T, D, F, seed=4)
    with cf.ThreadPoolExecutor(8) as pool:
        exp = _expected_operands(st, host, pool)
    _check_operands(st, exp)
    for label, (a, b, out, mnk) in GEMMS.items():
        M, N, K = mnk(T, D, F)
        qa, sfa, ga = exp[a]
        qb, sfb, gb = exp[b]
        ref, dabs = O.gemm_f64(qa, sfa, ga, qb, sfb, gb, M, N, K)
        got = _gpu_out(st, out)
        assert got.shape == (M, N)
        err = np.abs(got - ref)
        bound = 1e-5 * dabs + 2.0 ** -8 * np.abs(ref)
        assert np.all(err <= bound), (label, float(np.max(err - bound)))
        # a GEMM fed the wrong operand would not come near the reference
        assert np.any(ref != 0), label


def test_step_wiring_full_shape_sampled():
    # the 7B-MLP shape of the benchmark: every operand bit-exact, each GEMM
    # on 2048 sampled outputs plus one full row and one full column
    T, D, F = 8192, 4096, 11008
    st, host = _run(T, D, F, seed=4)
    with cf.ThreadPoolExecutor(10) as pool:
        exp = _expected_operands(st, host, pool)
    _check_operands(st, exp)
    rng = np.random.default_rng(11)
    for label, (a, b, out, mnk) in GEMMS.items():
        M, N, K = mnk(T, D, F)
        ms = np.concatenate([rng.integers(0, M, 2048), np.full(N, M - 1), np.arange(M)])
        ns = np.concatenate([rng.integers(0, N, 2048), np.arange(N), np.full(M, N - 1)])
        qa, sfa, ga = exp[a]
        qb, sfb, gb = exp[b]
        ref, dabs = O.gemm_f64_sampled(qa, sfa, ga, qb, sfb, gb, M, N, K, ms, ns)
        got = _gpu_out(st, out)[ms, ns]
        err = np.abs(got - ref)
        bound = 1e-5 * dabs + 2.0 ** -8 * np.abs(ref)
        assert np.all(err <= bound), (label, float(np.max(err - bound)))


def test_overlapped_schedule_writes_the_same_results():
    # the weight-gradient GEMMs on a second stream: every output and
    # intermediate bit-identical to the one-stream order, both workspaces clean
    T, D, F = 512, 256, 768
    st, host = _run(T, D, F, seed=6)
    names = ["H", "dH", "Y", "dX", "dW_up", "dW_down"]
    seq = {n: _bits(st.tensor(n)).copy() for n in names}
    for n in names:
        st.tensor(n).zero_()
    side = torch.cuda.Stream()
    st.run_overlapped(0, torch.cuda.current_stream(), side)
    torch.cuda.synchronize()
    assert nv.nvfp4_device_status(st.ws) == 0 and nv.nvfp4_device_status(st.ws_side) == 0
    for n in names:
        assert np.array_equal(_bits(st.tensor(n)), seq[n]), n
