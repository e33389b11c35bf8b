"""GPU parity at the benchmark's own sizes, against the fp64 oracle.

Every projection the benchmark step runs (Llama-3-8B's q/k/v/o, gate/up and
down at 2048 tokens, r = 16, NF4 + DQ) is run forward and backward through
the C ABI in the launch configuration the benchmark uses (full workspace,
the kernel selection of a default call).  Rows of y and dX are independent,
so the oracle computes 64 sampled rows of each (the first and last included);
t, dA and dB are checked in full.  One projection also runs at 8192 tokens,
the token count of the layer-set workload.
Tolerance: max |err| <= 2e-2 and relative Frobenius error <= 1e-2."""
import numpy as np
import pytest
import torch

from bit_nf4_quantized_35_b300 import capi, inputs
from oracle import oracle

from .helpers import assert_close, to_np_f32

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


def sample_rows(M, n=64, seed=0):
    rng = np.random.default_rng(seed)
    rows = np.sort(rng.choice(M, size=min(n, M), replace=False))
    rows[0], rows[-1] = 0, M - 1
    return np.unique(rows)


def run_layer(shape: inputs.LinearShape, seed_offset: int, rows_seed: int):
    d = inputs.linear_inputs(shape, seed_offset=seed_offset)
    g = {k: v.cuda().contiguous() for k, v in d.items()}
    q = capi.quantize_nf4(g["W"])
    ws = capi.Workspace(shape.M, shape.N, shape.K, shape.r)
    t = torch.empty(shape.M, shape.r, dtype=torch.float32, device="cuda")
    y = capi.linear_fwd(q, g["x"], g["A"], g["B"], shape.alpha, ws, t_save=t)
    dX, dA, dB = capi.linear_bwd(q, g["x"], g["dY"], g["A"], g["B"], shape.alpha, ws, t_saved=t)
    torch.cuda.synchronize()
    assert ws.device_status() == 0
    w_hat = oracle.dequant_f32(oracle.quantize_nf4(d["W"].float().numpy(), 64, 256,
                                                   want_idx=False))
    np_ = {k: v.float().numpy() for k, v in d.items()}
    rows = sample_rows(shape.M, 64, rows_seed)
    y_ref, t_ref = oracle.linear_fwd(np_["x"], w_hat, np_["A"], np_["B"], shape.alpha, rows=rows)
    ref = oracle.linear_bwd(np_["x"], np_["dY"], w_hat, np_["A"], np_["B"], shape.alpha,
                            rows=rows)
    name = shape.name
    assert_close(to_np_f32(y)[rows], y_ref, f"y {name} (64 sampled rows)")
    assert_close(to_np_f32(t), ref["t"], f"t {name}", max_abs=1e-3, rel_fro=1e-5)
    assert_close(to_np_f32(dX)[rows], ref["dX"], f"dX {name} (64 sampled rows)")
    assert_close(to_np_f32(dA), ref["dA"], f"dA {name}")
    assert_close(to_np_f32(dB), ref["dB"], f"dB {name}")


@pytest.mark.parametrize("li", range(len(inputs.LLAMA3_8B_PROJ)),
                         ids=list(inputs.LLAMA3_8B_PROJ))
def test_llama3_projection_fwd_bwd_M2048(li):
    name, (N, K) = list(inputs.LLAMA3_8B_PROJ.items())[li]
    shape = inputs.LinearShape(f"{name}_{N}x{K}_M2048_r16", N=N, K=K, M=2048, r=16, alpha=32.0)
    run_layer(shape, seed_offset=10 * li, rows_seed=li)


def test_down_proj_fwd_bwd_M8192():
    """down_proj 4096x14336 at 4 x 2048 tokens: the widest contraction of the
    forward (K = 14336) and the largest dA reduction (8192 tokens)."""
    shape = inputs.LinearShape("down_proj_4096x14336_M8192_r16", N=4096, K=14336, M=8192, r=16,
                               alpha=32.0)
    run_layer(shape, seed_offset=70, rows_seed=7)
