"""GPU parity of the fused QLoRA forward / backward against the fp64 oracle.

Inputs follow the seeded recipe of bit_nf4_quantized_35_b300.inputs.  The
weight seen by the oracle is the oracle's own dequantisation of the oracle's
own quantisation (bit-identical to the GPU's, as test_gpu_quantize checks).
Tolerance: max |err| <= 2e-2 and relative Frobenius error <= 1e-2."""
import numpy as np
import pytest
import torch

from bit_nf4_quantized_35_b300 import capi, inputs
from oracle import oracle

from .helpers import MAX_ABS, REL_FRO, assert_close, to_np_f32

pytestmark = pytest.mark.gpu

FORCE_GEMV, FORCE_GEMM = capi.QLORA_FLAG_FORCE_GEMV, capi.QLORA_FLAG_FORCE_GEMM


def _prep(shape: inputs.LinearShape, with_dy=True, zero_B=False, seed_offset=0):
    d = inputs.linear_inputs(shape, with_dy=with_dy, seed_offset=seed_offset)
    if zero_B:
        d["B"] = torch.zeros_like(d["B"])
    ref_q = oracle.quantize_nf4(d["W"].float().numpy(), 64, 256)
    w_hat = oracle.dequant_f32(ref_q)
    g = {k: v.cuda().contiguous() for k, v in d.items()}
    q = capi.quantize_nf4(g["W"])
    return d, g, q, w_hat


def _ws(shape):
    return capi.Workspace(shape.M, shape.N, shape.K, shape.r)


def _fwd(shape, g, q, ws, flags=0, y_dtype=torch.float32):
    t = torch.empty(shape.M, shape.r, dtype=torch.float32, device="cuda")
    y = capi.linear_fwd(q, g["x"], g["A"], g["B"], shape.alpha, ws, y_dtype=y_dtype, t_save=t,
                        flags=flags)
    torch.cuda.synchronize()
    assert ws.device_status() == 0
    return y, t


SMALL = [
    inputs.SINGLE_256,
    inputs.LinearShape("ragged_N520_K384_M200_r16", N=520, K=384, M=200, r=16, alpha=32.0),
    inputs.LinearShape("ragged_N264_K320_M129_r8", N=264, K=320, M=129, r=8, alpha=16.0),
    inputs.LinearShape("tiles_N768_K512_M384_r32", N=768, K=512, M=384, r=32, alpha=64.0),
    inputs.LinearShape("r64_N256_K256_M130_r64", N=256, K=256, M=130, r=64, alpha=128.0),
    inputs.LinearShape("r24_N136_K192_M17_r24", N=136, K=192, M=17, r=24, alpha=48.0),
    # 8192 columns or more: the down-projections stream through the TMA ring
    # kernel (u = dY B over N = 8200, t = x A^T over K = 8256; both end in a
    # partial 256-column stage)
    inputs.LinearShape("wideN_N8200_K256_M50_r40", N=8200, K=256, M=50, r=40, alpha=80.0),
    inputs.LinearShape("wideK_N136_K8256_M33_r16", N=136, K=8256, M=33, r=16, alpha=32.0),
]


@pytest.mark.parametrize("shape", SMALL, ids=lambda s: s.name)
@pytest.mark.parametrize("path", ["gemm", "gemv"])
def test_forward_small(shape, path):
    if path == "gemv" and shape.M > 16:
        shape = inputs.LinearShape(shape.name + "_M7", shape.N, shape.K, 7, shape.r, shape.alpha,
                                   shape.w_dtype)
    d, g, q, w_hat = _prep(shape, with_dy=False)
    ws = _ws(shape)
    y, t = _fwd(shape, g, q, ws, FORCE_GEMV if path == "gemv" else FORCE_GEMM)
    y_ref, t_ref = oracle.linear_fwd(d["x"].float().numpy(), w_hat, d["A"].float().numpy(),
                                     d["B"].float().numpy(), shape.alpha)
    assert_close(to_np_f32(y), y_ref, f"y {shape.name} {path}")
    assert_close(to_np_f32(t), t_ref, f"t {shape.name} {path}", max_abs=1e-3, rel_fro=1e-5)


@pytest.mark.parametrize("shape", SMALL, ids=lambda s: s.name)
def test_backward_small(shape):
    d, g, q, w_hat = _prep(shape)
    ws = _ws(shape)
    y, t = _fwd(shape, g, q, ws)
    before = [x.clone() for x in (q.packed, q.absmax_code, q.scale2)]
    dX, dA, dB = capi.linear_bwd(q, g["x"], g["dY"], g["A"], g["B"], shape.alpha, ws, t_saved=t)
    torch.cuda.synchronize()
    assert ws.device_status() == 0
    ref = oracle.linear_bwd(d["x"].float().numpy(), d["dY"].float().numpy(), w_hat,
                            d["A"].float().numpy(), d["B"].float().numpy(), shape.alpha)
    assert_close(to_np_f32(dX), ref["dX"], f"dX {shape.name}")
    assert_close(to_np_f32(dA), ref["dA"], f"dA {shape.name}")
    assert_close(to_np_f32(dB), ref["dB"], f"dB {shape.name}")
    # frozen base: the NF4 buffers are untouched
    for a, b in zip(before, (q.packed, q.absmax_code, q.scale2)):
        assert torch.equal(a, b)
    # recompute path (no saved t) gives the same gradients
    dX2, dA2, dB2 = capi.linear_bwd(q, g["x"], g["dY"], g["A"], g["B"], shape.alpha, ws)
    torch.cuda.synchronize()
    assert_close(to_np_f32(dB2), ref["dB"], f"dB recompute {shape.name}")
    assert torch.equal(dX, dX2)


def test_zero_B_gives_base_output_and_zero_dA():
    shape = inputs.LinearShape("zeroB_N256_K256_M64_r16", N=256, K=256, M=64, r=16, alpha=32.0)
    d, g, q, w_hat = _prep(shape, zero_B=True)
    ws = _ws(shape)
    y, t = _fwd(shape, g, q, ws)
    # base-only reference: A = 0 gives the same zero LoRA branch
    y_base = capi.linear_fwd(q, g["x"], torch.zeros_like(g["A"]), g["B"], shape.alpha, ws)
    torch.cuda.synchronize()
    assert torch.equal(y, y_base)
    dX, dA, dB = capi.linear_bwd(q, g["x"], g["dY"], g["A"], g["B"], shape.alpha, ws, t_saved=t)
    torch.cuda.synchronize()
    assert torch.count_nonzero(dA).item() == 0
    assert torch.count_nonzero(dB).item() > 0


def test_nonzero_B_changes_output():
    shape = inputs.LinearShape("lora_changes_y", N=256, K=256, M=32, r=8, alpha=16.0)
    d, g, q, w_hat = _prep(shape)
    ws = _ws(shape)
    y, _ = _fwd(shape, g, q, ws)
    y0 = capi.linear_fwd(q, g["x"], g["A"], torch.zeros_like(g["B"]), shape.alpha, ws)
    torch.cuda.synchronize()
    assert not torch.equal(y, y0)


def test_bf16_outputs_within_one_ulp_of_fp32_path():
    shape = inputs.LinearShape("bf16_out", N=512, K=512, M=256, r=16, alpha=32.0)
    d, g, q, w_hat = _prep(shape)
    ws = _ws(shape)
    y32, t = _fwd(shape, g, q, ws)
    y16, _ = _fwd(shape, g, q, ws, y_dtype=torch.bfloat16)
    assert torch.equal(y16, y32.to(torch.bfloat16))
    dX32, _, _ = capi.linear_bwd(q, g["x"], g["dY"], g["A"], g["B"], shape.alpha, ws, t_saved=t)
    dX16, _, _ = capi.linear_bwd(q, g["x"], g["dY"], g["A"], g["B"], shape.alpha, ws, t_saved=t,
                                 dx_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    assert torch.equal(dX16, dX32.to(torch.bfloat16))


def test_deterministic():
    shape = inputs.LinearShape("det", N=384, K=320, M=150, r=16, alpha=32.0)
    d, g, q, w_hat = _prep(shape)
    ws = _ws(shape)
    outs = []
    for _ in range(2):
        y, t = _fwd(shape, g, q, ws)
        dX, dA, dB = capi.linear_bwd(q, g["x"], g["dY"], g["A"], g["B"], shape.alpha, ws, t_saved=t)
        torch.cuda.synchronize()
        outs.append([y.clone(), dX.clone(), dA.clone(), dB.clone()])
    for a, b in zip(*outs):
        assert torch.equal(a, b)


# ------------------------------------------------------------ full-size cases
def _sample_rows(M, n=64, seed=0):
    rng = np.random.default_rng(seed)
    rows = np.sort(rng.choice(M, size=min(n, M), replace=False))
    rows[0], rows[-1] = 0, M - 1
    return np.unique(rows)


def test_qproj_prefill_forward_full_size():
    shape = inputs.QPROJ_2048
    d, g, q, w_hat = _prep(shape, with_dy=False)
    ws = _ws(shape)
    y, t = _fwd(shape, g, q, ws)
    rows = _sample_rows(shape.M)
    y_ref, t_ref = oracle.linear_fwd(d["x"].float().numpy(), w_hat, d["A"].float().numpy(),
                                     d["B"].float().numpy(), shape.alpha, rows=rows)
    assert_close(to_np_f32(y)[rows], y_ref, "y q_proj sampled rows")
    assert_close(to_np_f32(t)[rows], t_ref, "t q_proj sampled rows", max_abs=1e-3, rel_fro=1e-5)


@pytest.mark.parametrize("M", [1, 4, 16])
def test_gate_decode_gemv_full_size(M):
    shape = inputs.gate_decode(M)
    d, g, q, w_hat = _prep(shape, with_dy=False)
    ws = _ws(shape)
    y, t = _fwd(shape, g, q, ws)
    y_ref, _ = oracle.linear_fwd(d["x"].float().numpy(), w_hat, d["A"].float().numpy(),
                                 d["B"].float().numpy(), shape.alpha)
    assert_close(to_np_f32(y), y_ref, f"y gate decode M={M}")


GEMV_WIDE_K = [
    # K = 14336: the K slices of one row range spread over a cluster of 7 CTAs
    inputs.LinearShape("down_proj_4096x14336_M3_r16", N=4096, K=14336, M=3, r=16, alpha=32.0),
    # K = 4160 = 65 x 64 over 3 CTAs (the last slice shorter than the others),
    # r = 40 (three 16-wide tiles of t, the last one ragged), N = 1032 (a
    # ragged last row pair), 9 tokens (two 8-token tiles)
    inputs.LinearShape("ragged_N1032_K4160_M9_r40", N=1032, K=4160, M=9, r=40, alpha=80.0),
    # 2000 16-row tiles: 14 or 13 tiles per CTA
    inputs.LinearShape("tall_N32000_K4096_M1_r16", N=32000, K=4096, M=1, r=16, alpha=32.0),
]


@pytest.mark.parametrize("shape", GEMV_WIDE_K, ids=lambda s: s.name)
def test_decode_gemv_wide_k(shape):
    d, g, q, w_hat = _prep(shape, with_dy=False)
    ws = _ws(shape)
    y, t = _fwd(shape, g, q, ws, FORCE_GEMV)
    y_ref, t_ref = oracle.linear_fwd(d["x"].float().numpy(), w_hat, d["A"].float().numpy(),
                                     d["B"].float().numpy(), shape.alpha)
    assert_close(to_np_f32(y), y_ref, f"y {shape.name}")
    assert_close(to_np_f32(t), t_ref, f"t {shape.name}", max_abs=1e-3, rel_fro=1e-5)
    y16, _ = _fwd(shape, g, q, ws, FORCE_GEMV, y_dtype=torch.bfloat16)
    assert torch.equal(y16, y.to(torch.bfloat16)), "bf16 output is not the rounded fp32 result"


def test_gate_prefill_forward_full_size():
    """gate_proj 14336x4096 at 2048 tokens: the widest layer of the layer set
    (its pair tiles are 224 columns wide), y checked on sampled rows."""
    shape = inputs.LinearShape("gate_proj_14336x4096_M2048_r16", N=14336, K=4096, M=2048, r=16,
                               alpha=32.0)
    d, g, q, w_hat = _prep(shape, with_dy=False)
    ws = _ws(shape)
    y, t = _fwd(shape, g, q, ws)
    rows = _sample_rows(shape.M, n=16, seed=3)
    y_ref, t_ref = oracle.linear_fwd(d["x"].float().numpy(), w_hat, d["A"].float().numpy(),
                                     d["B"].float().numpy(), shape.alpha, rows=rows)
    assert_close(to_np_f32(y)[rows], y_ref, "y gate sampled rows")


def test_kproj_backward_full_size():
    """k_proj 1024x4096 at 2048 tokens: dX on sampled rows, dA and dB in full."""
    shape = inputs.LinearShape("k_proj_1024x4096_M2048_r16", N=1024, K=4096, M=2048, r=16,
                               alpha=32.0)
    d, g, q, w_hat = _prep(shape)
    ws = _ws(shape)
    y, t = _fwd(shape, g, q, ws)
    dX, dA, dB = capi.linear_bwd(q, g["x"], g["dY"], g["A"], g["B"], shape.alpha, ws, t_saved=t)
    torch.cuda.synchronize()
    assert ws.device_status() == 0
    rows = _sample_rows(shape.M, n=16, seed=4)
    ref = oracle.linear_bwd(d["x"].float().numpy(), d["dY"].float().numpy(), w_hat,
                            d["A"].float().numpy(), d["B"].float().numpy(), shape.alpha,
                            rows=rows)
    assert_close(to_np_f32(dX)[rows], ref["dX"], "dX k_proj sampled rows")
    assert_close(to_np_f32(dA), ref["dA"], "dA k_proj")
    assert_close(to_np_f32(dB), ref["dB"], "dB k_proj")
