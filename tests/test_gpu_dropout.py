"""GPU parity of LoRA dropout on the bypass input against the oracle
("QLoRA and 4bit Quantization | QLoRA 与 4-bit 量化", Step 5 training config;
"第 09 期 | QLoRA 4-bit 量化微调" LoraConfig lora_dropout).

  * the keep mask (Philox4x64-10) bit for bit against the oracle's;
  * forward (tensor-core GEMM and decode GEMV paths) and backward (dX fp32,
    dA, dB; saved and recomputed t) against the fp64 oracle with that mask;
  * p = 0 gives exactly the results of the calls without dropout;
  * the full gate projection at 2048 tokens.
Tolerance: max |err| <= 2e-2 and relative Frobenius error <= 1e-2."""
import numpy as np
import pytest
import torch

from bit_nf4_quantized_35_b300 import capi, inputs
from oracle import oracle

from .helpers import assert_close, to_np_f32

pytestmark = pytest.mark.gpu


def _unpack(mask: torch.Tensor, K: int) -> np.ndarray:
    words = mask.cpu().numpy().view(np.uint32)
    bits = ((words[:, :, None] >> np.arange(32, dtype=np.uint32)) & 1).astype(np.uint8)
    return bits.reshape(words.shape[0], -1)[:, :K]


@pytest.mark.parametrize("M,K,p,seed", [(37, 320, 0.1, 7), (5, 4224, 0.5, 8), (300, 1024, 0.0, 9),
                                        (2048, 4096, 0.05, 2 ** 40 + 3)])
def test_mask_bits_equal_oracle(M, K, p, seed):
    capi.load()
    mask = capi.dropout_mask(seed, p, M, K)
    torch.cuda.synchronize()
    keep = _unpack(mask, K)
    assert np.array_equal(keep, oracle.dropout_keep(seed, np.float32(p), M, K))
    w = mask.shape[1]
    assert w == capi.dropout_mask_words(K)
    tail = mask.cpu().numpy().view(np.uint32)[:, (K + 31) // 32:]
    assert not tail.any()  # words past K are zero


def _run(shape, p, seed, flags=0, t_saved=True):
    d = inputs.linear_inputs(shape, seed_offset=31)
    g = {k: v.cuda().contiguous() for k, v in d.items()}
    q = capi.quantize_nf4(g["W"])
    w_hat = oracle.dequant_f32(oracle.quantize_nf4(d["W"].float().numpy(), 64, 256))
    mask = capi.dropout_mask(seed, p, shape.M, shape.K)
    ws = capi.Workspace(shape.M, shape.N, shape.K, shape.r)
    t = torch.empty(shape.M, shape.r, dtype=torch.float32, device="cuda")
    y = capi.linear_fwd(q, g["x"], g["A"], g["B"], shape.alpha, ws, t_save=t, flags=flags,
                        dropout=(mask, p))
    dX, dA, dB = capi.linear_bwd(q, g["x"], g["dY"], g["A"], g["B"], shape.alpha, ws,
                                 t_saved=t if t_saved else None, dropout=(mask, p))
    torch.cuda.synchronize()
    assert ws.device_status() == 0
    keep = oracle.dropout_keep(seed, np.float32(p), shape.M, shape.K)
    np_ = {k: v.float().numpy() for k, v in d.items()}
    return g, q, ws, mask, (y, t, dX, dA, dB), keep, np_, w_hat


SHAPES = [
    inputs.LinearShape("drop_N520_K384_M200_r16", N=520, K=384, M=200, r=16, alpha=32.0),
    inputs.LinearShape("drop_N264_K1024_M129_r8", N=264, K=1024, M=129, r=8, alpha=16.0),
    # r = 40 and 64: three and four 16-wide rank steps in the dX correction
    inputs.LinearShape("drop_N136_K512_M77_r40", N=136, K=512, M=77, r=40, alpha=80.0),
    inputs.LinearShape("drop_N256_K320_M64_r64", N=256, K=320, M=64, r=64, alpha=128.0),
    # K >= 8192: t = x A^T with the keep mask through the TMA ring kernel
    inputs.LinearShape("drop_N136_K8256_M40_r24", N=136, K=8256, M=40, r=24, alpha=48.0),
]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: s.name)
@pytest.mark.parametrize("p", [0.1, 0.5])
@pytest.mark.parametrize("t_saved", [True, False])
def test_dropout_forward_backward(shape, p, t_saved):
    g, q, ws, mask, out, keep, np_, w_hat = _run(shape, p, 123, t_saved=t_saved)
    y, t, dX, dA, dB = out
    y_ref, t_ref = oracle.linear_fwd(np_["x"], w_hat, np_["A"], np_["B"], shape.alpha,
                                     keep=keep, p=np.float32(p))
    ref = oracle.linear_bwd(np_["x"], np_["dY"], w_hat, np_["A"], np_["B"], shape.alpha,
                            keep=keep, p=np.float32(p))
    assert_close(to_np_f32(y), y_ref, f"y {shape.name} p={p}")
    assert_close(to_np_f32(t), t_ref, f"t {shape.name}", max_abs=1e-3, rel_fro=1e-5)
    for name, got in (("dX", dX), ("dA", dA), ("dB", dB)):
        assert_close(to_np_f32(got), ref[name], f"{name} {shape.name} p={p}")


def test_dropout_decode_gemv():
    shape = inputs.LinearShape("drop_gemv_N520_K4224_M5", N=520, K=4224, M=5, r=16, alpha=32.0)
    d = inputs.linear_inputs(shape, with_dy=False, seed_offset=32)
    g = {k: v.cuda().contiguous() for k, v in d.items()}
    q = capi.quantize_nf4(g["W"])
    w_hat = oracle.dequant_f32(oracle.quantize_nf4(d["W"].float().numpy(), 64, 256))
    mask = capi.dropout_mask(5, 0.2, shape.M, shape.K)
    ws = capi.Workspace(shape.M, shape.N, shape.K, shape.r)
    t = torch.empty(shape.M, shape.r, dtype=torch.float32, device="cuda")
    y = capi.linear_fwd(q, g["x"], g["A"], g["B"], shape.alpha, ws, t_save=t,
                        flags=capi.QLORA_FLAG_FORCE_GEMV, dropout=(mask, 0.2))
    torch.cuda.synchronize()
    keep = oracle.dropout_keep(5, np.float32(0.2), shape.M, shape.K)
    y_ref, t_ref = oracle.linear_fwd(d["x"].float().numpy(), w_hat, d["A"].float().numpy(),
                                     d["B"].float().numpy(), shape.alpha, keep=keep,
                                     p=np.float32(0.2))
    assert_close(to_np_f32(y), y_ref, "y gemv dropout")
    assert_close(to_np_f32(t), t_ref, "t gemv dropout", max_abs=1e-3, rel_fro=1e-5)


def test_zero_probability_equals_the_plain_calls():
    shape = SHAPES[0]
    g, q, ws, mask, out, keep, np_, w_hat = _run(shape, 0.0, 1)
    y, t, dX, dA, dB = out
    t2 = torch.empty_like(t)
    y2 = capi.linear_fwd(q, g["x"], g["A"], g["B"], shape.alpha, ws, t_save=t2)
    dX2, dA2, dB2 = capi.linear_bwd(q, g["x"], g["dY"], g["A"], g["B"], shape.alpha, ws,
                                    t_saved=t2)
    torch.cuda.synchronize()
    for a, b in ((y, y2), (t, t2), (dX, dX2), (dA, dA2), (dB, dB2)):
        assert torch.equal(a, b)


@pytest.mark.slow
def test_dropout_gate_proj_full_size():
    shape = inputs.LinearShape("drop_gate_14336x4096_M2048", N=14336, K=4096, M=2048, r=16,
                               alpha=32.0)
    g, q, ws, mask, out, keep, np_, w_hat = _run(shape, 0.1, 2024)
    y, t, dX, dA, dB = out
    rng = np.random.default_rng(0)
    rows = np.unique(np.concatenate([[0, shape.M - 1], rng.choice(shape.M, 62, replace=False)]))
    y_ref, _ = oracle.linear_fwd(np_["x"], w_hat, np_["A"], np_["B"], shape.alpha, rows=rows,
                                 keep=keep, p=np.float32(0.1))
    ref = oracle.linear_bwd(np_["x"], np_["dY"], w_hat, np_["A"], np_["B"], shape.alpha,
                            rows=rows, keep=keep, p=np.float32(0.1))
    assert_close(to_np_f32(y)[rows], y_ref, "y gate dropout (64 rows)")
    assert_close(to_np_f32(t), ref["t"], "t gate dropout", max_abs=1e-3, rel_fro=1e-5)
    assert_close(to_np_f32(dX)[rows], ref["dX"], "dX gate dropout (64 rows)")
    assert_close(to_np_f32(dA), ref["dA"], "dA gate dropout")
    assert_close(to_np_f32(dB), ref["dB"], "dB gate dropout")
