"""GPU parity of the adapter merge W_out = bf16(W_hat + alpha/r B A) against
the oracle ("QLoRA and 4bit Quantization | QLoRA 与 4-bit 量化", Step 5
conclusion: adapter merge before deployment).

The oracle rounds the binary64 sum once; the kernel rounds an fp32 sum
(w_hat exact, B A accumulated in fp32, fp32 multiply-add with alpha/r) once.
The two agree bit for bit except where the exact value lies within the fp32
arithmetic's error of a bf16 rounding midpoint; there both neighbours are
correct roundings.  So every element must equal the oracle's, or be its
adjacent bf16 value with the exact sum within 2^-20 (relative) of the
midpoint between the two; and such elements must be rare."""
import numpy as np
import pytest
import torch

from bit_nf4_quantized_35_b300 import capi, inputs
from oracle import oracle

from .helpers import bf16_bits

pytestmark = pytest.mark.gpu


def _check_merge(shape, block=64, group=256, zero_B=False, codebook=0):
    d = inputs.linear_inputs(shape, with_dy=False, seed_offset=7)
    if zero_B:
        d["B"] = torch.zeros_like(d["B"])
    g = {k: v.cuda().contiguous() for k, v in d.items()}
    q = capi.quantize_nf4(g["W"], group=group, block=block, codebook=codebook)
    before = [t.clone() for t in (q.packed,) + tuple(x for x in (q.absmax_code, q.scale2,
                                                                    q.absmax_f32) if x is not None)]
    got = capi.merge_lora(q, g["A"], g["B"], shape.alpha)
    torch.cuda.synchronize()
    ref_q = oracle.quantize_nf4(d["W"].float().numpy(), block, group, codebook=codebook)
    w_hat = oracle.dequant_f32(ref_q)
    ref_bits, exact = oracle.merge_bf16(w_hat, d["A"].float().numpy(), d["B"].float().numpy(),
                                        shape.alpha)
    gb = bf16_bits(got)
    diff = gb != ref_bits
    if diff.any():
        gv = oracle.bf16_bits_to_f32(gb[diff]).astype(np.float64)
        rv = oracle.bf16_bits_to_f32(ref_bits[diff]).astype(np.float64)
        ex = exact[diff]
        assert np.all(np.abs(gb[diff].astype(np.int64) - ref_bits[diff].astype(np.int64)) == 1)
        assert np.all(np.abs(ex - (gv + rv) / 2) <= 2.0 ** -20 * np.abs(ex)), "not a near-tie"
        assert diff.mean() <= 1e-4, diff.mean()
    for a, b in zip(before, (q.packed,) + tuple(x for x in (q.absmax_code, q.scale2,
                                                             q.absmax_f32) if x is not None)):
        assert torch.equal(a, b)  # the NF4 buffers are const
    if zero_B:
        assert np.array_equal(gb, bf16_bits(capi.dequant(q)))
    return int(diff.sum())


SHAPES = [
    inputs.LinearShape("merge_N1032_K1024_r16", N=1032, K=1024, M=1, r=16, alpha=32.0),
    inputs.LinearShape("merge_N264_K4160_r8", N=264, K=4160, M=1, r=8, alpha=16.0),
    inputs.LinearShape("merge_N136_K384_r24", N=136, K=384, M=1, r=24, alpha=48.0),
    inputs.LinearShape("merge_N520_K512_r64", N=520, K=512, M=1, r=64, alpha=128.0),
]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: s.name)
def test_merge_small(shape):
    _check_merge(shape)


@pytest.mark.parametrize("fmt", [(64, 0, 0), (128, 256, 0), (128, 0, 0), (64, 256, 1)],
                         ids=lambda f: f"b{f[0]}g{f[1]}cb{f[2]}")
def test_merge_storage_formats(fmt):
    _check_merge(SHAPES[0], block=fmt[0], group=fmt[1], codebook=fmt[2])


def test_merge_zero_B_is_the_dequantised_weight():
    _check_merge(SHAPES[0], zero_B=True)


def test_merge_gate_proj_full_size():
    _check_merge(inputs.LinearShape("merge_gate_14336x4096_r16", N=14336, K=4096, M=1, r=16,
                                    alpha=32.0))
