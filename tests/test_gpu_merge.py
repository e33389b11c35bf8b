"""GPU parity of the adapter merge W_out = bf16(W_hat + alpha/r B A) against
the oracle ("QLoRA and 4bit Quantization | QLoRA 与 4-bit 量化", Step 5
conclusion: adapter merge before deployment).

The oracle rounds the binary64 sum once; the kernel rounds an fp32 value v
once (w_hat exact, B A from bf16 products accumulated in fp32 on the tensor
cores, then an fp32 multiply-add with s = alpha/r).  Every product of two bf16
values is exact in fp32, so v differs from the exact sum e by at most
  E = 2 (r + 2) 2^-23 (|w_hat| + s sum_j |B[n, j] A[j, k]|)
(r - 1 accumulation steps and the multiply-add, each off by at most 2^-23 of
the running magnitude bound, doubled for tensor-core accumulation that
truncates instead of rounding).  Rounding to nearest is monotonic, so every
element must lie between the bf16 roundings of e - E and e + E (this covers a
neighbouring value at a near-tie, and a sign flip where e is within E of 0);
and elements that differ from the oracle's must be rare.
"""
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
        ns, ks = np.nonzero(diff)
        A64 = np.abs(d["A"].double().numpy())
        B64 = np.abs(d["B"].double().numpy())
        s = shape.alpha / shape.r
        mag = np.abs(w_hat[ns, ks].astype(np.float64)) + s * np.einsum("ij,ji->i", B64[ns],
                                                                         A64[:, ks])
        bound = 2.0 * (shape.r + 2) * 2.0 ** -23 * mag
        lo = oracle.bf16_bits_to_f32(np.array([oracle.bf16_rne_double(float(v))
                                               for v in ex - bound], dtype=np.uint16))
        hi = oracle.bf16_bits_to_f32(np.array([oracle.bf16_rne_double(float(v))
                                               for v in ex + bound], dtype=np.uint16))
        inside = (gv >= lo.astype(np.float64)) & (gv <= hi.astype(np.float64))
        assert np.all(inside), (
            f"{int((~inside).sum())} elements outside the rounding interval, e.g. "
            f"got {gv[~inside][:4]} ref {rv[~inside][:4]} exact {ex[~inside][:4]}")
        assert diff.mean() <= 1e-3, diff.mean()
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


@pytest.mark.parametrize("shape", [
    inputs.LinearShape("merge_N8_K64_r8", N=8, K=64, M=1, r=8, alpha=16.0),
    inputs.LinearShape("merge_N24_K192_r16", N=24, K=192, M=1, r=16, alpha=32.0),
    inputs.LinearShape("merge_N1_K128_r8", N=1, K=128, M=1, r=8, alpha=8.0),
], ids=lambda s: s.name)
def test_merge_smaller_than_one_store_tile(shape):
    """Weights smaller than one 16-row x 256-column output tile (fewer rows
    than 16, fewer than four 64-column blocks): the parts of the tile past
    the weight must not be written."""
    d = inputs.linear_inputs(shape, with_dy=False, seed_offset=7)
    g = {k: v.cuda().contiguous() for k, v in d.items()}
    q = capi.quantize_nf4(g["W"])
    guard = torch.full((shape.N * shape.K + 4096,), 0x7fc1, dtype=torch.int16, device="cuda")
    out = guard[:shape.N * shape.K].view(torch.bfloat16).view(shape.N, shape.K)
    capi.merge_lora(q, g["A"], g["B"], shape.alpha, out=out)
    torch.cuda.synchronize()
    assert torch.all(guard[shape.N * shape.K:] == 0x7fc1)  # nothing past the weight
    ref = capi.merge_lora(q, g["A"], g["B"], shape.alpha)
    assert torch.equal(out, ref)
    _check_merge(shape)


def test_merge_zero_B_is_the_dequantised_weight():
    _check_merge(SHAPES[0], zero_B=True)


def test_merge_gate_proj_full_size():
    _check_merge(inputs.LinearShape("merge_gate_14336x4096_r16", N=14336, K=4096, M=1, r=16,
                                    alpha=32.0))
