"""GPU parity of the fused GEMM when output tiles are split across clusters.

A layer whose output tiles do not fill the SMs' waves is spread over all of
them: each cluster takes an equal share of (tile, 64-wide contraction block)
units and a tile shared by several clusters is summed from fp32 partials by
the last of them to finish.  These tests pick shapes that split (ragged rows,
columns and contraction), check forward and dX against the fp64 oracle with
the full workspace (split tiles) and with the minimal one (whole tiles only),
and check that repeated calls give bit-identical results, which also shows
that the per-tile counters return to zero after every call.
Tolerance: max |err| <= 2e-2 and relative Frobenius error <= 1e-2."""
import pytest
import torch

from bit_nf4_quantized_35_b300 import capi, inputs
from oracle import oracle

from .helpers import assert_close, to_np_f32

pytestmark = pytest.mark.gpu

FORCE_GEMM = capi.QLORA_FLAG_FORCE_GEMM


def _splits(M, out_cols, kdim, dx=False, clusters=74):
    """Mirror of the launch plan's rule: whole tiles (of the width the plan
    picks) that would keep fewer than half of the clusters' wave slots busy,
    and at least 8 contraction blocks of 256-column tiles per cluster."""
    mp = -(-M // 256)
    cands = (256, 128) if dx else (256, 224, 192, 160, 128)
    cost = lambda c: -(-(mp * -(-out_cols // c)) // clusters) * (c + 1100)
    bn = min(cands, key=lambda c: (cost(c), cands.index(c)))
    T = mp * -(-out_cols // bn)
    waves = -(-T // clusters)
    U = mp * -(-out_cols // 256) * -(-kdim // 64)
    return T * 2 < waves * clusters and U // clusters >= 8


SPLIT = [
    # rows 300 = 256 + 44, N = 6 x 256 + 8, K = 15 x 256 + 192: the forward
    # splits 14 tiles over 63 blocks each; dX (32 tiles of 25 blocks, the
    # last one ragged) keeps whole tiles
    inputs.LinearShape("split_N1544_K4032_M300_r16", N=1544, K=4032, M=300, r=16, alpha=32.0),
    # one ragged row tile of 16 tokens through the tensor-core path; forward
    # and dX both split
    inputs.LinearShape("split_N4096_K4096_M16_r8", N=4096, K=4096, M=16, r=8, alpha=16.0),
]


def _prep(shape):
    d = inputs.linear_inputs(shape, with_dy=True)
    ref_q = oracle.quantize_nf4(d["W"].float().numpy(), 64, 256)
    w_hat = oracle.dequant_f32(ref_q)
    g = {k: v.cuda().contiguous() for k, v in d.items()}
    q = capi.quantize_nf4(g["W"])
    return d, g, q, w_hat


@pytest.mark.parametrize("shape", SPLIT, ids=lambda s: s.name)
def test_split_tiles_forward_and_dx(shape):
    assert _splits(shape.M, shape.N, shape.K)
    assert shape.M > 16 or _splits(shape.M, shape.K, shape.N, dx=True)
    d, g, q, w_hat = _prep(shape)
    y_ref, _ = oracle.linear_fwd(d["x"].float().numpy(), w_hat, d["A"].float().numpy(),
                                 d["B"].float().numpy(), shape.alpha)
    ref = oracle.linear_bwd(d["x"].float().numpy(), d["dY"].float().numpy(), w_hat,
                            d["A"].float().numpy(), d["B"].float().numpy(), shape.alpha)
    for minimal in (False, True):
        ws = capi.Workspace(shape.M, shape.N, shape.K, shape.r, minimal=minimal)
        tag = f"{shape.name} {'whole tiles' if minimal else 'split tiles'}"
        outs = []
        for _ in range(3):
            t = torch.empty(shape.M, shape.r, dtype=torch.float32, device="cuda")
            y = capi.linear_fwd(q, g["x"], g["A"], g["B"], shape.alpha, ws, t_save=t,
                                flags=FORCE_GEMM)
            dX, dA, dB = capi.linear_bwd(q, g["x"], g["dY"], g["A"], g["B"], shape.alpha, ws,
                                         t_saved=t)
            torch.cuda.synchronize()
            assert ws.device_status() == 0
            outs.append((y, dX))
        assert_close(to_np_f32(outs[0][0]), y_ref, f"y {tag}")
        assert_close(to_np_f32(outs[0][1]), ref["dX"], f"dX {tag}")
        for y, dX in outs[1:]:
            assert torch.equal(y, outs[0][0]), f"y not repeatable ({tag})"
            assert torch.equal(dX, outs[0][1]), f"dX not repeatable ({tag})"


def test_split_tiles_bf16_output_is_rounded_fp32_sum():
    shape = SPLIT[0]
    d, g, q, w_hat = _prep(shape)
    ws = capi.Workspace(shape.M, shape.N, shape.K, shape.r)
    y32 = capi.linear_fwd(q, g["x"], g["A"], g["B"], shape.alpha, ws)
    y16 = capi.linear_fwd(q, g["x"], g["A"], g["B"], shape.alpha, ws, y_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    assert torch.equal(y16, y32.to(torch.bfloat16))
