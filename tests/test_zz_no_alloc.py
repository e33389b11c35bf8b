"""The allocation-free backward entry point.

qlora_linear_bwd_noalloc serves callers that cannot allocate device memory
(graph capture, restrictive allocators, hosts that pass only inputs and
outputs).  It keeps its workspace in one fixed device array shared by every
call, so the test runs calls of different sizes back to back (a large shape,
a small one, the large one again, then a third shape without a saved t):
each call, made through the C ABI, must give the gradients of the fp64
oracle within the tolerance of the other parity tests, and the same
gradients as qlora_linear_bwd on a freshly initialised workspace.  Sizes
beyond the fixed array are refused.  This file is collected last so that a
failure here never hides another test.
"""
import ctypes

import pytest
import torch

from bit_nf4_quantized_35_b300 import capi, inputs
from oracle import oracle

from .helpers import assert_close, to_np_f32

pytestmark = pytest.mark.gpu

LARGE = inputs.LinearShape("noalloc_N1032_K1024_M640_r16", N=1032, K=1024, M=640, r=16,
                           alpha=32.0)
SMALL = inputs.LinearShape("noalloc_N264_K320_M33_r8", N=264, K=320, M=33, r=8, alpha=16.0)
OTHER = inputs.LinearShape("noalloc_N520_K384_M200_r16", N=520, K=384, M=200, r=16, alpha=32.0)
# (shape, pass the forward's saved t?)
SEQUENCE = [(LARGE, True), (SMALL, True), (LARGE, True), (OTHER, False)]


def _case(shape):
    d = inputs.linear_inputs(shape)
    g = {k: v.cuda().contiguous() for k, v in d.items()}
    q = capi.quantize_nf4(g["W"])
    ref_q = oracle.quantize_nf4(d["W"].float().numpy(), 64, 256)
    ref = oracle.linear_bwd(d["x"].float().numpy(), d["dY"].float().numpy(),
                            oracle.dequant_f32(ref_q), d["A"].float().numpy(),
                            d["B"].float().numpy(), shape.alpha)
    ws = capi.Workspace(shape.M, shape.N, shape.K, shape.r)
    t = torch.empty(shape.M, shape.r, dtype=torch.float32, device="cuda")
    capi.linear_fwd(q, g["x"], g["A"], g["B"], shape.alpha, ws, t_save=t)
    fresh = capi.linear_bwd(q, g["x"], g["dY"], g["A"], g["B"], shape.alpha, ws, t_saved=t)
    torch.cuda.synchronize()
    assert ws.device_status() == 0
    return g, q, t, ref, [x.clone() for x in fresh]


def test_noalloc_backward_over_a_sequence_of_shapes():
    capi.load()
    cases = {s.name: _case(s) for s in (LARGE, SMALL, OTHER)}
    for call, (shape, saved) in enumerate(SEQUENCE):
        g, q, t, ref, fresh = cases[shape.name]
        got = capi.linear_bwd_noalloc(q, g["x"], g["dY"], g["A"], g["B"], shape.alpha,
                                      t_saved=t if saved else None)
        torch.cuda.synchronize()
        tag = f"call {call} {shape.name} t_saved={saved}"
        for name, a, b in zip(("dX", "dA", "dB"), got, fresh):
            assert_close(to_np_f32(a), ref[name], f"{name} vs oracle, {tag}")
            assert_close(to_np_f32(a), to_np_f32(b), f"{name} vs workspace call, {tag}")


def test_noalloc_backward_rejects_sizes_beyond_its_scratch():
    """A size whose workspace exceeds the fixed scratch is refused with
    QLORA_ERR_WORKSPACE before any device memory is touched."""
    lib = capi.load()
    N, K, M, r = 14336, 4096, 65536, 64
    assert capi.workspace_size_min(M, N, K, r) > 16 << 20
    q = capi.quantize_nf4(torch.zeros(64, 64, dtype=torch.bfloat16, device="cuda"))
    big = capi.NF4Weight(N, K, q.packed, q.absmax_code, q.scale2, None)  # never read
    x = torch.zeros(8, dtype=torch.bfloat16, device="cuda")
    p = capi._ptr(x)
    status = lib.qlora_linear_bwd_noalloc(ctypes.byref(big.struct()), p, p, M, p, p, r, 1.0,
                                          None, p, capi.QLORA_F32, p, p, 0, capi._stream(None))
    assert status == 8  # QLORA_ERR_WORKSPACE
