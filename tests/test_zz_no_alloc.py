"""The allocation-free backward entry point.

qlora_linear_bwd_noalloc serves callers that cannot allocate device memory
(graph capture, restrictive allocators, hosts that pass only inputs and
outputs).  Called through the C ABI twice in a row, it must give the same
gradients as qlora_linear_bwd with a caller workspace, within the tolerance
the other parity tests use, and must refuse sizes beyond its fixed scratch.
This file is collected last so that a failure here never hides another test.
"""
import ctypes

import pytest
import torch

from bit_nf4_quantized_35_b300 import capi, inputs

from .helpers import assert_close, to_np_f32

pytestmark = pytest.mark.gpu


def test_noalloc_backward_matches_workspace_backward_twice():
    capi.load()
    shape = inputs.LinearShape("noalloc_N520_K384_M200_r16", N=520, K=384, M=200, r=16,
                               alpha=32.0)
    d = inputs.linear_inputs(shape)
    g = {k: v.cuda().contiguous() for k, v in d.items()}
    q = capi.quantize_nf4(g["W"])
    ws = capi.Workspace(shape.M, shape.N, shape.K, shape.r)
    t = torch.empty(shape.M, shape.r, dtype=torch.float32, device="cuda")
    capi.linear_fwd(q, g["x"], g["A"], g["B"], shape.alpha, ws, t_save=t)
    ref = capi.linear_bwd(q, g["x"], g["dY"], g["A"], g["B"], shape.alpha, ws, t_saved=t)
    torch.cuda.synchronize()
    for call in range(2):
        got = capi.linear_bwd_noalloc(q, g["x"], g["dY"], g["A"], g["B"], shape.alpha,
                                      t_saved=t)
        torch.cuda.synchronize()
        for name, a, b in zip(("dX", "dA", "dB"), got, ref):
            assert_close(to_np_f32(a), to_np_f32(b), f"{name} (no-alloc call {call})")


def test_noalloc_backward_rejects_sizes_beyond_its_scratch():
    """A size whose workspace exceeds the fixed scratch is refused with
    QLORA_ERR_WORKSPACE before any device memory is touched."""
    lib = capi.load()
    N, K, M, r = 14336, 4096, 65536, 64
    assert capi.workspace_size(M, N, K, r) > 16 << 20
    q = capi.quantize_nf4(torch.zeros(64, 64, dtype=torch.bfloat16, device="cuda"))
    big = capi.NF4Weight(N, K, q.packed, q.absmax_code, q.scale2, None)  # never read
    x = torch.zeros(8, dtype=torch.bfloat16, device="cuda")
    p = capi._ptr(x)
    status = lib.qlora_linear_bwd_noalloc(ctypes.byref(big.struct()), p, p, M, p, p, r, 1.0,
                                          None, p, capi.QLORA_F32, p, p, 0, capi._stream(None))
    assert status == 8  # QLORA_ERR_WORKSPACE
