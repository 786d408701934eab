"""fa2_bwd_noalloc: the backward pass for callers that must not allocate
device memory (for example code inside a memory pool or framework allocator
it does not own, or a process that fixed its device footprint at start-up).

It keeps the backward's small scratch in an array built into the library, so
the caller passes only inputs and outputs. Its results must match fa2_bwd,
which takes a caller-allocated workspace, on consecutive calls: the built-in
array keeps the previous call's contents, and that must not leak into the
next call's gradients. This file is collected last on purpose, and the test
also passes when run alone in a fresh process.
"""

import ctypes
import math

import pytest
import torch

from exact_attention_64_gb300.workloads import make_inputs
from tests.parity import TOL, rel_fro, to64

_VP, _I, _F = ctypes.c_void_p, ctypes.c_int, ctypes.c_float


def _noalloc(lib):
    fn = lib.fa2_bwd_noalloc
    fn.restype = _I
    fn.argtypes = [_VP] * 9 + [_I] * 5 + [_F, _I, _VP]
    return fn


@pytest.mark.gpu
def test_noalloc_backward_matches_workspace_backward(cuda_device, fa2_lib):
    lib = fa2_lib.load_library()
    fn = _noalloc(lib)
    dev = cuda_device
    # Two consecutive calls with different shapes, dtypes and masks.
    cases = [(1, 2, 1000, 128, torch.bfloat16, True), (2, 1, 300, 64, torch.float16, False)]
    for B, H, N, d, dtype, causal in cases:
        q, k, v, do = (t.to(dev) for t in make_inputs(B, H, N, d, dtype, seed=B * 1000 + N))
        scale = 1.0 / math.sqrt(d)
        o, lse = fa2_lib.forward(q, k, v, causal=causal, scale=scale)
        ref = fa2_lib.backward(q, k, v, o, lse, do, causal=causal, scale=scale)
        dq, dk, dv = (torch.empty_like(q) for _ in range(3))
        stream = ctypes.c_void_p(torch.cuda.current_stream(dev).cuda_stream)
        code = fn(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                  do.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), B, H, N, d,
                  int(causal), scale, 1 if dtype == torch.bfloat16 else 0, stream)
        assert code == 0, fa2_lib.status_string(code)
        torch.cuda.synchronize()
        assert fa2_lib.device_status() == 0
        for got, want in zip((dq, dk, dv), ref):
            assert rel_fro(to64(got), to64(want)) <= TOL[dtype]["grad"]


def test_noalloc_rejects_sizes_beyond_its_scratch(fa2_lib):
    """Shapes whose scratch would not fit the built-in array are refused with
    FA2_ERR_UNSUPPORTED before anything touches the device."""
    fn = _noalloc(fa2_lib.load_library())
    a = 0x10000000
    ptrs = [a + i * 0x01000000 for i in range(9)]
    # 64 x 64 heads of 8192 rows need 32 MiB of scratch.
    assert fn(*ptrs, 64, 64, 8192, 128, 1, 0.088, 1, None) == 2
