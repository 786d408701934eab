"""fa2_bwd_noalloc: the backward pass for callers that must not allocate
device memory (for example code inside a memory pool or framework allocator
it does not own, or a process that fixed its device footprint at start-up).

It keeps the backward's small scratch in an array built into the library, so
the caller passes only inputs and outputs. It runs the same kernels as
fa2_bwd, which takes a caller-allocated workspace, so on the same inputs the
gradients must be equal bit for bit, call after call: the built-in array keeps
the previous call's contents, and none of that may leak into the next call's
gradients. The calls below change the data at a fixed shape, shrink the shape
and grow it again, so stale row sums or logsumexps in the array would change
bits. This file is collected last on purpose, and the test also passes when
run alone in a fresh process.
"""

import ctypes
import math

import pytest
import torch

from exact_attention_64_gb300.workloads import make_inputs

_VP, _I, _F = ctypes.c_void_p, ctypes.c_int, ctypes.c_float

FA2_ERR_INVALID_ARG, FA2_ERR_UNSUPPORTED, FA2_ERR_CUDA = 1, 2, 5


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
    cases = [
        # (B, H, N, d, dtype, causal, seed)
        (1, 2, 1000, 128, torch.bfloat16, True, 1),
        (1, 2, 1000, 128, torch.bfloat16, True, 2),   # same shape, new data
        (2, 1, 300, 64, torch.float16, False, 3),     # smaller
        (1, 3, 2000, 128, torch.bfloat16, True, 4),   # larger again
        (1, 3, 2000, 128, torch.bfloat16, True, 4),   # the same call twice
    ]
    for B, H, N, d, dtype, causal, seed in cases:
        q, k, v, do = (t.to(dev) for t in make_inputs(B, H, N, d, dtype, seed=seed))
        scale = 1.0 / math.sqrt(d)
        o, lse = fa2_lib.forward(q, k, v, causal=causal, scale=scale)
        ref = fa2_lib.backward(q, k, v, o, lse, do, causal=causal, scale=scale)
        dq, dk, dv = (torch.full_like(q, float("nan")) for _ in range(3))
        stream = ctypes.c_void_p(torch.cuda.current_stream(dev).cuda_stream)
        code = fn(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                  do.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), B, H, N, d,
                  int(causal), scale, 1 if dtype == torch.bfloat16 else 0, stream)
        assert code == 0, fa2_lib.status_string(code)
        torch.cuda.synchronize()
        assert fa2_lib.device_status() == 0
        for name, got, want in zip(("dq", "dk", "dv"), (dq, dk, dv), ref):
            assert torch.equal(got, want), (name, B, H, N, seed)


def test_noalloc_size_limit_at_its_boundary(fa2_lib):
    """The built-in array holds 16 MiB + 256 bytes: 8 bytes per padded query row
    and the work counter. B*H = 256 heads of N = 8192 need exactly that and pass
    the size check (this call
    then fails on its invalid dtype, or on a machine without a GPU on the
    device lookup, but never with FA2_ERR_UNSUPPORTED); 257 heads, or N = 8193
    (one more 128-row tile per head), are refused with FA2_ERR_UNSUPPORTED
    before anything touches the device."""
    lib = fa2_lib.load_library()
    fn = _noalloc(lib)
    a = 0x10000000
    ptrs = [a + i * 0x01000000 for i in range(9)]
    assert lib.fa2_bwd_workspace_size(16, 16, 8192, 128) == (16 << 20) + 256
    bad_dtype = 7
    assert fn(*ptrs, 16, 16, 8192, 128, 1, 0.088, bad_dtype, None) in (FA2_ERR_INVALID_ARG,
                                                                        FA2_ERR_CUDA)
    assert fn(*ptrs, 1, 257, 8192, 128, 1, 0.088, 1, None) == FA2_ERR_UNSUPPORTED
    assert fn(*ptrs, 16, 16, 8193, 64, 1, 0.088, 1, None) == FA2_ERR_UNSUPPORTED
    assert fn(*ptrs, 64, 64, 8192, 128, 1, 0.088, 1, None) == FA2_ERR_UNSUPPORTED
