"""Guard canaries: every output and workspace of the library's entry points is
placed inside a larger buffer whose margins hold a known byte pattern, and the
margins must come back untouched. Element parity only sees the outputs
themselves; a stray store past an output's end (a padded row, a split part's
fp32 rows, the merge, the preprocessing pass's padded rows, a host-buffer
chunk copy) would only show up here. The outputs are also checked against
the oracle, and their interiors are pre-filled with the same pattern so that
an unwritten output element would fail that check."""

import ctypes
import math

import numpy as np
import pytest
import torch

from exact_attention_64_gb300.workloads import make_inputs
from tests.parity import TOL, max_abs, oracle_bwd, oracle_fwd, rel_fro, to64

pytestmark = pytest.mark.gpu

MARGIN = 1 << 16          # bytes of canary on each side (a multiple of 256)
POISON = 0xA5             # 0xA5A5 is a finite bf16 / fp16 value; 0xA5A5A5A5 a finite fp32


class Guarded:
    """`nbytes` usable bytes at a 256-byte aligned offset inside a buffer of
    poison, on `device` (or pinned host memory for device=None)."""

    def __init__(self, nbytes: int, device):
        self.n = nbytes
        total = MARGIN + ((nbytes + 255) // 256) * 256 + MARGIN
        if device is None:
            self.buf = torch.full((total,), POISON, dtype=torch.uint8).pin_memory()
        else:
            self.buf = torch.full((total,), POISON, dtype=torch.uint8, device=device)
        assert self.buf.data_ptr() % 256 == 0

    def tensor(self, shape, dtype):
        t = self.buf[MARGIN:MARGIN + self.n].view(dtype).view(shape)
        assert t.data_ptr() % 256 == 0
        return t

    @property
    def ptr(self) -> int:
        return self.buf.data_ptr() + MARGIN

    def margins_intact(self) -> bool:
        head = self.buf[:MARGIN]
        tail = self.buf[MARGIN + self.n:]
        return bool((head == POISON).all()) and bool((tail == POISON).all())


def _nbytes(shape, dtype):
    return int(np.prod(shape)) * torch.tensor([], dtype=dtype).element_size()


SHAPES = [(N, d) for N in (1, 127, 129, 1000) for d in (64, 128)]


def _guarded_fwd_outputs(B, H, N, d, dtype, dev):
    go = Guarded(_nbytes((B, H, N, d), dtype), dev)
    gl = Guarded(_nbytes((B, H, N), torch.float32), dev)
    return go, gl, go.tensor((B, H, N, d), dtype), gl.tensor((B, H, N), torch.float32)


@pytest.mark.parametrize("N,d", SHAPES)
@pytest.mark.parametrize("S", [1, 2, 5, 128])
def test_forward_writes_nothing_outside_its_outputs(cuda_device, fa2_lib, N, d, S):
    B, H, dt = 1, 3, torch.bfloat16
    dev = cuda_device
    q, k, v, _ = make_inputs(B, H, N, d, dt, seed=N + d + S)
    scale = 1.0 / math.sqrt(d)
    lib = fa2_lib.load_library()
    qd, kd, vd = (t.to(dev) for t in (q, k, v))
    for causal in (False, True):
        go, gl, o, lse = _guarded_fwd_outputs(B, H, N, d, dt, dev)
        stream = ctypes.c_void_p(torch.cuda.current_stream(dev).cuda_stream)
        if S == 1:
            code = lib.fa2_fwd(qd.data_ptr(), kd.data_ptr(), vd.data_ptr(), o.data_ptr(),
                               lse.data_ptr(), B, H, N, d, int(causal), scale, 1, stream)
            gw = None
        else:
            nbytes = lib.fa2_fwd_split_workspace_size(B, H, N, d, S)
            gw = Guarded(nbytes, dev)
            code = lib.fa2_fwd_split(qd.data_ptr(), kd.data_ptr(), vd.data_ptr(), o.data_ptr(),
                                     lse.data_ptr(), B, H, N, d, int(causal), scale, 1, S,
                                     gw.ptr, nbytes, stream)
        assert code == 0
        torch.cuda.synchronize()
        assert fa2_lib.device_status() == 0
        assert go.margins_intact() and gl.margins_intact(), (causal, "outputs")
        assert gw is None or gw.margins_intact(), (causal, "split workspace")
        o_ref, lse_ref = oracle_fwd(q, k, v, causal, scale)
        assert max_abs(to64(o.cpu()), o_ref) <= TOL[dt]["o"]
        assert max_abs(to64(lse.cpu()), lse_ref) <= TOL[dt]["lse"]


@pytest.mark.parametrize("N,d", SHAPES)
@pytest.mark.parametrize("Nk_delta", [0, 1, -1])
def test_backward_writes_nothing_outside_its_outputs(cuda_device, fa2_lib, N, d, Nk_delta):
    """fa2_bwd (equal lengths) and fa2_bwd_qk (one key more or fewer)."""
    Nk = max(1, N + Nk_delta)
    B, H, dt = 2, 1, torch.float16
    dev = cuda_device
    q, _, _, do = make_inputs(B, H, N, d, dt, seed=5 * N + d)
    _, k, v, _ = make_inputs(B, H, Nk, d, dt, seed=5 * N + d + 1)
    scale = 1.0 / math.sqrt(d)
    lib = fa2_lib.load_library()
    qd, kd, vd, dod = (t.to(dev) for t in (q, k, v, do))
    for causal in (False, True):
        o, lse = fa2_lib.forward(qd, kd, vd, causal=causal, scale=scale)
        gq = Guarded(_nbytes((B, H, N, d), dt), dev)
        gk = Guarded(_nbytes((B, H, Nk, d), dt), dev)
        gv = Guarded(_nbytes((B, H, Nk, d), dt), dev)
        wbytes = lib.fa2_bwd_workspace_size(B, H, N, d)
        gw = Guarded(wbytes, dev)
        dq = gq.tensor((B, H, N, d), dt)
        dk = gk.tensor((B, H, Nk, d), dt)
        dv = gv.tensor((B, H, Nk, d), dt)
        stream = ctypes.c_void_p(torch.cuda.current_stream(dev).cuda_stream)
        code = lib.fa2_bwd_qk(qd.data_ptr(), kd.data_ptr(), vd.data_ptr(), o.data_ptr(),
                              lse.data_ptr(), dod.data_ptr(), dq.data_ptr(), dk.data_ptr(),
                              dv.data_ptr(), B, H, N, Nk, d, int(causal), scale, 0, gw.ptr,
                              wbytes, stream)
        assert code == 0
        torch.cuda.synchronize()
        assert fa2_lib.device_status() == 0
        for g, name in ((gq, "dq"), (gk, "dk"), (gv, "dv"), (gw, "workspace")):
            assert g.margins_intact(), (causal, name)
        ref = oracle_bwd(q, k, v, do, causal, scale)
        for g, r, name in zip((dq, dk, dv), ref, ("dq", "dk", "dv")):
            assert rel_fro(to64(g.cpu()), r) <= TOL[dt]["grad"], (causal, name)


@pytest.mark.parametrize("N,d", [(1, 64), (129, 128), (1000, 64)])
def test_step_host_writes_nothing_outside_its_buffers(cuda_device, fa2_lib, N, d):
    """fa2_step_host: host outputs (pinned) and the device workspace."""
    B, H, dt, hpc = 1, 5, torch.bfloat16, 2
    dev = cuda_device
    q, k, v, do = make_inputs(B, H, N, d, dt, seed=N + 3 * d)
    scale = 1.0 / math.sqrt(d)
    lib = fa2_lib.load_library()
    shape = (B, H, N, d)
    guards = {n: Guarded(_nbytes(shape, dt), None) for n in ("o", "dq", "dk", "dv")}
    guards["lse"] = Guarded(_nbytes((B, H, N), torch.float32), None)
    outs = {n: g.tensor(shape, dt) for n, g in guards.items() if n != "lse"}
    outs["lse"] = guards["lse"].tensor((B, H, N), torch.float32)
    wbytes = lib.fa2_step_host_workspace_size(B, H, N, d, hpc)
    gw = Guarded(wbytes, dev)
    ws = gw.buf[MARGIN:MARGIN + wbytes]
    with torch.cuda.device(dev):
        fa2_lib.step_host(q.pin_memory(), k.pin_memory(), v.pin_memory(), do.pin_memory(),
                          causal=True, scale=scale, heads_per_chunk=hpc, device=dev,
                          out=(outs["o"], outs["lse"], outs["dq"], outs["dk"], outs["dv"]),
                          workspace=ws)
    assert fa2_lib.device_status() == 0
    for name, g in list(guards.items()) + [("workspace", gw)]:
        assert g.margins_intact(), name
    o_ref, lse_ref = oracle_fwd(q, k, v, True, scale)
    assert max_abs(to64(outs["o"]), o_ref) <= TOL[dt]["o"]
    assert max_abs(to64(outs["lse"]), lse_ref) <= TOL[dt]["lse"]
    ref = oracle_bwd(q, k, v, do, True, scale)
    for name, r in zip(("dq", "dk", "dv"), ref):
        assert rel_fro(to64(outs[name]), r) <= TOL[dt]["grad"], name
