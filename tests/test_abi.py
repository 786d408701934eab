"""The C ABI without a GPU: the library loads, exports every symbol the
header declares, and rejects bad arguments before touching the device."""

import re
from pathlib import Path

HEADER = Path(__file__).resolve().parent.parent / "include" / "fa2.h"


def _declared():
    text = HEADER.read_text()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(fa2_\w+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = _declared()
    for required in ("fa2_fwd", "fa2_bwd", "fa2_bwd_workspace_size", "fa2_get_device_status",
                     "fa2_status_string"):
        assert required in names


def test_library_exports_every_declared_symbol(fa2_lib):
    lib = fa2_lib.load_library()
    missing = [n for n in _declared() if not hasattr(lib, n)]
    assert not missing, missing


def test_status_strings(fa2_lib):
    names = ["FA2_OK", "FA2_ERR_INVALID_ARG", "FA2_ERR_UNSUPPORTED", "FA2_ERR_ALIGNMENT",
             "FA2_ERR_ARCH", "FA2_ERR_CUDA", "FA2_ERR_DEVICE_TIMEOUT", "FA2_ERR_WORKSPACE",
             "FA2_ERR_OVERLAP"]
    for code, name in enumerate(names):
        assert fa2_lib.status_string(code) == name
    assert fa2_lib.status_string(99) == "FA2_ERR_UNKNOWN"


# Fake, never-dereferenced device addresses: validation fails before any CUDA call.
A = 0x10000000
STEP = 0x01000000


def _fwd(lib, q=A, k=A + STEP, v=A + 2 * STEP, o=A + 3 * STEP, lse=A + 4 * STEP, B=1, H=1, N=128,
         d=64, causal=0, scale=0.125, dtype=1):
    return lib.fa2_fwd(q, k, v, o, lse, B, H, N, d, causal, scale, dtype, None)


def test_fwd_rejects_bad_arguments(fa2_lib):
    lib = fa2_lib.load_library()
    assert _fwd(lib, q=0) == 1
    assert _fwd(lib, lse=0) == 1
    assert _fwd(lib, B=0) == 1
    assert _fwd(lib, N=0) == 1
    assert _fwd(lib, causal=2) == 1
    assert _fwd(lib, dtype=5) == 1
    assert _fwd(lib, scale=float("nan")) == 1
    assert _fwd(lib, scale=-1.0) == 1
    assert _fwd(lib, d=96) == 2
    assert _fwd(lib, d=256) == 2
    assert _fwd(lib, B=70000) == 2
    assert _fwd(lib, q=A + 8) == 3
    assert _fwd(lib, o=A + 3 * STEP + 2) == 3
    assert _fwd(lib, lse=A + 4 * STEP + 2) == 3
    assert _fwd(lib, o=A) == 8            # output aliases q
    assert _fwd(lib, lse=A + STEP + 64) == 8


def test_bwd_rejects_bad_arguments(fa2_lib):
    lib = fa2_lib.load_library()
    ws = lib.fa2_bwd_workspace_size(1, 1, 128, 64)
    base = [A + i * STEP for i in range(10)]

    def call(ptrs=base, wsz=ws, d=64, **kw):
        p = list(ptrs)
        return lib.fa2_bwd(p[0], p[1], p[2], p[3], p[4], p[5], p[6], p[7], p[8], 1, 1, 128, d,
                           kw.get("causal", 0), kw.get("scale", 0.125), 1, p[9], wsz, None)

    assert call([0] + base[1:]) == 1
    assert call(d=80) == 2
    assert call(wsz=ws - 1) == 7
    assert call(base[:9] + [0]) == 7
    bad = list(base)
    bad[9] = base[9] + 16
    assert call(bad) == 3                 # workspace must be 256-byte aligned
    bad = list(base)
    bad[6] = base[0]                      # dq aliases q
    assert call(bad) == 8


def test_workspace_size(fa2_lib):
    lib = fa2_lib.load_library()
    for fn in (lib.fa2_bwd_workspace_size, lib.fa2_bwd_atomic_workspace_size):
        assert fn(0, 1, 1, 64) == 0
        assert fn(1, 1, 1, 96) == 0
    # D and L*log2e, each [B*H][N rounded up to 128] fp32, then 256 bytes for
    # the persistent main launch's work counter
    assert lib.fa2_bwd_workspace_size(1, 1, 100, 64) == 2 * 512 + 256
    B, H, N, d = 4, 32, 8192, 128
    assert lib.fa2_bwd_workspace_size(B, H, N, d) == 2 * B * H * N * 4 + 256
    # fa2_bwd_atomic: the same, then the fp32 dQ accumulator [B*H][N rounded up to 128][d]
    assert lib.fa2_bwd_atomic_workspace_size(1, 1, 100, 64) == 2 * 512 + 256 + 128 * 64 * 4
    assert lib.fa2_bwd_atomic_workspace_size(B, H, N, d) == 2 * B * H * N * 4 + 256 + B * H * N * d * 4
    assert lib.fa2_bwd_atomic_workspace_size(3, 1, 129, 128) == 2 * 3 * 256 * 4 + 256 + 3 * 256 * 128 * 4


def test_fault_arming_validates(fa2_lib):
    lib = fa2_lib.load_library()
    assert lib.fa2_debug_arm_fault(5, 10) == 1
    assert lib.fa2_debug_arm_fault(-1, 10) == 1
    for kind in (1, 2, 3, 4):
        assert lib.fa2_debug_arm_fault(kind, 0) == 1
        assert lib.fa2_debug_arm_fault(kind, 5001) == 1
        assert lib.fa2_debug_arm_fault(kind, 10) == 0
    assert lib.fa2_debug_arm_fault(0, 0) == 0   # disarm again


def test_kv_outer_rejects_bad_arguments(fa2_lib):
    lib = fa2_lib.load_library()
    ws = lib.fa2_fwd_kv_outer_workspace_size(1, 1, 128, 64)
    base = [A + i * STEP for i in range(6)]

    def call(ptrs=base, wsz=ws, d=64, causal=0):
        p = list(ptrs)
        return lib.fa2_fwd_kv_outer(p[0], p[1], p[2], p[3], p[4], 1, 1, 128, d, causal, 0.125, 1,
                                    p[5], wsz, None)

    assert call([0] + base[1:]) == 1
    assert call(causal=3) == 1
    assert call(d=80) == 2
    assert call(wsz=ws - 1) == 7
    assert call(base[:5] + [0]) == 7
    assert call(base[:5] + [base[5] + 16]) == 3   # workspace must be 256-byte aligned
    assert call(base[:3] + [base[0]] + base[4:]) == 8  # o aliases q
    assert call(base[:5] + [base[1]]) == 8             # workspace overlaps k


def test_step_host_rejects_bad_arguments(fa2_lib):
    lib = fa2_lib.load_library()
    ws = lib.fa2_step_host_workspace_size(1, 2, 128, 64, 1)
    assert ws > 0
    base = [A + i * STEP for i in range(10)]

    def call(ptrs=base, wsz=ws, d=64, hpc=1, causal=0, dtype=1):
        p = list(ptrs)
        return lib.fa2_step_host(p[0], p[1], p[2], p[3], p[4], p[5], p[6], p[7], p[8], 1, 2, 128, d,
                                 causal, 0.125, dtype, hpc, p[9], wsz, None)

    assert call([0] + base[1:]) == 1
    assert call(causal=2) == 1
    assert call(dtype=7) == 1
    assert call(hpc=-1) == 1
    assert call(hpc=3) == 1               # more heads per chunk than heads
    assert call(d=96) == 2
    assert call(wsz=ws - 1) == 7
    assert call(base[:9] + [0]) == 7
    assert call(base[:9] + [base[9] + 16]) == 3
    assert lib.fa2_step_host_workspace_size(1, 2, 128, 96, 1) == 0
    assert lib.fa2_step_host_workspace_size(1, 2, 128, 64, 3) == 0
    # auto chunking: ceil(B*H / 8) heads per chunk
    assert lib.fa2_step_host_workspace_size(4, 32, 1024, 128, 0) == \
        lib.fa2_step_host_workspace_size(4, 32, 1024, 128, 16)
