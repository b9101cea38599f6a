"""The C ABI without a GPU: the library loads, exports what include/kda.h
declares, and rejects bad arguments before touching the device."""
import os
import re

import pytest

import prefill_kda_chunk_gb300 as K
from prefill_kda_chunk_gb300 import build as B

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    B.build()
    return K.lib()


def declared_symbols():
    names = []
    for fn in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if fn.endswith(".h"):
            text = open(os.path.join(ROOT, "include", fn)).read()
            names += re.findall(r"KDA_API\s+[\w\s\*]*?\b(kda_\w+)\s*\(", text)
    return names


def test_every_declared_symbol_is_exported(lib):
    names = declared_symbols()
    assert "kda_chunk_prefill" in names and len(names) >= 6
    for n in names:
        assert hasattr(lib, n), n


def test_status_strings(lib):
    for code, name in K.STATUS.items():
        s = K.kda_status_string(code)
        assert s and s != "unknown status", name
    assert K.kda_status_string(12345) == "unknown status"


def test_workspace_bytes(lib):
    REC = 17408

    def lst(items):                            # exact-form list: one int32 per chunk-head
        return -(-(items * 4) // 256) * 256

    # 512 chunks x 64 heads x 17408 B + the flag block + the list
    assert K.kda_workspace_bytes(1, 8192, 64, 1, 0) == 256 + 512 * 64 * REC + lst(512 * 64)
    assert K.kda_workspace_bytes(1, 256, 2, 1, 0) == 256 + 16 * 2 * REC + lst(32)  # small
    # packed batches: the chunk offsets after the flag block
    pc = (8192 + 15 * 16) // 16
    assert K.kda_workspace_bytes(1, 8192, 64, 16, 1) == 256 + 256 + pc * 64 * REC + lst(pc * 64)
    # long sequences with few heads: records plus the segment scan's entry
    # states, offsets and maps (3 P - 5 planes of N H 64 KiB); without a GPU
    # the library sizes for 152 SMs: with 4 N H <= 148, P = 3 (152 - 4) // (2 N H),
    # at most 16 and at least 16 chunks per segment, then no segment left empty
    def planes(nh, cps):
        if cps < 64 or 4 * nh > 148:
            return 0
        P = min(3 * (152 - 4) // (2 * nh), 16, cps // 16)
        if P < 2:
            return 0
        L = -(-cps // P)
        P = -(-cps // L)
        return 3 * P - 5 if P >= 2 else 0

    assert planes(32, 8192) == 13                    # P = 6
    assert K.kda_workspace_bytes(1, 131072, 32, 1, 0) == (256 + 8192 * 32 * REC + 13 * 32 * 65536
                                                         + lst(8192 * 32))
    assert planes(64, 512) == 0                      # T8192 H64: the plain chains fill the SMs
    assert K.kda_workspace_bytes(1, 8192, 64, 1, 0) == 256 + 512 * 64 * REC + lst(512 * 64)
    assert planes(6, 125) == 16                      # P = 7
    assert K.kda_workspace_bytes(2, 2000, 3, 2, 0) == (256 + 2 * 125 * 3 * REC + 16 * 6 * 65536
                                                      + lst(2 * 125 * 3))
    # forced segment counts, and off
    try:
        for P, expect in ((3, 4), (8, 19), (1, 0)):
            assert K.kda_set_scan_segments(P) == 0
            assert K.kda_workspace_bytes(1, 131072, 32, 1, 0) == (256 + 8192 * 32 * REC
                                                                 + expect * 32 * 65536
                                                                 + lst(8192 * 32))
        assert K.kda_set_scan_segments(200) == 0     # more segments than 125 chunks allow
        assert K.kda_workspace_bytes(2, 2000, 3, 2, 0) == (256 + 2 * 125 * 3 * REC
                                                          + (3 * 125 - 5) * 6 * 65536
                                                          + lst(2 * 125 * 3))
        assert K.kda_set_scan_segments(-1) != 0 and K.kda_set_scan_segments(5000) != 0
    finally:
        K.kda_set_scan_segments(0)
    assert K.kda_workspace_bytes(1, 1008, 3, 1, 0) == 256 + 63 * 3 * REC + lst(63 * 3)  # < 64 chunks
    assert K.kda_workspace_bytes(1, 8192, 38, 1, 0) == 256 + 512 * 38 * REC + lst(512 * 38)  # 4*38 > 152 - 4 (no device here: sized for 152 SMs)
    assert K.kda_workspace_bytes(1, 8192, 64, 2, 0) == 0      # N != B without cu_seqlens
    assert K.kda_workspace_bytes(2, 100, 0, 2, 0) == 0        # H < 1


A = 1 << 20  # an aligned fake address; validation fails before any dereference


def call(**kw):
    args = dict(q=A, k=A + 0x100000, v=A + 0x200000, g=A + 0x300000, beta=A + 0x400000,
                initial_state=0, cu_seqlens=0, B=1, T=16, H=1, K=128, V=128, N=1, scale=1.0,
                out=A + 0x500000, final_state=0, stream=0)
    args.update(kw)
    return K.kda_chunk_prefill(**args)


@pytest.mark.parametrize("kw,code", [
    (dict(q=0), "KDA_ERR_NULL_ARG"),
    (dict(out=0), "KDA_ERR_NULL_ARG"),
    (dict(K=64), "KDA_ERR_UNSUPPORTED_DIM"),
    (dict(V=256), "KDA_ERR_UNSUPPORTED_DIM"),
    (dict(H=0), "KDA_ERR_BAD_SHAPE"),
    (dict(T=-1), "KDA_ERR_BAD_SHAPE"),
    (dict(N=2), "KDA_ERR_BAD_SHAPE"),
    (dict(B=2, N=2, cu_seqlens=A + 0x600000), "KDA_ERR_BAD_SHAPE"),
    (dict(q=A + 2), "KDA_ERR_MISALIGNED"),
    (dict(g=A + 0x300004), "KDA_ERR_MISALIGNED"),
    (dict(beta=A + 0x400002), "KDA_ERR_MISALIGNED"),
    (dict(out=A), "KDA_ERR_ALIAS"),
    (dict(out=A + 0x300000 + 4096), "KDA_ERR_ALIAS"),
    (dict(final_state=A + 0x200000), "KDA_ERR_ALIAS"),
    (dict(initial_state=A + 0x700000, final_state=A + 0x700000 + 4096), "KDA_ERR_ALIAS"),
])
def test_host_validation_rejects(lib, kw, code):
    assert call(**kw) == K.STATUS_CODE[code]


def decode_call(**kw):
    args = dict(q=A, k=A + 0x100000, v=A + 0x200000, g=A + 0x300000, beta=A + 0x400000,
                state_in=A + 0x800000, state_out=A + 0x800000, N=2, H=3, K=128, V=128,
                scale=1.0, flags=0, out=A + 0x500000, stream=0)
    args.update(kw)
    return K.kda_decode_step(**args)


@pytest.mark.parametrize("kw,code", [
    (dict(q=0), "KDA_ERR_NULL_ARG"),
    (dict(state_out=0), "KDA_ERR_NULL_ARG"),
    (dict(out=0), "KDA_ERR_NULL_ARG"),
    (dict(K=64), "KDA_ERR_UNSUPPORTED_DIM"),
    (dict(V=64), "KDA_ERR_UNSUPPORTED_DIM"),
    (dict(H=0), "KDA_ERR_BAD_SHAPE"),
    (dict(N=-1), "KDA_ERR_BAD_SHAPE"),
    (dict(N=1 << 30, H=4), "KDA_ERR_BAD_SHAPE"),
    (dict(k=A + 0x100002), "KDA_ERR_MISALIGNED"),
    (dict(state_in=A + 0x800004, state_out=A + 0x900000), "KDA_ERR_MISALIGNED"),
    (dict(beta=A + 0x400001), "KDA_ERR_MISALIGNED"),
    (dict(out=A + 0x100000), "KDA_ERR_ALIAS"),
    (dict(out=A + 0x800000 + 256), "KDA_ERR_ALIAS"),
    (dict(state_out=A + 0x300000), "KDA_ERR_ALIAS"),
    (dict(state_out=A + 0x800000 + 4096), "KDA_ERR_ALIAS"),
    (dict(flags=4), "KDA_ERR_BAD_FLAGS"),
    (dict(flags=-1), "KDA_ERR_BAD_FLAGS"),
])
def test_decode_host_validation_rejects(lib, kw, code):
    assert decode_call(**kw) == K.STATUS_CODE[code]


def test_decode_empty_batch_is_a_no_op(lib):
    # N = 0: nothing to do, and no pointer is needed
    assert K.kda_decode_step(0, 0, 0, 0, 0, 0, 0, 0, 4, 128, 128, 1.0, 0, 0, 0) == 0


def test_prefill_ex_flags(lib):
    args = dict(q=A, k=A + 0x100000, v=A + 0x200000, g=A + 0x300000, beta=A + 0x400000,
                initial_state=0, cu_seqlens=0, B=1, T=16, H=1, K=128, V=128, N=1, scale=1.0,
                out=A + 0x500000, final_state=0, stream=0)
    assert K.kda_chunk_prefill_ex(**args, flags=8) == K.STATUS_CODE["KDA_ERR_BAD_FLAGS"]
    # known flags pass the host checks and reach the argument checks after them
    assert K.kda_chunk_prefill_ex(**dict(args, K=64), flags=3) == K.STATUS_CODE["KDA_ERR_UNSUPPORTED_DIM"]


def bwd(**kw):
    args = dict(q=A, k=A + 0x100000, v=A + 0x200000, g=A + 0x300000, beta=A + 0x400000,
                initial_state=0, cu_seqlens=0, B=1, T=16, H=1, K=128, V=128, N=1, scale=1.0,
                d_out=A + 0x500000, d_final_state=0, dq=A + 0x600000, dk=A + 0x700000,
                dv=A + 0x800000, dg=A + 0x900000, dbeta=A + 0xA00000, d_initial_state=0,
                stream=0)
    args.update(kw)
    return K.kda_chunk_prefill_backward(**args)


def test_backward_argument_checks(lib):
    S = K.STATUS_CODE
    assert bwd(K=64) == S["KDA_ERR_UNSUPPORTED_DIM"]
    assert bwd(H=0) == S["KDA_ERR_BAD_SHAPE"]
    assert bwd(N=2) == S["KDA_ERR_BAD_SHAPE"]              # N != B without cu_seqlens
    assert bwd(d_out=0) == S["KDA_ERR_NULL_ARG"]
    assert bwd(dbeta=0) == S["KDA_ERR_NULL_ARG"]
    assert bwd(dq=A + 0x600004) == S["KDA_ERR_MISALIGNED"]
    assert bwd(dbeta=A + 0xA00002) == S["KDA_ERR_MISALIGNED"]
    assert bwd(dk=A) == S["KDA_ERR_ALIAS"]                  # output over q
    assert bwd(dv=A + 0x600000) == S["KDA_ERR_ALIAS"]       # two outputs overlap
    assert bwd(d_initial_state=A + 0x500000) == S["KDA_ERR_ALIAS"]   # over d_out


def test_backward_workspace_bytes(lib):
    # chunked (default): per chunk-head a record, a list entry (rounded up in
    # all), (I + A)^-1 in fp32 and two bf16 states
    REC, ST2 = 17408 + 1280, 2 * 32768

    def lst(items):
        return -(-(items * 4) // 256) * 256

    ch = 512 * 64
    assert K.kda_backward_workspace_bytes(1, 8192, 64, 1, 0) == 256 + ch * REC + lst(ch) + ch * ST2
    pc = (8192 + 15 * 16) // 16
    assert K.kda_backward_workspace_bytes(1, 8192, 64, 16, 1) == (256 + 256 + pc * 64 * REC
                                                                 + lst(pc * 64) + pc * 64 * ST2)
    assert K.kda_backward_workspace_bytes(1, 8192, 64, 2, 0) == 0   # N != B
    # token-serial
    assert K.kda_set_backward_impl(1) == 0
    try:
        _token_serial_workspace_bytes()
    finally:
        K.kda_set_backward_impl(0)
    assert K.kda_set_backward_impl(2) != 0


def _token_serial_workspace_bytes():
    st, mib = 65536, 1 << 20
    assert K.kda_backward_workspace_bytes(1, 8192, 64, 1, 0) == 256 + 512 * 64 * st + 64 * mib
    assert K.kda_backward_workspace_bytes(2, 17, 3, 2, 0) == 256 + 2 * 2 * 3 * st + 6 * mib
    pc = (8192 + 15 * 16) // 16                       # packed: chunk bound, offsets table
    assert K.kda_backward_workspace_bytes(1, 8192, 64, 16, 1) == (256 + 256 + pc * 64 * st
                                                                 + 16 * 64 * mib)
    # more (sequence, head) pairs than the persistent kernel has CTAs: 1024 rings
    assert K.kda_backward_workspace_bytes(32, 16, 64, 32, 0) == 256 + 32 * 64 * st + 1024 * mib
    assert K.kda_backward_workspace_bytes(1, 8192, 64, 2, 0) == 0   # N != B
    assert K.kda_backward_workspace_bytes(1, 100, 0, 1, 0) == 0     # H < 1


def test_header_is_plain_c(tmp_path):
    """include/kda.h compiles as strict C99 (no C++ or torch types leak into
    the boundary), and a C caller can take every entry point's address."""
    import shutil
    import subprocess
    if shutil.which("gcc") is None:
        pytest.skip("gcc not found")
    names = declared_symbols()
    src = tmp_path / "use_kda.c"
    src.write_text('#include "kda.h"\n'
                   "typedef void (*fp)(void);\n"
                   "fp table[] = {\n" + "".join(f"    (fp){n},\n" for n in names) + "};\n")
    inc = os.path.join(ROOT, "include")
    r = subprocess.run(["gcc", "-std=c99", "-pedantic", "-Wall", "-Wextra", "-Werror",
                        "-I", inc, "-c", str(src), "-o", str(tmp_path / "use_kda.o")],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr


def test_noalloc_scratch_limit_boundary(lib):
    """The allocation-free entry point holds a 256 B flag block, every chunk
    record (17,408 B per 16-token chunk per head) and a 4 B list entry per
    chunk-head (rounded up to 256 B) in its fixed 64 MiB array. 3854 chunks
    of one head fit (67,106,304 B), 3855 do not (67,123,712 B). The size
    check comes before any CUDA call, so this needs no GPU: a call that fits
    goes on to the device checks, which fail here (no device) or, on a GPU,
    refuse the fake pointers, and nothing is launched either way."""
    def need(c):
        return 256 + c * 17408 + -(-(4 * c) // 256) * 256
    assert need(3854) <= (64 << 20) < need(3855)

    def na(T):
        return K.kda_chunk_prefill_noalloc(A, A + (8 << 20), A + (16 << 20), A + (24 << 20),
                                           A + (48 << 20), 0, 0, 1, T, 1, 128, 128, 1, 1.0,
                                           A + (64 << 20), 0, 0)
    assert na(3855 * 16) == K.STATUS_CODE["KDA_ERR_SCRATCH_LIMIT"]
    assert na(3854 * 16 + 1) == K.STATUS_CODE["KDA_ERR_SCRATCH_LIMIT"]
    assert na(3854 * 16) in (K.STATUS_CODE["KDA_ERR_CUDA"],
                             K.STATUS_CODE["KDA_ERR_NOT_DEVICE_MEMORY"],
                             K.STATUS_CODE["KDA_ERR_NO_DEVICE_SUPPORT"])
