"""The C ABI without a GPU: the library builds and loads, exports every function
include/mg_attn.h declares, and rejects bad arguments on the host before any
CUDA call (the fake pointers below are never dereferenced)."""
import ctypes
import os
import re

import pytest

import attention_forward_backward_gb300 as mg
from attention_forward_backward_gb300 import build as mgbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "mg_attn.h")


@pytest.fixture(scope="module")
def lib():
    mgbuild.build()
    return mg.load_library()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"\b(mg_[a-z0-9_]+)\s*\(", text)
    return sorted(set(names))


def test_header_declares_the_abi():
    names = declared_functions()
    for n in ("mg_attn_fwd", "mg_attn_bwd", "mg_attn_bwd_workspace_bytes", "mg_status_string",
              "mg_get_device_error"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    raw = ctypes.CDLL(mg.LIB_PATH)
    for name in declared_functions():
        assert hasattr(raw, name), name


# Fake, 16-byte aligned, distinct, non-overlapping "device" addresses.
BASE = 1 << 40
STEP = 1 << 36


def P(i):
    return BASE + i * STEP


def fwd(lib, Q=P(0), K=P(1), V=P(2), O=P(3), LSE=P(4), B=1, H=2, L=64, D=64, causal=1,
        scale=0.125, contract=0):
    return lib.mg_attn_fwd(Q, K, V, O, LSE, B, H, L, D, causal, scale, contract, None)


def bwd(lib, Q=P(0), K=P(1), V=P(2), O=P(3), dO=P(4), LSE=P(5), dQ=P(6), dK=P(7), dV=P(8),
        B=1, H=2, L=64, D=64, causal=1, scale=0.125, contract=0, ws=P(9), ws_bytes=1 << 20):
    return lib.mg_attn_bwd(Q, K, V, O, dO, LSE, dQ, dK, dV, B, H, L, D, causal, scale, contract,
                           ws, ws_bytes, None)


@pytest.mark.parametrize("kw,code", [
    (dict(Q=None), mg.MG_ERR_INVALID_ARG),
    (dict(O=None), mg.MG_ERR_INVALID_ARG),
    (dict(LSE=None), mg.MG_ERR_INVALID_ARG),
    (dict(K=P(1) + 4), mg.MG_ERR_INVALID_ARG),      # misaligned
    (dict(B=0), mg.MG_ERR_INVALID_ARG),
    (dict(H=-1), mg.MG_ERR_INVALID_ARG),
    (dict(L=0), mg.MG_ERR_INVALID_ARG),
    (dict(L=(1 << 20) + 1), mg.MG_ERR_INVALID_ARG),
    (dict(D=48), mg.MG_ERR_UNSUPPORTED),
    (dict(D=256), mg.MG_ERR_UNSUPPORTED),
    (dict(causal=2), mg.MG_ERR_INVALID_ARG),
    (dict(scale=0.0), mg.MG_ERR_INVALID_ARG),
    (dict(scale=-1.0), mg.MG_ERR_INVALID_ARG),
    (dict(scale=float("nan")), mg.MG_ERR_INVALID_ARG),
    (dict(scale=float("inf")), mg.MG_ERR_INVALID_ARG),
    (dict(contract=3), mg.MG_ERR_INVALID_ARG),
    (dict(contract=0x400 | 1), mg.MG_ERR_INVALID_ARG),  # unknown flag
    (dict(contract=0x100), mg.MG_ERR_UNSUPPORTED),      # 16-bit outputs under STRICT_F32
    (dict(contract=0x200), mg.MG_ERR_UNSUPPORTED),      # hi/lo dS split under STRICT_F32
    (dict(O=P(0)), mg.MG_ERR_INVALID_ARG),          # output aliases Q
    (dict(LSE=P(3) + 1024), mg.MG_ERR_INVALID_ARG),  # LSE inside O
])
def test_fwd_rejects(lib, kw, code):
    assert fwd(lib, **kw) == code


@pytest.mark.parametrize("kw,code", [
    (dict(dO=None), mg.MG_ERR_INVALID_ARG),
    (dict(dV=P(8) + 8), mg.MG_ERR_INVALID_ARG),
    (dict(D=16), mg.MG_ERR_UNSUPPORTED),
    (dict(ws=None), mg.MG_ERR_WORKSPACE),
    (dict(ws_bytes=16), mg.MG_ERR_WORKSPACE),
    (dict(ws=P(9) + 4), mg.MG_ERR_WORKSPACE),
    (dict(dQ=P(0)), mg.MG_ERR_INVALID_ARG),          # dQ aliases Q
    (dict(dK=P(6)), mg.MG_ERR_INVALID_ARG),          # dK aliases dQ
    (dict(ws=P(8)), mg.MG_ERR_INVALID_ARG),          # workspace aliases dV
    (dict(contract=1, ws=P(4)), mg.MG_ERR_INVALID_ARG),  # workspace aliases dO
    (dict(contract=0x200), mg.MG_ERR_UNSUPPORTED),      # hi/lo dS split under STRICT_F32
    (dict(contract=0x200 | 0x100 | 3), mg.MG_ERR_INVALID_ARG),  # no such base contract
])
def test_bwd_rejects(lib, kw, code):
    assert bwd(lib, **kw) == code


def test_workspace_bytes(lib):
    for contract in (0, 1):
        n = lib.mg_attn_bwd_workspace_bytes(2, 32, 8192, 128, contract)
        assert n >= 2 * 32 * 8192 * 4 and n % 256 == 0
        assert lib.mg_attn_bwd_workspace_bytes(1, 1, 1, 32, contract) == 256
    assert lib.mg_attn_bwd_workspace_bytes(1, 1, 1, 48, 0) == 0
    assert lib.mg_attn_bwd_workspace_bytes(0, 1, 1, 64, 0) == 0
    assert lib.mg_attn_bwd_workspace_bytes(1, 1, 1, 64, 5) == 0


def test_status_strings(lib):
    for code in range(6):
        s = lib.mg_status_string(code).decode()
        assert s.startswith("MG_")
    assert lib.mg_status_string(99).decode() == "unknown mg_status_t"


def test_kernel_names(lib):
    n = lib.mg_attn_kernel_count()
    names = [lib.mg_attn_kernel_name(i).decode() for i in range(n)]
    assert len(set(names)) == n and "accel_dkdv_dq" in names and "strict_fwd" in names
    assert lib.mg_attn_kernel_name(n).decode() == "unknown"


def test_binding_raises_on_error(lib):
    class FakeT:
        def __init__(self, p, shape):
            self.p, self.shape = p, shape

        def dim(self):
            return len(self.shape)

        def data_ptr(self):
            return self.p

    q = FakeT(P(0), (1, 2, 8, 48))
    with pytest.raises(mg.MgError) as ei:
        mg.mg_attn_fwd(q, FakeT(P(1), q.shape), FakeT(P(2), q.shape), FakeT(P(3), q.shape),
                       FakeT(P(4), q.shape[:3]), True, 0.1, "strict", stream=0)
    assert ei.value.status == mg.MG_ERR_UNSUPPORTED


# ---------------------------------------------------------------- cross attention (_ex calls)
def fwd_ex(lib, Q=P(0), K=P(1), V=P(2), O=P(3), LSE=P(4), B=1, H=2, Lq=64, Lk=96, D=64, mask=2,
           scale=0.125, contract=0):
    return lib.mg_attn_fwd_ex(Q, K, V, O, LSE, B, H, Lq, Lk, D, mask, scale, contract, None)


def bwd_ex(lib, Q=P(0), K=P(1), V=P(2), O=P(3), dO=P(4), LSE=P(5), dQ=P(6), dK=P(7), dV=P(8),
           B=1, H=2, Lq=64, Lk=96, D=64, mask=2, scale=0.125, contract=0, ws=P(9),
           ws_bytes=1 << 20):
    return lib.mg_attn_bwd_ex(Q, K, V, O, dO, LSE, dQ, dK, dV, B, H, Lq, Lk, D, mask, scale,
                              contract, ws, ws_bytes, None)


@pytest.mark.parametrize("kw,code", [
    (dict(mask=3), mg.MG_ERR_INVALID_ARG),
    (dict(mask=-1), mg.MG_ERR_INVALID_ARG),
    (dict(Lk=0), mg.MG_ERR_INVALID_ARG),
    (dict(Lq=0), mg.MG_ERR_INVALID_ARG),
    (dict(Lk=(1 << 20) + 1), mg.MG_ERR_INVALID_ARG),
    (dict(D=96), mg.MG_ERR_UNSUPPORTED),
    (dict(V=P(1) + 8), mg.MG_ERR_INVALID_ARG),       # misaligned
    (dict(O=P(2)), mg.MG_ERR_INVALID_ARG),           # O aliases V
])
def test_fwd_ex_rejects(lib, kw, code):
    assert fwd_ex(lib, **kw) == code


@pytest.mark.parametrize("kw,code", [
    (dict(mask=7), mg.MG_ERR_INVALID_ARG),
    (dict(Lk=0), mg.MG_ERR_INVALID_ARG),
    (dict(ws_bytes=64 * 4 * 2 - 16), mg.MG_ERR_WORKSPACE),  # Dvec is [B][H][Lq]
    (dict(dK=P(1)), mg.MG_ERR_INVALID_ARG),          # dK aliases K
])
def test_bwd_ex_rejects(lib, kw, code):
    assert bwd_ex(lib, **kw) == code


def test_workspace_bytes_ex_follows_the_query_length(lib):
    for contract in (0, 1):
        assert lib.mg_attn_bwd_workspace_bytes_ex(2, 3, 1000, 7, 64, contract) == \
            lib.mg_attn_bwd_workspace_bytes(2, 3, 1000, 64, contract)
        assert lib.mg_attn_bwd_workspace_bytes_ex(2, 3, 7, 1000, 64, contract) == \
            lib.mg_attn_bwd_workspace_bytes(2, 3, 7, 64, contract)
        assert lib.mg_attn_bwd_workspace_bytes_ex(1, 1, 1, 0, 64, contract) == 0


# ---------------------------------------------------------------- decode forward
def fwd_decode(lib, Q=P(0), K=P(1), V=P(2), O=P(3), LSE=P(4), B=1, H=2, Lq=4, Lk=1000, D=64,
               mask=2, scale=0.125, contract=0, ws=P(5), ws_bytes=1 << 24):
    return lib.mg_attn_fwd_decode(Q, K, V, O, LSE, B, H, Lq, Lk, D, mask, scale, contract, ws,
                                  ws_bytes, None)


@pytest.mark.parametrize("kw,code", [
    (dict(Lq=9), mg.MG_ERR_UNSUPPORTED),             # more rows than the decode schedule takes
    (dict(Lq=0), mg.MG_ERR_INVALID_ARG),
    (dict(Lk=0), mg.MG_ERR_INVALID_ARG),
    (dict(D=48), mg.MG_ERR_UNSUPPORTED),
    (dict(mask=3), mg.MG_ERR_INVALID_ARG),
    (dict(scale=0.0), mg.MG_ERR_INVALID_ARG),
    (dict(contract=3), mg.MG_ERR_INVALID_ARG),
    (dict(contract=0x100 | 1), mg.MG_ERR_UNSUPPORTED),  # decode writes O in f32 only
    (dict(ws=None), mg.MG_ERR_WORKSPACE),
    (dict(ws=P(5) + 8), mg.MG_ERR_WORKSPACE),        # misaligned workspace
    (dict(ws_bytes=16), mg.MG_ERR_WORKSPACE),
    (dict(K=P(1) + 4), mg.MG_ERR_INVALID_ARG),       # misaligned
    (dict(O=P(0)), mg.MG_ERR_INVALID_ARG),           # O aliases Q
    (dict(ws=P(2)), mg.MG_ERR_INVALID_ARG),          # workspace aliases V
])
def test_fwd_decode_rejects(lib, kw, code):
    assert fwd_decode(lib, **kw) == code


def test_decode_workspace_bytes(lib):
    """One record of D + 4 floats per (head, key split, query row); the split
    count is at least one, at most one per 256 keys, and the size is a multiple
    of 256 bytes. Worked cases with 152 SMs (the count assumed without a GPU):
    STRICT_F32, B=1, H=8, Lk=32768 asks for ceil(1216 / 8) = 152 splits, capped
    at 32768 / 256 = 128 splits of 256 keys: 8 * 128 * 1 * 132 floats = 540,672
    bytes. B=1, H=8, Lk=100000 keeps 152 splits of ceil(100000 / 152) = 658 ->
    672 keys (whole 32-key tiles), which cover the keys in 149 splits:
    8 * 149 * 3 * 132 floats (Lq = 3) = 1,888,128 bytes, rounded up to 1,888,256.
    The 16-bit contracts (tensor-core partials, one CTA per SM) take the split
    count s minimising ceil(8 s / 152) * (256 + 32768 / s): s = 19 (one wave),
    19 splits of 1792 keys (whole 128-key tiles): 8 * 19 * 132 floats = 80,256
    bytes, rounded up to 80,384."""
    assert lib.mg_attn_fwd_decode_workspace_bytes(1, 8, 1, 32768, 128, 0) == 540672
    assert lib.mg_attn_fwd_decode_workspace_bytes(1, 8, 1, 32768, 128, 1) == 80384
    assert lib.mg_attn_fwd_decode_workspace_bytes(1, 8, 1, 32768, 128, 2) == 80384
    assert lib.mg_attn_fwd_decode_workspace_bytes(1, 8, 3, 100000, 128, 0) == 1888256
    for (B, H, Lq, Lk, D) in [(1, 1, 1, 1, 32), (2, 3, 8, 5000, 64), (4, 32, 3, 100000, 128),
                              (64, 64, 1, 4096, 128)]:
        for contract in (0, 1):
            n = lib.mg_attn_fwd_decode_workspace_bytes(B, H, Lq, Lk, D, contract)
            rec = B * H * Lq * (D + 4) * 4
            assert n % 256 == 0 and rec <= n < rec * max(1, -(-Lk // 256)) + 256, (B, H, Lq, Lk)
    assert lib.mg_attn_fwd_decode_workspace_bytes(1, 1, 9, 100, 64, 0) == 0
    assert lib.mg_attn_fwd_decode_workspace_bytes(1, 1, 1, 0, 64, 0) == 0
    assert lib.mg_attn_fwd_decode_workspace_bytes(1, 1, 1, 100, 96, 0) == 0


# ---------------------------------------------------------------- key padding (_padded calls)
def fwd_pad(lib, Q=P(0), K=P(1), V=P(2), O=P(3), LSE=P(4), kv=P(10), B=2, H=2, Lq=64, Lk=96,
            D=64, mask=1, scale=0.125, contract=1):
    return lib.mg_attn_fwd_padded(Q, K, V, O, LSE, kv, B, H, Lq, Lk, D, mask, scale, contract,
                                  None)


def bwd_pad(lib, Q=P(0), K=P(1), V=P(2), O=P(3), dO=P(4), LSE=P(5), dQ=P(6), dK=P(7), dV=P(8),
            kv=P(10), B=2, H=2, Lq=64, Lk=96, D=64, mask=1, scale=0.125, contract=1, ws=P(9),
            ws_bytes=1 << 20):
    return lib.mg_attn_bwd_padded(Q, K, V, O, dO, LSE, dQ, dK, dV, kv, B, H, Lq, Lk, D, mask,
                                  scale, contract, ws, ws_bytes, None)


@pytest.mark.parametrize("kw,code", [
    (dict(kv=P(10) + 2), mg.MG_ERR_INVALID_ARG),    # lengths not 4-byte aligned
    (dict(O=P(10)), mg.MG_ERR_INVALID_ARG),         # O overlaps the lengths
    (dict(mask=5), mg.MG_ERR_INVALID_ARG),
    (dict(D=48), mg.MG_ERR_UNSUPPORTED),
    (dict(Q=0), mg.MG_ERR_INVALID_ARG),
])
def test_fwd_padded_rejects(lib, kw, code):
    assert fwd_pad(lib, **kw) == code


@pytest.mark.parametrize("kw,code", [
    (dict(kv=P(10) + 1), mg.MG_ERR_INVALID_ARG),
    (dict(dV=P(10)), mg.MG_ERR_INVALID_ARG),        # dV overlaps the lengths
    (dict(ws=P(10)), mg.MG_ERR_INVALID_ARG),        # workspace overlaps the lengths
    (dict(ws_bytes=16), mg.MG_ERR_WORKSPACE),
    (dict(B=0), mg.MG_ERR_INVALID_ARG),
])
def test_bwd_padded_rejects(lib, kw, code):
    assert bwd_pad(lib, **kw) == code


def test_workspace_bytes_with_16_bit_outputs(lib):
    """MG_OUT_16 adds an f32 dQ accumulator [B][H][Lq][D] after Dvec, each part
    rounded up to 256 bytes: B=1, H=2, Lq=100, D=64 -> 1024 + 51200 bytes."""
    dvec = lib.mg_attn_bwd_workspace_bytes_ex(1, 2, 100, 70, 64, 1)
    assert dvec == 1024
    assert lib.mg_attn_bwd_workspace_bytes_ex(1, 2, 100, 70, 64, 0x100 | 1) == 1024 + 51200
    assert lib.mg_attn_bwd_workspace_bytes_ex(1, 2, 100, 70, 64, 0x100 | 2) == 1024 + 51200
    assert lib.mg_attn_bwd_workspace_bytes_ex(1, 2, 100, 70, 64, 0x100) == 0  # STRICT
    # the hi/lo dS policy needs no workspace of its own
    assert lib.mg_attn_bwd_workspace_bytes_ex(1, 2, 100, 70, 64, 0x200 | 1) == 1024
    assert lib.mg_attn_bwd_workspace_bytes_ex(1, 2, 100, 70, 64, 0x200 | 0x100 | 1) == 1024 + 51200


def test_16_bit_outputs_size_their_buffers(lib):
    """With 16-bit outputs O (and dQ, dK, dV) take 2 bytes per element: an LSE
    placed right after a 16-bit O is no overlap, one placed inside it is; in the
    backward a dK right after a 16-bit dQ likewise."""
    n = 1 * 2 * 64 * 64
    assert fwd(lib, O=P(3), LSE=P(3) + 2 * n, contract=0x100 | 1) != mg.MG_ERR_INVALID_ARG
    assert fwd(lib, O=P(3), LSE=P(3) + 2 * n - 16, contract=0x100 | 1) == mg.MG_ERR_INVALID_ARG
    assert fwd(lib, O=P(3), LSE=P(3) + 2 * n, contract=1) == mg.MG_ERR_INVALID_ARG  # f32 O
    assert bwd(lib, dQ=P(6), dK=P(6) + 2 * n, contract=0x100 | 1) != mg.MG_ERR_INVALID_ARG
    assert bwd(lib, dQ=P(6), dK=P(6) + 2 * n - 16, contract=0x100 | 1) == mg.MG_ERR_INVALID_ARG


def test_noalloc_rejects_16_bit_outputs(lib):
    import ctypes
    f = lib.mg_attn_bwd_noalloc
    vp, i, fl = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    f.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, fl, i, vp]
    f.restype = i
    args = [P(k) for k in range(9)]
    assert f(*args, 1, 2, 64, 64, 1, 0.125, 0x100 | 1, None) == mg.MG_ERR_UNSUPPORTED


# ---------------------------------------------------------------- convolution derivatives
def conv(lib, which, a=P(0), b=P(1), out=P(2), N=2, H=8, W=8, C=64, K=64, R=3, S=3, stride=1,
         pad=1, contract=1):
    fn = lib.mg_conv2d_grad_input if which == "dgrad" else lib.mg_conv2d_grad_weight
    return fn(a, b, out, N, H, W, C, K, R, S, stride, pad, contract, None)


@pytest.mark.parametrize("which", ["dgrad", "wgrad"])
@pytest.mark.parametrize("kw,code", [
    (dict(a=None), mg.MG_ERR_INVALID_ARG),
    (dict(out=None), mg.MG_ERR_INVALID_ARG),
    (dict(b=P(1) + 8), mg.MG_ERR_INVALID_ARG),           # misaligned
    (dict(out=P(0)), mg.MG_ERR_INVALID_ARG),             # output aliases an input
    (dict(out=P(1) + 1024), mg.MG_ERR_INVALID_ARG),      # output inside an input
    (dict(N=0), mg.MG_ERR_INVALID_ARG),
    (dict(C=-8), mg.MG_ERR_INVALID_ARG),
    (dict(R=11, pad=1), mg.MG_ERR_INVALID_ARG),          # kernel larger than the padded image
    (dict(pad=-1), mg.MG_ERR_INVALID_ARG),
    (dict(stride=0), mg.MG_ERR_INVALID_ARG),
    (dict(H=70000), mg.MG_ERR_INVALID_ARG),
    (dict(N=1 << 16, H=256, W=256, C=64), mg.MG_ERR_INVALID_ARG),  # X beyond 2^31 elements
    (dict(stride=3), mg.MG_ERR_UNSUPPORTED),
    (dict(C=12), mg.MG_ERR_UNSUPPORTED),                 # channels not in 16-byte rows
    (dict(K=20), mg.MG_ERR_UNSUPPORTED),
    (dict(contract=0), mg.MG_ERR_UNSUPPORTED),           # STRICT_F32: tensor cores only
    (dict(contract=0x100 | 1), mg.MG_ERR_UNSUPPORTED),   # no 16-bit outputs
    (dict(contract=3), mg.MG_ERR_INVALID_ARG),
    (dict(contract=0x400 | 1), mg.MG_ERR_INVALID_ARG),
])
def test_conv_rejects(lib, which, kw, code):
    assert conv(lib, which, **kw) == code
