"""The C-ABI library without a GPU: it loads, exports every symbol the
header declares, validates arguments before touching CUDA, and its ring
schedule is bit-exact against the oracle's visit list."""
import ctypes
import os
import re

import pytest

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "ring_attn.h")


@pytest.fixture(scope="module")
def lib():
    from long_context_exact_ring_gb300 import build
    build.build()
    from long_context_exact_ring_gb300 import load_library
    return load_library()


def _declared():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[a-z_0-9]+\s*\*?\s*([a-z_0-9]+)\s*\(",
                                 text, flags=re.M)))


def test_header_declares_the_boundary():
    names = _declared()
    for want in ("ring_attn_fwd", "ring_attn_bwd", "attn_merge_partials", "ring_attn_schedule",
                 "ring_attn_check_status", "ring_attn_status_string",
                 "ring_attn_bwd_workspace_size"):
        assert want in names


def test_library_exports_every_declared_symbol(lib):
    for name in _declared():
        assert hasattr(lib, name), name


def test_binding_names_match_header():
    from long_context_exact_ring_gb300 import EXPORTED
    assert sorted(EXPORTED) == sorted(n for n in _declared() if n in EXPORTED)
    assert set(EXPORTED) <= set(_declared())


@pytest.mark.parametrize("P", [1, 2, 3, 4, 5, 8, 16, 33])
@pytest.mark.parametrize("causal", [0, 1])
def test_schedule_bit_exact_against_oracle(lib, P, causal):
    for i in range(P):
        n = lib.ring_attn_schedule(P, causal, i, None, None, 0)
        js = (ctypes.c_int * max(n, 1))()
        ks = (ctypes.c_int * max(n, 1))()
        assert lib.ring_attn_schedule(P, causal, i, js, ks, n) == n
        want = [(j, kind) for _, j, kind in oracle.ring_visits(P, bool(causal), i)
                if kind != oracle.KIND_SKIP]
        assert [(js[t], ks[t]) for t in range(n)] == want


def test_schedule_rejects_bad_arguments(lib):
    js = (ctypes.c_int * 4)()
    ks = (ctypes.c_int * 4)()
    assert lib.ring_attn_schedule(0, 0, 0, js, ks, 4) == -1
    assert lib.ring_attn_schedule(4, 0, 4, js, ks, 4) == -1
    assert lib.ring_attn_schedule(4, 0, -1, js, ks, 4) == -1
    assert lib.ring_attn_schedule(4, 2, 0, js, ks, 4) == -1
    assert lib.ring_attn_schedule(8, 0, 0, js, ks, 4) == -1      # cap too small


def test_status_strings(lib):
    for code, name in ((0, b"RA_OK"), (-1, b"RA_ERR_INVALID_ARG"), (-2, b"RA_ERR_UNSUPPORTED"),
                       (-3, b"RA_ERR_CUDA"), (-4, b"RA_ERR_DEVICE_TIMEOUT")):
        assert lib.ring_attn_status_string(code) == name


FAKE = 1 << 20    # a 16-byte aligned non-null value; never dereferenced below


def _fwd(lib, B=1, H=1, S=256, d=128, P=4, causal=1, scale=0.1, ptr=FAKE, lse=FAKE):
    return lib.ring_attn_fwd(ptr, ptr, ptr, ptr, lse, B, H, S, d, P, causal, scale, None)


def test_fwd_validates_before_any_launch(lib):
    assert _fwd(lib, S=250, P=4) == -1                 # unequal split
    assert _fwd(lib, P=0) == -1
    assert _fwd(lib, B=-1) == -1
    assert _fwd(lib, causal=2) == -1
    assert _fwd(lib, scale=float("nan")) == -1
    assert _fwd(lib, scale=float("inf")) == -1
    assert _fwd(lib, d=96) == -2                       # unsupported head dim
    assert _fwd(lib, d=256) == -2
    assert _fwd(lib, ptr=FAKE + 8) == -1               # misaligned
    assert _fwd(lib, ptr=0) == -1                      # null
    assert _fwd(lib, lse=FAKE + 2) == -1
    # empty shapes are a no-op and touch nothing
    assert _fwd(lib, B=0, ptr=0, lse=0) == 0
    assert _fwd(lib, S=0, ptr=0, lse=0) == 0


def test_bwd_validates_before_any_launch(lib):
    ws = lib.ring_attn_bwd_workspace_size(1, 2, 1024, 128)
    assert ws == 1 * 2 * 1024 * 128 * 4 + 2 * 2 * 1024 * 4
    assert lib.ring_attn_bwd_workspace_size(0, 2, 1024, 128) == 0

    def call(S=1024, P=4, d=128, ws_ptr=FAKE, ws_bytes=ws, ptr=FAKE):
        return lib.ring_attn_bwd(ptr, ptr, ptr, ptr, ptr, ptr, ptr, ptr, ptr, 1, 2, S, d, P, 1,
                                 0.1, ws_ptr, ws_bytes, None)
    assert call(S=1000, P=3) == -1
    assert call(d=80) == -2
    assert call(ws_bytes=ws - 1) == -1
    assert call(ws_ptr=FAKE + 16) == -1                # workspace must be 256-byte aligned
    assert call(ws_ptr=0) == -1
    assert call(ptr=FAKE + 4) == -1


def test_gqa_validates_before_any_launch(lib):
    def fwd(H=4, Hkv=2, ptr=FAKE, S=256, P=4):
        return lib.ring_attn_fwd_gqa(ptr, ptr, ptr, ptr, ptr, 1, H, Hkv, S, 128, P, 1, 0.1, None)
    assert fwd(H=4, Hkv=3) == -1                       # H not a multiple of H_kv
    assert fwd(Hkv=0) == -1
    assert fwd(Hkv=-2) == -1
    assert fwd(S=250) == -1
    assert fwd(ptr=FAKE + 8) == -1
    assert fwd(H=0, Hkv=0, ptr=0) == 0                 # empty
    ws = lib.ring_attn_bwd_workspace_size(1, 4, 256, 128)
    assert lib.ring_attn_bwd_gqa(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1, 4, 3, 256,
                                 128, 4, 1, 0.1, FAKE, ws, None) == -1


def test_merge_validates_before_any_launch(lib):
    def call(a=FAKE, b=FAKE * 2, out=FAKE * 3, la=FAKE * 4, lb=FAKE * 5, lout=FAKE * 6, d=64):
        return lib.attn_merge_partials(a, la, b, lb, out, lout, 1, 2, 8, d, None)
    assert call(d=0) == -1
    assert call(a=FAKE + 4) == -1
    assert call(out=FAKE * 2) == -1                    # o_out may alias only o_a
    assert call(lout=FAKE * 5) == -1
    assert lib.attn_merge_partials(0, 0, 0, 0, 0, 0, 0, 2, 8, 64, None) == 0


def test_strided_entry_points_validate_layouts(lib):
    ll3 = ctypes.c_longlong * 3
    B, H, S, d = 1, 2, 256, 128
    bshd = ll3(S * H * d, d, H * d)

    def fwd(qs=None, os_=None, ptr=FAKE):
        return lib.ring_attn_fwd_strided(ptr, qs, ptr, bshd, ptr, bshd, ptr, os_, FAKE, B, H, H, S,
                                         d, 4, 1, ctypes.c_float(0.1), None)
    assert fwd(qs=ll3(S * H * d, d, H * d + 4)) == -1       # row stride not 16-byte aligned
    assert fwd(qs=ll3(S * H * d, -d, H * d)) == -1          # negative stride
    assert fwd(qs=ll3(S * H * d, 0, H * d)) == -1           # zero stride over 2 heads
    assert fwd(os_=ll3(S * H * d, d, 1 << 37)) == -1        # beyond the stride limit
    assert fwd(ptr=FAKE + 8, qs=bshd) == -1                 # misaligned pointer
    # empty shape: nothing is launched or read
    assert lib.ring_attn_fwd_strided(0, None, 0, None, 0, None, 0, None, 0, 0, H, H, S, d, 4, 1,
                                     ctypes.c_float(0.1), None) == 0
    ws = lib.ring_attn_bwd_workspace_size(B, H, S, d)

    def bwd(dks=None):
        return lib.ring_attn_bwd_strided(FAKE, bshd, FAKE, bshd, FAKE, bshd, FAKE, bshd, FAKE,
                                         FAKE, bshd, FAKE, bshd, FAKE, dks, FAKE, bshd, B, H, H, S,
                                         d, 4, 1, ctypes.c_float(0.1), FAKE, ws, None)
    assert bwd(dks=ll3(S * H * d, d, H * d + 2)) == -1
    assert bwd(dks=ll3(S * H * d, d, 0)) == -1


def test_f32_forward_validates_before_any_launch(lib):
    B, H, S, d = 1, 2, 256, 64
    ws = lib.ring_attn_fwd_f32_workspace_size(B, H, H, S, d)
    assert ws == 3 * B * H * S * d * 2
    assert lib.ring_attn_fwd_f32_workspace_size(B, 4, 2, S, d) == (4 + 2 * 2) * S * d * 2
    assert lib.ring_attn_fwd_f32_workspace_size(0, H, H, S, d) == 0

    def call(q=FAKE, k=FAKE * 2, v=FAKE * 3, o=FAKE * 4, ws_ptr=FAKE * 5, ws_bytes=ws, Hkv=H, S_=S):
        return lib.ring_attn_fwd_f32(q, k, v, o, FAKE * 6, B, H, Hkv, S_, d, 4, 0,
                                     ctypes.c_float(0.125), ws_ptr, ws_bytes, None)
    assert call(ws_bytes=ws - 1) == -1                  # workspace too small
    assert call(ws_ptr=FAKE * 5 + 16) == -1             # workspace not 256-byte aligned
    assert call(o=FAKE * 2) == -1                       # o may not alias k
    assert call(o=FAKE * 3) == -1                       # ... or v
    assert call(q=FAKE + 8) == -1                       # misaligned
    assert call(Hkv=3) == -1                            # H not a multiple of H_kv
    assert call(S_=250) == -1                           # unequal split
    assert call(S_=0, ws_ptr=0, ws_bytes=0) == 0        # empty: nothing launched


def test_ulysses_validates_before_any_launch(lib):
    B, H, S, d = 1, 8, 1024, 128
    ws = lib.ring_attn_fwd_ulysses_workspace_size(B, H, H, S, d)
    assert ws == 4 * B * H * S * d * 2 + B * H * S * 4
    assert lib.ring_attn_fwd_ulysses_workspace_size(B, H, 0, S, d) == 0

    def call(H_=H, Hkv=H, P=4, ws_bytes=ws, ws_ptr=FAKE * 5, q=FAKE):
        return lib.ring_attn_fwd_ulysses_emulated(q, FAKE * 2, FAKE * 3, FAKE * 4, FAKE * 6, B, H_,
                                                  Hkv, S, d, P, 1, ctypes.c_float(0.1), ws_ptr,
                                                  ws_bytes, None)
    assert call(H_=6, Hkv=6) == -2                      # 6 heads cannot split over 4 ranks
    assert call(Hkv=2) == -2                            # 2 key/value heads cannot feed 4 ranks
    assert call(Hkv=3) == -1                            # 8 query heads over 3 key/value heads
    assert call(ws_bytes=ws - 1) == -1
    assert call(ws_ptr=FAKE * 5 + 64) == -1             # workspace not 256-byte aligned
    assert call(q=FAKE + 8) == -1
    assert call(P=3) == -1                              # 1024 tokens do not split in 3


def test_trace_visits_validates_before_any_cuda_call(lib):
    # NULL with a capacity, a buffer without one, a negative capacity and a
    # misaligned buffer are refused before the device is touched
    assert lib.ring_attn_trace_visits(None, 16) == -1
    assert lib.ring_attn_trace_visits(ctypes.c_void_p(FAKE), 0) == -1
    assert lib.ring_attn_trace_visits(ctypes.c_void_p(FAKE), -8) == -1
    assert lib.ring_attn_trace_visits(ctypes.c_void_p(FAKE + 4), 64) == -1
