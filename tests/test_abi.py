"""The C-ABI library loads, exports every symbol include/moex.h declares, and
rejects bad arguments on the host before touching the GPU (CPU-only)."""
import ctypes
import os
import re

import pytest

from helpers import ROOT, ensure_lib

HEADER = os.path.join(ROOT, "include", "moex.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(moex_\w+)\s*\(", text)))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for n in ["moex_quantize_q8_1", "moex_qgemv", "moex_moe_decode", "moex_weight_pack", "moex_route_topk",
              "moex_device_status"]:
        assert n in names


def test_library_exports_every_declared_symbol():
    L = ensure_lib()
    missing = [n for n in declared_functions() if not hasattr(L, n)]
    assert not missing, missing


def test_binding_covers_every_declared_symbol():
    import moe_expert_gb300 as mx
    assert set(declared_functions()) <= set(mx.SIGNATURES)


def test_status_strings_and_version():
    L = ensure_lib()
    assert L.moex_version() == 1
    assert L.moex_status_string(0) == b"ok"
    assert L.moex_status_string(7) == b"workspace too small"


def test_plane_bytes():
    import moe_expert_gb300 as mx
    L = ensure_lib()
    q, s = ctypes.c_size_t(), ctypes.c_size_t()
    assert L.moex_weight_plane_bytes(1, 1, 8192, 2560, ctypes.byref(q), ctypes.byref(s)) == 0
    assert (q.value, s.value) == (8192 * 2560, 8192 * 160)
    assert L.moex_weight_plane_bytes(2, 128, 2560, 1536, ctypes.byref(q), ctypes.byref(s)) == 0
    assert (q.value, s.value) == (128 * 2560 * 768, 128 * 2560 * 96)
    # K = 96: 3 scales = 6 bytes, padded to 16
    assert L.moex_weight_plane_bytes(1, 1, 4, 96, ctypes.byref(q), ctypes.byref(s)) == 0
    assert s.value == 4 * 16
    assert L.moex_weight_plane_bytes(1, 1, 4, 100, ctypes.byref(q), ctypes.byref(s)) == 1   # K % 32
    assert L.moex_weight_plane_bytes(9, 1, 4, 96, ctypes.byref(q), ctypes.byref(s)) == 3    # bad fmt


def test_host_validation_rejects_before_launch():
    import moe_expert_gb300 as mx
    L = ensure_lib()
    null = ctypes.c_void_p(0)
    buf = ctypes.create_string_buffer(4096 + 16)
    base = (ctypes.addressof(buf) + 15) // 16 * 16
    p = ctypes.c_void_p(base)
    # null pointers
    assert L.moex_quantize_q8_1(null, 64, 1, 64, p, p, null) == 1
    assert L.moex_qgemv(None, p, p, 1, p, 8, null) == 1
    # K not a multiple of 32, ncols out of range
    assert L.moex_quantize_q8_1(p, 48, 1, 48, p, p, null) == 1
    assert L.moex_quantize_q8_1(p, 64, 0, 64, p, p, null) == 1
    assert L.moex_quantize_q8_1(p, 64, 65, 64, p, p, null) == 1
    # misaligned activation pointer
    assert L.moex_quantize_q8_1(ctypes.c_void_p(base + 4), 64, 1, 64, p, p, null) == 2
    w = mx.QWeight(1, 1, 8, 64, base, base)
    assert L.moex_qgemv(ctypes.byref(w), p, p, 1, p, 4, null) == 1          # ldy < rows
    w_bad = mx.QWeight(1, 1, 8, 64, base + 8, base)
    assert L.moex_qgemv(ctypes.byref(w_bad), p, p, 1, p, 8, null) == 2      # misaligned plane
    w_fmt = mx.QWeight(5, 1, 8, 64, base, base)
    assert L.moex_qgemv(ctypes.byref(w_fmt), p, p, 1, p, 8, null) == 3
    # routing
    assert L.moex_route_topk(p, 4, 8, 9, p, p, null) == 1                   # k > E
    assert L.moex_route_topk(p, 4, 2048, 8, p, p, null) == 1                # E too large


def test_decode_validation_and_workspace():
    import moe_expert_gb300 as mx
    L = ensure_lib()
    null = ctypes.c_void_p(0)
    buf = ctypes.create_string_buffer(4096 + 16)
    base = (ctypes.addressof(buf) + 15) // 16 * 16
    p = ctypes.c_void_p(base)
    need = L.moex_moe_decode_workspace_bytes(3, 8, 2560, 1536)
    assert need >= 24 * 1536 + 24 * 48 * 8
    gu = mx.QWeight(1, 128, 3072, 2560, base, base)
    dn = mx.QWeight(2, 128, 2560, 1536, base, base)
    assert L.moex_moe_decode(ctypes.byref(gu), ctypes.byref(dn), p, 3, p, p, 8, p, p, need - 1, null) == 7
    assert L.moex_moe_decode(ctypes.byref(gu), ctypes.byref(dn), p, 9, p, p, 8, p, p, 1 << 30, null) == 1
    dn_bad = mx.QWeight(2, 128, 2560, 1024, base, base)                    # inter mismatch
    assert L.moex_moe_decode(ctypes.byref(gu), ctypes.byref(dn_bad), p, 3, p, p, 8, p, p, 1 << 30, null) == 1
    gu_iq = mx.QWeight(2, 128, 3072, 2560, base, base)                     # gate/up must be Q8_0
    assert L.moex_moe_decode(ctypes.byref(gu_iq), ctypes.byref(dn), p, 3, p, p, 8, p, p, 1 << 30, null) == 3


def test_prefill_and_dense_validation():
    """The prefill entry points reject bad arguments on the host, in the
    order their checks run, before anything is enqueued."""
    import moe_expert_gb300 as mx
    L = ensure_lib()
    null = ctypes.c_void_p(0)
    buf = ctypes.create_string_buffer(4096 + 16)
    base = (ctypes.addressof(buf) + 15) // 16 * 16
    p = ctypes.c_void_p(base)
    odd = ctypes.c_void_p(base + 4)
    E, H, I, T, k = 4, 256, 128, 8, 2
    gu = mx.QWeight(2, E, 2 * I, H, base, base)
    dn = mx.QWeight(2, E, H, I, base, base)
    need = L.moex_moe_prefill_workspace_bytes(T, k, E, H, I)
    assert need > 0
    assert L.moex_moe_prefill_workspace_bytes(0, k, E, H, I) == 0
    big = 1 << 40

    def pf(g=gu, d=dn, x=p, t=T, kk=k, out=p, ws=p, nbytes=big):
        return L.moex_moe_prefill(ctypes.byref(g), ctypes.byref(d), x, t, p, p, kk, out, ws, nbytes, null)

    assert pf(x=null) == 1
    assert pf(t=0) == 1
    assert pf(kk=17) == 1
    assert pf(d=mx.QWeight(2, E + 1, H, I, base, base)) == 1            # expert counts differ
    assert pf(d=mx.QWeight(2, E, H, 2 * I, base, base)) == 1            # down K != inter
    assert pf(g=mx.QWeight(2, E, 2 * I, 96, base, base),
              d=mx.QWeight(2, E, 96, I, base, base)) == 3               # hidden not a multiple of 128
    assert pf(nbytes=need - 1) == 7
    assert pf(x=odd) == 2
    assert pf(out=odd) == 2
    assert L.moex_moe_prefill_residual(ctypes.byref(gu), ctypes.byref(dn), p, T, p, p, k, null, p, p, big,
                                       null) == 1
    assert L.moex_moe_prefill_residual(ctypes.byref(gu), ctypes.byref(dn), p, T, p, p, k, odd, p, p, big,
                                       null) == 2

    W = mx.QWeight(2, 1, 256, 128, base, base)
    dneed = L.moex_dense_prefill_workspace_bytes(T, 256, 128)
    assert dneed > 0 and L.moex_dense_prefill_workspace_bytes(T, 64, 128) == 0

    def dp(w=W, x=p, y=p, ldy=256, ws=p, nbytes=big):
        return L.moex_dense_prefill(ctypes.byref(w), x, T, y, ldy, ws, nbytes, null)

    assert dp(w=mx.QWeight(2, 2, 256, 128, base, base)) == 3          # one matrix only
    assert dp(y=null) == 1
    assert dp(ldy=255) == 1
    assert dp(w=mx.QWeight(2, 1, 192, 128, base, base), ldy=192) == 3  # rows not a multiple of 128
    assert dp(w=mx.QWeight(2, 1, 256, 96, base, base)) == 3           # K not a multiple of 64
    assert dp(nbytes=dneed - 1) == 7
    assert dp(x=odd) == 2


def test_prefill_q8_validation():
    """The integer-route prefill rejects bad arguments on the host, in the
    order its checks run, before anything is enqueued."""
    import moe_expert_gb300 as mx
    L = ensure_lib()
    null = ctypes.c_void_p(0)
    buf = ctypes.create_string_buffer(4096 + 16)
    base = (ctypes.addressof(buf) + 15) // 16 * 16
    p = ctypes.c_void_p(base)
    odd = ctypes.c_void_p(base + 4)
    E, H, I, T, k = 4, 256, 128, 8, 2
    gu = mx.QWeight(2, E, 2 * I, H, base, base)
    dn = mx.QWeight(2, E, H, I, base, base)
    need = L.moex_moe_prefill_q8_workspace_bytes(T, k, E, H, I)
    assert need > 0 and L.moex_moe_prefill_q8_workspace_bytes(T, k, E, H, 32) == 0
    off = mx.moe_prefill_q8_workspace_layout(T, k, E, H, I)
    assert off[9] == need and all(off[i] <= off[i + 1] and off[i] % 256 == 0 for i in range(9))
    assert off[8] - off[7] >= T * k * I and off[9] - off[8] >= 8 * T * k * (I // 32)
    big = 1 << 40

    def pf(g=gu, d=dn, x=p, t=T, kk=k, out=p, ws=p, nbytes=big, h=None):
        if h is None:
            return L.moex_moe_prefill_q8(ctypes.byref(g), ctypes.byref(d), x, t, p, p, kk, out, ws, nbytes, null)
        return L.moex_moe_prefill_q8_debug(ctypes.byref(g), ctypes.byref(d), x, t, p, p, kk, out, ws, nbytes, h,
                                           null)

    assert pf(x=null) == 1
    assert pf(t=0) == 1
    assert pf(kk=17) == 1
    assert pf(d=mx.QWeight(2, E + 1, H, I, base, base)) == 1            # expert counts differ
    assert pf(d=mx.QWeight(2, E, H, 2 * I, base, base)) == 1            # down K != inter
    assert pf(g=mx.QWeight(2, E, 2 * I, 96, base, base),
              d=mx.QWeight(2, E, 96, I, base, base)) == 3               # hidden not a multiple of 128
    assert pf(nbytes=need - 1) == 7
    assert pf(x=odd) == 2
    assert pf(out=odd) == 2
    assert pf(h=odd) == 2                                               # H output misaligned


def test_decode_residual_validation():
    import moe_expert_gb300 as mx
    L = ensure_lib()
    null = ctypes.c_void_p(0)
    buf = ctypes.create_string_buffer(4096 + 16)
    base = (ctypes.addressof(buf) + 15) // 16 * 16
    p = ctypes.c_void_p(base)
    gu = mx.QWeight(1, 16, 512, 256, base, base)
    dn = mx.QWeight(2, 16, 256, 256, base, base)
    big = 1 << 30
    assert L.moex_moe_decode_residual(ctypes.byref(gu), ctypes.byref(dn), p, 2, p, p, 4, null, p, p, big, null) == 1
    assert L.moex_moe_decode_residual(ctypes.byref(gu), ctypes.byref(dn), p, 2, p, p, 4, ctypes.c_void_p(base + 8),
                                      p, p, big, null) == 2
