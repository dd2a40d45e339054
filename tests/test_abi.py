"""The C ABI on the CPU: the library loads, exports every declared symbol, plans
on the host, and rejects bad arguments with the documented status before any
launch.

Calls that pass fake (never dereferenced) device pointers are written so that
argument validation fails first; no call here reaches a CUDA launch.
"""
import ctypes
import os
import re

import numpy as np
import pytest

import kv_cache_decode_gb300 as kvd

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "kvdecode.h")


@pytest.fixture(scope="module")
def lib():
    from kv_cache_decode_gb300 import _build
    _build.build()
    return kvd.load()


def test_exports_every_declared_symbol(lib):
    text = open(HEADER).read()
    declared = set(re.findall(r"^\s*(?:kvd_status|const char\*|size_t)\s+(kvd_\w+)\s*\(", text, re.M))
    assert declared == set(kvd.EXPORTED)
    for name in declared:
        assert hasattr(lib, name), name
    assert kvd.version().startswith("kvdecode")


def test_status_strings(lib):
    for code in range(5):
        assert kvd.status_string(code)
    assert kvd.status_string(99) == "unknown status"


@pytest.mark.parametrize("shape,expect", [
    ((1, 8, 1, 128, 256), kvd.OK),
    ((0, 8, 1, 128, 256), kvd.OK),
    ((1, 8, 3, 128, 256), kvd.ERR_INVALID_ARG),    # group does not divide
    ((1, 8, 1, 96, 256), kvd.ERR_UNSUPPORTED),     # head_dim
    ((1, 130, 2, 128, 256), kvd.ERR_UNSUPPORTED),  # group 65 > 64
    ((1, 0, 1, 128, 256), kvd.ERR_INVALID_ARG),
    ((1, 8, 1, 128, -1), kvd.ERR_INVALID_ARG),
    ((-1, 8, 1, 128, 256), kvd.ERR_INVALID_ARG),
])
def test_plan_validation(lib, shape, expect):
    n = ctypes.c_int(0)
    ws = ctypes.c_size_t(0)
    rc = lib.kvd_decode_plan(*shape, 152, 0, 0, ctypes.byref(n), ctypes.byref(ws))
    assert rc == expect


def test_plan_null_outputs(lib):
    assert lib.kvd_decode_plan(1, 8, 1, 128, 256, 152, 0, 0, None, None) == kvd.ERR_INVALID_ARG


def test_plan_heuristic_and_workspace(lib):
    # One CTA per resident slot, capped by the work; workspace formula.
    for name, B, Hq, Hkv, D, L in [("palm", 64, 48, 1, 256, 2048), ("mha", 32, 40, 40, 128, 4096),
                                    ("gqa", 128, 32, 8, 128, 8192), ("long", 4, 48, 1, 256, 65536)]:
        info = kvd.kernel_info(Hq, Hkv, D)
        n, ws = kvd.decode_plan(B, Hq, Hkv, D, L, num_sms=152)
        assert n == 152 * info["ctas_per_sm"], name
        G, P = Hq // Hkv, B * Hkv
        slots = n + P - 1
        r = lambda x: (x + 255) // 256 * 256
        assert ws == r(slots * G * D * 4) + r(slots * G * 8), name
    # tiny: capped by work (256 tokens, two tiles per CTA minimum)
    info = kvd.kernel_info(8, 1, 128)
    n, ws = kvd.decode_plan(1, 8, 1, 128, 256, num_sms=152)
    assert n == 256 // (2 * info["tile_tokens"])
    assert kvd.decode_plan(1, 8, 1, 128, 256, num_sms=152, n_split=1) == (1, 0)
    assert kvd.decode_plan(2, 8, 1, 128, 256, num_sms=152, n_split=5)[0] == 5


def test_kernel_info_fits_smem(lib):
    for D in (64, 128, 256):
        for G in (1, 4, 8, 16, 17, 32, 48, 64):
            for dt in ("bf16", "f32"):
                info = kvd.kernel_info(G, 1, D, dt)
                assert info["smem_bytes"] <= 227 * 1024
                assert info["smem_bytes"] * info["ctas_per_sm"] <= 228 * 1024
                assert info["threads"] % 32 == 0


FAKE = 0x100000  # aligned, never dereferenced: every call below fails validation first


def _dec_args(**over):
    a = dict(q=FAKE, k=FAKE, v=FAKE, lens=FAKE, B=2, S=64, maxlen=64, Hq=8, Hkv=2, D=128,
             scale=0.088, n_split=4, ws=FAKE, ws_bytes=0, out=FAKE, dt=0, lse=None, status=None,
             stream=None)
    a.update(over)
    return [a[k] for k in ("q", "k", "v", "lens", "B", "S", "maxlen", "Hq", "Hkv", "D", "scale",
                           "n_split", "ws", "ws_bytes", "out", "dt", "lse", "status", "stream")]


@pytest.mark.parametrize("fn", ["kvd_decode_attention", "kvd_split_kv_chunk", "kvd_split_kv_merge"])
@pytest.mark.parametrize("over,expect", [
    (dict(q=None), kvd.ERR_INVALID_ARG),
    (dict(k=None), kvd.ERR_INVALID_ARG),
    (dict(v=None), kvd.ERR_INVALID_ARG),
    (dict(lens=None), kvd.ERR_INVALID_ARG),
    (dict(out=None), kvd.ERR_INVALID_ARG),
    (dict(q=FAKE + 8), kvd.ERR_INVALID_ARG),        # not 16-byte aligned
    (dict(k=FAKE + 2), kvd.ERR_INVALID_ARG),
    (dict(out=FAKE + 4), kvd.ERR_INVALID_ARG),
    (dict(lens=FAKE + 2), kvd.ERR_INVALID_ARG),
    (dict(B=-1), kvd.ERR_INVALID_ARG),
    (dict(S=0), kvd.ERR_INVALID_ARG),
    (dict(maxlen=65), kvd.ERR_INVALID_ARG),         # max_seq_len > s_max
    (dict(maxlen=-1), kvd.ERR_INVALID_ARG),
    (dict(Hq=7), kvd.ERR_INVALID_ARG),              # group does not divide
    (dict(D=100), kvd.ERR_UNSUPPORTED),
    (dict(Hq=130, Hkv=2), kvd.ERR_UNSUPPORTED),
    (dict(scale=float("nan")), kvd.ERR_INVALID_ARG),
    (dict(scale=float("inf")), kvd.ERR_INVALID_ARG),
    (dict(n_split=-2), kvd.ERR_INVALID_ARG),
    (dict(dt=7), kvd.ERR_INVALID_ARG),
    (dict(ws_bytes=16), kvd.ERR_WORKSPACE_TOO_SMALL),
    (dict(ws=None, ws_bytes=1 << 30), kvd.ERR_WORKSPACE_TOO_SMALL),
    (dict(ws=FAKE + 16, ws_bytes=1 << 30), kvd.ERR_INVALID_ARG),  # workspace not 256-aligned
])
def test_decode_rejects(lib, fn, over, expect):
    assert getattr(lib, fn)(*_dec_args(**over)) == expect


@pytest.mark.parametrize("args,expect", [
    ((None, FAKE, FAKE, FAKE, FAKE, 2, 8, 1, 128, None, None), kvd.ERR_INVALID_ARG),
    ((FAKE, FAKE, FAKE, FAKE + 8, FAKE, 2, 8, 1, 128, None, None), kvd.ERR_INVALID_ARG),
    ((FAKE, FAKE, FAKE, FAKE, None, 2, 8, 1, 128, None, None), kvd.ERR_INVALID_ARG),
    ((FAKE, FAKE, FAKE, FAKE, FAKE, 2, 8, 1, 100, None, None), kvd.ERR_INVALID_ARG),
    ((FAKE, FAKE, FAKE, FAKE, FAKE, -1, 8, 1, 128, None, None), kvd.ERR_INVALID_ARG),
    ((FAKE, FAKE, FAKE, FAKE, FAKE, 2, 8, 0, 128, None, None), kvd.ERR_INVALID_ARG),
    ((FAKE, FAKE, FAKE, FAKE, FAKE, 0, 8, 1, 128, None, None), kvd.OK),  # batch 0: no-op
])
def test_append_rejects(lib, args, expect):
    assert lib.kvd_kv_append(*args) == expect


def test_decode_batch_zero_is_noop(lib):
    assert lib.kvd_decode_attention(*_dec_args(B=0, n_split=3, ws=None)) == kvd.OK


def _step_args(kn=FAKE, vn=FAKE, pos=FAKE, **over):
    a = _dec_args(**over)
    # (k_cache, v_cache, k_new, v_new, pos, q, seq_lens) + the rest of kvd_decode_attention's
    return [a[1], a[2], kn, vn, pos, a[0], a[3]] + a[4:]


@pytest.mark.parametrize("over,expect", [
    (dict(q=None), kvd.ERR_INVALID_ARG),
    (dict(k=None), kvd.ERR_INVALID_ARG),
    (dict(lens=None), kvd.ERR_INVALID_ARG),
    (dict(out=FAKE + 4), kvd.ERR_INVALID_ARG),
    (dict(B=-1), kvd.ERR_INVALID_ARG),
    (dict(S=0), kvd.ERR_INVALID_ARG),
    (dict(maxlen=65), kvd.ERR_INVALID_ARG),
    (dict(Hq=7), kvd.ERR_INVALID_ARG),
    (dict(Hq=130, Hkv=2), kvd.ERR_UNSUPPORTED),
    (dict(scale=float("nan")), kvd.ERR_INVALID_ARG),
    (dict(ws_bytes=16), kvd.ERR_WORKSPACE_TOO_SMALL),
    (dict(kn=None), kvd.ERR_INVALID_ARG),
    (dict(vn=FAKE + 8), kvd.ERR_INVALID_ARG),
    (dict(pos=FAKE + 2), kvd.ERR_INVALID_ARG),
    (dict(pos=None), kvd.ERR_INVALID_ARG),
])
def test_decode_step_rejects(lib, over, expect):
    # Nothing is launched when either half's arguments are rejected (fake pointers).
    assert lib.kvd_decode_step(*_step_args(**over)) == expect


def test_decode_step_batch_zero_is_noop(lib):
    assert lib.kvd_decode_step(*_step_args(B=0, n_split=3, ws=None)) == kvd.OK


def _paged_args(bt=FAKE, B=2, max_blocks=4, page=16, num_pages=10, maxlen=64, **over):
    a = _dec_args(maxlen=maxlen, **over)
    # (q, k_pages, v_pages, block_table, seq_lens, batch, max_blocks, page_size, num_pages) + the rest
    return [a[0], a[1], a[2], bt, a[3], B, max_blocks, page, num_pages] + a[6:]


@pytest.mark.parametrize("over,expect", [
    (dict(), None),                                    # valid up to the launch (not made here)
    (dict(bt=None), kvd.ERR_INVALID_ARG),
    (dict(bt=FAKE + 2), kvd.ERR_INVALID_ARG),          # table not 4-byte aligned
    (dict(page=48), kvd.ERR_INVALID_ARG),              # not a power of two
    (dict(page=8), kvd.ERR_INVALID_ARG),               # below 16
    (dict(page=8192), kvd.ERR_INVALID_ARG),            # above 4096
    (dict(max_blocks=0), kvd.ERR_INVALID_ARG),
    (dict(num_pages=0), kvd.ERR_INVALID_ARG),
    (dict(num_pages=1 << 27, page=16), kvd.ERR_INVALID_ARG),   # pool rows reach 2^31
    (dict(maxlen=65), kvd.ERR_INVALID_ARG),            # above max_blocks * page_size
    (dict(q=None), kvd.ERR_INVALID_ARG),
    (dict(Hq=7), kvd.ERR_INVALID_ARG),
    (dict(ws_bytes=16), kvd.ERR_WORKSPACE_TOO_SMALL),
])
def test_decode_paged_rejects(lib, over, expect):
    if expect is None:
        return  # the valid case would launch; the GPU tests cover it
    assert lib.kvd_decode_attention_paged(*_paged_args(**over)) == expect
    a = _paged_args(**over)
    # step: (k_pages, v_pages, k_new, v_new, pos, q, block_table, seq_lens, batch, ...)
    step = [a[1], a[2], FAKE, FAKE, FAKE, a[0], a[3], a[4]] + a[5:]
    assert lib.kvd_decode_step_paged(*step) == expect


def test_decode_paged_batch_zero_is_noop(lib):
    assert lib.kvd_decode_attention_paged(*_paged_args(B=0, n_split=3, ws=None)) == kvd.OK


@pytest.mark.parametrize("args,expect", [
    ((None, FAKE, FAKE, FAKE, FAKE, FAKE, 2, 4, 16, 10, 1, 128, None, None), kvd.ERR_INVALID_ARG),
    ((FAKE, FAKE, FAKE, FAKE, None, FAKE, 2, 4, 16, 10, 1, 128, None, None), kvd.ERR_INVALID_ARG),
    ((FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 2, 4, 24, 10, 1, 128, None, None), kvd.ERR_INVALID_ARG),
    ((FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 2, 0, 16, 10, 1, 128, None, None), kvd.ERR_INVALID_ARG),
    ((FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 2, 4, 16, 0, 1, 128, None, None), kvd.ERR_INVALID_ARG),
    ((FAKE, FAKE, FAKE, FAKE, FAKE, None, 2, 4, 16, 10, 1, 128, None, None), kvd.ERR_INVALID_ARG),
    ((FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 0, 4, 16, 10, 1, 128, None, None), kvd.OK),  # batch 0: no-op
])
def test_append_paged_rejects(lib, args, expect):
    assert lib.kvd_kv_append_paged(*args) == expect


@pytest.mark.parametrize("args,expect", [
    # (k_codes, v_codes, k_scales, v_scales, k_new, v_new, table, pos, B, max_blocks, page, num_pages, Hkv, D, status, stream)
    ((FAKE, FAKE, None, FAKE, FAKE, FAKE, FAKE, FAKE, 2, 4, 16, 10, 1, 128, None, None), kvd.ERR_INVALID_ARG),
    ((FAKE, FAKE, FAKE, FAKE + 2, FAKE, FAKE, FAKE, FAKE, 2, 4, 16, 10, 1, 128, None, None), kvd.ERR_INVALID_ARG),
    ((FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None, FAKE, 2, 4, 16, 10, 1, 128, None, None), kvd.ERR_INVALID_ARG),
    ((FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 2, 4, 24, 10, 1, 128, None, None), kvd.ERR_INVALID_ARG),
    ((FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 2, 4, 16, 10, 1, 96, None, None), kvd.ERR_UNSUPPORTED),
    ((FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 0, 4, 16, 10, 1, 128, None, None), kvd.OK),  # batch 0
])
def test_append_q8_paged_rejects(lib, args, expect):
    assert lib.kvd_kv_append_q8_paged(*args) == expect


def _q8_args(ks=FAKE, vs=FAKE, **over):
    a = _dec_args(**over)
    # (q, k_codes, v_codes, k_scales, v_scales, seq_lens, batch, ...) as kvd_decode_attention after the cache
    return [a[0], a[1], a[2], ks, vs] + a[3:]


@pytest.mark.parametrize("over,expect", [
    (dict(ks=None), kvd.ERR_INVALID_ARG),
    (dict(vs=FAKE + 2), kvd.ERR_INVALID_ARG),          # scales not 4-byte aligned
    (dict(Hq=130, Hkv=2), kvd.ERR_UNSUPPORTED),        # group 65 > KVD_MAX_GROUP
    (dict(D=96), kvd.ERR_UNSUPPORTED),
    (dict(q=None), kvd.ERR_INVALID_ARG),
    (dict(k=FAKE + 8), kvd.ERR_INVALID_ARG),
    (dict(ws_bytes=16), kvd.ERR_WORKSPACE_TOO_SMALL),
])
def test_decode_q8_rejects(lib, over, expect):
    assert lib.kvd_decode_attention_q8(*_q8_args(**over)) == expect
    a = _q8_args(**over)
    # step: (k_codes, v_codes, k_scales, v_scales, k_new, v_new, pos, q, seq_lens, batch, ...)
    step = [a[1], a[2], a[3], a[4], FAKE, FAKE, FAKE, a[0], a[5]] + a[6:]
    assert lib.kvd_decode_step_q8(*step) == expect


def test_decode_q8_batch_zero_is_noop(lib):
    assert lib.kvd_decode_attention_q8(*_q8_args(B=0, n_split=3, ws=None)) == kvd.OK


@pytest.mark.parametrize("args,expect", [
    ((None, FAKE, FAKE, FAKE, 2, 8, 8, 1, 128, None), kvd.ERR_INVALID_ARG),
    ((FAKE, FAKE, None, FAKE, 2, 8, 8, 1, 128, None), kvd.ERR_INVALID_ARG),
    ((FAKE, FAKE + 8, FAKE, FAKE, 2, 8, 8, 1, 128, None), kvd.ERR_INVALID_ARG),
    ((FAKE, FAKE, FAKE, FAKE, 2, 8, 9, 1, 128, None), kvd.ERR_INVALID_ARG),   # max_seq_len > s_max
    ((FAKE, FAKE, FAKE, FAKE, 2, 8, 8, 1, 96, None), kvd.ERR_UNSUPPORTED),
    ((FAKE, FAKE, FAKE, FAKE, 0, 8, 8, 1, 128, None), kvd.OK),               # batch 0: no-op
])
def test_quantize_q8_rejects(lib, args, expect):
    assert lib.kvd_kv_quantize_q8(*args) == expect


@pytest.mark.parametrize("args,expect", [
    ((FAKE, FAKE, None, FAKE, FAKE, FAKE, FAKE, 2, 8, 1, 128, None, None), kvd.ERR_INVALID_ARG),
    ((FAKE, FAKE, FAKE, FAKE + 2, FAKE, FAKE, FAKE, 2, 8, 1, 128, None, None), kvd.ERR_INVALID_ARG),
    ((FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None, 2, 8, 1, 128, None, None), kvd.ERR_INVALID_ARG),
    ((FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 2, 8, 1, 96, None, None), kvd.ERR_UNSUPPORTED),
    ((FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 0, 8, 1, 128, None, None), kvd.OK),
])
def test_append_q8_rejects(lib, args, expect):
    assert lib.kvd_kv_append_q8(*args) == expect


@pytest.mark.parametrize("T,Hq,Hkv,expect", [
    (0, 8, 2, kvd.ERR_INVALID_ARG),
    (4, 8, 2, kvd.OK),          # T * G = 16: one block of rows
    (5, 8, 2, kvd.OK),          # T * G = 20: two blocks of rows
    (2, 48, 1, kvd.OK),         # MQA, T * G = 96: six blocks
    (64, 64, 1, kvd.OK),        # the largest: KVD_MAX_TOKENS x KVD_MAX_GROUP
    (65, 8, 2, kvd.ERR_UNSUPPORTED),  # T > KVD_MAX_TOKENS
    (2, 130, 2, kvd.ERR_UNSUPPORTED),  # group 65
    (1, 48, 1, kvd.OK),         # T = 1: any group, as the single-token plan
])
def test_plan_multi(lib, T, Hq, Hkv, expect):
    n = ctypes.c_int(0)
    ws = ctypes.c_size_t(0)
    assert lib.kvd_decode_plan_multi(2, T, Hq, Hkv, 128, 1000, 152, 0, 0, ctypes.byref(n), ctypes.byref(ws)) == expect
    if expect == kvd.OK and T > 1:
        n1, ws1 = kvd.decode_plan(2, Hq, Hkv, 128, 1000, 152)
        assert n.value == n1 and ws.value >= T * (ws1 - 512)


@pytest.mark.parametrize("T,over,expect", [
    (0, dict(), kvd.ERR_INVALID_ARG),
    (65, dict(), kvd.ERR_UNSUPPORTED),      # T > KVD_MAX_TOKENS
    (2, dict(q=None), kvd.ERR_INVALID_ARG),
    (2, dict(ws_bytes=16), kvd.ERR_WORKSPACE_TOO_SMALL),
])
def test_decode_multi_rejects(lib, T, over, expect):
    a = _dec_args(**over)
    assert lib.kvd_decode_attention_multi(*(a[:5] + [T] + a[5:])) == expect


@pytest.mark.parametrize("phi,over,expect", [
    (float("inf"), dict(), kvd.ERR_INVALID_ARG),
    (float("nan"), dict(), kvd.ERR_INVALID_ARG),
    (3e38, dict(), kvd.ERR_INVALID_ARG),              # phi * log2(e) overflows float
    (0.0, dict(q=None), kvd.ERR_INVALID_ARG),
    (0.0, dict(D=96), kvd.ERR_UNSUPPORTED),
    (0.0, dict(ws_bytes=16), kvd.ERR_WORKSPACE_TOO_SMALL),
])
def test_decode_umax_rejects(lib, phi, over, expect):
    a = _dec_args(**over)
    assert lib.kvd_decode_attention_umax(*(a[:11] + [phi] + a[11:])) == expect
    step = [a[1], a[2], FAKE, FAKE, FAKE, a[0], a[3]] + a[4:11] + [phi] + a[11:]
    assert lib.kvd_decode_step_umax(*step) == expect


def test_step_staging_bytes(lib):
    al = lambda x: -(-x // 256) * 256
    # q | k_new | v_new | pos | seq_lens, each 256-byte aligned
    assert lib.kvd_step_staging_bytes(3, 2, 8, 2, 128) == al(6 * 8 * 128 * 2) + 2 * al(6 * 2 * 128 * 2) + 2 * al(12)
    assert lib.kvd_step_staging_bytes(3, 0, 8, 2, 128) == 0


def _host_step_args(**over):
    a = dict(k=FAKE, v=FAKE, qh=FAKE, knh=FAKE, vnh=FAKE, posh=FAKE, lensh=FAKE, stg=FAKE, stg_bytes=1 << 20, B=2,
             T=1, S=64, maxlen=64, Hq=8, Hkv=2, D=128, scale=0.088, n_split=4, ws=FAKE, ws_bytes=1 << 20,
             out=FAKE, outh=FAKE, dt=0, lse=None, status=None, stream=None)
    a.update(over)
    return list(a.values())


@pytest.mark.parametrize("over,expect", [
    (dict(qh=None), kvd.ERR_INVALID_ARG),
    (dict(lensh=None), kvd.ERR_INVALID_ARG),
    (dict(outh=None), kvd.ERR_INVALID_ARG),
    (dict(stg=None), kvd.ERR_INVALID_ARG),
    (dict(stg=FAKE + 16), kvd.ERR_INVALID_ARG),       # staging not 256-byte aligned
    (dict(stg_bytes=1024), kvd.ERR_INVALID_ARG),      # staging too small
    (dict(T=0), kvd.ERR_INVALID_ARG),
    (dict(D=96), kvd.ERR_UNSUPPORTED),
    (dict(k=None), kvd.ERR_INVALID_ARG),
    (dict(ws_bytes=16), kvd.ERR_WORKSPACE_TOO_SMALL),
    (dict(B=0), kvd.OK),                              # nothing to copy or launch
    (dict(out=None), kvd.ERR_INVALID_ARG),            # direct write needs pinned host memory
])
def test_decode_step_host_rejects(lib, over, expect):
    # every rejection comes before any copy is queued (the pointers are fake)
    assert lib.kvd_decode_step_host(*_host_step_args(**over)) == expect


@pytest.mark.parametrize("fn", ["kvd_kv_quantize_fp8", "kvd_kv_quantize_q8"])
@pytest.mark.parametrize("args,expect", [
    ((None, FAKE, FAKE, FAKE, 2, 8, 8, 1, 128, None), kvd.ERR_INVALID_ARG),
    ((FAKE, FAKE, FAKE, FAKE, 2, 8, 8, 1, 96, None), kvd.ERR_UNSUPPORTED),
    ((FAKE, FAKE + 8, FAKE, FAKE, 2, 8, 8, 1, 128, None), kvd.ERR_INVALID_ARG),
    ((FAKE, FAKE, FAKE, FAKE, 0, 8, 8, 1, 128, None), kvd.OK),
])
def test_quantize_8bit_rejects(lib, fn, args, expect):
    assert getattr(lib, fn)(*args) == expect


@pytest.mark.parametrize("args,expect", [
    ((FAKE, FAKE, None, FAKE, FAKE, FAKE, FAKE, 2, 8, 1, 128, None, None), kvd.ERR_INVALID_ARG),
    ((FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 2, 8, 1, 96, None, None), kvd.ERR_UNSUPPORTED),
    ((FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 0, 8, 1, 128, None, None), kvd.OK),
])
def test_append_fp8_rejects(lib, args, expect):
    assert lib.kvd_kv_append_fp8(*args) == expect


def test_append_fp8_paged_rejects(lib):
    ok = (FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 0, 4, 16, 10, 1, 128, None, None)
    assert lib.kvd_kv_append_fp8_paged(*ok) == kvd.OK
    bad_page = ok[:10] + (24,) + ok[11:]
    assert lib.kvd_kv_append_fp8_paged(*bad_page) == kvd.ERR_INVALID_ARG


@pytest.mark.parametrize("args,expect", [
    # (outs, lses, n_shards, rows, head_dim, in_dtype, out, out_dtype, lse_out, stream)
    ((None, FAKE, 2, 10, 128, 1, FAKE, 0, None, None), kvd.ERR_INVALID_ARG),
    ((FAKE, FAKE, 0, 10, 128, 1, FAKE, 0, None, None), kvd.ERR_INVALID_ARG),     # no shard
    ((FAKE, FAKE, 2, -1, 128, 1, FAKE, 0, None, None), kvd.ERR_INVALID_ARG),
    ((FAKE, FAKE, 2, 10, 96, 1, FAKE, 0, None, None), kvd.ERR_UNSUPPORTED),
    ((FAKE + 8, FAKE, 2, 10, 128, 1, FAKE, 0, None, None), kvd.ERR_INVALID_ARG),  # outs not 16-byte aligned
    ((FAKE, FAKE, 2, 10, 128, 7, FAKE, 0, None, None), kvd.ERR_INVALID_ARG),      # bad dtype
    ((FAKE, FAKE, 2, 0, 128, 1, FAKE, 0, None, None), kvd.OK),                    # no rows: no-op
    # written ranges overlapping read ones (in place), or each other; outs
    # [2, 10, 128] fp32 is 10240 bytes, out [10, 128] bf16 2560
    ((FAKE, FAKE + (1 << 24), 2, 10, 128, 1, FAKE, 0, None, None), kvd.ERR_INVALID_ARG),         # out = outs[0]
    ((FAKE, FAKE + (1 << 24), 2, 10, 128, 1, FAKE + 5120, 0, None, None), kvd.ERR_INVALID_ARG),  # out = outs[1]
    ((FAKE, FAKE + (1 << 24), 2, 10, 128, 1, FAKE + (2 << 24), 0, FAKE + (1 << 24), None),
     kvd.ERR_INVALID_ARG),                                                                       # lse_out = lses[0]
    ((FAKE, FAKE + (1 << 24), 2, 10, 128, 1, FAKE + (2 << 24), 0, FAKE + (2 << 24) + 2048, None),
     kvd.ERR_INVALID_ARG),                                                                       # lse_out inside out
])
def test_merge_attention_rejects(lib, args, expect):
    assert lib.kvd_merge_attention(*args) == expect


def test_decode_ex_rejects(lib):
    c = kvd._CCache(k=FAKE, v=FAKE, s_max=64)
    a = _dec_args()  # q, k, v, lens, B, S, maxlen, Hq, Hkv, D, scale, n_split, ws, ws_bytes, out, dt, lse, status, stream
    def call(cache, kn=None, vn=None, pos=None, T=1, **over):
        b = _dec_args(**over)
        return lib.kvd_decode_ex(cache, b[0], b[3], b[4], T, b[6], b[7], b[8], b[9], b[10], b[11], b[12], b[13],
                                 b[14], b[15], b[16], kn, vn, pos, b[17], b[18])
    assert call(None) == kvd.ERR_INVALID_ARG
    assert call(ctypes.byref(c), kn=FAKE) == kvd.ERR_INVALID_ARG            # only part of the append
    cq = kvd._CCache(k=FAKE, v=FAKE, k_scales=FAKE, s_max=64)
    assert call(ctypes.byref(cq)) == kvd.ERR_INVALID_ARG                    # one scale array only
    cf = kvd._CCache(k=FAKE, v=FAKE, s_max=64, fp8=1)
    assert call(ctypes.byref(cf)) == kvd.ERR_INVALID_ARG                    # fp8 codes without scales
    cpq = kvd._CCache(k=FAKE, v=FAKE, k_scales=FAKE, v_scales=FAKE, block_table=FAKE, max_blocks=4,
                      page_size=16, num_pages=10)
    # paged int8 passes every check up to the workspace (none given here)
    assert call(ctypes.byref(cpq)) == kvd.ERR_WORKSPACE_TOO_SMALL
    cpq2 = kvd._CCache(k=FAKE, v=FAKE, k_scales=FAKE, v_scales=FAKE + 2, block_table=FAKE, max_blocks=4,
                       page_size=16, num_pages=10)
    assert call(ctypes.byref(cpq2)) == kvd.ERR_INVALID_ARG                   # scales not 4-byte aligned
    cp = kvd._CCache(k=FAKE, v=FAKE, block_table=FAKE, max_blocks=4, page_size=24, num_pages=10)
    assert call(ctypes.byref(cp)) == kvd.ERR_INVALID_ARG                     # page size not a power of two
    assert call(ctypes.byref(c), T=65) == kvd.ERR_UNSUPPORTED                # T > KVD_MAX_TOKENS
    assert call(ctypes.byref(c), B=0, ws=None, n_split=3) == kvd.OK          # batch 0: no-op


@pytest.mark.parametrize("args,expect", [
    # (src, bytes, ctas, sink, status_word, stream)
    ((None, 1 << 20, 0, None, None, None), kvd.ERR_INVALID_ARG),
    ((FAKE + 8, 1 << 20, 0, None, None, None), kvd.ERR_INVALID_ARG),    # src not 16-byte aligned
    ((FAKE, 1 << 20, -1, None, None, None), kvd.ERR_INVALID_ARG),
    ((FAKE, 1 << 20, 0, FAKE + 4, None, None), kvd.ERR_INVALID_ARG),    # sink not 8-byte aligned
    ((FAKE, 15, 0, None, None, None), kvd.OK),                          # under 16 bytes: nothing to read
])
def test_probe_read_rejects(lib, args, expect):
    assert lib.kvd_probe_read(*args) == expect
