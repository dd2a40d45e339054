"""fp8 (E4M3) KV cache on the GPU, through the C ABI: the bulk quantizer and
the quantizing appends against the oracle's E4M3 quantizer bit for bit
(every code and scale), and attention over the fp8 cache (kvd_decode_ex with
kvd_cache.fp8) against the oracle's attention over the rows read back.
Shapes cover the head dimensions and groups from MHA to MQA, ragged and empty
sequences, contiguous and paged caches, one and several query tokens; rows
past each sequence's end hold NaN codes and scales, so any over-read fails."""
import numpy as np
import pytest

import oracle
import workloads
from gpu_helpers import assert_close, bf16_tensor_bits, cuda_or_skip, to_dev_bf16
from workloads import bf16_bits_to_f32

pytestmark = pytest.mark.gpu

NAN8 = 0x7F  # an E4M3 NaN code

CASES = [
    # name, B, Hq, Hkv, D, S, lengths lo..hi, seed
    ("gqa4", 9, 32, 8, 128, 900, 0, 900, 121),
    ("mha64", 5, 6, 6, 64, 400, 1, 400, 122),
    ("g8d256", 4, 16, 2, 256, 300, 1, 300, 123),
    ("mqa48", 4, 48, 1, 256, 700, 1, 700, 124),
    ("g64d128", 3, 64, 1, 128, 500, 1, 500, 126),
    ("g24d128kv3", 3, 72, 3, 128, 400, 0, 400, 127),
]


def _gpu_fp8(inp, dev, n_cached):
    """Codes and scales of rows t < n_cached[b] from the GPU quantizer; other
    rows hold NaN codes and NaN scales."""
    import torch
    import kv_cache_decode_gb300 as kvd
    B, S, Hkv, D = inp.k_cache.shape
    cached = torch.from_numpy(n_cached.astype(np.int32)).to(dev)
    res = []
    for c in (inp.k_cache, inp.v_cache):
        codes = torch.full((B, S, Hkv, D), NAN8, dtype=torch.uint8, device=dev)
        scales = torch.full((B, S, Hkv), float("nan"), dtype=torch.float32, device=dev)
        kvd.kv_quantize_fp8(to_dev_bf16(c, dev), codes, scales, cached, S)
        res += [codes, scales]
    return res  # kc, ks, vc, vs


def _oracle_fp8(inp, n_cached):
    B, S, Hkv, D = inp.k_cache.shape
    out = []
    for c in (inp.k_cache, inp.v_cache):
        codes = np.full((B, S, Hkv, D), NAN8, np.uint8)
        scales = np.full((B, S, Hkv), np.nan, np.float32)
        for b in range(B):
            n = int(n_cached[b])
            if n:
                codes[b, :n], scales[b, :n] = oracle.quantize_fp8(c[b, :n])
        out += [codes, scales]
    return out


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_fp8_quantize_matches_oracle(case):
    import torch
    dev = cuda_or_skip()
    name, B, Hq, Hkv, D, S, lo, hi, seed = case
    inp = workloads.step_inputs(workloads.Workload(name, B, Hq, Hkv, D, S, lo, hi, seed))
    n_cached = np.maximum(inp.seq_lens - 1, 0)
    got = [x.cpu().numpy() for x in _gpu_fp8(inp, dev, n_cached)]
    torch.cuda.synchronize()
    want = _oracle_fp8(inp, n_cached)
    for g, w, what in zip(got, want, ("k codes", "k scales", "v codes", "v scales")):
        assert np.array_equal(g.view(np.uint8), w.view(np.uint8)), what


def _step(inp, dev, out_dtype, n_split, paged_page=0, codes_dtype=None):
    """The fp8 step through kvd_decode_ex (append included); returns
    (out f64, lse, status, host cache after the step: kc, ks, vc, vs)."""
    import torch
    import kv_cache_decode_gb300 as kvd
    n_cached = np.maximum(inp.seq_lens - 1, 0)
    kc, ks, vc, vs = _gpu_fp8(inp, dev, n_cached)
    B, Hq, D = inp.q.shape
    S = inp.k_cache.shape[1]
    q, kn, vn = (to_dev_bf16(x, dev) for x in (inp.q, inp.k_new, inp.v_new))
    pos = torch.from_numpy(inp.pos).to(dev)
    lens = torch.from_numpy(inp.seq_lens).to(dev)
    tdt = torch.bfloat16 if out_dtype == "bf16" else torch.float32
    out = torch.full(inp.q.shape, float("nan"), dtype=tdt, device=dev)
    lse = torch.full((B, Hq), float("nan"), dtype=torch.float32, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    ws = kvd.alloc_workspace(q, inp.k_cache, S, n_split, out_dtype)
    kw = dict(k_new=kn, v_new=vn, pos=pos, workspace=ws, n_split=n_split, lse=lse, status=status)
    if codes_dtype is not None:
        kc, vc = kc.view(codes_dtype), vc.view(codes_dtype)
    if paged_page:
        pin = workloads.paged_step_inputs(inp, paged_page, seed=paged_page)
        table, P, npg = pin.block_table, paged_page, pin.k_pages.shape[0]

        def pool(x, fill):
            h = x.cpu().numpy()
            p = np.full((npg, P) + h.shape[2:], fill, dtype=h.dtype)
            for b in range(table.shape[0]):
                for j in range(table.shape[1]):
                    if table[b, j] >= 0:
                        blk = h[b, j * P:(j + 1) * P]
                        p[table[b, j], :blk.shape[0]] = blk
            return torch.from_numpy(p).to(dev)
        kc, vc = pool(kc.view(torch.uint8), NAN8), pool(vc.view(torch.uint8), NAN8)
        ks, vs = pool(ks, np.nan), pool(vs, np.nan)
        kvd.decode_ex(q, kc, vc, lens, S, inp.workload.scale, out, k_scales=ks, v_scales=vs,
                      block_table=torch.from_numpy(table).to(dev), **kw)
    else:
        kvd.decode_ex(q, kc, vc, lens, S, inp.workload.scale, out, k_scales=ks, v_scales=vs, **kw)
    torch.cuda.synchronize()
    o = bf16_bits_to_f32(bf16_tensor_bits(out)) if out_dtype == "bf16" else out.cpu().numpy()
    return (o.astype(np.float64), lse.cpu().numpy(), int(status.item()),
            [x.view(torch.uint8).cpu().numpy() if x.dtype != torch.float32 else x.cpu().numpy()
             for x in (kc, ks, vc, vs)])


def _oracle_step(inp):
    n_cached = np.maximum(inp.seq_lens - 1, 0)
    kc, ks, vc, vs = _oracle_fp8(inp, n_cached)
    kc, vc, ks, vs, _ = oracle.kv_append_q8(kc, vc, ks, vs, inp.k_new, inp.v_new, inp.pos, fmt="fp8")
    out, lse = oracle.decode_attention_q8(inp.q, kc, vc, ks, vs, inp.seq_lens, inp.workload.scale, fmt="fp8")
    return out, lse, (kc, ks, vc, vs)


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
@pytest.mark.parametrize("out_dtype", ["bf16", "f32"])
def test_fp8_step_matches_oracle(case, out_dtype):
    dev = cuda_or_skip()
    name, B, Hq, Hkv, D, S, lo, hi, seed = case
    inp = workloads.step_inputs(workloads.Workload(name, B, Hq, Hkv, D, S, lo, hi, seed))
    want, want_lse, wcache = _oracle_step(inp)
    for n_split in (0, 7):
        o, l, status, gcache = _step(inp, dev, out_dtype, n_split)
        assert status == 0
        for b in range(B):
            n = int(inp.seq_lens[b])
            for g, w in zip(gcache, wcache):
                assert np.array_equal(g[b, :n].view(np.uint8), w[b, :n].view(np.uint8)), "appended rows"
        assert_close(o, want, out_dtype, f"{name} fp8 n_split {n_split}")
        finite = np.isfinite(want_lse)
        assert np.max(np.abs(l[finite] - want_lse[finite]), initial=0.0) < (4e-3 if out_dtype == "bf16" else 1e-4)
        assert np.all(np.isneginf(l[~finite]))


@pytest.mark.parametrize("case", [CASES[0], CASES[3]], ids=["gqa4", "mqa48"])
@pytest.mark.parametrize("page", [16, 64])
def test_fp8_paged_equals_contiguous(case, page):
    dev = cuda_or_skip()
    name, B, Hq, Hkv, D, S, lo, hi, seed = case
    inp = workloads.step_inputs(workloads.Workload(name, B, Hq, Hkv, D, S, lo, hi, seed))
    o1, l1, s1, _ = _step(inp, dev, "f32", 5)
    o2, l2, s2, _ = _step(inp, dev, "f32", 5, paged_page=page)
    assert s1 == s2 == 0
    assert np.array_equal(o1, o2) and np.array_equal(l1.view(np.uint32), l2.view(np.uint32))


def test_fp8_codes_as_float8_tensors():
    """Codes held in torch float8_e4m3fn tensors (the same bits) give the same step."""
    import torch
    dev = cuda_or_skip()
    name, B, Hq, Hkv, D, S, lo, hi, seed = CASES[0]
    inp = workloads.step_inputs(workloads.Workload(name, B, Hq, Hkv, D, S, lo, hi, seed))
    a = _step(inp, dev, "f32", 0)
    b = _step(inp, dev, "f32", 0, codes_dtype=torch.float8_e4m3fn)
    assert np.array_equal(a[0], b[0]) and a[2] == b[2] == 0


def test_fp8_multi_token_matches_oracle():
    import torch
    import kv_cache_decode_gb300 as kvd
    dev = cuda_or_skip()
    T = 3
    w = workloads.Workload("fm", 5, 48, 1, 256, 600, T, 600, 125)
    mi = workloads.multi_step_inputs(w, T)
    B, _, Hq, D = mi.q.shape
    S, Hkv = mi.k_cache.shape[1], mi.k_cache.shape[2]
    cached = np.maximum(mi.seq_lens - T, 0).astype(np.int32)
    codes, scales = [], []
    for c in (mi.k_cache, mi.v_cache):
        cd = torch.full((B, S, Hkv, D), NAN8, dtype=torch.uint8, device=dev)
        sc = torch.full((B, S, Hkv), float("nan"), dtype=torch.float32, device=dev)
        kvd.kv_quantize_fp8(to_dev_bf16(c, dev), cd, sc, torch.from_numpy(cached).to(dev), S)
        codes.append(cd)
        scales.append(sc)
    q, kn, vn = (to_dev_bf16(x, dev) for x in (mi.q, mi.k_new, mi.v_new))
    out = torch.full(mi.q.shape, float("nan"), dtype=torch.float32, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    _, nbytes = kvd.decode_plan_multi(B, T, Hq, Hkv, D, S, 0, 0, "f32")
    ws = torch.empty(max(nbytes, 1), dtype=torch.uint8, device=dev)
    kvd.decode_ex(q, codes[0], codes[1], torch.from_numpy(mi.seq_lens).to(dev), S, w.scale, out,
                  k_scales=scales[0], v_scales=scales[1], k_new=kn, v_new=vn, pos=torch.from_numpy(mi.pos).to(dev),
                  workspace=ws, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    kc = np.full((B, S, Hkv, D), NAN8, np.uint8)
    vc = np.full((B, S, Hkv, D), NAN8, np.uint8)
    ks = np.full((B, S, Hkv), np.nan, np.float32)
    vs = np.full((B, S, Hkv), np.nan, np.float32)
    for b in range(B):
        n = int(cached[b])
        if n:
            kc[b, :n], ks[b, :n] = oracle.quantize_fp8(mi.k_cache[b, :n])
            vc[b, :n], vs[b, :n] = oracle.quantize_fp8(mi.v_cache[b, :n])
    for i in range(T):
        kc, vc, ks, vs, _ = oracle.kv_append_q8(kc, vc, ks, vs, mi.k_new[:, i], mi.v_new[:, i], mi.pos + i, fmt="fp8")
    ok = np.isfinite(ks)
    kd = oracle.dequantize_fp8(np.where(ok[..., None], kc, 0), np.where(ok, ks, 0))
    vd = oracle.dequantize_fp8(np.where(ok[..., None], vc, 0), np.where(ok, vs, 0))
    got = out.cpu().numpy().astype(np.float64)
    for i in range(T):
        Li = np.clip(mi.seq_lens - T + 1 + i, 0, None).astype(np.int32)
        want, _ = oracle.decode_attention_f64kv(mi.q[:, i], kd, vd, Li, w.scale)
        assert_close(got[:, i], want, "f32", f"fp8 multi token {i}")


def test_fp8_paged_append_edges():
    """kvd_kv_append_fp8_paged: rows at page boundaries, past the capacity and
    into an entry that names no page, against the oracle byte for byte."""
    import torch
    import kv_cache_decode_gb300 as kvd
    dev = cuda_or_skip()
    P = 16
    w = workloads.Workload("app8f", 6, 8, 2, 128, 64, 1, 64, 126)
    inp = workloads.step_inputs(w, lens=np.array([16, 17, 32, 1, 64, 40], np.int32))
    pin = workloads.paged_step_inputs(inp, P, seed=7)
    table = pin.block_table.copy()
    pos = inp.pos.copy()
    pos[4] = 64
    table[5, 39 // P] = pin.k_pages.shape[0] + 5
    num_pages = pin.k_pages.shape[0]
    r = np.random.default_rng(127)
    host = [r.integers(0, 256, (num_pages, P, 2, 128), dtype=np.uint8) for _ in range(2)]
    host += [r.random((num_pages, P, 2), dtype=np.float32) for _ in range(2)]
    pools = [torch.from_numpy(h.copy()).to(dev) for h in host]
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    kvd.kv_append_fp8_paged(pools[0], pools[1], pools[2], pools[3], to_dev_bf16(inp.k_new, dev),
                            to_dev_bf16(inp.v_new, dev), torch.from_numpy(table).to(dev),
                            torch.from_numpy(pos).to(dev), status=status)
    torch.cuda.synchronize()
    want = oracle.kv_append_q8_paged(host[0], host[1], host[2], host[3], inp.k_new, inp.v_new, table, pos, fmt="fp8")
    assert want[4] == 2 and want[5] == 1
    for g, x, what in zip(pools, want[:4], ("k codes", "v codes", "k scales", "v scales")):
        assert np.array_equal(g.cpu().numpy().view(np.uint8), x.view(np.uint8)), what
    assert int(status.item()) == (0x2 | 0x8)
