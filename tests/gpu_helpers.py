"""Shared helpers for the GPU parity tests: run one decode step through the C
ABI and compare it with the CPU oracle."""
from __future__ import annotations

import json
import os

import numpy as np
import pytest

import kv_cache_decode_gb300 as kvd
import oracle
from workloads import StepInputs, bf16_bits_to_f32, f32_to_bf16_bits

GUARD = 256  # elements of canary on each side of every output buffer
CANARY_BF16 = 0x7F81  # a signalling-NaN bit pattern nobody writes
CANARY_F32 = -12345.678
WS_GUARD = 4096
WS_CANARY = 0xA5


def cuda_or_skip():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from kv_cache_decode_gb300 import _build
    _build.build()
    kvd.load()
    return torch.device("cuda:0")


def to_dev_bf16(bits: np.ndarray, dev):
    import torch
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(dev).view(torch.bfloat16)


def bf16_tensor_bits(t) -> np.ndarray:
    import torch
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def guarded(shape, dtype, dev):
    """A buffer with GUARD canary elements on each side; returns (full, view)."""
    import torch
    n = int(np.prod(shape))
    if dtype == torch.bfloat16:
        full = torch.full((n + 2 * GUARD,), CANARY_BF16, dtype=torch.int16, device=dev).view(torch.bfloat16)
    else:
        full = torch.full((n + 2 * GUARD,), CANARY_F32, dtype=dtype, device=dev)
    return full, full[GUARD:GUARD + n].view(*shape)


def guards_intact(full) -> bool:
    import torch
    if full.dtype == torch.bfloat16:
        g = full.view(torch.int16)
        ok = (g[:GUARD] == CANARY_BF16).all() and (g[-GUARD:] == CANARY_BF16).all()
    else:
        ok = (full[:GUARD] == CANARY_F32).all() and (full[-GUARD:] == CANARY_F32).all()
    return bool(ok)


class StepResult:
    pass


def run_step(inp: StepInputs, dev, out_dtype="bf16", n_split=0, max_seq_len=None,
             seq_lens_override=None, append=True, keep_cache=False):
    """Upload the pre-append cache, append the new token on the GPU, then run
    decode attention through the C ABI. Returns host copies of the results."""
    import torch
    w = inp.workload
    B, Hq, D = inp.q.shape
    S_max, Hkv = inp.k_cache.shape[1], inp.k_cache.shape[2]
    q = to_dev_bf16(inp.q, dev)
    kc = to_dev_bf16(inp.k_cache, dev)
    vc = to_dev_bf16(inp.v_cache, dev)
    kn = to_dev_bf16(inp.k_new, dev)
    vn = to_dev_bf16(inp.v_new, dev)
    pos = torch.from_numpy(inp.pos).to(dev)
    lens_np = inp.seq_lens if seq_lens_override is None else np.asarray(seq_lens_override, np.int32)
    lens = torch.from_numpy(lens_np).to(dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    if append:
        # A sequence of length 0 has no new token; its (zero) row goes to slot 0,
        # which attention never reads. The oracle side does the same.
        kvd.kv_append(kc, vc, kn, vn, pos)
    tdt = torch.bfloat16 if out_dtype == "bf16" else torch.float32
    out_full, out = guarded((B, Hq, D), tdt, dev)
    lse_full, lse = guarded((B, Hq), torch.float32, dev)
    mx = int(lens_np.max(initial=0)) if max_seq_len is None else max_seq_len
    mx = min(max(mx, 0), S_max)
    n_eff, ws_bytes = kvd.decode_plan(B, Hq, Hkv, D, mx, 0, n_split, out_dtype)
    ws_full = torch.full((ws_bytes + 2 * WS_GUARD,), WS_CANARY, dtype=torch.uint8, device=dev)
    ws = ws_full[WS_GUARD:WS_GUARD + ws_bytes] if ws_bytes else None
    kvd.decode_attention(q, kc, vc, lens, mx, w.scale, out, workspace=ws, n_split=n_split,
                         lse=lse, status=status)
    torch.cuda.synchronize()
    r = StepResult()
    r.n_split = n_eff
    r.out = (bf16_bits_to_f32(bf16_tensor_bits(out)) if out_dtype == "bf16"
             else out.cpu().numpy()).astype(np.float64)
    r.lse = lse.cpu().numpy().astype(np.float64)
    r.status = int(status.item())
    r.guards_ok = guards_intact(out_full) and guards_intact(lse_full)
    wsh = ws_full.cpu().numpy()
    r.ws_guards_ok = bool((wsh[:WS_GUARD] == WS_CANARY).all() and (wsh[-WS_GUARD:] == WS_CANARY).all())
    if keep_cache:
        r.k_cache = bf16_tensor_bits(kc)
        r.v_cache = bf16_tensor_bits(vc)
    return r


def oracle_step(inp: StepInputs, batch_rows=None, lens=None):
    """Oracle output for the post-append cache of the given batch rows."""
    rows = np.arange(inp.q.shape[0]) if batch_rows is None else np.asarray(batch_rows)
    L = inp.seq_lens[rows] if lens is None else np.asarray(lens, np.int32)[rows]
    kc = inp.k_cache[rows].copy()
    vc = inp.v_cache[rows].copy()
    kc, vc, _ = oracle.kv_append(kc, vc, inp.k_new[rows], inp.v_new[rows], inp.pos[rows])
    return oracle.decode_attention(inp.q[rows], kc, vc, L, inp.workload.scale)


def bf16_ulp(x: np.ndarray) -> np.ndarray:
    """Spacing of bf16 numbers at |x| (8 significant bits)."""
    ax = np.maximum(np.abs(x), np.finfo(np.float32).tiny)
    return np.exp2(np.floor(np.log2(ax)) - 7)


#: bf16 unit roundoff: a weight rounded to bf16 (round to nearest even) carries
#: a relative error of at most 2^-9.
BF16_U = 2.0 ** -9
#: Slack for the float32 parts of the kernels (scores, exponentials, sums),
#: the level the fp32-output mode is held to everywhere.
F32_SLACK = 1e-4

#: One record per assert_close call: what was compared and how many bf16
#: elements needed the rounding allowance above 1e-2.
PARITY_LOG = []


def weight_rounding_bound(spread: np.ndarray) -> np.ndarray:
    """Bound on what rounding the softmax weights to bf16 moves an output.

    With exact weights w_t and rounded ones w_t (1 + d_t), |d_t| <= u, the
    normalised output moves by sum_t (w'_t - w_t)(v_t - out), and
    |w'_t - w_t| <= w_t * 2u / (1 - u); so the move is at most
    2u / (1 - u) * sum_t w_t |v_t - out| = that factor times ``spread``."""
    return 2.0 * BF16_U / (1.0 - BF16_U) * spread


def assert_close(got: np.ndarray, ref: np.ndarray, out_dtype: str, what: str = "", spread=None):
    """Compare a GPU result with the oracle's.

    fp32 output: max-abs error 1e-4 everywhere.
    bf16 output: max-abs error 1e-2. An element above 1e-2 is accepted only
    if its error is within what the kernels' bf16 roundings can produce: half
    a bf16 step at its magnitude (the output's own rounding), plus the bound
    on the weights' rounding to bf16 (``weight_rounding_bound``), plus the
    fp32 slack. ``spread(flat_indices)`` gives sum_t w_t |v_t - ref| for those
    elements (exact weights); without it the weight term is taken as zero.
    The number of elements that needed the allowance and their largest |ref|
    are recorded (``PARITY_LOG``; also appended as JSON lines to the file
    named by KVD_PARITY_LOG, if set)."""
    assert got.shape == ref.shape
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    err = np.abs(got - ref)
    rec = {"what": what, "dtype": out_dtype, "n": int(err.size), "max_err": float(err.max(initial=0.0))}
    if out_dtype == "bf16":
        over = np.flatnonzero(err.ravel() > 1e-2)
        tol = np.full(err.shape, 1e-2)
        if over.size:
            r = ref.ravel()[over]
            mag = np.maximum(np.abs(r), np.abs(got.ravel()[over]))
            allow = 0.5 * bf16_ulp(mag) + F32_SLACK
            if spread is not None:
                allow = allow + weight_rounding_bound(np.asarray(spread(over), np.float64))
            tol.ravel()[over] = np.maximum(1e-2, allow)
        rec["n_over_1e-2"] = int(over.size)
        rec["max_abs_ref_over"] = float(np.abs(ref.ravel()[over]).max(initial=0.0))
    else:
        tol = np.full_like(ref, 1e-4)
        rec["n_over_1e-2"] = 0
    bad = err > tol
    rec["n_bad"] = int(bad.sum())
    PARITY_LOG.append(rec)
    path = os.environ.get("KVD_PARITY_LOG")
    if path:
        with open(path, "a") as f:
            f.write(json.dumps(rec) + "\n")
    if bad.any():
        i = np.unravel_index(np.argmax(err - tol), err.shape)
        raise AssertionError(f"{what}: {int(bad.sum())} elements out of tolerance; worst at {i}: "
                             f"got {got[i]!r} ref {ref[i]!r} err {err[i]:.3e} tol {tol[i]:.3e}")
    return float(err.max(initial=0.0))


def spread_step(inp: StepInputs, rows=None, lens=None):
    """``spread`` for assert_close over oracle_step(inp, rows, lens): for the
    flat indices of elements (row i, query head h, column d) of the [rows, Hq,
    D] output, sum_t w_t |v_t[d] - ref| with the oracle's exact weights of
    (rows[i], h) over the post-append cache."""
    rows = np.arange(inp.q.shape[0]) if rows is None else np.asarray(rows)
    L_all = inp.seq_lens if lens is None else np.asarray(lens, np.int32)
    _, Hq, D = inp.q.shape
    Hkv = inp.k_cache.shape[2]
    G = Hq // Hkv
    ref_cache = {}

    def fn(flat):
        out = np.empty(len(flat))
        for j, f in enumerate(flat):
            i, rem = divmod(int(f), Hq * D)
            h, d = divmod(rem, D)
            b = int(rows[i])
            key = (b, h)
            if key not in ref_cache:
                L = int(L_all[b])
                kc = inp.k_cache[b:b + 1].copy()
                vc = inp.v_cache[b:b + 1].copy()
                kc, vc, _ = oracle.kv_append(kc, vc, inp.k_new[b:b + 1], inp.v_new[b:b + 1], inp.pos[b:b + 1])
                w = oracle.attention_weights(inp.q[b:b + 1], kc, np.array([L], np.int32), inp.workload.scale, 0, h)
                v = bf16_bits_to_f32(vc[0, :L, h // G, :]).astype(np.float64)
                ref_cache[key] = (w, v, w @ v)
            w, v, o = ref_cache[key]
            out[j] = float(w @ np.abs(v[:, d] - o[d]))
        return out
    return fn
